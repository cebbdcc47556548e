// Launch of one instantiation of the tcgen05 fused attention kernel, shared
// by the translation unit of the plain kernels and that of the traced ones.
#pragma once

#include <cuda_runtime.h>

#include "attn_a2a.h"
#include "fa_tc.cuh"

namespace attn_a2a {

// PAIR: the CTA-pair kernel, launched in clusters of two; `grid` is then the
// CTAs wanted, cut to an even count of at most twice the clusters that can be
// resident at once (every cluster's CTAs wait on each other) and twice the
// work units.
template <int D, int MODE, int NMAP, bool TRACE = false, bool SPLIT = false, bool PAIR = false>
int launch_t(const tc::Maps<NMAP>& maps, const tc::Params& p, int grid, cudaStream_t stream, bool pdl = false) {
  auto kern = tc::fa_fwd_tc_kernel<D, MODE, NMAP, TRACE, SPLIT, PAIR>;
  using C = tc::Cfg<D, PAIR>;
  constexpr int smem = tc::kStagedStores<MODE> ? C::SMEM_ALLOC_STG : C::SMEM_ALLOC;
  // The in-kernel register split assumes exactly this launch register count;
  // with fewer registers at launch the softmax warpgroups could never obtain
  // their share, so refuse to launch rather than risk a stuck kernel.
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return ATTN_A2A_ECUDA;
  if (attr.numRegs != tc::kLaunchRegs) return ATTN_A2A_EUNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_A2A_ECUDA;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute cl[1];
    cl[0].id = cudaLaunchAttributeClusterDimension;
    cl[0].val.clusterDim.x = 2;
    cl[0].val.clusterDim.y = 1;
    cl[0].val.clusterDim.z = 1;
    cfg.attrs = cl;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * (grid / 2 > 0 ? grid / 2 : 1));
    int resident = 0;
    if (cudaOccupancyMaxActiveClusters(&resident, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_A2A_ECUDA;
    }
    int clusters = grid / 2;
    if (clusters > resident) clusters = resident;
    if (clusters > p.total) clusters = p.total;
    if (clusters < 1) return ATTN_A2A_EUNSUPPORTED;
    cfg.gridDim = dim3(2 * clusters);
    if (cudaLaunchKernelEx(&cfg, kern, maps, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_A2A_ECUDA;
    }
    return ATTN_A2A_OK;
  }
  if (pdl) {
    // launched with programmatic stream serialisation: the tail kernel's CTAs
    // start as the plain kernel's CTAs exit; a call's first kernel (p.pdl has
    // kPdlWait) runs its set-up as the previous kernel's CTAs exit and waits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, maps, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_A2A_ECUDA;
    }
    return ATTN_A2A_OK;
  }
  kern<<<grid, tc::kThreads, smem, stream>>>(maps, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_A2A_OK : ATTN_A2A_ECUDA;
}

// The traced instantiations (per-tile stamps into p.trace) of the four
// head-sharded modes: kModeContig, kModeA2A, kModeA2AT, kModeContigT.
int launch_fa_tc_traced(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid,
                        cudaStream_t stream);

// The split instantiation (pieces of items tail_first .. total - 1, workspace
// in p) of the same four modes: the tail kernel behind the plain kernel that
// runs items 0 .. tail_first - 1, or the whole schedule on its own; with
// pdl, launched with programmatic stream serialisation (p.pdl says what the
// kernel waits for).
int launch_fa_tc_split(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid,
                       cudaStream_t stream, bool pdl);

// The CTA-pair instantiation (d = 128) of the two bulk-store modes,
// kModeA2AT and kModeContigT; p counts work units (p.nquad per head) and
// maps.k has 64-row boxes.
int launch_fa_tc_pair(const tc::Maps<1>& maps, const tc::Params& p, int mode, int grid, cudaStream_t stream);

// The split instantiation of the whole layer's global-tile modes (kModeS2SG,
// kModeS2SGT; sequence-sharded inputs loaded in segments), as
// launch_fa_tc_split.
int launch_fa_tc_split_s2s(const tc::Maps<tc::kMaxS2SRanks>& maps, const tc::Params& p, int d, int mode, int grid,
                           cudaStream_t stream, bool pdl);

}  // namespace attn_a2a

// Launch of one instantiation of the tcgen05 fused attention kernel, shared
// by the translation unit of the plain kernels and that of the traced ones.
#pragma once

#include <cuda_runtime.h>

#include "attn_a2a.h"
#include "fa_tc.cuh"

namespace attn_a2a {

template <int D, int MODE, int NMAP, bool TRACE = false, bool SPLIT = false>
int launch_t(const tc::Maps<NMAP>& maps, const tc::Params& p, int grid, cudaStream_t stream, bool pdl = false) {
  auto kern = tc::fa_fwd_tc_kernel<D, MODE, NMAP, TRACE, SPLIT>;
  constexpr int smem = tc::kStagedStores<MODE> ? tc::Cfg<D>::SMEM_ALLOC_STG : tc::Cfg<D>::SMEM_ALLOC;
  // The in-kernel register split assumes exactly this launch register count;
  // with fewer registers at launch the softmax warpgroups could never obtain
  // their share, so refuse to launch rather than risk a stuck kernel.
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return ATTN_A2A_ECUDA;
  if (attr.numRegs != tc::kLaunchRegs) return ATTN_A2A_EUNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_A2A_ECUDA;
  if (pdl) {
    // the tail kernel, queued behind the plain one: launched with programmatic
    // stream serialisation, so its CTAs start as the plain kernel's CTAs exit
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
// in p) of the same four modes: with pdl, the tail kernel launched behind the
// plain kernel that runs items 0 .. tail_first - 1; without, the whole
// schedule on its own.
int launch_fa_tc_split(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid,
                       cudaStream_t stream, bool pdl);

}  // namespace attn_a2a

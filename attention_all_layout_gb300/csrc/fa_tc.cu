// Host launcher of the tcgen05 fused attention kernel: TMA descriptors for
// Q, K and V with the caller's strides, the persistent grid, the launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "fa_tc.cuh"
#include "internal.h"

namespace attn_a2a {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B, H, S, d] bf16 with element strides (sb, sh, ss), d contiguous; box of
// 64 x 128 rows with the 128-byte swizzle the MMA descriptors expect.
// Rows beyond S read as zeros.
bool make_map(CUtensorMap* m, const void* base, int B, int H, int S, int d, long long sb,
              long long sh, long long ss) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  // A size-1 dimension's stride is never used to address memory; give it a
  // legal value so the encoder accepts it.
  if (S == 1) ss = d;
  if (H == 1) sh = ss * S;
  if (B == 1) sb = sh * H;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(ss) * 2, static_cast<cuuint64_t>(sh) * 2,
                           static_cast<cuuint64_t>(sb) * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool A2A>
int launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const tc::Params& p,
             int grid, cudaStream_t stream) {
  auto kern = tc::fa_fwd_tc_kernel<D, A2A>;
  constexpr int smem = tc::Cfg<D>::SMEM_ALLOC;
  // The in-kernel register split assumes exactly this launch register count;
  // with fewer registers at launch the softmax warpgroups could never obtain
  // their share, so refuse to launch rather than risk a stuck kernel.
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return ATTN_A2A_ECUDA;
  if (attr.numRegs != tc::kLaunchRegs) return ATTN_A2A_EUNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_A2A_ECUDA;
  kern<<<grid, tc::kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_A2A_OK : ATTN_A2A_ECUDA;
}

}  // namespace

int launch_fa_tc(const void* q, const void* k, const void* v, const attn_a2a_shape& shp,
                 float scale, bool a2a, const EpiParams& epi, int* dev_status,
                 const attn_a2a_opts& opts, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, shp.B, shp.H, shp.S, shp.d, shp.q_sb, shp.q_sh, shp.q_ss) ||
      !make_map(&mk, k, shp.B, shp.H, shp.S, shp.d, shp.k_sb, shp.k_sh, shp.k_ss) ||
      !make_map(&mv, v, shp.B, shp.H, shp.S, shp.d, shp.v_sb, shp.v_sh, shp.v_ss))
    return ATTN_A2A_ECUDA;
  tc::Params p{};
  p.B = shp.B;
  p.H = shp.H;
  p.S = shp.S;
  p.nblk = (shp.S + tc::kBM - 1) / tc::kBM;
  p.npair = (p.nblk + 1) / 2;
  p.total = shp.B * shp.H * p.npair;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.dev_status = dev_status;
  p.timeout_ns = opts.timeout_ns > 0 ? static_cast<unsigned long long>(opts.timeout_ns) : 2000000000ull;
  p.inject_stall = opts.inject_stall;
  p.store_kind = opts.store_kind;
  p.epi = epi;
  int grid = opts.grid > 0 ? opts.grid : num_sms_current_device();
  if (grid <= 0) return ATTN_A2A_ECUDA;
  if (grid > p.total) grid = p.total;
  if (shp.d == 128)
    return a2a ? launch_t<128, true>(mq, mk, mv, p, grid, stream)
               : launch_t<128, false>(mq, mk, mv, p, grid, stream);
  return a2a ? launch_t<64, true>(mq, mk, mv, p, grid, stream)
             : launch_t<64, false>(mq, mk, mv, p, grid, stream);
}

}  // namespace attn_a2a

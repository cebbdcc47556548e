// Slow SIMT attention (no tensor cores) with the all-to-all epilogue: one warp
// per query row, fp32 online softmax, probabilities kept in fp32. A bring-up
// and cross-check path for small problems; the product path is fa_tc.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace attn_a2a {
namespace {

constexpr int kRowsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(256) fa_fwd_simt_kernel(const __nv_bfloat16* __restrict__ q,
                                                          const __nv_bfloat16* __restrict__ k,
                                                          const __nv_bfloat16* __restrict__ v,
                                                          attn_a2a_shape shp, float scale_log2,
                                                          EpiParams epi) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  if (row >= shp.S) return;
  const __nv_bfloat16* qp = q + b * shp.q_sb + h * shp.q_sh + row * shp.q_ss;
  const __nv_bfloat16* kp = k + b * shp.k_sb + h * shp.k_sh;
  const __nv_bfloat16* vp = v + b * shp.v_sb + h * shp.v_sh;
  float qv[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qv[e] = __bfloat162float(qp[lane + 32 * e]);
    o[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int key = 0; key < shp.S; ++key) {
    const __nv_bfloat16* kr = kp + key * shp.k_ss;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(qv[e], __bfloat162float(kr[lane + 32 * e]), dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float x = dot * scale_log2;
    const float m_new = fmaxf(m, x);
    const float corr = exp2f(m - m_new);
    const float pr = exp2f(x - m_new);
    l = l * corr + pr;
    const __nv_bfloat16* vr = vp + key * shp.v_ss;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = fmaf(pr, __bfloat162float(vr[lane + 32 * e]), o[e] * corr);
    m = m_new;
  }
  uint16_t* dst = out_row_ptr<D, true>(epi, shp.B, shp.H, shp.S, b, h, row);
  __nv_bfloat16* d16 = reinterpret_cast<__nv_bfloat16*>(dst);
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < E; ++e) d16[lane + 32 * e] = __float2bfloat16_rn(o[e] * inv);
}

}  // namespace

int launch_fa_simt(const void* q, const void* k, const void* v, const attn_a2a_shape& shp,
                   float scale, const EpiParams& epi, cudaStream_t stream) {
  const dim3 grid((shp.S + kRowsPerBlock - 1) / kRowsPerBlock, shp.H, shp.B);
  const float sl2 = scale * 1.4426950408889634f;
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  if (shp.d == 128)
    fa_fwd_simt_kernel<128><<<grid, 256, 0, stream>>>(qb, kb, vb, shp, sl2, epi);
  else
    fa_fwd_simt_kernel<64><<<grid, 256, 0, stream>>>(qb, kb, vb, shp, sl2, epi);
  return cudaGetLastError() == cudaSuccess ? ATTN_A2A_OK : ATTN_A2A_ECUDA;
}

}  // namespace attn_a2a

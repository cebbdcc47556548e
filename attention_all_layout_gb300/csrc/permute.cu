// The serial all-to-all on its own: copy a contiguous [B, H, S, d] output
// into P sequence-sharded partitions [B, c_j, H, d]. Pure data movement
// (HBM bound): each thread moves 16-byte vectors; reads are fully coalesced,
// writes land as whole 2*d-byte rows.
#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace attn_a2a {
namespace {

template <int D>
__global__ void __launch_bounds__(256) permute_h2s_kernel(const uint4* __restrict__ o, int B, int H,
                                                          int S, EpiParams epi, int64_t total_vec) {
  constexpr int kVecPerRow = D / 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total_vec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / kVecPerRow;
    const int c = static_cast<int>(i - row * kVecPerRow);
    const int s = static_cast<int>(row % S);
    const int64_t bh = row / S;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    const uint4 val = o[i];
    uint16_t* dst = out_row_ptr<D, true>(epi, B, H, S, b, h, s);
    reinterpret_cast<uint4*>(dst)[c] = val;
  }
}

}  // namespace

int launch_permute(const void* o, const attn_a2a_shape& shp, const EpiParams& epi,
                   cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(shp.B) * shp.H * shp.S * (shp.d / 8);
  if (total == 0) return ATTN_A2A_OK;
  int grid = num_sms_current_device() * 8;
  if (grid <= 0) grid = 1024;
  const int64_t need = (total + 255) / 256;
  if (need < grid) grid = static_cast<int>(need);
  const auto* src = static_cast<const uint4*>(o);
  if (shp.d == 128)
    permute_h2s_kernel<128><<<grid, 256, 0, stream>>>(src, shp.B, shp.H, shp.S, epi, total);
  else
    permute_h2s_kernel<64><<<grid, 256, 0, stream>>>(src, shp.B, shp.H, shp.S, epi, total);
  return cudaGetLastError() == cudaSuccess ? ATTN_A2A_OK : ATTN_A2A_ECUDA;
}

}  // namespace attn_a2a

// CTA-pair instantiations of the fused attention kernel (d = 128): a cluster
// of two CTAs on two SMs runs each work unit of four 128-row query tiles of
// one head with M = 256 tensor-core MMAs (cta_group::2), each CTA holding its
// own two query tiles and half of every K/V block, so that each SM reads
// half the K and V bytes from shared memory per block. A translation unit of
// its own, so that it compiles in parallel with the others.
#include "fa_tc_launch.cuh"

namespace attn_a2a {

int launch_fa_tc_pair(const tc::Maps<1>& maps, const tc::Params& p, int mode, int grid, cudaStream_t stream) {
  switch (mode) {
    case tc::kModeA2AT: return launch_t<128, tc::kModeA2AT, 1, false, false, true>(maps, p, grid, stream);
    case tc::kModeContigT: return launch_t<128, tc::kModeContigT, 1, false, false, true>(maps, p, grid, stream);
    default: return ATTN_A2A_EUNSUPPORTED;
  }
}

}  // namespace attn_a2a

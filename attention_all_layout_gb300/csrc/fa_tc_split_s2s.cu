// Split instantiations of the whole Ulysses layer's kernels whose tiles are
// counted over the whole sequence (kModeS2SG, kModeS2SGT): the same split
// schedule as the fused call's (tail_piece and merge_partials in fa_tc.cuh),
// its pieces loaded from the sequence-sharded partitions in segments. A
// translation unit of its own, so that it compiles in parallel.
#include "fa_tc_launch.cuh"

namespace attn_a2a {

int launch_fa_tc_split_s2s(const tc::Maps<tc::kMaxS2SRanks>& maps, const tc::Params& p, int d, int mode, int grid,
                           cudaStream_t stream, bool pdl) {
  constexpr int N = tc::kMaxS2SRanks;
  if (d == 128) {
    switch (mode) {
      case tc::kModeS2SGT: return launch_t<128, tc::kModeS2SGT, N, false, true>(maps, p, grid, stream, pdl);
      case tc::kModeS2SG: return launch_t<128, tc::kModeS2SG, N, false, true>(maps, p, grid, stream, pdl);
      default: return ATTN_A2A_EUNSUPPORTED;
    }
  }
  switch (mode) {
    case tc::kModeS2SGT: return launch_t<64, tc::kModeS2SGT, N, false, true>(maps, p, grid, stream, pdl);
    case tc::kModeS2SG: return launch_t<64, tc::kModeS2SG, N, false, true>(maps, p, grid, stream, pdl);
    default: return ATTN_A2A_EUNSUPPORTED;
  }
}

}  // namespace attn_a2a

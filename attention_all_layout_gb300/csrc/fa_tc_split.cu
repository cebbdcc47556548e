// Split instantiations of the fused attention kernel: work items divided over
// all CTAs by key blocks (the last wave's, or all of them), partial results
// merged through the caller's workspace (tail_piece and merge_partials in
// fa_tc.cuh).
// Separate from the plain kernels, whose code (and registers) the split paths
// would otherwise change, and a translation unit of its own so that it
// compiles in parallel.
#include "fa_tc_launch.cuh"

namespace attn_a2a {

int launch_fa_tc_split(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid,
                       cudaStream_t stream, bool pdl) {
  if (d == 128) {
    switch (mode) {
      case tc::kModeContig: return launch_t<128, tc::kModeContig, 1, false, true>(maps, p, grid, stream, pdl);
      case tc::kModeA2A: return launch_t<128, tc::kModeA2A, 1, false, true>(maps, p, grid, stream, pdl);
      case tc::kModeA2AT: return launch_t<128, tc::kModeA2AT, 1, false, true>(maps, p, grid, stream, pdl);
      case tc::kModeContigT: return launch_t<128, tc::kModeContigT, 1, false, true>(maps, p, grid, stream, pdl);
      case tc::kModeA2AC: return launch_t<128, tc::kModeA2AC, 1, false, true>(maps, p, grid, stream, pdl);
      default: return ATTN_A2A_EUNSUPPORTED;
    }
  }
  switch (mode) {
    case tc::kModeContig: return launch_t<64, tc::kModeContig, 1, false, true>(maps, p, grid, stream, pdl);
    case tc::kModeA2A: return launch_t<64, tc::kModeA2A, 1, false, true>(maps, p, grid, stream, pdl);
    case tc::kModeA2AT: return launch_t<64, tc::kModeA2AT, 1, false, true>(maps, p, grid, stream, pdl);
    case tc::kModeContigT: return launch_t<64, tc::kModeContigT, 1, false, true>(maps, p, grid, stream, pdl);
    case tc::kModeA2AC: return launch_t<64, tc::kModeA2AC, 1, false, true>(maps, p, grid, stream, pdl);
    default: return ATTN_A2A_EUNSUPPORTED;
  }
}

}  // namespace attn_a2a

// Traced instantiations of the fused attention kernel: the same kernel with
// per-tile %globaltimer stamps written to a caller buffer (the record layout
// is described at kTraceRecord in fa_tc.cuh). A translation unit of its own so
// that it compiles in parallel with the plain kernels.
#include "fa_tc_launch.cuh"

namespace attn_a2a {

static_assert(ATTN_A2A_TRACE_RECORD == tc::kTraceRecord, "trace record size of the header and the kernel");

int launch_fa_tc_traced(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid,
                        cudaStream_t stream) {
  if (d == 128) {
    switch (mode) {
      case tc::kModeContig: return launch_t<128, tc::kModeContig, 1, true>(maps, p, grid, stream);
      case tc::kModeA2A: return launch_t<128, tc::kModeA2A, 1, true>(maps, p, grid, stream);
      case tc::kModeA2AT: return launch_t<128, tc::kModeA2AT, 1, true>(maps, p, grid, stream);
      case tc::kModeContigT: return launch_t<128, tc::kModeContigT, 1, true>(maps, p, grid, stream);
      case tc::kModeA2AC: return launch_t<128, tc::kModeA2AC, 1, true>(maps, p, grid, stream);
      default: return ATTN_A2A_EUNSUPPORTED;
    }
  }
  switch (mode) {
    case tc::kModeContig: return launch_t<64, tc::kModeContig, 1, true>(maps, p, grid, stream);
    case tc::kModeA2A: return launch_t<64, tc::kModeA2A, 1, true>(maps, p, grid, stream);
    case tc::kModeA2AT: return launch_t<64, tc::kModeA2AT, 1, true>(maps, p, grid, stream);
    case tc::kModeContigT: return launch_t<64, tc::kModeContigT, 1, true>(maps, p, grid, stream);
    case tc::kModeA2AC: return launch_t<64, tc::kModeA2AC, 1, true>(maps, p, grid, stream);
    default: return ATTN_A2A_EUNSUPPORTED;
  }
}

}  // namespace attn_a2a

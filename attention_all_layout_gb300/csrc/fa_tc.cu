// Host launcher of the tcgen05 fused attention kernel: TMA descriptors for
// Q, K and V with the caller's strides, the persistent grid, the launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "fa_tc_launch.cuh"
#include "internal.h"

namespace attn_a2a {
namespace {

// Longest sequence, in 128-row key blocks, for which the automatic store kind
// picks bulk tensor stores for the all-to-all layout: every length. Measured
// at H = 40, d = 128, P = 8 with the current kernel, where warp 3 issues the
// stores (bulk / row stores, calls alternating, median of pairs): S = 32768
// 0.979, 49152 0.978, 75600 0.989. (Before the store warp: 0.988 at 24576,
// 0.993 at 32768, 1.003 at 75600, and the boundary was S = 32768; with the
// first kernel 1.008 at 24576, 1.004 at 32768, and it was S = 16384.)
constexpr int kBulkA2AMaxBlocks = INT_MAX;
// The same boundary for the whole Ulysses layer (sequence-sharded inputs):
// there bulk stores also mean tiles counted over the whole sequence
// (kModeS2SGT) instead of the per-partition tiles of kModeS2S with row
// stores, for equal partitions (ragged ones always take kModeS2S). Measured
// with warp 3 issuing the stores (H = 40, d = 128, P = 8, builds
// alternating): S = 32768 13.60-13.65 against 13.78-13.82 ms, the same bytes;
// every length, as for the fused call.
constexpr int kBulkS2SMaxBlocks = INT_MAX;

}  // namespace

// store_kind 0: bulk tensor stores where they are built and measured faster -
// the contiguous layout, and the all-to-all layout with up to kMaxStoreMaps
// partitions and at most max_bulk_blocks key blocks (at longer sequences its
// strided tile stores measured level with or slower than row stores) - else
// row stores;
// 1: bulk stores, or 0 where they are not built; 2: row stores; 3: row stores
// written as whole lines through shared memory (all-to-all layout only, else 0).
int resolve_store_kind(int S, int P, bool a2a, int store_kind, int max_bulk_blocks) {
  const bool built = !a2a || P <= tc::kMaxStoreMaps;
  if (store_kind == 1) return built ? 1 : 0;
  if (store_kind == 2) return 2;
  if (store_kind == 3) return a2a ? 3 : 0;
  const bool faster = !a2a || (S + tc::kBM - 1) / tc::kBM <= max_bulk_blocks;
  return built && faster ? 1 : 2;
}

int resolve_store_kind(int S, int P, bool a2a, int store_kind) {
  return resolve_store_kind(S, P, a2a, store_kind, kBulkA2AMaxBlocks);
}

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
// 64 columns x box_rows rows with the 128-byte swizzle the MMA descriptors
// expect. Rows beyond S read as zeros.
bool make_map(CUtensorMap* m, const void* base, int B, int H, int S, int d, long long sb,
              long long sh, long long ss, int box_rows = 128) {
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
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output partition j, [B, c_j, H_row, d] bf16 contiguous, addressed as
// (d, head, row, batch) with heads [0, H) of a row of H_row heads; box of 64
// columns x 1 head x 128 rows, 128-byte swizzle (the staging buffer's
// layout). Rows past c_j are not written by a store.
bool make_out_map(CUtensorMap* m, void* base, int B, int H, int H_row, int c, int d, int box_rows = 128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(c),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H_row) * d * 2,
                           static_cast<cuuint64_t>(c) * H_row * d * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void common_params(tc::Params& p, const attn_a2a_shape& shp, float scale, int* dev_status,
                   const attn_a2a_opts& opts) {
  p.B = shp.B;
  p.H = shp.H;
  p.S = shp.S;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.dev_status = dev_status;
  p.timeout_ns = opts.timeout_ns > 0 ? static_cast<unsigned long long>(opts.timeout_ns) : 2000000000ull;
  p.inject_stall = opts.inject_stall;
}

// Launch ids for the split tail's workspace flags: every launch that splits its
// tail gets a new one (never 0, the value of a zeroed workspace), so flags left
// by an earlier launch - finished or aborted - never match.
std::atomic<unsigned> g_epoch{0};

unsigned next_epoch() {
  unsigned e;
  do {
    e = g_epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
  } while (e == 0u);
  return e;
}

// Fewest key blocks per CTA that a split tail must save over the unsplit last
// wave (nblk - tail_len) before the automatic choice uses it. A tail piece
// restarts the two-tile pipeline (Q loads, first block, drain) and a split
// item pays for its partials' writes and merge: measured on GB300, a tail of
// 17-block ranges instead of 32-block items (the image preset) ran 42 us
// without the merge instead of about 30, and the partials' write and merge
// added about 17 us, so that the split lost 6 % there (joint, 31 of 36
// blocks: lost 10 %); at the video and long presets (80 and 62 blocks saved)
// it gained 0.3-0.8 %.
constexpr int kSplitMinSavedBlocks = 32;

// Fewest key blocks per CTA that the whole-schedule split must save over the
// unsplit waves before the automatic choice uses it, and only where the K and
// V of every head fit in half of L2: its ranges walk through all heads at
// once, so with more K/V than L2 holds every range re-reads its heads' K and
// V from HBM (measured on GB300: video and long presets 20 % slower). A cut
// item costs a partial write (3.6 us) and a merge (2-3 us) on the critical
// path: measured with warp 3 issuing the bulk stores, the image preset (15
// blocks saved of 96) ran 7 % faster split (0.144 against 0.154 ms), the
// joint preset (5 of 108) no faster (0.178 against 0.177-0.179 ms).
constexpr int kSplitAllMinSavedBlocks = 8;

}  // namespace

// The split decision for `total` work items of `nblk` key blocks on `grid`
// CTAs of a GPU with num_sms SMs and l2_bytes of L2, kv_bytes the K and V
// bytes of every head (the rule described at plan_split_tail):
// ATTN_A2A_SPLIT_ALL or ATTN_A2A_SPLIT_TAIL with the first split item and the
// blocks per range, or 0 (nothing split: tail_first = total, tail_len = 0).
int split_decision(int total, int nblk, int grid, int num_sms, long long kv_bytes, long long l2_bytes, int split,
                   int& tail_first, int& tail_len) {
  tail_first = total;
  tail_len = 0;
  if (split == ATTN_A2A_SPLIT_NONE || total <= 0 || grid <= 0 || nblk < 2 || nblk > (1 << 20)) return 0;
  const long long blocks = static_cast<long long>(total) * nblk;
  if (blocks > INT_MAX / 2 || grid > num_sms) return 0;  // every range's CTA must be resident at once
  const int waves = (total + grid - 1) / grid;
  const int all_len = static_cast<int>((blocks + grid - 1) / grid);
  const bool all_pays = 2 * kv_bytes <= l2_bytes && waves * nblk - all_len >= kSplitAllMinSavedBlocks;
  if (split == ATTN_A2A_SPLIT_ALL || (split == ATTN_A2A_SPLIT_AUTO && all_pays)) {
    tail_first = 0;
    tail_len = all_len;
    return ATTN_A2A_SPLIT_ALL;
  }
  const int r = total - (waves - 1) * grid;
  if (r >= grid) return 0;  // the last wave is full
  const int len = static_cast<int>((static_cast<long long>(r) * nblk + grid - 1) / grid);
  if (split == ATTN_A2A_SPLIT_AUTO && nblk - len < kSplitMinSavedBlocks) return 0;
  tail_first = (waves - 1) * grid;
  tail_len = len;
  return ATTN_A2A_SPLIT_TAIL;
}

namespace {

// Split schedule (the kernel's tail_piece), with the caller's workspace:
// ATTN_A2A_SPLIT_TAIL divides a last wave of r < grid items into ranges of
// ceil(r * nblk / grid) <= nblk key blocks, one per CTA, run by a second
// kernel behind the plain one; ATTN_A2A_SPLIT_ALL divides all items into
// ranges of ceil(total * nblk / grid) blocks in one kernel (whole = true);
// ATTN_A2A_SPLIT_AUTO takes the whole-schedule split where K and V fit in
// half of L2 and it saves at least kSplitAllMinSavedBlocks blocks per CTA,
// else the tail split where that saves at least kSplitMinSavedBlocks blocks
// per CTA. Every range's CTA must be resident
// at once (a final piece waits for other ranges), so a grid larger than the
// SM count is not split. Returns ATTN_A2A_EINVAL if the workspace is too small.
int plan_split_tail(tc::Params& p, int grid, int d, const attn_a2a_opts& opts, bool& whole) {
  p.tail_first = p.total;
  p.tail_len = 0;
  whole = false;
  if (opts.workspace == nullptr || opts.split == ATTN_A2A_SPLIT_NONE) return ATTN_A2A_OK;
  if (opts.workspace_bytes < ATTN_A2A_WORKSPACE_BYTES(grid, d)) return ATTN_A2A_EINVAL;
  if (opts.trace != nullptr || p.interleave > 1) return ATTN_A2A_OK;
  const int kind = split_decision(p.total, p.nblk, grid, num_sms_current_device(), 4LL * p.B * p.H * p.S * d,
                                  l2_bytes_current_device(), opts.split, p.tail_first, p.tail_len);
  if (kind == 0) return ATTN_A2A_OK;
  whole = kind == ATTN_A2A_SPLIT_ALL;
  uint8_t* base = static_cast<uint8_t*>(opts.workspace);
  const size_t flags = (static_cast<size_t>(grid) * 32u + 255u) / 256u * 256u;
  p.ws_flags = reinterpret_cast<unsigned*>(base);
  p.ws_o = reinterpret_cast<float*>(base + flags);
  p.ws_ml = p.ws_o + static_cast<size_t>(grid) * 2 * tc::kBM * d;
  p.epoch = next_epoch();
  return ATTN_A2A_OK;
}

int grid_for(const tc::Params& p, const attn_a2a_opts& opts) {
  int grid = opts.grid > 0 ? opts.grid : num_sms_current_device();
  if (grid <= 0) return 0;
  return grid > p.total ? p.total : grid;
}

// 1 when every output buffer that receives rows (the partitions with rows, or
// the contiguous output) is memory of the current device, 0 when one is not
// (host memory, including pinned or coherent host memory the device can
// store to, managed memory, another device's memory), -1 on a CUDA error.
int outputs_in_device_memory(bool a2a, const EpiParams& epi, const attn_a2a_shape& shp) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  auto on_device = [dev](const void* ptr) -> int {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    return attr.type == cudaMemoryTypeDevice && attr.device == dev ? 1 : 0;
  };
  if (!a2a) return on_device(epi.out);
  for (int j = 0; j < epi.P; ++j) {
    const int c = epi.cbase + (j < epi.crem ? 1 : 0);
    if (c == 0) continue;
    const int r = on_device(epi.part[j]);
    if (r != 1) return r;
  }
  (void)shp;
  return 1;
}

}  // namespace

int launch_plain(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid, cudaStream_t stream);

int launch_fa_tc(const void* q, const void* k, const void* v, const attn_a2a_shape& shp,
                 float scale, bool a2a, const EpiParams& epi, int* dev_status,
                 const attn_a2a_opts& opts, cudaStream_t stream) {
  tc::Maps<1> maps;
  std::memset(&maps, 0, sizeof(maps));
  int kind = resolve_store_kind(shp.S, epi.P, a2a, opts.store_kind);
  if (kind == 0) return ATTN_A2A_EUNSUPPORTED;
  if (kind == 1 || (opts.store_kind == 0 && a2a)) {
    // Bulk tensor stores go through tensor maps made for this device's memory:
    // outputs elsewhere (host memory the device can address, for one) take the
    // whole-line row stores (all-to-all) or the row stores (contiguous) when
    // the kind is automatic, and are refused when bulk stores were asked for.
    // The automatic all-to-all kind also takes whole-line row stores instead
    // of row stores there, which such links drain far faster.
    const int dev_rc = outputs_in_device_memory(a2a, epi, shp);
    if (dev_rc < 0) return ATTN_A2A_ECUDA;
    if (dev_rc == 0) {
      if (opts.store_kind == 1) return ATTN_A2A_EUNSUPPORTED;
      kind = a2a ? 3 : 2;
    }
  }
  const bool bulk = kind == 1;
  // Equal partitions of an odd multiple of 64 rows (the joint preset's 576)
  // cut every other partition boundary through a 128-row tile; every 64-row
  // half of a tile then lies in one partition, so each tile goes out as two
  // half-tile tensor stores instead of row stores for the cut tiles.
  const bool halves = bulk && a2a && epi.P > 1 && epi.crem == 0 && epi.cbase % tc::kBM == tc::kBM / 2;
  if (bulk && a2a) {
    const int h_row = epi.hstride > 0 ? epi.hstride : shp.H;
    for (int j = 0; j < epi.P; ++j) {
      const int c = epi.cbase + (j < epi.crem ? 1 : 0);
      if (c == 0) continue;
      if (!make_out_map(&maps.o[j], epi.part[j], shp.B, shp.H, h_row, c, shp.d, halves ? tc::kBM / 2 : tc::kBM))
        return ATTN_A2A_ECUDA;
    }
  }
  if (bulk && !a2a) {  // [B, H, S, d] contiguous, addressed like the inputs
    const long long ss = shp.d, sh = ss * shp.S, sb = sh * shp.H;
    if (!make_map(&maps.o[0], epi.out, shp.B, shp.H, shp.S, shp.d, sb, sh, ss)) return ATTN_A2A_ECUDA;
  }
  if (!make_map(&maps.q[0], q, shp.B, shp.H, shp.S, shp.d, shp.q_sb, shp.q_sh, shp.q_ss) ||
      !make_map(&maps.k[0], k, shp.B, shp.H, shp.S, shp.d, shp.k_sb, shp.k_sh, shp.k_ss) ||
      !make_map(&maps.v[0], v, shp.B, shp.H, shp.S, shp.d, shp.v_sb, shp.v_sh, shp.v_ss))
    return ATTN_A2A_ECUDA;
  tc::Params p{};
  common_params(p, shp, scale, dev_status, opts);
  p.nblk = (shp.S + tc::kBM - 1) / tc::kBM;
  p.npair = (p.nblk + 1) / 2;
  p.total = shp.B * shp.H * p.npair;
  p.epi = epi;
  p.half_stores = halves ? 1 : 0;
  // chunk-interleaved order: only when every chunk holds the same whole number of pairs
  if (opts.tile_order == 1 && a2a && epi.P > 1 && epi.crem == 0 && epi.cbase % (2 * tc::kBM) == 0)
    p.interleave = epi.cbase / (2 * tc::kBM);
  // CTA pairs (cta_group::2 MMAs over two SMs): d = 128, bulk-store
  // epilogue, sequence order, untraced, and no split schedule
  const bool pair_ok = shp.d == 128 && bulk && p.interleave <= 1 && opts.trace == nullptr;
  if (opts.cta_pairs == 1 && !pair_ok) return ATTN_A2A_EUNSUPPORTED;
  if (pair_ok && opts.cta_pairs == 1) {
    // each CTA of a pair loads half of every key block: K in 64-row boxes
    if (!make_map(&maps.k[0], k, shp.B, shp.H, shp.S, shp.d, shp.k_sb, shp.k_sh, shp.k_ss, 64))
      return ATTN_A2A_ECUDA;
    p.nquad = (p.npair + 1) / 2;
    p.total = shp.B * shp.H * p.nquad;
    p.tail_first = p.total;
    p.tail_len = 0;
    const int want = opts.grid > 0 ? opts.grid : num_sms_current_device();
    if (want <= 0) return ATTN_A2A_ECUDA;
    return launch_fa_tc_pair(maps, p, a2a ? tc::kModeA2AT : tc::kModeContigT, want, stream);
  }
  const int grid = grid_for(p, opts);
  if (grid <= 0) return ATTN_A2A_ECUDA;
  bool whole = false;
  const int split_rc = plan_split_tail(p, grid, shp.d, opts, whole);
  if (split_rc != ATTN_A2A_OK) return split_rc;
  const int mode = a2a ? (bulk ? tc::kModeA2AT : kind == 3 ? tc::kModeA2AC : tc::kModeA2A)
                       : (bulk ? tc::kModeContigT : tc::kModeContig);
  if (opts.trace != nullptr) {
    p.trace = opts.trace;
    return launch_fa_tc_traced(maps, p, shp.d, mode, grid, stream);
  }
  // Every call's first kernel goes behind the stream's previous work with
  // programmatic serialisation and waits for it after its set-up (kPdlWait):
  // where that work is a kernel, its launch and set-up overlap the previous
  // kernel's last CTAs (the next call of a short problem starts on the SMs
  // that a call's last wave leaves idle).
  if (whole) {
    p.pdl = tc::kPdlWait | tc::kPdlTrigger;
    return launch_fa_tc_split(maps, p, shp.d, mode, grid, stream, true);
  }
  if (p.tail_first < p.total) {
    // the full waves in the plain kernel, then the tail kernel behind it
    tc::Params pm = p;
    pm.total = p.tail_first;
    pm.tail_first = pm.total;
    pm.pdl = tc::kPdlWait;
    const int rc = launch_plain(maps, pm, shp.d, mode, grid, stream);
    if (rc != ATTN_A2A_OK) return rc;
    p.pdl = tc::kPdlWaitEnd;
    return launch_fa_tc_split(maps, p, shp.d, mode, grid, stream, true);
  }
  p.pdl = tc::kPdlWait;
  return launch_plain(maps, p, shp.d, mode, grid, stream);
}

// The plain kernel, launched with programmatic serialisation when p.pdl asks
// its CTAs to wait for the stream's previous kernel.
int launch_plain(const tc::Maps<1>& maps, const tc::Params& p, int d, int mode, int grid, cudaStream_t stream) {
  const bool pdl = (p.pdl & tc::kPdlWait) != 0;
  switch (mode) {
    case tc::kModeA2AT:
      return d == 128 ? launch_t<128, tc::kModeA2AT, 1>(maps, p, grid, stream, pdl)
                      : launch_t<64, tc::kModeA2AT, 1>(maps, p, grid, stream, pdl);
    case tc::kModeContigT:
      return d == 128 ? launch_t<128, tc::kModeContigT, 1>(maps, p, grid, stream, pdl)
                      : launch_t<64, tc::kModeContigT, 1>(maps, p, grid, stream, pdl);
    case tc::kModeA2A:
      return d == 128 ? launch_t<128, tc::kModeA2A, 1>(maps, p, grid, stream, pdl)
                      : launch_t<64, tc::kModeA2A, 1>(maps, p, grid, stream, pdl);
    case tc::kModeA2AC:
      return d == 128 ? launch_t<128, tc::kModeA2AC, 1>(maps, p, grid, stream, pdl)
                      : launch_t<64, tc::kModeA2AC, 1>(maps, p, grid, stream, pdl);
    default:
      return d == 128 ? launch_t<128, tc::kModeContig, 1>(maps, p, grid, stream, pdl)
                      : launch_t<64, tc::kModeContig, 1>(maps, p, grid, stream, pdl);
  }
}

int launch_fa_tc_s2s(const void* const* qp, const void* const* kp, const void* const* vp,
                     const attn_a2a_shape& shp, float scale, const EpiParams& epi, int* dev_status,
                     const attn_a2a_opts& opts, cudaStream_t stream) {
  if (epi.P > tc::kMaxS2SRanks) return ATTN_A2A_EUNSUPPORTED;
  tc::Maps<tc::kMaxS2SRanks> maps;
  std::memset(&maps, 0, sizeof(maps));
  // Equal partitions whose length is a multiple of 64 but not of 128 would end
  // every partition in a half-empty block: count tiles over the whole sequence
  // and load each as two 64-row pieces, each inside one partition, and store
  // each tile as two 64-row halves (kModeS2SGT with half_stores: the joint
  // preset's layer 0.1773-0.1818 ms against 0.1836-0.1891 with row stores,
  // kModeS2SG). Partitions of a multiple of 128 rows tile the same either way;
  // they take the global tiles with one 128-row piece where the automatic
  // store kind is bulk (kModeS2SGT: the image preset's layer measured 1.4 %
  // faster than with row stores), else the per-partition tiles of kModeS2S.
  // Other partition lengths count tiles per partition (kModeS2S).
  int auto_kind = resolve_store_kind(shp.S, epi.P, true, opts.store_kind, kBulkS2SMaxBlocks);
  if (auto_kind == 0) return ATTN_A2A_EUNSUPPORTED;
  if (auto_kind == 1) {  // bulk stores only into this device's memory (see launch_fa_tc)
    const int dev_rc = outputs_in_device_memory(true, epi, shp);
    if (dev_rc < 0) return ATTN_A2A_ECUDA;
    if (dev_rc == 0) {
      if (opts.store_kind == 1) return ATTN_A2A_EUNSUPPORTED;
      auto_kind = 2;
    }
  }
  const bool equal64 = epi.crem == 0 && epi.cbase > 0 && epi.cbase % (tc::kBM / 2) == 0;
  const int seg = epi.cbase % tc::kBM == 0 ? tc::kBM : tc::kBM / 2;
  const bool global_tiles = equal64 && (seg < tc::kBM || auto_kind == 1);
  const int kind = auto_kind;
  // partitions of an odd multiple of 64 rows: tiles stored in two 64-row halves
  const bool halves = kind == 1 && global_tiles && seg < tc::kBM;
  const long long row = static_cast<long long>(shp.H) * shp.d;  // partition j is [B, c_j, H, d]
  for (int j = 0; j < epi.P; ++j) {
    const int c = epi.cbase + (j < epi.crem ? 1 : 0);
    if (c == 0) continue;
    const long long sb = row * c;
    const int box = global_tiles ? seg : tc::kBM;
    if (!make_map(&maps.q[j], qp[j], shp.B, shp.H, c, shp.d, sb, shp.d, row, box) ||
        !make_map(&maps.k[j], kp[j], shp.B, shp.H, c, shp.d, sb, shp.d, row, box) ||
        !make_map(&maps.v[j], vp[j], shp.B, shp.H, c, shp.d, sb, shp.d, row, box))
      return ATTN_A2A_ECUDA;
  }
  tc::Params p{};
  common_params(p, shp, scale, dev_status, opts);
  if (global_tiles) {
    p.seg = seg;
    p.half_stores = halves ? 1 : 0;
    p.nblk = (shp.S + tc::kBM - 1) / tc::kBM;
    p.npair = (p.nblk + 1) / 2;
    p.total = shp.B * shp.H * p.npair;
    p.epi = epi;
    const int grid = grid_for(p, opts);
    if (grid <= 0) return ATTN_A2A_ECUDA;
    // the split schedule, with a workspace, as for the fused call, except that
    // the automatic choice takes only the whole-schedule split here: measured on
    // GB300, the image layer ran 0.1507 ms split against 0.1582, while the video
    // layer's last-wave split ran 13.63 ms against 13.45 unsplit
    bool whole = false;
    const int split_rc = plan_split_tail(p, grid, shp.d, opts, whole);
    if (split_rc != ATTN_A2A_OK) return split_rc;
    if (!whole && opts.split == ATTN_A2A_SPLIT_AUTO) {
      p.tail_first = p.total;
      p.tail_len = 0;
    }
    if (kind == 1) {
      for (int j = 0; j < epi.P; ++j)
        if (!make_out_map(&maps.o[j], epi.part[j], shp.B, shp.H, shp.H, epi.cbase, shp.d,
                          halves ? tc::kBM / 2 : tc::kBM))
          return ATTN_A2A_ECUDA;
    }
    const int mode = kind == 1 ? tc::kModeS2SGT : tc::kModeS2SG;
    // programmatic serialisation behind the stream's previous kernel, as in launch_fa_tc
    auto plain = [&](const tc::Params& pp) -> int {
      if (kind == 1)
        return shp.d == 128 ? launch_t<128, tc::kModeS2SGT, tc::kMaxS2SRanks>(maps, pp, grid, stream, true)
                            : launch_t<64, tc::kModeS2SGT, tc::kMaxS2SRanks>(maps, pp, grid, stream, true);
      return shp.d == 128 ? launch_t<128, tc::kModeS2SG, tc::kMaxS2SRanks>(maps, pp, grid, stream, true)
                          : launch_t<64, tc::kModeS2SG, tc::kMaxS2SRanks>(maps, pp, grid, stream, true);
    };
    if (whole) {
      p.pdl = tc::kPdlWait | tc::kPdlTrigger;
      return launch_fa_tc_split_s2s(maps, p, shp.d, mode, grid, stream, true);
    }
    if (p.tail_first < p.total) {
      tc::Params pm = p;
      pm.total = p.tail_first;
      pm.tail_first = pm.total;
      pm.pdl = tc::kPdlWait;
      const int rc = plain(pm);
      if (rc != ATTN_A2A_OK) return rc;
      p.pdl = tc::kPdlWaitEnd;
      return launch_fa_tc_split_s2s(maps, p, shp.d, mode, grid, stream, true);
    }
    p.pdl = tc::kPdlWait;
    return plain(p);
  }
  p.nb_big = (epi.cbase + 1 + tc::kBM - 1) / tc::kBM;
  p.nb_small = (epi.cbase + tc::kBM - 1) / tc::kBM;
  p.nblk = epi.crem * p.nb_big + (epi.P - epi.crem) * p.nb_small;
  p.npair = (p.nblk + 1) / 2;
  p.total = shp.B * shp.H * p.npair;
  p.epi = epi;
  p.tail_first = p.total;  // no split schedule with per-partition tiles
  p.pdl = tc::kPdlWait;
  const int grid = grid_for(p, opts);
  if (grid <= 0) return ATTN_A2A_ECUDA;
  if (shp.d == 128) return launch_t<128, tc::kModeS2S, tc::kMaxS2SRanks>(maps, p, grid, stream, true);
  return launch_t<64, tc::kModeS2S, tc::kMaxS2SRanks>(maps, p, grid, stream, true);
}

}  // namespace attn_a2a

// Fused attention forward + post-attention all-to-all epilogue on tcgen05.
//
// X-Stage pages ("Key Contributions", FlashAttention-A2A piggybacking;
// "Results", FlashAttention-A2A optimisation): the owner of each output tile
// stores it straight into its destination layout and immediately resumes the
// Q loop of its next tile; there is no dedicated communication warp or SM and
// no separate permute pass. Here the tile owner is the softmax warpgroup that
// holds the tile's rows: it normalises its O rows, issues their stores into
// the sequence-sharded partitions and goes back to the next work item's
// softmax, while the stores drain (the X-stage) behind the next Q loop.
//
// CTA layout (384 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: Q tiles once per work item, then K_j, V_j
//               through a ring of shared-memory stages
//   warp 1      MMA issuer (one thread) and TMEM allocator
//   warp 2      relay: waits on the TMA and O-free barriers on the issuer's
//               behalf; with the softmax threads' own arrivals it completes
//               one event barrier phase per group of MMAs
//   warp 3      bulk-store modes: issues the output tiles' tensor stores
//               (store_role); otherwise idle
//   warps 4-7   softmax/correction/epilogue for query tile 0 (128 rows)
//   warps 8-11  the same for query tile 1
// A work item is (b, h, pair of adjacent 128-row query blocks), so each K/V
// tile read from L2 serves 256 query rows.
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256) fp32 scores; the
// bf16 probabilities P_t are written over the first 64 columns of S_t;
// O0 [256,256+d), O1 [256+d, 256+2d) fp32 accumulators.
//
// MMA order per key block j (skewed so each softmax has two MMAs of slack):
//   S0_j = Q0 K_j^T ; O1 += P1_{j-1} V_{j-1} ; S1_j = Q1 K_j^T ; O0 += P0_j V_j
// and a final O1 += P1 V after the loop (S0_{j+1} follows O0 += P0_j V_j
// directly, in the same issue group). Because tcgen05 operations of one
// thread complete in order, the commit after S_t_j also means that the
// previous P_t V product is done, so the softmax role may rescale O_t in
// place before it publishes P_t_j.
//
// Why a relay: on GB300 any shared-memory load or mbarrier query in the
// thread that issues tcgen05.mma stalls it behind its queued MMAs. The issuer
// therefore syncs twice per key block - before O1 += P1 V (P1 ready), and
// before O0 += P0 V together with the next S0 (V_j landed, P0 ready and
// K_{j+1} landed, one event) - each on one mbarrier phase. The relay thread
// does the waits on the TMA and O-free barriers and arrives on the event's
// barrier; the softmax threads that wrote P arrive on it directly. A parity
// wait on an mbarrier measured cheaper in the issuer (about 55 cycles per
// sync between groups of eight 128x128x16 MMAs) than a load of a
// shared-memory counter with a branch on it (about 120).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "epilogue.cuh"
#include "ptx.cuh"

namespace attn_a2a {
namespace tc {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per block
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
// A block's probabilities are taken against the row's running maximum m as
// long as their sum stays within kSpecBound (then no single p exceeds it and
// the fp32 accumulators stay far from overflow); past it the block's own
// maximum is taken and O and l are rescaled.
constexpr float kSpecBound = 4096.0f;  // 2^12
// Register split (setmaxnreg): the kernel launches with kLaunchRegs per thread;
// warpgroup 0 (producer, MMA issuer, relay, store warp) gives registers back and
// the two softmax warpgroups take them: 128*kRegsLow + 256*kRegsHigh must not
// exceed 384*kLaunchRegs, else setmaxnreg.inc would wait forever. The launcher
// refuses to launch unless the compiled launch register count is kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 80;
constexpr int kRegsHigh = 208;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs, "register split exceeds the launch budget");

// PAIR: the CTA-pair kernel (d = 128), whose K/V stages hold this CTA's
// half of a block - keys 64 r .. 64 r + 63 of K (two 64-row atoms), columns
// 64 r .. 64 r + 63 of V (one 128-row atom) for rank r - so twice as many
// stages fit in the same shared memory.
template <int D, bool PAIR = false>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!PAIR || D == 128, "CTA pairs split V by 64-column atoms: d = 128 only");
  static constexpr int TILE_BYTES = 128 * D * 2;  // one Q, K or V tile (128 rows x d bf16)
  static constexpr int KV_BYTES = PAIR ? TILE_BYTES / 2 : TILE_BYTES;  // one K/V stage
  static constexpr int NSTAGE = PAIR ? 8 : (D == 128) ? 4 : 6;
  static constexpr int ATOM_BYTES = 128 * 128;    // 128 rows x one 128-byte swizzle column
  static constexpr int K_ATOM_BYTES = KV_BYTES / (D / 64);  // a K stage's 128-byte swizzle column
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSTAGE * KV_BYTES;
  // barrier slots
  static constexpr int QF = 0, QE = 2, SF = 4, OF = 6, OE = 8, KVF = 10;
  static constexpr int KVE = KVF + NSTAGE;
  static constexpr int DONE = KVE + NSTAGE;
  // store-warp epilogue: STG + t = warp 3 is done with the staging buffer
  // after tile t's use (one phase per work item); STGW + t = the four warps of
  // tile t have written their rows
  static constexpr int STG = DONE + 1, STGW = DONE + 3;
  // the MMA issuer's events (see relay_role): EVA = A (the relay's arrival),
  // EVB = B_j (tile 0's 128 softmax threads + the relay), EVC = C_j and E
  // (tile 1's 128 softmax threads + the relay). Each kind's next event depends
  // on MMAs issued after the issuer consumed the previous one, so no event
  // barrier completes two phases ahead of the issuer's parity wait.
  static constexpr int EVA = STGW + 2, EVB = EVA + 1, EVC = EVA + 2;
  static constexpr int NBAR = EVC + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  // MISC: +0 abort flag, +4 TMEM base
  static constexpr int SMEM_USED = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
  // the bulk-store epilogue's staging buffer: one 128-row output tile in
  // 128-byte-swizzled 64-column atoms, shared by the two query tiles in turn
  static constexpr int STG_OFF = (SMEM_USED + 1023) / 1024 * 1024;
  static constexpr int SMEM_ALLOC_STG = STG_OFF + TILE_BYTES + 1024;
  static_assert(SMEM_ALLOC_STG <= 227 * 1024, "staging buffer does not fit");
};

// Where the output tile goes and where the inputs come from:
//   kModeContig  inputs [B,H,S,d] (strided), output [B,H,S,d] contiguous;
//   kModeA2A     inputs [B,H,S,d] (strided), output P sequence-sharded
//                partitions [B,c_j,H,d] (the post-attention all-to-all);
//   kModeS2S     inputs AND output P sequence-sharded partitions: the
//                pre-attention all-to-all is folded into the loads as well.
//                Query tiles and key blocks are then counted per partition,
//                starting at each partition's row 0, so that none straddles two
//                partitions; only a partition's last block can be partial.
//   kModeA2AT    as kModeA2A, but each output tile goes out as bulk tensor
//                stores (TMA) from a shared-memory staging buffer: the owner
//                warps stage the tile and resume; one thread of warp 3 issues
//                the tile's stores, and only the buffer's reuse waits, for the
//                stores' shared-memory reads. A tile that
//                straddles two partitions is stored row by row as in kModeA2A.
//   kModeContigT as kModeContig, with the bulk-store epilogue.
//   kModeS2SG    as kModeS2S (sequence-sharded in and out), for partitions of
//                equal length c, a multiple of 64: tiles and key blocks are
//                counted over the whole sequence as in kModeA2A, and every
//                128-row tile is loaded in p.seg-row pieces (128, or 64 when c
//                is not a multiple of 128), each lying inside one partition, so
//                no block is half empty and the result equals kModeA2A's bit
//                for bit. Output as kModeA2A (row stores).
//   kModeS2SGT   as kModeS2SG, with kModeA2AT's bulk-store epilogue.
//   kModeA2AC    as kModeA2A, but each warp writes its 32 rows as whole lines:
//                it puts 16 rows at a time into its own slice of the staging
//                buffer, then every store instruction of the warp covers whole
//                rows (2 of 256 bytes, or 4 of 128), so a destination reached
//                over a slower link (another device's or the host's memory)
//                receives full lines instead of 16-byte pieces of 32 rows.
//                No barrier with other warps: each warp's slice is its own.
// (kModeS2S keeps the row stores: with the staging path its register
// pressure grew and the whole layer measured ≈ 3 % slower.)
enum : int {
  kModeContig = 0,
  kModeA2A = 1,
  kModeS2S = 2,
  kModeA2AT = 3,
  kModeContigT = 4,
  kModeS2SG = 5,
  kModeS2SGT = 6,
  kModeA2AC = 7
};
template <int MODE>
constexpr bool kBulkStores = MODE == kModeA2AT || MODE == kModeContigT || MODE == kModeS2SGT;
// modes that use the staging buffer (bulk tensor stores, or whole-line row stores)
template <int MODE>
constexpr bool kStagedStores = kBulkStores<MODE> || MODE == kModeA2AC;
template <int MODE>
constexpr bool kSegLoads = MODE == kModeS2SG || MODE == kModeS2SGT;
constexpr int kMaxS2SRanks = 8;
constexpr int kMaxStoreMaps = 8;  // output partitions with a tensor map (bulk-store epilogue)

template <int N>
struct Maps {
  CUtensorMap q[N], k[N], v[N];
  CUtensorMap o[kMaxStoreMaps];  // output partitions, bulk-store epilogue only
};

// Params::pdl (programmatic dependent launch). kPdlWait: the kernel was
// launched with programmatic stream serialisation behind whatever ran before
// it on the stream, and every thread waits for that grid's completion
// (griddepcontrol.wait) after the set-up and before its first access to
// global memory. kPdlTrigger: a split kernel lets the next kernel of the
// stream launch once all its CTAs have started
// (griddepcontrol.launch_dependents); the plain kernel always does.
// kPdlWaitEnd: the tail kernel, which runs beside the plain kernel ahead of
// it without waiting for it, waits for it before exiting, so that the tail
// kernel's completion - all that a kernel queued behind it with programmatic
// serialisation waits for - covers the plain kernel's stores too.
constexpr int kPdlWait = 1, kPdlTrigger = 2, kPdlWaitEnd = 4;

struct Params {
  int B, H, S;
  int nblk;   // query tiles per head = key blocks per head (ceil(S/128), or the per-partition count)
  int npair;  // ceil(nblk / 2): work items per head
  int total;  // B * H * npair, or B * H * nquad for the CTA-pair kernel
  int nquad;  // CTA-pair kernel: ceil(npair / 2) units of two pairs per head, one pair per CTA
  float scale_log2;
  int* dev_status;
  unsigned long long timeout_ns;
  int inject_stall;
  int nb_big, nb_small;  // kModeS2S: 128-row blocks of a longer / shorter chunk
  int interleave;        // > 1: chunk-interleaved item order with this many pairs per chunk
  int seg;               // kModeS2SG(T): rows per TMA box of the sequence-sharded loads (128 or 64)
  int half_stores;       // kModeA2AT, kModeS2SGT: every tile stored as two 64-row halves, each into the partition
                         // holding it (equal partitions of an odd multiple of 64 rows; 64-row output boxes)
  long long* trace;      // traced instantiations only: kTraceRecord int64 per (item, tile, warp)
  int pdl;               // kPdlWait | kPdlTrigger: programmatic dependent launch (see the kernel's set-up)
  // Split schedule (see tail_piece): the key blocks of items [tail_first,
  // total) are divided over the CTAs, tail_len blocks per CTA; tail_first =
  // total when nothing is split. Partial results go through the caller's
  // workspace, one slot per range.
  int tail_first, tail_len;
  unsigned epoch;        // this launch's id, written to the workspace flags
  float* ws_o;           // [grid][2 tiles][D/4][128 rows] float4: a partial piece's O (unnormalised);
                         // row-minor, so that a warp's 32 rows are 512 contiguous bytes
  float* ws_ml;          // [grid][2][128][2] fp32: its running maximum (log2 domain) and row sum
  unsigned* ws_flags;    // [grid][2][4 warps]: epoch once that warp's rows are written
  EpiParams epi;
};

// 128-row block `idx` of a head: which tensor map holds it, its first row
// there, and the row count of that map (so rows >= c do not exist).
struct Blk {
  int map, row, c;
};

template <int MODE>
__device__ __forceinline__ Blk locate_block(const Params& p, int idx) {
  Blk r;
  if constexpr (MODE == kModeS2S) {
    const int nbig = p.epi.crem * p.nb_big;
    int j, blk;
    if (idx < nbig) {
      j = idx / p.nb_big;
      blk = idx - j * p.nb_big;
      r.c = p.epi.cbase + 1;
    } else {
      const int t = idx - nbig;
      const int k = p.nb_small > 0 ? t / p.nb_small : 0;
      j = p.epi.crem + k;
      blk = t - k * p.nb_small;
      r.c = p.epi.cbase;
    }
    r.map = j;
    r.row = blk * kBM;
  } else {
    r.map = 0;
    r.row = idx * kBM;
    r.c = p.S;
  }
  return r;
}

// The key blocks in order, without the division locate_block needs: the
// softmax and the producer visit blocks 0, 1, 2, ... of every item, and in the
// sequence-sharded mode a runtime division per block costs the softmax (whose
// warps keep their sub-partitions busy) several percent.
template <int MODE>
struct BlockWalker {
  int k = 0, b = 0, nbk = 0, ck = 0;  // partition, block in it, its blocks, its rows
  __device__ __forceinline__ void reset(const Params& p) {
    k = 0;
    b = 0;
    if constexpr (MODE == kModeS2S) {
      ck = p.epi.crem > 0 ? p.epi.cbase + 1 : p.epi.cbase;
      nbk = p.epi.crem > 0 ? p.nb_big : p.nb_small;
    }
  }
  __device__ __forceinline__ Blk block(const Params& p) const {
    Blk r;
    if constexpr (MODE == kModeS2S) {
      r.map = k;
      r.row = b * kBM;
      r.c = ck;
    } else {
      r.map = 0;
      r.row = b * kBM;
      r.c = p.S;
    }
    return r;
  }
  __device__ __forceinline__ void next(const Params& p) {
    ++b;
    if constexpr (MODE == kModeS2S) {
      if (b == nbk) {  // partitions without rows only follow the last block
        b = 0;
        if (++k == p.epi.crem) {
          ck = p.epi.cbase;
          nbk = p.nb_small;
        }
      }
    }
  }
};

struct Item {
  int b, h, pair;
};

// ------------------------------------------------------------------ split schedule
// Work items are pairs of 128-row query tiles with nblk key blocks each; a
// wave holds one item per CTA. When the number of items is not a multiple of
// the grid, the last wave leaves CTAs idle (the image preset: 384 items on
// 152 CTAs, a last wave of 80). A split launch instead counts the key blocks
// of items [tail_first, total) one item after the other (u = (item -
// tail_first) * nblk + key block) and gives each CTA one range of tail_len
// consecutive blocks. Two uses: the tail kernel behind the plain one, with
// tail_first = the last wave's first item and tail_len <= nblk; and the whole
// schedule in one kernel (tail_first = 0, tail_len = ceil(total * nblk /
// grid), usually more than nblk).
// A range cuts items into pieces [k0, k1) of their key blocks, run in the
// range's order. A piece that starts inside its item (k0 > 0, the range's
// first) is "partial": it writes its unnormalised O, running maximum and row
// sum to the workspace slot of its range and raises per-warp flags. The piece
// holding the item's first key block but not its last (k0 = 0, k1 < nblk, the
// range's last) is "final": it waits for the flags of the ranges after its
// own that hold the rest of the item, merges their partials into its
// accumulator and stores the tile as usual. A range thus has at most one
// partial piece, run first, and one final piece, run last; partial pieces
// never wait. Range g runs on CTA grid - 1 - g, so a final piece waits only
// for CTAs of lower index, which the hardware dispatches no later.
// In the tail kernel (SPLIT = true, launched right behind the plain kernel
// with programmatic dependent launch) each CTA starts on the SM that a plain
// CTA leaves; it reads only q, k and v, which the plain kernel does not write,
// so it needs no wait for the plain kernel's results. Keeping the split paths
// in their own instantiation leaves the plain kernel's code and registers as
// they are.
struct Piece {
  int item, k0, k1;
  int kind;  // 0: a whole item; 1: partial (to the workspace); 2: final piece of a split item
};

// The range this CTA runs (the split schedule's g).
__device__ __forceinline__ int split_range() { return static_cast<int>(gridDim.x - 1 - blockIdx.x); }

// Piece k (0, 1, ...) of this CTA's range, in order; false past its last.
__device__ __forceinline__ bool tail_piece(const Params& p, int k, Piece& out) {
  const int R = (p.total - p.tail_first) * p.nblk;
  const int u0 = split_range() * p.tail_len;
  const int u1 = min(u0 + p.tail_len, R);
  if (u0 >= u1) return false;
  const int i0 = u0 / p.nblk, i = i0 + k;
  if (i > (u1 - 1) / p.nblk) return false;
  const int k0 = k == 0 ? u0 - i0 * p.nblk : 0;
  const int k1 = min(u1 - i * p.nblk, p.nblk);
  out = Piece{p.tail_first + i, k0, k1, k0 > 0 ? 1 : (k1 < p.nblk ? 2 : 0)};
  return true;
}

// This CTA's piece number `it` (0, 1, ...), a function of it alone, so the
// roles keep no other loop state; false past the last piece. The plain kernel
// (SPLIT = false) runs whole items blockIdx.x, blockIdx.x + grid, ... below
// p.total; the tail kernel (SPLIT = true) runs only this CTA's tail pieces.
// The CTA-pair kernel (PAIR = true) runs one unit per cluster at a time: both
// CTAs of cluster c run units c, c + grid / 2, ...
template <bool SPLIT, bool PAIR = false>
__device__ __forceinline__ bool piece_at(const Params& p, int it, Piece& out) {
  if constexpr (PAIR) {
    static_assert(!SPLIT, "the CTA-pair kernel has no split schedule");
    const int n = static_cast<int>(gridDim.x) / 2;
    const int item = static_cast<int>(blockIdx.x) / 2 + it * n;
    out = Piece{item, 0, p.nblk, 0};
    return item < p.total;
  } else if constexpr (!SPLIT) {
    const int item = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
    out = Piece{item, 0, p.nblk, 0};
    return item < p.total;
  } else {
    return tail_piece(p, it, out);
  }
}

// For the CTA-pair kernel `item` is a unit (b, h, quad): rank r of the
// cluster takes query-tile pair 2 quad + r (past the head's last pair when
// npair is odd: rows beyond S, read as zeros and never stored).
template <bool PAIR = false>
__device__ __forceinline__ Item decode_item(const Params& p, int item) {
  Item it;
  if constexpr (PAIR) {
    it.pair = 2 * (item % p.nquad) + static_cast<int>(cluster_ctarank());
    const int bh = item / p.nquad;
    it.h = bh % p.H;
    it.b = bh / p.H;
    return it;
  }
  it.pair = item % p.npair;
  if (p.interleave > 1) {
    // i-th item of a head -> pair (i mod P) * pairs_per_chunk + i / P: neighbouring
    // items (run at the same time by neighbouring CTAs) land in different chunks
    const int P = p.npair / p.interleave;
    it.pair = (it.pair % P) * p.interleave + it.pair / P;
  }
  const int bh = item / p.npair;
  it.h = bh % p.H;
  it.b = bh / p.H;
  return it;
}

// ------------------------------------------------------------------ producer
// PAIR: each CTA loads its own Q tiles and its half of every K/V block into
// its own shared memory; all of them complete on the leader's QF/KVF
// barriers, on which only the leader announces the pair's bytes.
template <int D, int MODE, int NMAP, bool SPLIT, bool PAIR = false>
__device__ void producer_role(const Params& p, const Maps<NMAP>* maps, uint32_t sbase, uint32_t bar0,
                              const WaitCtl& w) {
  using C = Cfg<D, PAIR>;
  static_assert(!PAIR || (!kSegLoads<MODE> && MODE != kModeS2S), "CTA pairs load head-sharded inputs only");
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool lead = rank == 0;
  // the barrier a load completes on: the leader's for a pair
  auto FBAR = [&](int i) { return PAIR ? mapa_shared(BAR(i), 0) : BAR(i); };
  const uint64_t pol_kv = l2_policy_evict_last();  // K/V are re-read by every query tile of the head
  const uint64_t pol_q = l2_policy_evict_first();  // each Q tile is read once
  uint32_t kv_it = 0;
  uint32_t q_loads[2] = {0, 0};
  bool ok = true;
  int it = 0;
  // kModeS2SG(T): rows [row, row + 128) of the sequence as 128 / p.seg boxes of
  // p.seg rows (128, or 64), each from the partition that holds it (equal
  // partitions of p.epi.cbase rows, a multiple of p.seg), at row offset
  // k * p.seg of every 128-row swizzle atom column (a multiple of 8 KB, so each
  // piece starts on a 1 KB swizzle boundary). Rows past S fall past the last
  // partition's end and read as zeros.
  auto load_segments = [&](uint32_t dst, const CUtensorMap* tmaps, uint32_t bar, int row, const Item& wi,
                           uint64_t pol) {
    for (int off = 0; off < kBM; off += p.seg) {
      const int g = row + off;
      int j = g / p.epi.cbase;
      if (j > p.epi.P - 1) j = p.epi.P - 1;
      const int l = g - j * p.epi.cbase;
      const uint32_t piece = dst + static_cast<uint32_t>(off) * 128u;
#pragma unroll
      for (int a = 0; a < D / 64; ++a)
        tma_load_4d(piece + a * C::ATOM_BYTES, &tmaps[j], bar, a * 64, l, wi.h, wi.b, pol);
    }
  };
  for (Piece pc; ok && piece_at<SPLIT, PAIR>(p, it, pc); ++it) {
    const int k0 = pc.k0, nb = pc.k1 - pc.k0;
    const Item wi = decode_item<PAIR>(p, pc.item);
    auto load_q = [&](int t) -> bool {
      if (!mbar_wait(BAR(C::QE + t), (it & 1) ^ 1, w)) return false;
      if (lead) mbar_arrive_expect_tx(BAR(C::QF + t), PAIR ? 2 * C::TILE_BYTES : C::TILE_BYTES);
      const uint32_t dst = sbase + C::Q_OFF + t * C::TILE_BYTES;
      int qt = 2 * wi.pair + t;  // past the last tile (odd count): rows past S read as zeros,
      if (MODE == kModeS2S && qt >= p.nblk) qt = p.nblk - 1;  // or a real tile whose rows are not stored
      const Blk bq = locate_block<MODE>(p, qt);
      if constexpr (kSegLoads<MODE>) {
        load_segments(dst, maps->q, BAR(C::QF + t), bq.row, wi, pol_q);
      } else if constexpr (PAIR) {
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_4d_pair(dst + a * C::ATOM_BYTES, &maps->q[0], FBAR(C::QF + t), a * 64, bq.row, wi.h, wi.b, pol_q);
      } else {
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_4d(dst + a * C::ATOM_BYTES, &maps->q[bq.map], BAR(C::QF + t), a * 64, bq.row, wi.h, wi.b, pol_q);
      }
      ++q_loads[t];
      return true;
    };
    BlockWalker<MODE> kw;
    kw.reset(p);
    if constexpr (MODE != kModeS2S) kw.b = k0;  // (the split tail is not used with per-partition blocks)
    auto load_kv = [&](bool is_v) -> bool {  // the walker's current key block
      const Blk bk = kw.block(p);
      const CUtensorMap* m = is_v ? &maps->v[bk.map] : &maps->k[bk.map];
      const uint32_t s = kv_it % C::NSTAGE;
      const uint32_t ph = (kv_it / C::NSTAGE) & 1;
      if (!mbar_wait(BAR(C::KVE + s), ph ^ 1, w)) return false;
      if (lead) mbar_arrive_expect_tx(BAR(C::KVF + s), C::TILE_BYTES);  // the pair's two halves make one tile
      const uint32_t dst = sbase + C::KV_OFF + s * C::KV_BYTES;
      if constexpr (kSegLoads<MODE>) {
        load_segments(dst, is_v ? maps->v : maps->k, BAR(C::KVF + s), bk.row, wi, pol_kv);
      } else if constexpr (PAIR) {
        // K: keys 64 r .. 64 r + 63 (the map's box is 64 rows), both column
        // atoms; V: all 128 keys of column atom r
        if (is_v) {
          tma_load_4d_pair(dst, m, FBAR(C::KVF + s), static_cast<int>(rank) * 64, bk.row, wi.h, wi.b, pol_kv);
        } else {
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_4d_pair(dst + a * C::K_ATOM_BYTES, m, FBAR(C::KVF + s), a * 64,
                             bk.row + static_cast<int>(rank) * 64, wi.h, wi.b, pol_kv);
        }
      } else {
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_4d(dst + a * C::ATOM_BYTES, m, BAR(C::KVF + s), a * 64, bk.row, wi.h, wi.b, pol_kv);
      }
      ++kv_it;
      return true;
    };
    ok = load_q(0) && load_kv(false) && load_q(1) && load_kv(true);
    kw.next(p);
    for (int j = 1; ok && j < nb; ++j, kw.next(p)) ok = load_kv(false) && load_kv(true);
  }
  if (!ok && lead) {
    // Aborting: wait (bounded) for the copies this thread started, so none
    // lands in shared memory after the CTA has exited. (A pair's copies all
    // complete on the leader's barriers, and neither CTA of a pair exits
    // before the other has finished.)
    const uint32_t n = kv_it < static_cast<uint32_t>(C::NSTAGE) ? kv_it : C::NSTAGE;
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t idx = kv_it - 1 - i;
      mbar_wait_drain(BAR(C::KVF + idx % C::NSTAGE), (idx / C::NSTAGE) & 1, 100000000ull);
    }
    for (int t = 0; t < 2; ++t)
      if (q_loads[t] > 0) mbar_wait_drain(BAR(C::QF + t), (q_loads[t] - 1) & 1, 100000000ull);
  }
}

// ------------------------------------------------------------------ MMA issuer
// PAIR: run by the leader alone; every MMA spans both CTAs (M = 256: 128 query
// rows of each, K and V from both halves) and every commit arrives on the
// barrier of both CTAs.
template <int D, bool SPLIT, bool PAIR = false>
__device__ void mma_role(const Params& p, uint32_t sbase, uint32_t bar0, uint32_t tmem,
                         const WaitCtl& w) {
  using C = Cfg<D, PAIR>;
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  constexpr int kM = PAIR ? 2 * kBM : kBM;
  constexpr uint32_t kIdescQK = idesc_bf16_f32(kM, kBN, false, false);  // Q, K both K-major
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kM, D, false, true);     // V is MN-major (d contiguous)
  auto umma_commit = [](uint32_t bar) {
    if constexpr (PAIR) umma_commit_pair(bar);
    else ::attn_a2a::umma_commit(bar);
  };
  uint32_t kv_it = 0;
  uint32_t ev_a = 0, ev_b = 0, ev_c = 0;  // events consumed per kind
  bool ok = true;

  auto issue_qk = [&](int t, uint32_t sK) {
    const uint32_t qa = sbase + C::Q_OFF + t * C::TILE_BYTES;
    const uint32_t kb = sbase + C::KV_OFF + sK * C::KV_BYTES;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk / 4) * C::ATOM_BYTES + (kk % 4) * 32;
      const uint32_t offk = (kk / 4) * C::K_ATOM_BYTES + (kk % 4) * 32;
      const uint64_t da = sdesc_sw128(qa + off, 16, 1024), db = sdesc_sw128(kb + offk, 16, 1024);
      if constexpr (PAIR) umma_ss_pair(tmem + t * 128, da, db, kIdescQK, kk > 0 ? 1u : 0u);
      else umma_ss(tmem + t * 128, da, db, kIdescQK, kk > 0 ? 1u : 0u);
    }
  };
  // O_t (+)= P_t V_j for key block j (counted from the piece's first) of a
  // piece of nb blocks; the relay has already seen P_t ready and O_t free.
  auto issue_pv = [&](int t, int j, uint32_t sV, int nb) {
    const uint32_t vb = sbase + C::KV_OFF + sV * C::KV_BYTES;
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk) {
      const uint64_t dv = sdesc_sw128(vb + kk * 2048, C::ATOM_BYTES, 1024);
      if constexpr (PAIR)
        umma_ts_pair(tmem + 256 + t * D, tmem + t * 128 + kk * 8, dv, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      else
        umma_ts(tmem + 256 + t * D, tmem + t * 128 + kk * 8, dv, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
    }
    if (t == 1) umma_commit(BAR(C::KVE + sV));  // V_j now read by both tiles
    if (j == nb - 1) umma_commit(BAR(C::OF + t));
  };
  // wait for the relay's next event of one kind (its barrier's next phase)
  auto sync = [&](int bar, uint32_t& n) -> bool {
    if (!mbar_wait(BAR(bar), n++ & 1u, w)) return false;
    tc_fence_after();
    return true;
  };

  for (int it = 0; ok; ++it) {
    Piece pc;
    if (!piece_at<SPLIT, PAIR>(p, it, pc)) break;
    const int nb = pc.k1 - pc.k0;
    uint32_t sVprev = 0;
    if (!sync(C::EVA, ev_a)) { ok = false; break; }  // A: both Q tiles and the piece's first K
    issue_qk(0, kv_it % C::NSTAGE);
    umma_commit(BAR(C::SF + 0));
    for (int j = 0; j < nb; ++j) {  // the piece's key blocks, counted from its first
      const uint32_t sK = kv_it % C::NSTAGE;
      if (j > 0) {
        if (!sync(C::EVC, ev_c)) { ok = false; break; }  // C_j: P1_{j-1} (and O1 free at j = 1)
        issue_pv(1, j - 1, sVprev, nb);
      }
      issue_qk(1, sK);
      umma_commit(BAR(C::SF + 1));
      umma_commit(BAR(C::KVE + sK));  // K_j read by both tiles
      if (j == nb - 1) {
        umma_commit(BAR(C::QE + 0));
        umma_commit(BAR(C::QE + 1));
      }
      ++kv_it;
      const uint32_t sV = kv_it % C::NSTAGE;
      // B_j: V_j and P0_j (and O0 free at j = 0), and K_{j+1}, so that
      // O0 += P0 V_j and S0_{j+1} go to the tensor core back to back
      if (!sync(C::EVB, ev_b)) { ok = false; break; }
      issue_pv(0, j, sV, nb);
      sVprev = sV;
      ++kv_it;
      if (j + 1 < nb) {
        issue_qk(0, kv_it % C::NSTAGE);
        umma_commit(BAR(C::SF + 0));
      }
    }
    if (ok && !sync(C::EVC, ev_c)) ok = false;  // E: P1 of the last block (and O1 free if there is one block)
    if (ok) issue_pv(1, nb - 1, sVprev, nb);
  }
  if (!ok) {
    // Aborting: let every MMA already issued finish before TMEM is freed.
    umma_commit(BAR(C::DONE));
    mbar_wait_drain(BAR(C::DONE), 0, 100000000ull);
  }
}

// ------------------------------------------------------------------ relay
// Completes the MMA issuer's events, one barrier phase per event, in issue
// order:
//   A    EVA, the relay's arrival: both Q tiles and the piece's first K landed -> S0_0
//   C_j  EVC, tile 1's 128 softmax threads (P1_{j-1} written) and the relay
//        (O1 free at j = 1), j > 0                                 -> O1 += P1 V, S1_j
//   B_j  EVB, tile 0's 128 softmax threads (P0_j written) and the relay (V_j
//        landed, O0 free at j = 0, K_{j+1} landed unless j is last) -> O0 += P0 V, S0_{j+1}
//   E    EVC, tile 1's softmax threads (P1 of the last block) and the relay
//        (O1 free if the piece has one block)                      -> last O1 += P1 V
// The probabilities' readiness thus reaches the issuer in one hop, while the
// relay takes the waits on the TMA and O-free barriers off the issuer. The
// relay arrives for an event only once the barrier's previous phase has
// completed, so its arrival cannot count toward the previous event; the
// softmax threads' arrivals for an event need an S that is issued only after
// the issuer consumed the previous one, so they cannot either.
// PAIR: run by the leader alone, on the leader's barriers, which count both
// CTAs' loads and both CTAs' softmax and O-free arrivals.
template <int D, bool SPLIT, bool PAIR = false>
__device__ void relay_role(const Params& p, uint32_t bar0, const WaitCtl& w) {
  using C = Cfg<D, PAIR>;
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t kv_it = 0;
  uint32_t n_b = 0, n_c = 0;  // EVB / EVC events arrived for so far
  int it = 0;
  auto kv_ready = [&]() -> bool {
    const bool r = mbar_wait(BAR(C::KVF + kv_it % C::NSTAGE), (kv_it / C::NSTAGE) & 1, w);
    ++kv_it;
    return r;
  };
  auto o_free = [&](int t) -> bool { return mbar_wait(BAR(C::OE + t), (it & 1) ^ 1, w); };
  // before arriving for an event of a barrier: its previous phase has completed
  auto after_previous = [&](int bar, uint32_t& n) -> bool {
    const bool r = n == 0 || mbar_wait(BAR(bar), (n - 1) & 1u, w);
    ++n;
    return r;
  };
  for (Piece pc; piece_at<SPLIT, PAIR>(p, it, pc); ++it) {
    const int nb = pc.k1 - pc.k0;
    if (!(mbar_wait(BAR(C::QF + 0), it & 1, w) && mbar_wait(BAR(C::QF + 1), it & 1, w))) return;
    if (!kv_ready()) return;
    mbar_arrive(BAR(C::EVA));  // A
    for (int j = 0; j < nb; ++j) {
      if (j > 0) {
        if (!after_previous(C::EVC, n_c)) return;
        if (j == 1 && !o_free(1)) return;
        mbar_arrive(BAR(C::EVC));  // C_j
      }
      if (!after_previous(C::EVB, n_b)) return;
      if (!kv_ready()) return;  // V_j
      if (j == 0 && !o_free(0)) return;
      if (j + 1 < nb && !kv_ready()) return;  // K_{j+1}
      mbar_arrive(BAR(C::EVB));  // B_j
    }
    if (!after_previous(C::EVC, n_c)) return;
    if (nb == 1 && !o_free(1)) return;
    mbar_arrive(BAR(C::EVC));  // E
  }
}

// ------------------------------------------------------------------ per-tile trace
// Traced instantiations (TRACE = true) record, per work item, query tile t and
// warp w of the tile's warpgroup, kTraceRecord int64 at
// trace[((item * 2 + t) * 4 + w) * kTraceRecord]:
//   0 %globaltimer when the tile's first scores are ready (its Q loop starts)
//   1 %globaltimer when its O accumulator is final (the Q loop ends)
//   2 %globaltimer when the warp starts issuing the tile's output stores
//   3 %globaltimer when the warp has issued them and resumes (for the bulk
//     stores' issuing thread: after the commit and the wait for the staging
//     tile to be read)
//   4 SM clock cycles between 2 and 3 (finer than the timer's resolution)
//   5 %smid, 6 blockIdx.x, 7 the tile's first sequence row
// This is the per-tile store-span record of the X-Stage pages' validation
// ("Results": tensor-core timelines and store-span distributions).
constexpr int kTraceRecord = 8;

__device__ __forceinline__ uint32_t smid_u32() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

// ------------------------------------------------------------------ softmax / epilogue
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Row maximum of the 128 scores (keys >= valid excluded when MASK).
template <bool MASK>
__device__ __forceinline__ float row_max(const uint32_t (&sr)[128], int valid) {
  float a[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 128; i += 2) {
    float x0 = __uint_as_float(sr[i]), x1 = __uint_as_float(sr[i + 1]);
    if (MASK) {
      x0 = i < valid ? x0 : -INFINITY;
      x1 = i + 1 < valid ? x1 : -INFINITY;
    }
    a[(i / 2) & 3] = max3f(a[(i / 2) & 3], x0, x1);
  }
  return max3f(a[0], a[1], fmaxf(a[2], a[3]));
}

// p_i = 2^(s_i * sl2 - m) for the 128 keys of the block, packed to bf16 pairs
// in pk; returns the fp32 sum of the p_i (FlashAttention's convention: the
// row sum is not rounded, the probabilities fed to P*V are). Keys >= valid
// get p = 0 when MASK.
template <bool MASK>
__device__ __forceinline__ float probs(const uint32_t (&sr)[128], uint32_t (&pk)[64], float sl2, float neg_m,
                                       int valid) {
  const uint64_t scale2 = f2_pack(sl2, sl2);
  const uint64_t bias2 = f2_pack(neg_m, neg_m);
  uint64_t acc[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) acc[a] = f2_pack(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    float x0, x1, p0, p1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), scale2, bias2), x0, x1);
    p0 = ex2_approx(x0);
    p1 = ex2_approx(x1);
    if (MASK) {
      p0 = 2 * i < valid ? p0 : 0.f;
      p1 = 2 * i + 1 < valid ? p1 : 0.f;
    }
    acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
  float s0, s1;
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
  return s0 + s1;
}

// Bulk-store epilogue of one tile (kModeA2AT, kModeContigT, kModeS2SGT), the
// owner threads' part: each writes its normalised bf16 row into the staging
// buffer (128-byte swizzle, as the tensor map expects) and hands it to the
// async proxy. The store role issues the tile's tensor stores.
template <int D>
__device__ __forceinline__ void stage_tile(uint32_t stg, int r, const uint32_t (&o)[D], float inv_l) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint32_t a = static_cast<uint32_t>(c / 8) * (128u * 128u);  // 64-column atom
    const uint32_t addr = stg + a + static_cast<uint32_t>(r) * 128u + static_cast<uint32_t>(((c % 8) ^ (r & 7)) * 16);
    const uint32_t x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
    const uint32_t y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
    const uint32_t z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
    const uint32_t v = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(v) : "memory");
  }
  fence_proxy_async_smem();
}

// Where tile t of work item wi goes by bulk tensor store: false when the tile
// has no rows or straddles two partitions (then its rows are stored from
// registers); else the output map and the coordinates (y, z) - (head, first
// row in the partition) for the all-to-all layout, (first row, head) for the
// contiguous one.
template <int MODE>
__device__ __forceinline__ bool tile_store_target(const Params& p, const Item& wi, int t, int& map, int& y, int& z) {
  const int s0 = (2 * wi.pair + t) * kBM;  // the tile's first sequence row
  map = 0;
  if (s0 >= p.S) return false;
  if constexpr (MODE == kModeContigT) {
    y = s0;
    z = wi.h;
    return true;
  } else {
    int j0, l0, c0, j1, l1, c1;
    chunk_of_row(p.epi, s0, j0, l0, c0);
    map = j0;
    y = wi.h;
    z = l0;
    if (p.half_stores) return true;  // two halves, each inside one partition (store_role)
    chunk_of_row(p.epi, min(s0 + kBM, p.S) - 1, j1, l1, c1);
    return j0 == j1 && j0 < kMaxStoreMaps;  // the whole tile lands in one partition
  }
}

// ------------------------------------------------------------------ store role
// Bulk-store modes: one thread of warp 3 issues every tile's tensor stores, so
// that the owner warps go back to their next work as soon as they have staged
// their rows. The staging buffer's uses run tile 0, then tile 1, of each
// piece; for every use, bulk or not, it waits until the four owner warps
// have arrived on STGW + t (after staging, or at once for a tile without bulk
// stores or a partial piece's), issues the tile's stores and waits until they
// have read the staging buffer, and then releases the buffer (STG + t, one
// phase per piece) to the next use, which waits for that release before it
// stages (stg_free in softmax_role).
// Before returning (also on an abort) it waits until its stores have read the
// staging buffer: shared memory must outlive those reads, while the writes
// themselves are complete, like any of the grid's, when the grid is.
template <int D, int MODE, int NMAP, bool SPLIT, bool PAIR = false>
__device__ void store_role(const Params& p, const Maps<NMAP>* maps, uint32_t stg, uint32_t bar0, const WaitCtl& w) {
  using C = Cfg<D, PAIR>;
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t n[2] = {0, 0};  // uses of each tile so far
  bool ok = true;
  for (int it = 0; ok; ++it) {
    Piece pc;
    if (!piece_at<SPLIT, PAIR>(p, it, pc)) break;
    const Item wi = decode_item<PAIR>(p, pc.item);
    for (int t = 0; t < 2; ++t) {
      if (!mbar_wait(BAR(C::STGW + t), n[t]++ & 1u, w)) {
        ok = false;
        break;
      }
      int map, y, z;
      if (!(SPLIT && pc.kind == 1) && tile_store_target<MODE>(p, wi, t, map, y, z)) {
        if (MODE != kModeContigT && p.half_stores) {
          // rows [s, s + 64) of each half into the partition that holds them
          // (a half starting at or past S has no rows)
          const int s0 = (2 * wi.pair + t) * kBM;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int s = s0 + h * (kBM / 2);
            if (s < p.S) {
              int j, l, c;
              chunk_of_row(p.epi, s, j, l, c);
#pragma unroll
              for (int a = 0; a < D / 64; ++a)
                tma_store_4d(&maps->o[j], stg + a * 128 * 128 + h * 64 * 128, a * 64, y, l, wi.b);
            }
          }
        } else {
#pragma unroll
          for (int a = 0; a < D / 64; ++a) tma_store_4d(&maps->o[map], stg + a * 128 * 128, a * 64, y, z, wi.b);
        }
        bulk_commit_group();
        bulk_wait_read_all();  // the buffer may be reused once the stores have read it
      }
      mbar_arrive(BAR(C::STG + t));
    }
  }
  bulk_wait_read_all();
}

// Partial piece of a split item: this thread's row of the tile - unnormalised
// O (read from TMEM, 32 columns at a time), running maximum m (log2 domain)
// and row sum l - into the workspace slot of this CTA's range; then the warp's
// flag is raised to this launch's epoch (every lane's stores fenced first).
// Measured on GB300: releasing O before the stores and raising the flag a
// piece later, after the stores had drained, made the split schedule 2 %
// slower (image preset) than waiting for them here.
template <int D>
__device__ __forceinline__ void write_partial(const Params& p, int t, int r, int lane, int w4, uint32_t tO, float m,
                                              float l) {
  const size_t tile = static_cast<size_t>(split_range()) * 2 + t;
  const size_t row = tile * kBM + r;
  float4* dst = reinterpret_cast<float4*>(p.ws_o) + tile * (D / 4) * kBM + r;  // column group g at dst[g * 128]
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t x[32];
    tmem_ld_x32(tO + c * 32, x);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      dst[(c * 8 + i) * kBM] = make_float4(__uint_as_float(x[4 * i]), __uint_as_float(x[4 * i + 1]),
                                           __uint_as_float(x[4 * i + 2]), __uint_as_float(x[4 * i + 3]));
  }
  *reinterpret_cast<float2*>(p.ws_ml + row * 2) = make_float2(m, l);
  __threadfence();
  __syncwarp();
  if (lane == 0) st_release_gpu_u32(p.ws_flags + tile * 4 + w4, p.epoch);
}

// Final piece of a split `item`: merge the partial pieces of the same item
// (ranges g + 1 .. g_last after this CTA's g, which cover the item's other key
// blocks) into this row's accumulator O in TMEM (tO) and its (m, l): with M
// the largest maximum, O = sum O_i 2^(m_i - M) and l = sum l_i 2^(m_i - M)
// over the pieces, the usual combination of softmax partial results. One
// partial at a time, 32 columns at a time, so that it needs few registers
// (loading the next 32 columns meanwhile measured no faster).
// Each warp waits only for the same warp of the other CTAs (it holds the same
// rows). Called before O is released to the next piece. False on abort.
template <int D>
__device__ __forceinline__ bool merge_partials(const Params& p, int item, int t, int r, int w4, uint32_t tO, float& m,
                                               float& l, const WaitCtl& w) {
  const int g_last = ((item - p.tail_first) * p.nblk + p.nblk - 1) / p.tail_len;
  for (int gs = split_range() + 1; gs <= g_last; ++gs) {
    const size_t tile = static_cast<size_t>(gs) * 2 + t;
    if (!__all_sync(0xffffffffu, flag_wait(p.ws_flags + tile * 4 + w4, p.epoch, w))) return false;
    const size_t row = tile * kBM + r;
    const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + row * 2);
    const float mx = fmaxf(m, ml.x);
    const float a = ex2_approx(m - mx), b = ex2_approx(ml.x - mx);
    const float4* src = reinterpret_cast<const float4*>(p.ws_o) + tile * (D / 4) * kBM + r;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t x[32];
      tmem_ld_x32(tO + c * 32, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 yy = src[(c * 8 + i) * kBM];
        x[4 * i + 0] = __float_as_uint(fmaf(__uint_as_float(x[4 * i + 0]), a, yy.x * b));
        x[4 * i + 1] = __float_as_uint(fmaf(__uint_as_float(x[4 * i + 1]), a, yy.y * b));
        x[4 * i + 2] = __float_as_uint(fmaf(__uint_as_float(x[4 * i + 2]), a, yy.z * b));
        x[4 * i + 3] = __float_as_uint(fmaf(__uint_as_float(x[4 * i + 3]), a, yy.w * b));
      }
      tmem_st_x32(tO + c * 32, x);
    }
    l = fmaf(l, a, ml.y * b);
    m = mx;
  }
  return true;
}

// kModeA2AC epilogue of one warp: its 32 rows (this lane's row in o, scaled
// by inv_l, going to dst, or nowhere when dst is null) in two passes of 16
// rows through the warp's own slice `wbuf` of the staging buffer (TILE_BYTES/8
// bytes: 16 rows). Each row is written into the slice with its 16-byte chunks
// rotated by the row index (chunk c at c ^ row, so that the 16 rows' stores
// spread over the banks), then read back so that the lanes of one store
// instruction hold consecutive chunks of whole rows: 512 bytes of
// consecutive addresses per row pair (d = 128) or row quadruple (d = 64).
template <int D>
__device__ __forceinline__ void line_store_rows(uint32_t wbuf, int lane, uint16_t* dst, const uint32_t (&o)[D],
                                                float inv_l) {
  constexpr int RB = D * 2;        // bytes per row
  constexpr int CH = RB / 16;      // 16-byte chunks per row
  constexpr int RP = 16;           // rows per pass: the slice holds 16 rows
  constexpr int RPI = 512 / RB;    // rows per store instruction
  static_assert(RP * RB == Cfg<D>::TILE_BYTES / 8, "slice size");
  const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int pass = 0; pass < 32 / RP; ++pass) {
    const int rr = lane - pass * RP;  // this lane's row within the pass, if it is in it
    if (rr >= 0 && rr < RP) {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const uint32_t x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
        const uint32_t y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
        const uint32_t z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
        const uint32_t w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
        const uint32_t a = wbuf + static_cast<uint32_t>(rr * RB + ((c ^ (rr & (CH - 1))) * 16));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
      }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < RP / RPI; ++i) {
      const int row = i * RPI + lane / CH;  // within the pass
      const int c = lane % CH;
      const unsigned long long rp = __shfl_sync(0xffffffffu, mine, pass * RP + row);
      const uint32_t a = wbuf + static_cast<uint32_t>(row * RB + ((c ^ (row & (CH - 1))) * 16));
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
      if (rp != 0ull) reinterpret_cast<uint4*>(rp)[c] = v;
    }
    __syncwarp();
  }
}

template <int D, int MODE, int NMAP, bool TRACE, bool SPLIT, bool PAIR = false>
__device__ void softmax_role(const Params& p, int t, uint32_t bar0, uint32_t tmem, const Maps<NMAP>* maps,
                             uint32_t stg, const WaitCtl& w) {
  using C = Cfg<D, PAIR>;
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  // The staging buffer is free for this tile's use at work item `it` once
  // warp 3 is done with the use before it, the other tile's: tile 1 waits for
  // tile 0's release at `it`, tile 0 for tile 1's at it - 1. Each tile waits
  // on the other tile's barrier, whose releases cannot run two phases ahead
  // of the waiter (the other tile's next use needs this one staged first), so
  // the parity wait is exact; one barrier for both tiles was not (a tile
  // could wait for phase u - 1 while its own use u - 2 was still unreleased).
  auto stg_free = [&](int item_it) -> bool {
    if (t == 0) return item_it == 0 || mbar_wait(BAR(C::STG + 1), (item_it - 1) & 1u, w);
    return mbar_wait(BAR(C::STG + 0), item_it & 1u, w);
  };
  // This thread's arrival on an event of the MMA issuer (EVB, EVC, OE): a
  // pair's events are the leader's barriers, on which the other CTA arrives
  // once per warp for its 32 threads (warp-uniform call).
  auto arrive_event = [&](int i) {
    if constexpr (PAIR) {
      if (rank != 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(BAR(i), 0), 32);
        return;
      }
    }
    mbar_arrive(BAR(i));
  };
  const int r = (warp & 3) * 32 + lane;  // this thread's row of the tile = its TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_off + t * 128;
  const uint32_t tO = tmem + lane_off + 256 + t * D;
  const float sl2 = p.scale_log2;
  uint32_t sf_cnt = 0;
  for (int it = 0;; ++it) {
    int item, nb;
    {
      Piece pc;
      if (!piece_at<SPLIT, PAIR>(p, it, pc)) break;
      item = pc.item;
      nb = pc.k1 - pc.k0;
    }
    const Item wi = decode_item<PAIR>(p, item);
    const int srow = (2 * wi.pair + t) * kBM + r;
    uint64_t tr_q0 = 0, tr_q1 = 0, tr_e0 = 0;  // trace stamps (TRACE only)
    long long tr_c0 = 0;
    // the warp's record: written by lane 0 once the warp has issued its stores
    auto trace_out = [&]() {
      if constexpr (TRACE) {
        if (lane == 0) {
          long long* rec = p.trace + ((static_cast<long long>(item) * 2 + t) * 4 + (warp & 3)) * kTraceRecord;
          const long long c1 = clock64();
          rec[0] = static_cast<long long>(tr_q0);
          rec[1] = static_cast<long long>(tr_q1);
          rec[2] = static_cast<long long>(tr_e0);
          rec[3] = static_cast<long long>(globaltimer_ns());
          rec[4] = c1 - tr_c0;
          rec[5] = smid_u32();
          rec[6] = blockIdx.x;
          rec[7] = (2 * wi.pair + t) * kBM;
        }
      }
    };
    float m_used = -INFINITY;
    float l = 0.f;
    BlockWalker<MODE> kb;
    kb.reset(p);
    if constexpr (MODE != kModeS2S) {
      Piece pc;
      piece_at<SPLIT, PAIR>(p, it, pc);
      kb.b = pc.k0;  // (the split tail is not used with per-partition blocks)
    }
    for (int j = 0; j < nb; ++j) {  // the piece's key blocks, counted from its first
      const bool got = __all_sync(0xffffffffu, mbar_wait(BAR(C::SF + t), sf_cnt & 1, w));
      if (!got) return;
      ++sf_cnt;
      if constexpr (TRACE) {
        if (j == 0) tr_q0 = globaltimer_ns();
      }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld_x128(tS, sr);
      const Blk bk = kb.block(p);
      kb.next(p);
      const int valid = bk.c - bk.row;  // keys of this block that exist (>= 128 except at the end)
      uint32_t pk[64];
      // Exponentiate against the running maximum m_used without first taking
      // this block's maximum (the maximum only guards against overflow, and
      // it moves rarely once a few blocks are in). Every p is at most the
      // block's row sum, so a sum within kSpecBound proves the stale maximum
      // safe; otherwise (and on the first block) take the block's maximum,
      // rescale O and l by 2^(m_used - m_new), and redo the block. The
      // decision is warp-uniform because the TMEM loads and stores are
      // warp-collective; rows whose maximum did not grow get alpha = 1.
      float ls = -1.0f;
      if (m_used != -INFINITY)
        ls = valid >= kBN ? probs<false>(sr, pk, sl2, -m_used, valid) : probs<true>(sr, pk, sl2, -m_used, valid);
      if (__any_sync(0xffffffffu, !(ls >= 0.0f && ls <= kSpecBound))) {
        const float mx = valid >= kBN ? row_max<false>(sr, valid) : row_max<true>(sr, valid);
        const float m_tgt = fmaxf(m_used, mx * sl2);
        // 0 on the first block (m_used = -inf); exactly 1 where the maximum did not move
        const float alpha = m_tgt == m_used ? 1.0f : ex2_approx(m_used - m_tgt);
        if (j > 0) {
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_x32(tO + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), x0, x1);
              o[i] = __float_as_uint(x0);
              o[i + 1] = __float_as_uint(x1);
            }
            tmem_st_x32(tO + c * 32, o);
          }
        }
        l *= alpha;
        m_used = m_tgt;
        ls = valid >= kBN ? probs<false>(sr, pk, sl2, -m_used, valid) : probs<true>(sr, pk, sl2, -m_used, valid);
      }
      l += ls;
      tmem_st_x64(tS, pk);
      tc_fence_before();
      // P_t written: this thread's arrival on the issuer's event (B_j for tile 0,
      // C_{j+1} or E for tile 1)
      if (!(p.inject_stall && t == 0 && j == 0 && it == 0)) arrive_event(t == 0 ? C::EVB : C::EVC);  // test hook
    }
    // ---- epilogue: the tile owner stores its rows to their destination and moves on
    const bool got = __all_sync(0xffffffffu, mbar_wait(BAR(C::OF + t), it & 1, w));
    if (!got) return;
    if constexpr (TRACE) tr_q1 = globaltimer_ns();
    tc_fence_after();
    if constexpr (SPLIT) {
      Piece pc;
      piece_at<SPLIT>(p, it, pc);
      if (pc.kind == 1) {
        // a partial piece of a split item: its O goes to the workspace, no
        // output; the staging buffer of the bulk-store epilogue is passed on in turn
        write_partial<D>(p, t, r, lane, warp & 3, tO, m_used, l);
        tc_fence_before();
        mbar_arrive(BAR(C::OE + t));
        if constexpr (kBulkStores<MODE>) {
          // no stores for the store role: this use only passes the staging buffer on
          if (lane == 0) {
            if (!stg_free(it)) return;
            mbar_arrive(BAR(C::STGW + t));
          }
        }
        continue;
      }
      if (pc.kind == 2 && !merge_partials<D>(p, item, t, r, warp & 3, tO, m_used, l, w)) return;
    }
    uint32_t o[D];
    if constexpr (D == 128) tmem_ld_x128(tO, o);
    else tmem_ld_x64(tO, o);
    tc_fence_before();
    arrive_event(C::OE + t);  // O_t may now be overwritten by the next item
    if constexpr (TRACE) {
      tr_e0 = globaltimer_ns();
      tr_c0 = clock64();
    }
    if constexpr (kBulkStores<MODE>) {
      // Each use waits until warp 3 is done with the staging buffer's
      // previous use (stg_free), stages the tile when it goes out by bulk
      // stores, and each warp arrives on STGW + t for the store role, which
      // issues them.
      int map, y, z;
      const bool bulk = tile_store_target<MODE>(p, wi, t, map, y, z);
      if (bulk) {
        if (!__all_sync(0xffffffffu, stg_free(it))) return;
        stage_tile<D>(stg, r, o, 1.0f / l);
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::STGW + t));
        trace_out();
        continue;
      }
      // no bulk store for this tile: its rows go from registers below
      if (lane == 0) {
        if (!stg_free(it)) return;
        mbar_arrive(BAR(C::STGW + t));
      }
    }
    uint16_t* dst = nullptr;
    if constexpr (MODE == kModeS2S) {
      const int qt = 2 * wi.pair + t;
      if (qt < p.nblk) {
        const Blk bq = locate_block<MODE>(p, qt);
        const int lrow = bq.row + r;
        if (lrow < bq.c)
          dst = static_cast<uint16_t*>(p.epi.part[bq.map]) +
                ((static_cast<int64_t>(wi.b) * bq.c + lrow) * p.H + wi.h) * D;
      }
    } else if (srow < p.S) {
      if constexpr (MODE == kModeA2A || MODE == kModeA2AC) {
        if (p.epi.crem == 0) {
          // equal partitions: the row's partition is one division away
          // (measured 0.3 % faster per launch at the video shape than the
          // general rule of out_row_ptr)
          const int j = srow / p.epi.cbase;
          const int lr = srow - j * p.epi.cbase;
          const int hs = p.epi.hstride > 0 ? p.epi.hstride : p.H;
          dst = static_cast<uint16_t*>(p.epi.part[j]) + ((static_cast<int64_t>(wi.b) * p.epi.cbase + lr) * hs + wi.h) * D;
        } else {
          dst = out_row_ptr<D, true>(p.epi, p.B, p.H, p.S, wi.b, wi.h, srow);
        }
      } else {
        dst = out_row_ptr<D, MODE != kModeContig && MODE != kModeContigT>(p.epi, p.B, p.H, p.S, wi.b, wi.h, srow);
      }
    }
    if constexpr (MODE == kModeA2AC) {
      line_store_rows<D>(stg + static_cast<uint32_t>(t * 4 + (warp & 3)) * (Cfg<D>::TILE_BYTES / 8), lane, dst, o,
                         1.0f / l);
    } else if (dst != nullptr) {
      const float inv_l = 1.0f / l;
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
        v.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
        v.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
        v.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
        d4[c] = v;
      }
    }
    trace_out();
  }
}

// ------------------------------------------------------------------ kernel
// PAIR: launched in clusters of two CTAs (the CTA-pair kernel); the leader's
// warps 1 and 2 run the pair's MMA issuer and relay, the other CTA's stay idle.
template <int D, int MODE, int NMAP, bool TRACE = false, bool SPLIT = false, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_tc_kernel(const __grid_constant__ Maps<NMAP> maps, const __grid_constant__ Params p) {
  static_assert(!PAIR || (!TRACE && !SPLIT && kBulkStores<MODE>), "CTA pairs: plain bulk-store kernels only");
  using C = Cfg<D, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::MISC_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::MISC_OFF + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(C::QF + t), 1);
      mbar_init(BAR(C::QE + t), 1);
      mbar_init(BAR(C::SF + t), 1);
      mbar_init(BAR(C::OF + t), 1);
      mbar_init(BAR(C::OE + t), PAIR ? 2 * kBM : kBM);  // a pair's: both CTAs' rows
    }
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(BAR(C::KVF + s), 1);
      mbar_init(BAR(C::KVE + s), 1);
    }
    mbar_init(BAR(C::DONE), 1);
    mbar_init(BAR(C::STG + 0), 1);
    mbar_init(BAR(C::STG + 1), 1);
    mbar_init(BAR(C::STGW + 0), 4);  // one arrive per warp of the tile
    mbar_init(BAR(C::STGW + 1), 4);
    mbar_init(BAR(C::EVA), 1);
    mbar_init(BAR(C::EVB), (PAIR ? 2 * kBM : kBM) + 1);
    mbar_init(BAR(C::EVC), (PAIR ? 2 * kBM : kBM) + 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    const int nmaps = MODE == kModeS2S || kSegLoads<MODE> ? p.epi.P : 1;
    if (MODE == kModeA2AT || MODE == kModeS2SGT)
      for (int i = 0; i < p.epi.P && i < kMaxStoreMaps; ++i)
        if (p.epi.cbase > 0 || i < p.epi.crem) tma_prefetch_desc(&maps.o[i]);  // partitions with rows only
    if (MODE == kModeContigT) tma_prefetch_desc(&maps.o[0]);
    for (int i = 0; i < nmaps; ++i) {
      tma_prefetch_desc(&maps.q[i]);
      tma_prefetch_desc(&maps.k[i]);
      tma_prefetch_desc(&maps.v[i]);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // a pair: neither CTA signals the other's barriers before they are
  // initialised, and the leader issues no MMA before both TMEMs are allocated
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // A kernel queued behind this one with programmatic serialisation may
  // launch now (no effect without one): a tail kernel takes each SM as this
  // kernel's CTA there exits; the next call's first kernel runs its set-up
  // there and waits. A dependent grid launches only once every CTA of this
  // one has started, so its waiting CTAs never keep one of this grid's off
  // an SM (a split kernel's ranges must all be resident at once).
  if (!SPLIT || (p.pdl & kPdlTrigger)) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched behind the previous kernel of the stream: the set-up above
  // overlapped its last CTAs; nothing global is touched before it has
  // completed and its memory operations are visible.
  if (p.pdl & kPdlWait) asm volatile("griddepcontrol.wait;" ::: "memory");
  const WaitCtl w{abort_flag, p.dev_status, p.timeout_ns};

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    const bool lead = !PAIR || cluster_ctarank() == 0;
    if (warp == 0) {
      if (lane == 0) producer_role<D, MODE, NMAP, SPLIT, PAIR>(p, &maps, sbase, bar0, w);
    } else if (warp == 1) {
      if (lane == 0 && lead) mma_role<D, SPLIT, PAIR>(p, sbase, bar0, tmem, w);
    } else if (warp == 2) {
      if (lane == 0 && lead) relay_role<D, SPLIT, PAIR>(p, bar0, w);
    } else if constexpr (kBulkStores<MODE>) {
      // every bulk store has read the staging buffer before the store role returns
      if (lane == 0) store_role<D, MODE, NMAP, SPLIT, PAIR>(p, &maps, sbase + C::STG_OFF, bar0, w);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    softmax_role<D, MODE, NMAP, TRACE, SPLIT, PAIR>(p, (warp - 4) / 4, bar0, tmem, &maps, sbase + C::STG_OFF, w);
  }
  if (p.pdl & kPdlWaitEnd) asm volatile("griddepcontrol.wait;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  // a pair: the leader's MMAs read the other CTA's shared memory and TMEM,
  // and the other CTA arrives on the leader's barriers, up to the end
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc
}  // namespace attn_a2a

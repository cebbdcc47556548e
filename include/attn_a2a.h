/*
 * attn_a2a.h - C ABI of libattn_a2a.so: non-causal bf16 attention forward on
 * NVIDIA GB300 (sm_103a) fused with the post-attention Ulysses all-to-all
 * layout change, plus a Burst-Gap store probe.
 *
 * Source of the operations (X-Stage: An Overlooked Pipeline Stage for
 * Communication-Computation Overlap in DiT Inference, gist.science
 * explanation):
 *   - "Key Contributions", FlashAttention-A2A (piggybacking): in Ulysses
 *     sequence-parallel attention the post-attention all-to-all is fused into
 *     FlashAttention; the owner of each output tile issues the stores of that
 *     tile to its destination and resumes the Q loop of its next tile, with no
 *     dedicated communication warp or SM.
 *   - Technical Summary, "Methodology", Burst-Gap equation
 *     T_iss(G; K, V) = max(T0_iss(K, V), V/R - G) with the measured
 *     quantities T0_iss, R and Q.
 *
 * Shapes and layouts (all tensors bf16, element strides in ELEMENTS):
 *   q, k, v : logical [B, H, S, d], innermost d contiguous; the caller gives
 *             the batch, head and sequence strides. "Head-sharded": virtual
 *             rank r holds heads [r*H/P, (r+1)*H/P) over the full sequence.
 *   output  : P partitions, partition j is a contiguous [B, c_j, H, d] array
 *             holding sequence rows [start_j, start_j + c_j) of every head
 *             ("sequence-sharded"). c_j = floor(S/P) + (j < S mod P ? 1 : 0),
 *             start_j = sum of the earlier c_i (torch.tensor_split rule).
 *   math    : O[b,h] = softmax(scale * Q[b,h] K[b,h]^T) V[b,h]; fp32
 *             accumulation and row sums, probabilities rounded to bf16
 *             before the P*V product, output rounded to bf16 (round to
 *             nearest even).
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns every buffer. The library allocates no
 *     device memory per call; it keeps small host-side state only (a cached
 *     driver entry point, the SM count per device, and the streams and
 *     events of attn_a2a_fwd_host), plus the fixed __device__ array of
 *     xstage_probe_run_noalloc.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream). Work is asynchronous on that stream and ordered with
 *     it as any kernel is. The attention calls launch their first kernel with
 *     programmatic stream serialisation: where the stream's previous work is
 *     a kernel that allows it (CUDA's programmatic dependent launch), their
 *     CTAs may start on SMs that kernel has left and run their set-up, but
 *     they wait for that kernel's completion before they read or write any
 *     buffer. A kernel the caller queues behind a call with programmatic
 *     serialisation waits, as usual, for the call's last kernel, whose
 *     completion covers all of the call's stores.
 *   - Errors: argument errors are detected on the host and returned
 *     synchronously before anything is launched (ATTN_A2A_EINVAL /
 *     ATTN_A2A_EUNSUPPORTED). A launch failure returns ATTN_A2A_ECUDA.
 *     Every in-kernel wait is bounded; if one expires the kernel stops all of
 *     its roles, writes ATTN_A2A_ETIMEOUT to *dev_status (when dev_status is
 *     not NULL) and returns, leaving the context usable. dev_status is a
 *     device int the caller clears to 0 beforehand and reads when it wants.
 *   - Alignment: every pointer 16-byte aligned; batch, head and sequence
 *     strides multiples of 8 elements (16 bytes).
 *   - Outputs must not alias inputs.
 */
#ifndef ATTN_A2A_H
#define ATTN_A2A_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_A2A_OK = 0,
  ATTN_A2A_EINVAL = 1,        /* bad argument (null, misaligned, out of range) */
  ATTN_A2A_EUNSUPPORTED = 2,  /* valid but not built (e.g. d not in {64,128}) */
  ATTN_A2A_ECUDA = 3,         /* CUDA runtime/driver error at launch */
  ATTN_A2A_ETIMEOUT = 4,      /* a bounded in-kernel wait expired (device status) */
  ATTN_A2A_ETOOLARGE = 5      /* request larger than the fixed scratch of an
                                 allocation-free entry point */
} attn_a2a_status;

/* Problem shape and input strides (elements). d is contiguous. */
typedef struct {
  int B, H, S, d;
  long long q_sb, q_sh, q_ss;
  long long k_sb, k_sh, k_ss;
  long long v_sb, v_sh, v_ss;
} attn_a2a_shape;

/* Tuning and test options for the *_ex entry points. Zero-initialised means
 * the defaults used by the plain entry points. */
typedef struct {
  int store_kind;       /* how the tile owner stores its output tile:
                           0 = automatic: 1 for the contiguous layout and for the
                               all-to-all layout with P <= 8 (where it measured
                               faster), else 2; where an output buffer
                               is not memory of the current device
                               (cudaPointerGetAttributes: host memory the device
                               can address, managed memory, another device's
                               memory), 3 for the all-to-all layout, and 2 for the
                               contiguous one;
                           1 = bulk tensor stores (TMA) from a shared-memory staging
                               tile: the owner commits the bulk group and resumes,
                               waiting only until the stores have read the staging
                               tile before reusing it; a tile that straddles two
                               partitions is stored as in 2. All-to-all layout
                               with P > 8, or an output buffer that is not memory
                               of the current device: ATTN_A2A_EUNSUPPORTED;
                           2 = vector st.global of each owned output row straight
                               from registers;
                           3 = whole-line row stores, all-to-all layout only (else
                               ATTN_A2A_EUNSUPPORTED): each warp passes its rows
                               through its own slice of a shared-memory staging
                               buffer, so that every store instruction writes
                               whole rows (512 consecutive bytes) instead of a
                               16-byte piece of each of 32 rows. For partitions
                               reached over a slower link than the GPU's own
                               memory, such as host memory that the device can
                               address (pinned, or coherent on a system with a
                               coherent host link) or another GPU's memory mapped
                               into this one's address space (1 uses tensor maps,
                               made for the device's own memory, and is refused
                               there; 2 stores 16-byte pieces of 32 rows at a time,
                               which such links drain far more slowly). Chosen
                               automatically for all-to-all outputs outside the
                               device's memory.
                           Results are identical; values > 3 are ATTN_A2A_EINVAL */
  int grid;             /* persistent CTAs; 0 = one per SM */
  long long timeout_ns; /* limit of every in-kernel wait; 0 = 2 000 000 000 ns */
  int inject_stall;     /* test hook, 0 in normal use. 1 = the softmax role of the first
                           query tile withholds its first "probabilities ready" signal,
                           so the MMA role's bounded wait expires and the kernel reports
                           ATTN_A2A_ETIMEOUT through dev_status and exits cleanly */
  int tile_order;       /* order of a head's work items (pairs of 128-row query tiles):
                           0 = sequence order (consecutive items write to the same
                           destination partition); 1 = chunk-interleaved: consecutive
                           items cycle through the P destination partitions, spreading
                           each wave's store burst over all of them (burst shaping).
                           Results are identical; only the store pattern changes */
  long long* trace;     /* NULL in normal use. Device int64 buffer of at least
                           ATTN_A2A_TRACE_BYTES(B, H, S) bytes, 8-byte aligned: runs
                           the traced instantiation of the same kernel, which records
                           per work item, query tile t and warp w of the tile owner
                           ATTN_A2A_TRACE_RECORD int64 at
                           trace[((item*2 + t)*4 + w) * ATTN_A2A_TRACE_RECORD]:
                           [0] %globaltimer ns when the tile's first scores are ready,
                           [1] when its output accumulator is final, [2] when the warp
                           starts issuing the tile's stores, [3] when it has issued them
                           and resumes; [4] SM cycles from [2] to [3]; [5] SM id;
                           [6] CTA index; [7] the tile's first sequence row. A work item
                           is a pair of 128-row query tiles of one (b, h):
                           item = (b*H + h) * ceil(ceil(S/128)/2) + pair, and CTA c runs
                           items c, c + grid, ... (the X-Stage pages' "Results":
                           per-tile store spans and tensor-core timelines). Results are
                           identical to the untraced call. attn_a2a_fwd_ex and
                           attn_a2a_fwd_contig_ex only */
  int part_heads;       /* 0 in normal use (= H). Ulysses head-group launch, all-to-all
                           layout only: the heads per row of each output partition,
                           >= H and a multiple of P. The call computes its H heads (one
                           rank's head group, e.g. heads [r*part_heads/P, (r+1)*part_heads/P)
                           of the layer) and stores head h of sequence row s at
                           out_partitions[j][(b*c_j + s - start_j)*part_heads + h] * d,
                           so the caller passes each partition pointer already offset
                           to the group's first head (h0 * d elements). P such calls,
                           one per head group, fill the partitions exactly as one call
                           over all part_heads heads does, byte for byte. Where the
                           partitions are another GPU's memory mapped into this one's
                           address space, this is the one-sided store of the pages'
                           FlashAttention-A2A ("Key Contributions") from rank r's tile
                           owners into rank j's buffer */
  int split;            /* 0 in normal use. With a workspace, how work items are divided
                           by key blocks (see workspace): ATTN_A2A_SPLIT_AUTO (0) lets
                           the library choose; ATTN_A2A_SPLIT_TAIL (1) divides only a
                           partial last wave, whenever there is one; ATTN_A2A_SPLIT_ALL
                           (2) divides every item's key blocks into equal ranges, one
                           per CTA, in one kernel; ATTN_A2A_SPLIT_NONE (3) divides
                           nothing. Other values: ATTN_A2A_EINVAL */
  void* workspace;      /* NULL in normal use. Device scratch of at least
                           ATTN_A2A_WORKSPACE_BYTES(grid, d) bytes (grid = the
                           persistent CTAs, attn_a2a_num_sms() by default), 256-byte
                           aligned, zeroed by the caller before its first use, not
                           overlapping any input or output. With it, when the last wave
                           of work items holds fewer items than there are CTAs, key
                           blocks of items are divided into equal ranges, one per CTA
                           (the split option): either the last wave's, in a second
                           kernel queued behind the first (programmatic dependent
                           launch), or every item's, in one kernel. A range that starts
                           inside an item writes that piece's partial result here; the
                           range holding the item's first key block merges the partials
                           and stores the tile. The automatic choice divides the last
                           wave when that saves each CTA at least 32 key blocks (long
                           sequences). Otherwise the call is the same as without a
                           workspace. The
                           kernel leaves the workspace valid for the next call; calls
                           that share one workspace must not run at the same time. Not
                           used with tile_order = 1 or trace. The split items agree with
                           the unsplit schedule to rounding (their key blocks are summed
                           in pieces); all other items are the same bytes.
                           attn_a2a_fwd_ex and attn_a2a_fwd_contig_ex only */
  long long workspace_bytes; /* size of workspace */
  int cta_pairs;        /* 0 in normal use: the library chooses. 1 = run the work on CTA
                           pairs: clusters of two CTAs on two SMs whose tensor cores
                           compute each pair of query tiles' scores and outputs as one
                           256-row MMA (tcgen05 cta_group::2), each CTA holding its own
                           query tiles and half of every K and V block, so that each SM
                           reads half the K/V bytes per key block from shared memory; a
                           work unit is then four 128-row query tiles of one (b, h).
                           Needs d = 128 and the bulk-store epilogue (store kind 1, or
                           the automatic kind into device memory), tile_order = 0 and no
                           trace; otherwise ATTN_A2A_EUNSUPPORTED. No split schedule:
                           the workspace is not used. grid then counts CTAs of pairs (an
                           odd count is cut to the even one below it). 2 = one CTA per
                           work item, as without this option. Results are the same bytes
                           as 2 (each row sums the same products in the same order).
                           Other values: ATTN_A2A_EINVAL */
} attn_a2a_opts;

/* attn_a2a_opts.split */
#define ATTN_A2A_SPLIT_AUTO 0
#define ATTN_A2A_SPLIT_TAIL 1
#define ATTN_A2A_SPLIT_ALL 2
#define ATTN_A2A_SPLIT_NONE 3

/* Workspace bytes of attn_a2a_opts.workspace for a grid of `grid` CTAs and
 * head dimension d: per CTA, a flag word per (query tile, warp), and one
 * partial result (O fp32, running maximum, row sum) of two 128-row tiles. */
#define ATTN_A2A_WORKSPACE_BYTES(grid, d) \
  (256LL + 32LL * (long long)(grid) + 1024LL * (long long)(grid) * ((long long)(d) + 2))

/* Trace record of attn_a2a_opts.trace: int64 per (work item, tile, warp), and
 * the buffer size in bytes for B, H, S. */
#define ATTN_A2A_TRACE_RECORD 8
#define ATTN_A2A_TRACE_BYTES(B, H, S) \
  ((long long)(B) * (H) * ((((long long)(S) + 127) / 128 + 1) / 2) * 2 * 4 * ATTN_A2A_TRACE_RECORD * 8)

/*
 * attn_a2a_fwd - fused attention + head-to-sequence all-to-all (the product).
 * The owner of each 128-row output tile of head h stores row s of that tile
 * to out_partitions[j][b, s - start_j, h, :] where j is the chunk holding s,
 * then returns to its next tile. A tile that straddles a chunk boundary is
 * split row by row; rows >= S are never stored.
 *   q, k, v        : device bf16, layout above, caller-owned, read only.
 *   shp            : host pointer to the shape/strides.
 *   P              : virtual ranks, 1 <= P <= 64, H % P == 0 (with
 *                    attn_a2a_opts.part_heads: part_heads % P == 0 instead).
 *   scale          : softmax scale, finite and >= 0 (1/sqrt(d) in DiT).
 *   out_partitions : HOST array of P device pointers, partition j is
 *                    [B, c_j, H, d] bf16 contiguous (may be NULL if c_j == 0).
 *   dev_status     : optional device int (NULL allowed), see conventions.
 * Returns an attn_a2a_status.
 */
int attn_a2a_fwd(const void* q, const void* k, const void* v, const attn_a2a_shape* shp,
                 int P, float scale, void* const* out_partitions, int* dev_status,
                 void* stream);

/* attn_a2a_fwd with options (NULL opts = defaults). */
int attn_a2a_fwd_ex(const void* q, const void* k, const void* v, const attn_a2a_shape* shp,
                    int P, float scale, void* const* out_partitions, int* dev_status,
                    const attn_a2a_opts* opts, void* stream);

/*
 * attn_a2a_fwd_contig - "attention alone": the same kernel and arithmetic
 * with the output tile stored contiguously to out = [B, H, S, d] bf16
 * (device, contiguous). Followed by attn_a2a_permute it is the serial
 * baseline (attention, then a separate all-to-all) of the pages' Results,
 * FlashAttention-A2A optimisation; its output is bit-identical to the fused
 * path's after the permutation.
 */
int attn_a2a_fwd_contig(const void* q, const void* k, const void* v, const attn_a2a_shape* shp,
                        float scale, void* out, int* dev_status, void* stream);

int attn_a2a_fwd_contig_ex(const void* q, const void* k, const void* v,
                           const attn_a2a_shape* shp, float scale, void* out, int* dev_status,
                           const attn_a2a_opts* opts, void* stream);

/*
 * attn_a2a_fwd_s2s - the whole Ulysses attention layer on virtual ranks:
 * sequence-sharded q, k, v in, sequence-sharded output out. Ulysses
 * sequence parallelism (the pages' FlashAttention-A2A setting) exchanges
 * twice around attention: sequence -> head sharding before it, head ->
 * sequence after it. attn_a2a_fwd folds the second exchange into the
 * epilogue; this call also folds the first one into the loads: each CTA
 * TMA-loads its Q, K and V tiles straight from the sequence-sharded input
 * partitions, so neither exchange is a separate pass.
 *   q_parts, k_parts, v_parts : HOST arrays of P device pointers; partition j
 *                    of each is [B, c_j, H, d] bf16 contiguous (chunk rule as
 *                    above; may be NULL if c_j == 0).
 *   shp            : B, H, S (= sum of c_j), d; the strides are ignored.
 *   P              : 1 <= P <= 8 (ATTN_A2A_EUNSUPPORTED beyond), H % P == 0.
 *   out_partitions : as for attn_a2a_fwd.
 * When all partitions have the same length and it is a multiple of 64 rows,
 * query tiles and key blocks are counted over the whole sequence and each
 * 128-row tile is loaded in pieces that lie inside one partition (one piece,
 * or two 64-row halves); the result is then bit-identical to attn_a2a_fwd's.
 * Otherwise tiles and key blocks are taken per partition (each starting at a
 * partition's first row), so the key blocks differ from attn_a2a_fwd's and
 * the rounding may differ in the last bits.
 */
int attn_a2a_fwd_s2s(const void* const* q_parts, const void* const* k_parts,
                     const void* const* v_parts, const attn_a2a_shape* shp, int P, float scale,
                     void* const* out_partitions, int* dev_status, void* stream);

/*
 * attn_a2a_fwd_s2s_ex - attn_a2a_fwd_s2s with options (opts may be NULL: as
 * attn_a2a_fwd_s2s). Taken: store_kind 0-2, grid, timeout_ns, inject_stall,
 * workspace / workspace_bytes and split, meaning what they mean for
 * attn_a2a_fwd_ex; the split schedule applies where tiles are counted over
 * the whole sequence (equal partitions of a multiple of 64 rows), and with
 * the same split the result is then the same bytes as attn_a2a_fwd_ex's. The
 * automatic choice (ATTN_A2A_SPLIT_AUTO) takes only the whole-schedule split
 * here (the last wave's split measured slower for the layer); an explicit
 * ATTN_A2A_SPLIT_TAIL is honoured. ATTN_A2A_EUNSUPPORTED for store_kind 3, tile_order 1, a
 * trace, part_heads or cta_pairs 1, which the whole-layer kernels do not
 * have; out-of-range values are ATTN_A2A_EINVAL. The workspace must not
 * overlap any input or output partition.
 */
int attn_a2a_fwd_s2s_ex(const void* const* q_parts, const void* const* k_parts,
                        const void* const* v_parts, const attn_a2a_shape* shp, int P, float scale,
                        void* const* out_partitions, int* dev_status, const attn_a2a_opts* opts,
                        void* stream);

/*
 * attn_a2a_permute - the serial all-to-all on its own: a pure copy of a
 * contiguous [B, H, S, d] bf16 device tensor o into the P partitions
 * (same layout and chunk rule as attn_a2a_fwd). shp supplies B, H, S, d; its
 * strides are ignored. H % P == 0 is required as for the fused call.
 */
int attn_a2a_permute(const void* o, const attn_a2a_shape* shp, int P,
                     void* const* out_partitions, void* stream);

/*
 * attn_a2a_fwd_simt - slow SIMT debug path (no tensor cores): the same
 * attention and the same partition epilogue computed by one warp per query
 * row in fp32 (probabilities are not rounded to bf16). For bring-up and
 * cross-checks on small problems only.
 */
int attn_a2a_fwd_simt(const void* q, const void* k, const void* v, const attn_a2a_shape* shp,
                      int P, float scale, void* const* out_partitions, void* stream);

/*
 * attn_a2a_fwd_host - the product call from host memory, for callers whose
 * data lives on the host: copies q, k, v (host, contiguous [B,H,S,d] bf16,
 * pinned for asynchronous copies) into the caller's device buffers dq, dk,
 * dv, runs the fused attention and delivers the partitions into hparts[j]
 * (host): when every hparts[j] with rows is pinned host memory
 * (cudaPointerGetAttributes type cudaMemoryTypeHost), the kernels store each
 * output row straight into it over the host link (whole-line row stores,
 * store_kind 3) and dparts is not written; otherwise they store into the
 * caller's device partitions dparts[j], copied back into hparts[j]. hparts
 * must not overlap hq, hk or hv. The heads are
 * processed in up to eight chunks - small first and last ones, so that
 * little copying is exposed before the first kernel and after the last - so
 * that the copies of one chunk overlap the kernel of another; the copies run
 * on two library-owned streams, and the chunks' kernels alternate between
 * `stream` and a third library-owned stream so that one kernel's last wave
 * overlaps the next kernel (the streams and four events are created on the
 * first call per device). Everything is ordered by events against `stream`:
 * it starts after the work already queued on `stream`, and `stream`
 * completes only after the last copy back. Returns after enqueueing;
 * synchronise `stream` before reading hparts. Calls on one device are
 * serialised while they enqueue.
 */
int attn_a2a_fwd_host(const void* hq, const void* hk, const void* hv, const attn_a2a_shape* shp,
                      int P, float scale, void* dq, void* dk, void* dv,
                      void* const* dparts, void* const* hparts, int* dev_status, void* stream);

/*
 * Burst-Gap probe (Technical Summary, "Methodology"; "Key Contributions",
 * characterisation by parameterised microbenchmarks). K producer CTAs run
 * `rounds` rounds; in each round every producer issues its share V/K of an
 * aggregate store burst of V bytes, then computes for a gap of G ns. Each
 * producer records three %globaltimer stamps per round into
 * stamps[(p * rounds + r) * 3 + {0,1,2}]: burst start, last store issued,
 * gap end. The issuer-visible issue time is stamp1 - stamp0. Destinations
 * advance through dst (dst_bytes, device, caller-owned scratch) so that
 * successive bursts do not hit the same lines; make dst_bytes several times
 * the L2 size to measure drain into HBM.
 */
typedef struct {
  int K;                 /* producer CTAs, 1 .. 1024 */
  int rounds;            /* rounds per producer, >= 1 */
  long long V_bytes;     /* aggregate burst volume per round; multiple of 4096*K */
  long long G_ns;        /* gap after each burst, ns, >= 0 */
  int store_kind;        /* 0: st.global.v4 by all producer threads, each producer's
                               share of the burst contiguous;
                            1: cp.async.bulk from shared memory, issued by one thread;
                            2: st.global.v4 of whole 256-byte rows, scattered, by
                               128 threads (one warpgroup) of each producer: the
                               burst is V/256 rows and producer p writes rows p,
                               p + K, p + 2K, ... (the pattern of the fused kernel's
                               whole-line row stores, store_kind 3 there, issued by
                               the tile owner's warpgroup) */
  int gap_kind;          /* 0: spin on %globaltimer for G_ns (the issuer stays idle);
                            1: dependent FMA chain on every producer thread sized by the
                               host to last about G_ns (the issuer computes);
                            2: tensor-core work: fma_iters tcgen05.mma of 128x128x16
                               (bf16, fp32 accumulate in TMEM) issued after the burst and
                               waited for, so each round's issue time is the MMA pipe's
                               stall (G_ns is ignored for kinds 1 and 2) */
  void* dst;             /* device scratch target, 16-byte aligned */
  long long dst_bytes;   /* >= V_bytes, multiple of 4096*K */
  long long* stamps;     /* device int64 [K][rounds][3] */
  long long fma_iters;   /* gap_kind 1: dependent FMAs per thread per gap; gap_kind 2: MMA
                            instructions per gap (both host-calibrated, <= 1e8) */
} xstage_probe_cfg;

int xstage_probe_run(const xstage_probe_cfg* cfg, void* stream);

/*
 * xstage_probe_run_noalloc - the same probe for callers that cannot allocate
 * device memory. (The pages have no counterpart: this is a deployment
 * convenience.) Some callers may not call cudaMalloc at the point where they
 * want to measure: a process whose device memory is owned entirely by another
 * allocator (a framework's caching pool, a fixed arena reserved at start-up),
 * or a runtime whose rules forbid allocation after initialisation. They still
 * own the small stamps buffer, but not a burst target.
 *
 * Instead of cfg->dst, this entry point stores into a fixed device array that
 * lives inside the library: XSTAGE_PROBE_NOALLOC_MAX_BYTES bytes (16 MiB),
 * reserved on every GPU that loads the library until the process exits.
 * cfg->dst and cfg->dst_bytes are ignored; every other field means what it
 * means for xstage_probe_run. V_bytes above XSTAGE_PROBE_NOALLOC_MAX_BYTES
 * returns ATTN_A2A_ETOOLARGE without launching. Because the target (16 MiB)
 * is smaller than L2, this variant measures stores absorbed by L2, not the
 * drain into HBM that a large caller-owned target measures.
 *
 * Argument checks are those of xstage_probe_run (same status for the same
 * fields, including the fma_iters bound and gap_kind 2), apart from dst.
 *
 * Set-up: the first call on each device looks up the device address of the
 * array (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Only a successful lookup is kept: if it fails,
 * the call returns ATTN_A2A_ECUDA and the next call on that device tries
 * again. The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine); like xstage_probe_run it raises the kernel's dynamic
 * shared-memory limit with cudaFuncSetAttribute for store_kind 1 and
 * gap_kind 2, which allocates nothing either.
 *
 * Sharing: all calls on a device use the same array and it keeps the last
 * call's contents. The probe only writes it, so nothing has to start at zero.
 * Calls that overlap on the GPU (different streams, no ordering) race on the
 * array, which makes their timings interfere; order them on one stream.
 */
#define XSTAGE_PROBE_NOALLOC_MAX_BYTES (16ll * 1024 * 1024)

int xstage_probe_run_noalloc(const xstage_probe_cfg* cfg, void* stream);

/*
 * moe_gemm_scatter - synthetic MegaMoE-style workload for the pages'
 * "reshaping" result ("Key Contributions", MegaMoE: an interleaved scheduler
 * mixes Linear-1 (compute) and Linear-2 (communication) work across expert
 * waves so that store bursts get larger gaps). A persistent tcgen05 grouped
 * GEMM runs a caller-ordered task list; each task is one 128 x 256 output
 * tile (128 token rows, 256 output columns) of one expert:
 *   kind 0 ("Linear-1"): h_out[e, rows, cols] = x[e] w1[e]^T, stored locally;
 *   kind 1 ("Linear-2"): y = x[e] w2[e]^T, each output row r of expert e
 *                        scattered to dst[rank][slot, cols] with
 *                        row_map[e*T + r] = (rank << 24) | slot.
 * Tasks at neighbouring list positions run at the same time on
 * neighbouring SMs, so the list order (Expert-Wave: each wave's kind-0 tasks,
 * then its kind-1 tasks; interleaved: kind-0 tasks of the next wave alternate
 * with kind-1 tasks of the current one) shapes the store bursts.
 *   x  : device bf16 [E, T, K]; w1, w2 : device bf16 [E, N, K] (K contiguous).
 *   T % 128 == 0, K % 64 == 0, N % 256 == 0.
 *   tasks   : device int32 [n_tasks][4] = (kind, expert, row block, column block):
 *             rows [128 m, 128 m + 128), columns [256 n, 256 n + 256).
 *   h_out   : device bf16 [E, T, N].  row_map : device int32 [E * T].
 *   dst     : HOST array of P device pointers, dst[j] = bf16 [dst_rows[j], N];
 *             dst_rows is a HOST array. 1 <= P <= 64.
 *   grid    : persistent CTAs, 0 = one per SM.
 * Malformed tasks and out-of-range row_map entries are skipped on the device
 * and reported as ATTN_A2A_EINVAL through dev_status. Every task writes its
 * own output tile, so the result does not depend on the order.
 */
int moe_gemm_scatter(const void* x, const void* w1, const void* w2, int E, int T, int K, int N,
                     const int* tasks, int n_tasks, void* h_out, const int* row_map, int P,
                     void* const* dst, const int* dst_rows, int* dev_status, int grid, void* stream);

/* Static description of a status code. Never NULL. */
const char* attn_a2a_strerror(int status);

/* Number of SMs the library sizes its persistent grid to on the current device
 * (0 if no device). Host-only query, no launch. */
int attn_a2a_num_sms(void);

/* The store kind (attn_a2a_opts.store_kind) an attn_a2a_fwd(_ex) (layout 1)
 * or attn_a2a_fwd_contig(_ex) (layout 0) call would use for its output
 * tiles: 1 = bulk tensor stores from a staging tile, 2 = row stores from
 * registers, 3 = whole-line row stores. S = sequence length, P = partitions
 * (1 for the contiguous layout), layout = 0 contiguous ("attention alone"),
 * 1 all-to-all; store_kind = the requested kind, 0 for the automatic choice.
 * Writes the kind to *resolved (host int) and returns ATTN_A2A_OK;
 * ATTN_A2A_EUNSUPPORTED where the kind is not built (1 for all-to-all with
 * P > 8, 3 for the contiguous layout); ATTN_A2A_EINVAL for arguments out of
 * range. Host-only, no launch. */
int attn_a2a_store_kind(int S, int P, int layout, int store_kind, int* resolved);

/* The split schedule (attn_a2a_opts.split, with a large enough workspace) an
 * attn_a2a_fwd_ex or attn_a2a_fwd_contig_ex call of B x H heads of length S,
 * head dimension d, would use on `grid` persistent CTAs (0 = one per SM) of a
 * GPU with num_sms SMs and l2_bytes of L2 (0 = those of the current device):
 * writes *kind = ATTN_A2A_SPLIT_ALL (every work item's key blocks in equal
 * ranges, one per CTA), ATTN_A2A_SPLIT_TAIL (the partial last wave's, in a
 * second kernel) or 0 (nothing split), *first_item = the first split work item
 * and *range_blocks = the key blocks per CTA range (0 when nothing is split).
 * Work items are pairs of 128-row query tiles, B*H*ceil(ceil(S/128)/2) of
 * them. Not split either way: trace calls and tile_order = 1. Returns
 * ATTN_A2A_OK; ATTN_A2A_EINVAL for arguments out of range (d other than 64 or
 * 128); ATTN_A2A_ECUDA if 0 asks for a device value and there is no device.
 * Host-only, no launch. */
int attn_a2a_split_plan(int B, int H, int S, int d, int grid, int num_sms, long long l2_bytes, int split,
                        int* kind, int* first_item, int* range_blocks);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_A2A_H */

// C ABI of libattn_a2a.so: argument validation, the chunk rule of the
// sequence-sharded partitions, and dispatch to the kernels' launchers.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <climits>

#include "attn_a2a.h"
#include "internal.h"

namespace attn_a2a {

int num_sms_current_device() {
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

long long l2_bytes_current_device() {
  static long long cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi; }

// Bytes spanned by a strided [B, H, S, d] bf16 tensor.
Span tensor_span(const void* p, int B, int H, int S, int d, long long sb, long long sh, long long ss) {
  const long long last = (B - 1) * sb + (H - 1) * sh + (S - 1) * ss + d;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + static_cast<uintptr_t>(last) * 2u};
}

bool stride_ok(long long s, int extent) {
  if (extent <= 1) return true;  // never used to address memory
  return s > 0 && (s % 8) == 0 && s * 2 < (1ll << 40);
}

// Shape, scale and input pointers. Sets *empty when there is nothing to do.
int check_inputs(const void* q, const void* k, const void* v, const attn_a2a_shape* shp, float scale,
                 bool* empty) {
  if (shp == nullptr) return ATTN_A2A_EINVAL;
  if (shp->B < 0 || shp->H < 0 || shp->S < 0 || shp->d <= 0) return ATTN_A2A_EINVAL;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_A2A_EINVAL;
  if (shp->d != 64 && shp->d != 128) return ATTN_A2A_EUNSUPPORTED;
  *empty = (shp->B == 0 || shp->H == 0 || shp->S == 0);
  if (*empty) return ATTN_A2A_OK;
  if (static_cast<long long>(shp->B) * shp->H * ((shp->S + 255) / 256) > (1ll << 30))
    return ATTN_A2A_EUNSUPPORTED;  // work-item count must fit an int
  if (q == nullptr || k == nullptr || v == nullptr) return ATTN_A2A_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_A2A_EINVAL;
  const long long st[9] = {shp->q_sb, shp->q_sh, shp->q_ss, shp->k_sb, shp->k_sh,
                           shp->k_ss, shp->v_sb, shp->v_sh, shp->v_ss};
  const int ext[3] = {shp->B, shp->H, shp->S};
  for (int i = 0; i < 9; ++i)
    if (!stride_ok(st[i], ext[i % 3])) return ATTN_A2A_EINVAL;
  return ATTN_A2A_OK;
}

// Partition pointers and the chunk rule: chunk j has floor(S/P) rows plus one
// for j < S mod P (torch.tensor_split).
// part_heads = heads per partition row (0 = H): a launch over one head group
// writes heads [0, H) of rows that hold part_heads heads (the caller offsets
// each partition pointer to the group's first head); the head-sharding rule
// then applies to the full row.
int make_partitions(const attn_a2a_shape& shp, int P, void* const* parts, EpiParams* e, int part_heads = 0) {
  if (P < 1 || P > kMaxRanks) return ATTN_A2A_EINVAL;
  const int h_row = part_heads > 0 ? part_heads : shp.H;
  if (h_row < shp.H || h_row % P != 0) return ATTN_A2A_EINVAL;
  if (parts == nullptr) return ATTN_A2A_EINVAL;
  std::memset(e, 0, sizeof(*e));
  e->P = P;
  e->cbase = shp.S / P;
  e->crem = shp.S % P;
  for (int j = 0; j < P; ++j) {
    const int c = e->cbase + (j < e->crem ? 1 : 0);
    const bool has_bytes = c > 0 && shp.B > 0 && shp.H > 0;
    if (has_bytes && (parts[j] == nullptr || !aligned16(parts[j]))) return ATTN_A2A_EINVAL;
    e->part[j] = parts[j];
  }
  e->hstride = part_heads > 0 ? part_heads : 0;
  return ATTN_A2A_OK;
}

bool partitions_alias_inputs(const attn_a2a_shape& shp, const EpiParams& e, const Span* in, int nin) {
  for (int j = 0; j < e.P; ++j) {
    const int c = e.cbase + (j < e.crem ? 1 : 0);
    if (c == 0) continue;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(e.part[j]);
    // rows of h_row heads, of which this call writes the first H
    const long long h_row = e.hstride > 0 ? e.hstride : shp.H;
    const long long last = (static_cast<long long>(shp.B) * c - 1) * h_row + shp.H;
    const Span out{lo, lo + static_cast<uintptr_t>(last) * shp.d * 2u};
    for (int i = 0; i < nin; ++i)
      if (overlaps(out, in[i])) return true;
  }
  return false;
}

// Copy streams and events of the host-buffer entry point, created once per
// device on first use (host-side resources; no device memory).
constexpr int kMaxHostChunks = 8;

struct HostPipe {
  std::once_flag once;
  std::mutex mu;
  bool ok = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp2 = nullptr;
  cudaEvent_t ev_start = nullptr, ev_h2d = nullptr, ev_comp = nullptr, ev_end = nullptr;
};

// Head counts of the chunks of one batch entry of the host-buffer call. The
// first chunk is small, so that little copying is exposed before the first
// kernel; each next chunk grows by at most 2.5x, so that its copy (about a
// third of its kernel's time per head at ~200 GB/s) finishes while the kernel
// before it runs; the last chunk is small again, so that little copying back
// is exposed after the last kernel. Returns the number of chunks (<= kMaxHostChunks).
int plan_head_chunks(int H, int* chunk) {
  if (H <= 4) {
    for (int i = 0; i < H; ++i) chunk[i] = 1;
    return H;
  }
  const int first = H / 32 > 1 ? H / 32 : 1;
  int n = 0, rem = H, prev = first;
  chunk[n++] = first;
  rem -= first;
  while (rem > first && n < kMaxHostChunks - 1) {
    int next = (5 * prev + 1) / 2;                  // at most 2.5x the previous chunk
    if (next > rem - first) next = rem - first;     // leave a small last chunk
    if (n == kMaxHostChunks - 2) next = rem - first;
    chunk[n++] = next;
    rem -= next;
    prev = next;
  }
  chunk[n++] = rem;
  return n;
}

HostPipe g_pipes[128];

HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  HostPipe* hp = &g_pipes[dev];
  std::call_once(hp->once, [hp] {
    const unsigned ef = cudaEventDisableTiming;
    hp->ok = cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&hp->comp2, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->ev_start, ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->ev_h2d, ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->ev_comp, ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->ev_end, ef) == cudaSuccess;
  });
  return hp->ok ? hp : nullptr;
}

attn_a2a_opts default_opts() {
  attn_a2a_opts o;
  std::memset(&o, 0, sizeof(o));
  return o;
}

int fwd_common(const void* q, const void* k, const void* v, const attn_a2a_shape* shp, int P,
               float scale, void* const* out_partitions, void* out_contig, bool a2a, int* dev_status,
               const attn_a2a_opts* opts, void* stream) {
  bool empty = false;
  int rc = check_inputs(q, k, v, shp, scale, &empty);
  if (rc != ATTN_A2A_OK) return rc;
  if (opts != nullptr && (opts->store_kind < 0 || opts->store_kind > 3 || opts->grid < 0 ||
                          opts->timeout_ns < 0 || opts->inject_stall < 0 || opts->inject_stall > 1 ||
                          opts->tile_order < 0 || opts->tile_order > 1 ||
                          (reinterpret_cast<uintptr_t>(opts->trace) & 7u) != 0 || opts->part_heads < 0 ||
                          (opts->part_heads > 0 && !a2a) || opts->split < ATTN_A2A_SPLIT_AUTO ||
                          opts->split > ATTN_A2A_SPLIT_NONE || opts->cta_pairs < 0 || opts->cta_pairs > 2))
    return ATTN_A2A_EINVAL;
  // the bulk-store epilogue exists for the contiguous layout and for the
  // all-to-all layout with up to 8 partitions
  if (opts != nullptr && opts->store_kind == 1 && a2a && P > 8) return ATTN_A2A_EUNSUPPORTED;
  EpiParams epi;
  std::memset(&epi, 0, sizeof(epi));
  if (a2a) {
    rc = make_partitions(*shp, P, out_partitions, &epi, opts != nullptr ? opts->part_heads : 0);
    if (rc != ATTN_A2A_OK) return rc;
  } else {
    epi.P = 1;
    epi.cbase = shp->S;
    epi.out = out_contig;
  }
  if (empty) return ATTN_A2A_OK;
  const Span in[3] = {
      tensor_span(q, shp->B, shp->H, shp->S, shp->d, shp->q_sb, shp->q_sh, shp->q_ss),
      tensor_span(k, shp->B, shp->H, shp->S, shp->d, shp->k_sb, shp->k_sh, shp->k_ss),
      tensor_span(v, shp->B, shp->H, shp->S, shp->d, shp->v_sb, shp->v_sh, shp->v_ss)};
  if (a2a) {
    if (partitions_alias_inputs(*shp, epi, in, 3)) return ATTN_A2A_EINVAL;
  } else {
    if (out_contig == nullptr || !aligned16(out_contig)) return ATTN_A2A_EINVAL;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(out_contig);
    const Span out{lo, lo + static_cast<uintptr_t>(shp->B) * shp->H * shp->S * shp->d * 2u};
    for (const Span& s : in)
      if (overlaps(out, s)) return ATTN_A2A_EINVAL;
  }
  if (opts != nullptr && opts->workspace != nullptr) {
    // split-tail scratch: aligned, and apart from every input and output
    const uintptr_t lo = reinterpret_cast<uintptr_t>(opts->workspace);
    if ((lo & 255u) != 0 || opts->workspace_bytes <= 0) return ATTN_A2A_EINVAL;
    const Span ws{lo, lo + static_cast<uintptr_t>(opts->workspace_bytes)};
    for (const Span& s : in)
      if (overlaps(ws, s)) return ATTN_A2A_EINVAL;
    if (a2a) {
      const long long h_row = epi.hstride > 0 ? epi.hstride : shp->H;
      for (int j = 0; j < epi.P; ++j) {
        const int c = epi.cbase + (j < epi.crem ? 1 : 0);
        if (c == 0) continue;
        const uintptr_t plo = reinterpret_cast<uintptr_t>(epi.part[j]);
        const long long last = (static_cast<long long>(shp->B) * c - 1) * h_row + shp->H;
        if (overlaps(ws, Span{plo, plo + static_cast<uintptr_t>(last) * shp->d * 2u})) return ATTN_A2A_EINVAL;
      }
    } else {
      const uintptr_t olo = reinterpret_cast<uintptr_t>(out_contig);
      if (overlaps(ws, Span{olo, olo + static_cast<uintptr_t>(shp->B) * shp->H * shp->S * shp->d * 2u}))
        return ATTN_A2A_EINVAL;
    }
  }
  const attn_a2a_opts o = opts ? *opts : default_opts();
  return launch_fa_tc(q, k, v, *shp, scale, a2a, epi, dev_status, o, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace attn_a2a

using namespace attn_a2a;

extern "C" {

const char* attn_a2a_strerror(int status) {
  switch (status) {
    case ATTN_A2A_OK: return "ok";
    case ATTN_A2A_EINVAL: return "invalid argument";
    case ATTN_A2A_EUNSUPPORTED: return "unsupported configuration";
    case ATTN_A2A_ECUDA: return "CUDA error";
    case ATTN_A2A_ETIMEOUT: return "bounded in-kernel wait expired";
    case ATTN_A2A_ETOOLARGE: return "request exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int attn_a2a_num_sms(void) { return num_sms_current_device(); }

int attn_a2a_split_plan(int B, int H, int S, int d, int grid, int num_sms, long long l2_bytes, int split,
                        int* kind, int* first_item, int* range_blocks) {
  if (kind == nullptr || first_item == nullptr || range_blocks == nullptr || B < 0 || H < 0 || S < 0 ||
      (d != 64 && d != 128) || grid < 0 || num_sms < 0 || l2_bytes < 0 || split < ATTN_A2A_SPLIT_AUTO ||
      split > ATTN_A2A_SPLIT_NONE)
    return ATTN_A2A_EINVAL;
  const int nblk = (S + 127) / 128;
  const long long total = static_cast<long long>(B) * H * ((nblk + 1) / 2);
  if (total > INT_MAX) return ATTN_A2A_EUNSUPPORTED;
  if (num_sms == 0) num_sms = num_sms_current_device();
  if (l2_bytes == 0) l2_bytes = l2_bytes_current_device();
  if (num_sms <= 0) return ATTN_A2A_ECUDA;
  int g = grid > 0 ? grid : num_sms;
  if (g > total) g = static_cast<int>(total);
  int first = 0, len = 0;
  *kind = split_decision(static_cast<int>(total), nblk, g, num_sms, 4LL * B * H * S * d, l2_bytes, split, first, len);
  *first_item = first;
  *range_blocks = len;
  return ATTN_A2A_OK;
}

int attn_a2a_store_kind(int S, int P, int layout, int store_kind, int* resolved) {
  if (resolved == nullptr || S < 0 || P < 1 || P > kMaxRanks || layout < 0 || layout > 1 || store_kind < 0 ||
      store_kind > 3)
    return ATTN_A2A_EINVAL;
  const int kind = resolve_store_kind(S, P, layout == 1, store_kind);
  if (kind == 0) return ATTN_A2A_EUNSUPPORTED;
  *resolved = kind;
  return ATTN_A2A_OK;
}

int attn_a2a_fwd_ex(const void* q, const void* k, const void* v, const attn_a2a_shape* shp, int P,
                    float scale, void* const* out_partitions, int* dev_status,
                    const attn_a2a_opts* opts, void* stream) {
  return fwd_common(q, k, v, shp, P, scale, out_partitions, nullptr, true, dev_status, opts, stream);
}

int attn_a2a_fwd(const void* q, const void* k, const void* v, const attn_a2a_shape* shp, int P,
                 float scale, void* const* out_partitions, int* dev_status, void* stream) {
  return fwd_common(q, k, v, shp, P, scale, out_partitions, nullptr, true, dev_status, nullptr, stream);
}

int attn_a2a_fwd_contig_ex(const void* q, const void* k, const void* v, const attn_a2a_shape* shp,
                           float scale, void* out, int* dev_status, const attn_a2a_opts* opts,
                           void* stream) {
  return fwd_common(q, k, v, shp, 1, scale, nullptr, out, false, dev_status, opts, stream);
}

int attn_a2a_fwd_contig(const void* q, const void* k, const void* v, const attn_a2a_shape* shp,
                        float scale, void* out, int* dev_status, void* stream) {
  return fwd_common(q, k, v, shp, 1, scale, nullptr, out, false, dev_status, nullptr, stream);
}

int attn_a2a_fwd_s2s(const void* const* q_parts, const void* const* k_parts,
                     const void* const* v_parts, const attn_a2a_shape* shp, int P, float scale,
                     void* const* out_partitions, int* dev_status, void* stream) {
  return attn_a2a_fwd_s2s_ex(q_parts, k_parts, v_parts, shp, P, scale, out_partitions, dev_status, nullptr, stream);
}

int attn_a2a_fwd_s2s_ex(const void* const* q_parts, const void* const* k_parts,
                        const void* const* v_parts, const attn_a2a_shape* shp, int P, float scale,
                        void* const* out_partitions, int* dev_status, const attn_a2a_opts* opts, void* stream) {
  if (shp == nullptr || q_parts == nullptr || k_parts == nullptr || v_parts == nullptr)
    return ATTN_A2A_EINVAL;
  if (opts != nullptr && (opts->store_kind < 0 || opts->store_kind > 3 || opts->grid < 0 || opts->timeout_ns < 0 ||
                          opts->inject_stall < 0 || opts->inject_stall > 1 || opts->tile_order < 0 ||
                          opts->tile_order > 1 || (reinterpret_cast<uintptr_t>(opts->trace) & 7u) != 0 ||
                          opts->part_heads < 0 || opts->split < ATTN_A2A_SPLIT_AUTO ||
                          opts->split > ATTN_A2A_SPLIT_NONE || opts->cta_pairs < 0 || opts->cta_pairs > 2))
    return ATTN_A2A_EINVAL;
  // what the whole-layer kernels do not have: whole-line row stores, the
  // chunk-interleaved order, a trace, head-group partitions, CTA pairs
  if (opts != nullptr && (opts->store_kind == 3 || opts->tile_order != 0 || opts->trace != nullptr ||
                          opts->part_heads != 0 || opts->cta_pairs == 1))
    return ATTN_A2A_EUNSUPPORTED;
  if (shp->B < 0 || shp->H < 0 || shp->S < 0 || shp->d <= 0) return ATTN_A2A_EINVAL;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_A2A_EINVAL;
  if (shp->d != 64 && shp->d != 128) return ATTN_A2A_EUNSUPPORTED;
  EpiParams epi;
  int rc = make_partitions(*shp, P, out_partitions, &epi);
  if (rc != ATTN_A2A_OK) return rc;
  if (P > 8) return ATTN_A2A_EUNSUPPORTED;
  if (static_cast<long long>(shp->B) * shp->H * shp->S == 0) return ATTN_A2A_OK;
  if (static_cast<long long>(shp->B) * shp->H * ((shp->S + 255) / 256 + P) > (1ll << 30))
    return ATTN_A2A_EUNSUPPORTED;
  Span in[3 * 8];
  int nin = 0;
  for (int j = 0; j < P; ++j) {
    const int c = epi.cbase + (j < epi.crem ? 1 : 0);
    if (c == 0) continue;
    const void* ptrs[3] = {q_parts[j], k_parts[j], v_parts[j]};
    for (const void* ptr : ptrs) {
      if (ptr == nullptr || !aligned16(ptr)) return ATTN_A2A_EINVAL;
      const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
      in[nin++] = Span{lo, lo + static_cast<uintptr_t>(shp->B) * c * shp->H * shp->d * 2u};
    }
  }
  if (partitions_alias_inputs(*shp, epi, in, nin)) return ATTN_A2A_EINVAL;
  if (opts != nullptr && opts->workspace != nullptr) {
    // split scratch: aligned, and apart from every input and output partition
    const uintptr_t lo = reinterpret_cast<uintptr_t>(opts->workspace);
    if ((lo & 255u) != 0 || opts->workspace_bytes <= 0) return ATTN_A2A_EINVAL;
    const Span ws{lo, lo + static_cast<uintptr_t>(opts->workspace_bytes)};
    for (int i = 0; i < nin; ++i)
      if (overlaps(ws, in[i])) return ATTN_A2A_EINVAL;
    for (int j = 0; j < epi.P; ++j) {
      const int c = epi.cbase + (j < epi.crem ? 1 : 0);
      if (c == 0) continue;
      const uintptr_t plo = reinterpret_cast<uintptr_t>(epi.part[j]);
      if (overlaps(ws, Span{plo, plo + static_cast<uintptr_t>(shp->B) * c * shp->H * shp->d * 2u}))
        return ATTN_A2A_EINVAL;
    }
  }
  const attn_a2a_opts o = opts ? *opts : default_opts();
  return launch_fa_tc_s2s(q_parts, k_parts, v_parts, *shp, scale, epi, dev_status, o,
                          static_cast<cudaStream_t>(stream));
}

int attn_a2a_permute(const void* o, const attn_a2a_shape* shp, int P, void* const* out_partitions,
                     void* stream) {
  if (shp == nullptr || shp->B < 0 || shp->H < 0 || shp->S < 0) return ATTN_A2A_EINVAL;
  if (shp->d != 64 && shp->d != 128) return ATTN_A2A_EUNSUPPORTED;
  EpiParams epi;
  int rc = make_partitions(*shp, P, out_partitions, &epi);
  if (rc != ATTN_A2A_OK) return rc;
  if (static_cast<long long>(shp->B) * shp->H * shp->S == 0) return ATTN_A2A_OK;
  if (o == nullptr || !aligned16(o)) return ATTN_A2A_EINVAL;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(o);
  const Span in{lo, lo + static_cast<uintptr_t>(shp->B) * shp->H * shp->S * shp->d * 2u};
  if (partitions_alias_inputs(*shp, epi, &in, 1)) return ATTN_A2A_EINVAL;
  return launch_permute(o, *shp, epi, static_cast<cudaStream_t>(stream));
}

int attn_a2a_fwd_simt(const void* q, const void* k, const void* v, const attn_a2a_shape* shp, int P,
                      float scale, void* const* out_partitions, void* stream) {
  bool empty = false;
  int rc = check_inputs(q, k, v, shp, scale, &empty);
  if (rc != ATTN_A2A_OK) return rc;
  EpiParams epi;
  rc = make_partitions(*shp, P, out_partitions, &epi);
  if (rc != ATTN_A2A_OK) return rc;
  if (empty) return ATTN_A2A_OK;
  if (shp->H > 65535 || shp->B > 65535) return ATTN_A2A_EUNSUPPORTED;
  return launch_fa_simt(q, k, v, *shp, scale, epi, static_cast<cudaStream_t>(stream));
}

int attn_a2a_fwd_host(const void* hq, const void* hk, const void* hv, const attn_a2a_shape* shp, int P,
                      float scale, void* dq, void* dk, void* dv, void* const* dparts,
                      void* const* hparts, int* dev_status, void* stream) {
  if (shp == nullptr) return ATTN_A2A_EINVAL;
  if (hq == nullptr || hk == nullptr || hv == nullptr || hparts == nullptr) return ATTN_A2A_EINVAL;
  // The device copies are contiguous [B, H, S, d].
  attn_a2a_shape s = *shp;
  s.q_ss = s.k_ss = s.v_ss = s.d;
  s.q_sh = s.k_sh = s.v_sh = static_cast<long long>(s.S) * s.d;
  s.q_sb = s.k_sb = s.v_sb = static_cast<long long>(s.H) * s.S * s.d;
  bool empty = false;
  int rc = check_inputs(dq, dk, dv, &s, scale, &empty);
  if (rc != ATTN_A2A_OK) return rc;
  EpiParams epi;
  rc = make_partitions(s, P, dparts, &epi);
  if (rc != ATTN_A2A_OK) return rc;
  if (empty) return ATTN_A2A_OK;
  for (int j = 0; j < P; ++j)
    if (epi.cbase + (j < epi.crem ? 1 : 0) > 0 && hparts[j] == nullptr) return ATTN_A2A_EINVAL;
  {
    const Span in[3] = {tensor_span(dq, s.B, s.H, s.S, s.d, s.q_sb, s.q_sh, s.q_ss),
                        tensor_span(dk, s.B, s.H, s.S, s.d, s.k_sb, s.k_sh, s.k_ss),
                        tensor_span(dv, s.B, s.H, s.S, s.d, s.v_sb, s.v_sh, s.v_ss)};
    if (partitions_alias_inputs(s, epi, in, 3)) return ATTN_A2A_EINVAL;
  }
  // Host partitions that are pinned host memory (which the device can store
  // to) receive the rows straight from the kernels, as whole-line row stores
  // over the host link, and no copy back is needed; otherwise the kernels
  // store into dparts and each chunk is copied back.
  bool direct = true;
  for (int j = 0; j < P && direct; ++j) {
    if (epi.cbase + (j < epi.crem ? 1 : 0) == 0) continue;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, hparts[j]) != cudaSuccess) {
      cudaGetLastError();
      direct = false;
    } else {
      direct = attr.type == cudaMemoryTypeHost;
    }
  }
  HostPipe* hp = host_pipe();
  if (hp == nullptr) return ATTN_A2A_ECUDA;
  std::lock_guard<std::mutex> lock(hp->mu);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Heads are processed in chunks (plan_head_chunks): the host->device copy
  // of the next chunk and the device->host copy of the previous one overlap
  // the kernel of this one, and consecutive chunks' kernels alternate between
  // the caller's stream and a second one, so that the next kernel's CTAs take
  // the SMs the last wave of the previous one leaves idle.
  int chunk[kMaxHostChunks];
  const int nchunk = plan_head_chunks(s.H, chunk);
  const size_t head_elems = static_cast<size_t>(s.S) * s.d;
  // device buffers may still be in use by earlier work on the caller's stream
  if (cudaEventRecord(hp->ev_start, st) != cudaSuccess || cudaStreamWaitEvent(hp->h2d, hp->ev_start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->comp2, hp->ev_start, 0) != cudaSuccess)
    return ATTN_A2A_ECUDA;
  attn_a2a_opts o = default_opts();
  if (direct) o.store_kind = 3;
  void* const* outs = direct ? hparts : dparts;
  int launch = 0;
  for (int b = 0; b < s.B; ++b) {
    for (int ci = 0, h0 = 0; ci < nchunk; h0 += chunk[ci], ++ci, ++launch) {
      const int h1 = h0 + chunk[ci];
      const cudaStream_t cs_stream = launch % 2 == 0 ? st : hp->comp2;
      const size_t off = (static_cast<size_t>(b) * s.H + h0) * head_elems;  // elements
      const size_t bytes = static_cast<size_t>(h1 - h0) * head_elems * 2u;
      const void* hsrc[3] = {hq, hk, hv};
      void* ddst[3] = {dq, dk, dv};
      for (int i = 0; i < 3; ++i)
        if (cudaMemcpyAsync(static_cast<uint16_t*>(ddst[i]) + off, static_cast<const uint16_t*>(hsrc[i]) + off, bytes,
                            cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
          return ATTN_A2A_ECUDA;
      if (cudaEventRecord(hp->ev_h2d, hp->h2d) != cudaSuccess ||
          cudaStreamWaitEvent(cs_stream, hp->ev_h2d, 0) != cudaSuccess)
        return ATTN_A2A_ECUDA;
      attn_a2a_shape cs = s;  // one batch entry, heads [h0, h1)
      cs.B = 1;
      cs.H = h1 - h0;
      EpiParams ce = epi;
      ce.hstride = s.H;
      for (int j = 0; j < P; ++j) {
        const int c = epi.cbase + (j < epi.crem ? 1 : 0);
        ce.part[j] = c > 0 ? static_cast<void*>(static_cast<uint16_t*>(outs[j]) +
                                                 (static_cast<size_t>(b) * c * s.H + h0) * s.d)
                           : nullptr;
      }
      rc = launch_fa_tc(static_cast<uint16_t*>(dq) + off, static_cast<uint16_t*>(dk) + off,
                        static_cast<uint16_t*>(dv) + off, cs, scale, true, ce, dev_status, o, cs_stream);
      if (rc != ATTN_A2A_OK) return rc;
      if (cudaEventRecord(hp->ev_comp, cs_stream) != cudaSuccess ||
          cudaStreamWaitEvent(hp->d2h, hp->ev_comp, 0) != cudaSuccess)
        return ATTN_A2A_ECUDA;
      for (int j = 0; j < P && !direct; ++j) {
        const int c = epi.cbase + (j < epi.crem ? 1 : 0);
        if (c == 0) continue;
        const size_t eoff = (static_cast<size_t>(b) * c * s.H + h0) * s.d;
        const size_t pitch = static_cast<size_t>(s.H) * s.d * 2u;
        if (cudaMemcpy2DAsync(static_cast<uint16_t*>(hparts[j]) + eoff, pitch,
                              static_cast<const uint16_t*>(dparts[j]) + eoff, pitch,
                              static_cast<size_t>(h1 - h0) * s.d * 2u, c, cudaMemcpyDeviceToHost,
                              hp->d2h) != cudaSuccess)
          return ATTN_A2A_ECUDA;
      }
    }
  }
  // the caller's stream completes only when the last copy back has (which
  // follows every chunk's kernel, on either stream; with direct stores the
  // copy stream only waits for the kernels)
  if (cudaEventRecord(hp->ev_end, hp->d2h) != cudaSuccess || cudaStreamWaitEvent(st, hp->ev_end, 0) != cudaSuccess)
    return ATTN_A2A_ECUDA;
  return ATTN_A2A_OK;
}

int moe_gemm_scatter(const void* x, const void* w1, const void* w2, int E, int T, int K, int N,
                     const int* tasks, int n_tasks, void* h_out, const int* row_map, int P,
                     void* const* dst, const int* dst_rows, int* dev_status, int grid, void* stream) {
  if (E < 1 || T < 128 || T % 128 != 0 || K < 64 || K % 64 != 0 || N < 256 || N % 256 != 0)
    return ATTN_A2A_EINVAL;
  if (static_cast<long long>(E) * T >= (1ll << 31) || static_cast<long long>(E) * T * N >= (1ll << 40))
    return ATTN_A2A_EUNSUPPORTED;
  if (n_tasks < 0 || grid < 0 || P < 1 || P > 64 || dst == nullptr || dst_rows == nullptr) return ATTN_A2A_EINVAL;
  if (n_tasks == 0) return ATTN_A2A_OK;
  if (x == nullptr || w1 == nullptr || w2 == nullptr || h_out == nullptr || tasks == nullptr || row_map == nullptr)
    return ATTN_A2A_EINVAL;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(h_out) || !aligned16(tasks) ||
      (reinterpret_cast<uintptr_t>(row_map) & 3u) != 0)
    return ATTN_A2A_EINVAL;
  for (int j = 0; j < P; ++j) {
    if (dst_rows[j] < 0 || dst_rows[j] >= (1 << 24)) return ATTN_A2A_EINVAL;
    if (dst_rows[j] > 0 && (dst[j] == nullptr || !aligned16(dst[j]))) return ATTN_A2A_EINVAL;
  }
  return launch_moe_gemm(x, w1, w2, E, T, K, N, tasks, n_tasks, h_out, row_map, P, dst, dst_rows, dev_status,
                         grid, static_cast<cudaStream_t>(stream));
}

int xstage_probe_run(const xstage_probe_cfg* cfg, void* stream) {
  if (cfg == nullptr) return ATTN_A2A_EINVAL;
  const xstage_probe_cfg& c = *cfg;
  const int bad = check_probe_cfg(c);
  if (bad != ATTN_A2A_OK) return bad;
  if (c.dst_bytes < c.V_bytes || c.dst == nullptr || !aligned16(c.dst)) return ATTN_A2A_EINVAL;
  return launch_probe(c, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

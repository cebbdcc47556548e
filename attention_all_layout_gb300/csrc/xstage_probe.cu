// Burst-Gap probe (X-Stage pages, Technical Summary, "Methodology": the
// Burst-Gap model T_iss(G; K, V) = max(T0_iss(K, V), V/R - G) and its measured
// quantities T0_iss, R and Q; "Key Contributions": characterisation through
// parameterised microbenchmarks).
//
// K producer CTAs repeat: issue a burst of V/K bytes of stores (the shape of
// the attention epilogue's output rows: 16-byte vector stores, or bulk
// asynchronous copies from shared memory), then spend a gap G not storing.
// Thread 0 of each producer stamps %globaltimer at burst start, after the
// last store of the burst has been issued by every thread of the CTA, and at
// gap end. Stores are never waited for inside a round: the issuer only sees
// the time it took to get them accepted, which is what the model predicts.
// The gap is either idle time, a dependent FMA chain, or tensor-core work
// (tcgen05.mma into TMEM, issued once the burst is out): with the latter the
// issue time of each round is exactly how long the MMA pipe stalls.
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

// Burst target of xstage_probe_run_noalloc: fixed device memory inside the
// library for callers that cannot allocate (include/attn_a2a.h explains who
// and why). Every GPU that loads the library holds these 16 MiB until exit.
static __device__ __align__(256) uint8_t g_noalloc_target[XSTAGE_PROBE_NOALLOC_MAX_BYTES];

namespace attn_a2a {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kRowThreads = 128;  // store_kind 2: the threads that store (one warpgroup)
constexpr int kBulkChunk = 32768;  // bytes of the shared-memory source of each bulk copy
// gap_kind 2: operands (two 128 x 64 bf16 swizzle atoms) at a 1024-byte aligned
// offset after the bulk source, then an mbarrier and the TMEM address slot.
constexpr int kMmaOperandBytes = 2 * 16384;
constexpr int kMmaSmem = kBulkChunk + 1024 + kMmaOperandBytes + 64;
constexpr uint32_t kMmaTmemCols = 128;

__global__ void __launch_bounds__(kProbeThreads)
    xstage_probe_kernel(uint8_t* __restrict__ dst, long long dst_bytes, long long V, int rounds,
                        long long G_ns, int store_kind, int gap_kind, long long fma_iters,
                        long long* __restrict__ stamps) {
  extern __shared__ __align__(128) uint8_t bulk_src[];
  const int K = gridDim.x, prod = blockIdx.x;
  const long long share = V / K;
  const long long nslots = dst_bytes / V;
  if (store_kind == 1) {
    for (int i = threadIdx.x; i < kBulkChunk / 4; i += blockDim.x)
      reinterpret_cast<uint32_t*>(bulk_src)[i] = 0x3c003c00u ^ static_cast<uint32_t>(i);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  float acc = 1.0f + 1e-3f * threadIdx.x;
  uint64_t t0 = 0, t1 = 0, t2 = 0;
  // gap_kind 2 set-up: zeroed operands, one mbarrier, 128 TMEM columns
  uint32_t ops = 0, mbar = 0, tmem = 0;
  uint32_t* tslot = nullptr;
  if (gap_kind == 2) {
    const uint32_t raw = smem_u32(bulk_src) + kBulkChunk;
    ops = (raw + 1023u) & ~1023u;
    uint8_t* gops = bulk_src + (ops - smem_u32(bulk_src));
    for (int i = threadIdx.x; i < kMmaOperandBytes / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(gops)[i] = 0u;
    mbar = ops + kMmaOperandBytes;
    tslot = reinterpret_cast<uint32_t*>(gops + kMmaOperandBytes + 8);
    if (threadIdx.x == 0) {
      mbar_init(mbar, 1);
      fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x < 32) {
      tmem_alloc(smem_u32(tslot), kMmaTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = *tslot;
  }
  uint32_t mma_phase = 0;
  for (int r = 0; r < rounds; ++r) {
    __syncthreads();
    if (threadIdx.x == 0) t0 = globaltimer_ns();
    uint8_t* base = dst + (r % nslots) * V + prod * share;
    if (store_kind == 0) {
      const uint4 val = make_uint4(static_cast<uint32_t>(r), static_cast<uint32_t>(prod), threadIdx.x, 0u);
      uint4* b4 = reinterpret_cast<uint4*>(base);
      const long long n = share / 16;
      for (long long i = threadIdx.x; i < n; i += blockDim.x) b4[i] = val;
    } else if (store_kind == 2) {
      // whole 256-byte rows, scattered, from one warpgroup: the round's V bytes
      // are V/256 rows and producer p writes rows p, p + K, p + 2K, ... with
      // its first 128 threads (16 per row, so a warp's store covers two rows
      // K * 256 bytes apart), as the fused kernel's tile owner - one
      // warpgroup - writes its rows with whole-line row stores
      if (threadIdx.x < kRowThreads) {
        const uint4 val = make_uint4(static_cast<uint32_t>(r), static_cast<uint32_t>(prod), threadIdx.x, 2u);
        uint8_t* slot = dst + (r % nslots) * V;
        const long long nrow = share / 256;
        for (long long i = threadIdx.x / 16; i < nrow; i += kRowThreads / 16)
          reinterpret_cast<uint4*>(slot + (i * K + prod) * 256)[threadIdx.x % 16] = val;
      }
    } else if (threadIdx.x == 0) {
      const uint32_t src = smem_u32(bulk_src);
      for (long long off = 0; off < share; off += kBulkChunk) {
        const long long left = share - off;
        const uint32_t size = static_cast<uint32_t>(left < kBulkChunk ? left : kBulkChunk);
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(base + off),
                     "r"(src), "r"(size)
                     : "memory");
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) t1 = globaltimer_ns();
    if (gap_kind == 0) {
      if (threadIdx.x == 0)
        while (globaltimer_ns() - t1 < static_cast<uint64_t>(G_ns)) {
        }
    } else if (gap_kind == 1) {
      for (long long i = 0; i < fma_iters; ++i) acc = fmaf(acc, 0.99999988f, 1.1920929e-7f);
    } else if (threadIdx.x == 0) {
      // fma_iters tcgen05.mma of 128 x 128 x 16 (bf16 in, fp32 in TMEM), then
      // wait (bounded, 1 s) for them to finish
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      tc_fence_after();
      for (long long i = 0; i < fma_iters; ++i) {
        const uint32_t off = static_cast<uint32_t>(i & 3) * 32;
        umma_ss(tmem, sdesc_sw128(ops + off, 16, 1024), sdesc_sw128(ops + 16384 + off, 16, 1024), idesc,
                i > 0 ? 1u : 0u);
      }
      umma_commit(mbar);
      mbar_wait_drain(mbar, mma_phase, 1000000000ull);
      mma_phase ^= 1u;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      t2 = globaltimer_ns();
      long long* st = stamps + (static_cast<long long>(prod) * rounds + r) * 3;
      st[0] = static_cast<long long>(t0);
      st[1] = static_cast<long long>(t1);
      st[2] = static_cast<long long>(t2);
    }
  }
  if (store_kind == 1 && threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if (acc == 1234.5f) dst[0] = 1;  // keeps the gap's FMA chain from being removed
  if (gap_kind == 2) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
      tc_fence_after();
      tmem_dealloc(tmem, kMmaTmemCols);
    }
  }
}

}  // namespace

int launch_probe(const xstage_probe_cfg& c, cudaStream_t stream) {
  const int smem = c.gap_kind == 2 ? kMmaSmem : (c.store_kind == 1 ? kBulkChunk : 0);
  if (smem > 0 &&
      cudaFuncSetAttribute(xstage_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
    return ATTN_A2A_ECUDA;
  xstage_probe_kernel<<<c.K, kProbeThreads, smem, stream>>>(
      static_cast<uint8_t*>(c.dst), c.dst_bytes, c.V_bytes, c.rounds, c.G_ns, c.store_kind,
      c.gap_kind, c.fma_iters, c.stamps);
  return cudaGetLastError() == cudaSuccess ? ATTN_A2A_OK : ATTN_A2A_ECUDA;
}

// Field checks shared by both probe entry points (everything except the
// caller's burst target, which only xstage_probe_run takes).
int check_probe_cfg(const xstage_probe_cfg& c) {
  if (c.K < 1 || c.K > 1024 || c.rounds < 1) return ATTN_A2A_EINVAL;
  if (c.V_bytes <= 0 || c.V_bytes % (4096ll * c.K) != 0) return ATTN_A2A_EINVAL;
  if (c.G_ns < 0 || c.store_kind < 0 || c.store_kind > 2 || c.gap_kind < 0 || c.gap_kind > 2)
    return ATTN_A2A_EINVAL;
  if (c.gap_kind >= 1 && (c.fma_iters < 0 || c.fma_iters > kProbeMaxGapIters)) return ATTN_A2A_EINVAL;
  if (c.stamps == nullptr || (reinterpret_cast<uintptr_t>(c.stamps) & 7u) != 0) return ATTN_A2A_EINVAL;
  return ATTN_A2A_OK;
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];

// Device address of g_noalloc_target on the current device. In host code the
// array's name is only a host-side stand-in, not an address a kernel may use;
// the usable address comes from cudaGetSymbolAddress, looked up with that
// device current by the first call on each device. Only a successful lookup
// is kept: after a failure the call returns ATTN_A2A_ECUDA and the next call
// tries again.
int noalloc_target(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();  // leave no stale error for the next launch check
    return ATTN_A2A_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_target) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ATTN_A2A_ECUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_A2A_OK;
}

}  // namespace
}  // namespace attn_a2a

// The probe without any device allocation: the same checks and the same
// launch as xstage_probe_run, with the burst target in the library's fixed
// array instead of a caller buffer. No cudaMalloc, cudaFree or allocating
// library call is made here (cudaFuncSetAttribute, which gap_kind 2 and the
// bulk-copy source need for their shared memory, allocates nothing).
extern "C" int xstage_probe_run_noalloc(const xstage_probe_cfg* cfg, void* stream) {
  using namespace attn_a2a;
  if (cfg == nullptr) return ATTN_A2A_EINVAL;
  const int bad = check_probe_cfg(*cfg);
  if (bad != ATTN_A2A_OK) return bad;
  if (cfg->V_bytes > XSTAGE_PROBE_NOALLOC_MAX_BYTES) return ATTN_A2A_ETOOLARGE;
  void* target = nullptr;
  const int rc = noalloc_target(&target);
  if (rc != ATTN_A2A_OK) return rc;
  xstage_probe_cfg c = *cfg;
  c.dst = target;
  c.dst_bytes = XSTAGE_PROBE_NOALLOC_MAX_BYTES;
  return launch_probe(c, static_cast<cudaStream_t>(stream));
}

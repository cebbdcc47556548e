// Synthetic MegaMoE-style workload for the Burst-Gap "reshaping" result
// (X-Stage pages, "Key Contributions", MegaMoE: an interleaved scheduler mixes
// Linear-1 (compute) and Linear-2 (communication) work across expert waves so
// that the bursts of remote stores get larger gaps; "Results", MegaMoE
// optimisation: 1.18x geomean over Expert-Wave). Not the DeepGEMM kernel:
// a grouped GEMM of our own whose tasks are
//   kind 0 ("Linear-1"):  H[e, rows, cols] = X_e W1_e^T, stored locally;
//   kind 1 ("Linear-2"):  Y_e = X_e W2_e^T, each output row scattered to its
//                         destination partition (rank, slot) - the store
//                         traffic that the pages' remote stores stand for.
// The task list fixes the order (Expert-Wave or interleaved); a persistent
// grid walks it with a static stride, so tasks at neighbouring positions run
// at the same time on neighbouring SMs.
//
// CTA: 256 threads. Warp 0 TMA producer, warp 1 MMA issuer (one thread) and
// TMEM owner, warps 4-7 epilogue (thread = output row). Tile 128 x 256 (one
// M=128 N=256 MMA per 16-wide K slice: at N=128 the shared-memory operand
// reads of a 128x128 MMA alone keep the tensor core from its peak), K in
// 64-element steps through a 4-stage shared-memory ring, two TMEM
// accumulators (512 columns) so the epilogue of one task overlaps the MMAs
// of the next; the epilogue drains each accumulator in two 128-column halves.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace attn_a2a {
namespace moe {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kHalf = 128;  // accumulator columns the epilogue holds in registers at a time
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileBytes = 128 * kBK * 2;       // one 128 x 64 bf16 operand tile (one swizzle atom wide)
constexpr int kStageBytes = 3 * kTileBytes;     // A and the two 128-row halves of B
constexpr int kBarOff = kStages * kStageBytes;  // 192 KB
// barrier slots: FULL[kStages], EMPTY[kStages], AFULL[2], AEMPTY[2], DONE
constexpr int FULL = 0, EMPTY = kStages, AFULL = 2 * kStages, AEMPTY = 2 * kStages + 2, DONE = 2 * kStages + 4;
constexpr int kNumBars = DONE + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmem = kMiscOff + 16 + 1024;
constexpr int kMaxParts = 64;

struct Maps {
  CUtensorMap x, w1, w2;
};

struct Params {
  const int4* tasks;  // (kind, expert, m_blk, n_blk)
  int n_tasks;
  int E, T, K, N;
  uint16_t* h_out;     // kind 0 output [E, T, N]
  const int* row_map;  // kind 1: (rank << 24) | slot for row e*T + t
  void* dst[kMaxParts];
  int dst_rows[kMaxParts];
  int P;
  int* dev_status;
  unsigned long long timeout_ns;
};

constexpr int kStatusInval = 1;  // ATTN_A2A_EINVAL

__device__ __forceinline__ bool task_ok(const Params& p, const int4& t) {
  return (t.x == 0 || t.x == 1) && t.y >= 0 && t.y < p.E && t.z >= 0 && t.z < p.T / kBM && t.w >= 0 &&
         t.w < p.N / kBN;
}

__device__ __forceinline__ void flag_bad_input(const Params& p) {
  if (p.dev_status != nullptr) atomicCAS(p.dev_status, 0, kStatusInval);
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + kBarOff;
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + kMiscOff + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nk = p.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(FULL + s), 1);
      mbar_init(BAR(EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(AFULL + b), 1);
      mbar_init(BAR(AEMPTY + b), kBM);
    }
    mbar_init(BAR(DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.w1);
    tma_prefetch_desc(&maps.w2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.dev_status, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- producer
      const uint64_t pol = l2_policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int ti = blockIdx.x; ok && ti < p.n_tasks; ti += gridDim.x) {
        const int4 t = p.tasks[ti];
        if (!task_ok(p, t)) continue;
        const CUtensorMap* wm = t.x == 0 ? &maps.w1 : &maps.w2;
        for (int kc = 0; ok && kc < nk; ++kc, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1;
          if (!mbar_wait(BAR(EMPTY + s), ph ^ 1, w)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR(FULL + s), kStageBytes);
          const uint32_t st = sbase + s * kStageBytes;
          tma_load_4d(st, &maps.x, BAR(FULL + s), kc * kBK, t.z * kBM, t.y, 0, pol);
          tma_load_4d(st + kTileBytes, wm, BAR(FULL + s), kc * kBK, t.w * kBN, t.y, 0, pol);
          tma_load_4d(st + 2 * kTileBytes, wm, BAR(FULL + s), kc * kBK, t.w * kBN + 128, t.y, 0, pol);  // B rows 128..255
        }
      }
      if (!ok) {  // wait (bounded) for the copies already started
        const uint32_t n = it < static_cast<uint32_t>(kStages) ? it : kStages;
        for (uint32_t i = 0; i < n; ++i) {
          const uint32_t idx = it - 1 - i;
          mbar_wait_drain(BAR(FULL + idx % kStages), (idx / kStages) & 1, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int ti = blockIdx.x; ok && ti < p.n_tasks; ti += gridDim.x) {
        const int4 t = p.tasks[ti];
        if (!task_ok(p, t)) continue;
        const uint32_t ab = tl & 1;
        if (!mbar_wait(BAR(AEMPTY + ab), ((tl >> 1) & 1) ^ 1, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1;
          if (!mbar_wait(BAR(FULL + s), ph, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = sbase + s * kStageBytes, b = a + kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_ss(tmem + ab * kBN, sdesc_sw128(a + kk * 32, 16, 1024), sdesc_sw128(b + kk * 32, 16, 1024), idesc,
                    (kc > 0 || kk > 0) ? 1u : 0u);
          umma_commit(BAR(EMPTY + s));
        }
        if (!ok) break;
        umma_commit(BAR(AFULL + ab));
        ++tl;
      }
      if (!ok) {
        umma_commit(BAR(DONE));
        mbar_wait_drain(BAR(DONE), 0, 100000000ull);
      }
    }
  } else if (warp >= 4) {  // ------------------------------------------ epilogue
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t tl = 0;
    for (int ti = blockIdx.x; ti < p.n_tasks; ti += gridDim.x) {
      const int4 t = p.tasks[ti];
      if (!task_ok(p, t)) {
        if (threadIdx.x == 128) flag_bad_input(p);
        continue;
      }
      const uint32_t ab = tl & 1;
      const bool got = __all_sync(0xffffffffu, mbar_wait(BAR(AFULL + ab), (tl >> 1) & 1, w));
      if (!got) break;
      tc_fence_after();
      const int row = t.z * kBM + r;  // row of expert t.y
      uint16_t* dst = nullptr;
      if (t.x == 0) {
        dst = p.h_out + ((static_cast<int64_t>(t.y) * p.T + row) * p.N + t.w * kBN);
      } else {
        const int rm = p.row_map[static_cast<int64_t>(t.y) * p.T + row];
        const int rank = rm >> 24, slot = rm & 0xFFFFFF;
        if (rm >= 0 && rank < p.P && slot < p.dst_rows[rank])
          dst = static_cast<uint16_t*>(p.dst[rank]) + (static_cast<int64_t>(slot) * p.N + t.w * kBN);
        else
          flag_bad_input(p);
      }
      for (int half = 0; half < kBN / kHalf; ++half) {
        uint32_t acc[kHalf];
        tmem_ld_x128(tmem + lane_off + ab * kBN + half * kHalf, acc);
        if (half == kBN / kHalf - 1) {  // the whole accumulator is in registers
          tc_fence_before();
          mbar_arrive(BAR(AEMPTY + ab));
        }
        if (dst == nullptr) continue;
        uint4* d4 = reinterpret_cast<uint4*>(dst + half * kHalf);
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c) {
          uint4 v;
          __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(acc[8 * c + 0]), __uint_as_float(acc[8 * c + 1]));
          __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(acc[8 * c + 2]), __uint_as_float(acc[8 * c + 3]));
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(acc[8 * c + 4]), __uint_as_float(acc[8 * c + 5]));
          __nv_bfloat162 h3 = __floats2bfloat162_rn(__uint_as_float(acc[8 * c + 6]), __uint_as_float(acc[8 * c + 7]));
          v.x = *reinterpret_cast<uint32_t*>(&h0);
          v.y = *reinterpret_cast<uint32_t*>(&h1);
          v.z = *reinterpret_cast<uint32_t*>(&h2);
          v.w = *reinterpret_cast<uint32_t*>(&h3);
          d4[c] = v;
        }
      }
      ++tl;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [E, rows, K] bf16 contiguous, box 64 x 128 rows, 128-byte swizzle.
bool map3(CUtensorMap* m, const void* base, int E, int rows, int K) {
  auto fn = encode();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(E), 1};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(rows) * K * 2,
                           static_cast<cuuint64_t>(E) * rows * K * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

int launch_moe_gemm(const void* x, const void* w1, const void* w2, int E, int T, int K, int N,
                    const int* tasks, int n_tasks, void* h_out, const int* row_map, int P,
                    void* const* dst, const int* dst_rows, int* dev_status, int grid, cudaStream_t stream) {
  moe::Maps maps;
  if (!moe::map3(&maps.x, x, E, T, K) || !moe::map3(&maps.w1, w1, E, N, K) || !moe::map3(&maps.w2, w2, E, N, K))
    return ATTN_A2A_ECUDA;
  moe::Params p;
  std::memset(&p, 0, sizeof(p));
  p.tasks = reinterpret_cast<const int4*>(tasks);
  p.n_tasks = n_tasks;
  p.E = E;
  p.T = T;
  p.K = K;
  p.N = N;
  p.h_out = static_cast<uint16_t*>(h_out);
  p.row_map = row_map;
  p.P = P;
  for (int j = 0; j < P; ++j) {
    p.dst[j] = dst[j];
    p.dst_rows[j] = dst_rows[j];
  }
  p.dev_status = dev_status;
  p.timeout_ns = 2000000000ull;
  int g = grid > 0 ? grid : num_sms_current_device();
  if (g <= 0) return ATTN_A2A_ECUDA;
  if (g > n_tasks) g = n_tasks;
  if (cudaFuncSetAttribute(moe::moe_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, moe::kSmem) !=
      cudaSuccess)
    return ATTN_A2A_ECUDA;
  moe::moe_gemm_kernel<<<g, moe::kThreads, moe::kSmem, stream>>>(maps, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_A2A_OK : ATTN_A2A_ECUDA;
}

}  // namespace attn_a2a

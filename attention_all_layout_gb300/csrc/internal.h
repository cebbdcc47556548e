// Host-side glue shared by the translation units of libattn_a2a.so.
#pragma once

#include <cuda_runtime.h>

#include "attn_a2a.h"
#include "epilogue.cuh"

namespace attn_a2a {

// Validated problem description handed to the launchers.
struct Problem {
  int B, H, S, d;
  float scale;
};

int num_sms_current_device();
// L2 cache bytes of the current device (0 if unknown).
long long l2_bytes_current_device();

// The epilogue's store kind for a request: 1 = bulk tensor stores, 2 = row
// stores, or 0 when store_kind 1 asks for bulk stores where they are not
// built (the all-to-all layout with P > 8). store_kind 0 picks what measured
// faster; it must be 0, 1 or 2.
int resolve_store_kind(int S, int P, bool a2a, int store_kind);
// The split schedule's decision (see fa_tc.cu): ATTN_A2A_SPLIT_ALL,
// ATTN_A2A_SPLIT_TAIL or 0, with the first split item and blocks per range.
int split_decision(int total, int nblk, int grid, int num_sms, long long kv_bytes, long long l2_bytes, int split,
                   int& tail_first, int& tail_len);

int launch_fa_tc(const void* q, const void* k, const void* v, const attn_a2a_shape& shp,
                 float scale, bool a2a, const EpiParams& epi, int* dev_status,
                 const attn_a2a_opts& opts, cudaStream_t stream);

// Sequence-sharded inputs (P partitions [B, c_j, H, d] each for q, k, v) and
// sequence-sharded output partitions in epi; P <= 8.
int launch_fa_tc_s2s(const void* const* q_parts, const void* const* k_parts,
                     const void* const* v_parts, const attn_a2a_shape& shp, float scale,
                     const EpiParams& epi, int* dev_status, const attn_a2a_opts& opts,
                     cudaStream_t stream);

int launch_fa_simt(const void* q, const void* k, const void* v, const attn_a2a_shape& shp,
                   float scale, const EpiParams& epi, cudaStream_t stream);

int launch_permute(const void* o, const attn_a2a_shape& shp, const EpiParams& epi,
                   cudaStream_t stream);

// Upper bound of xstage_probe_cfg.fma_iters (gap_kind 1 and 2), so that no
// probe holds the GPU for long.
constexpr long long kProbeMaxGapIters = 100000000ll;

// Argument checks of the probe entry points, apart from the burst target:
// ATTN_A2A_OK or ATTN_A2A_EINVAL.
int check_probe_cfg(const xstage_probe_cfg& cfg);

int launch_probe(const xstage_probe_cfg& cfg, cudaStream_t stream);

int launch_moe_gemm(const void* x, const void* w1, const void* w2, int E, int T, int K, int N,
                    const int* tasks, int n_tasks, void* h_out, const int* row_map, int P,
                    void* const* dst, const int* dst_rows, int* dev_status, int grid, cudaStream_t stream);

}  // namespace attn_a2a

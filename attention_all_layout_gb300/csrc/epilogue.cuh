// Destination of one output row: either the contiguous [B, H, S, d] layout
// ("attention alone") or the post-attention Ulysses all-to-all layout, P
// sequence-sharded partitions [B, c_j, H, d] (X-Stage pages, "Key
// Contributions", FlashAttention-A2A piggybacking: the tile owner stores the
// tile into its destination layout itself).
#pragma once

#include <cstdint>

namespace attn_a2a {

constexpr int kMaxRanks = 64;

struct EpiParams {
  void* out;                  // contiguous [B, H, S, d] (contiguous epilogue)
  void* part[kMaxRanks];      // partition j: [B, c_j, H, d] (all-to-all epilogue)
  int P;                      // virtual ranks
  int cbase;                  // floor(S / P)
  int crem;                   // S mod P: chunks 0 .. crem-1 hold cbase + 1 rows
  int hstride;                // heads per partition row when it exceeds the launch's H
                              // (a launch over a slice of the heads); 0 = H
};

// Chunk j holding sequence row s, its local row l and its length c_j.
__device__ __forceinline__ void chunk_of_row(const EpiParams& e, int s, int& j, int& l, int& c) {
  const int big = e.cbase + 1;
  const int split = e.crem * big;  // rows living in the longer chunks
  if (s < split) {
    j = s / big;
    l = s - j * big;
    c = big;
  } else {
    const int t = s - split;
    const int k = t / e.cbase;  // cbase > 0 here: s < S and S - split = (P-crem)*cbase
    j = e.crem + k;
    l = t - k * e.cbase;
    c = e.cbase;
  }
}

// Element pointer of output row s of head h, batch b (bf16 elements).
template <int D, bool A2A>
__device__ __forceinline__ uint16_t* out_row_ptr(const EpiParams& e, int B_unused, int H, int S,
                                                 int b, int h, int s) {
  (void)B_unused;
  if constexpr (A2A) {
    int j, l, c;
    chunk_of_row(e, s, j, l, c);
    uint16_t* base = static_cast<uint16_t*>(e.part[j]);
    const int hs = e.hstride > 0 ? e.hstride : H;
    return base + ((static_cast<int64_t>(b) * c + l) * hs + h) * D;
  } else {
    uint16_t* base = static_cast<uint16_t*>(e.out);
    return base + ((static_cast<int64_t>(b) * H + h) * S + s) * D;
  }
}

}  // namespace attn_a2a

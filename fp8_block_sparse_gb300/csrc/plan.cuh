// plan.cuh -- query-tile planning shared by the prefill kernels: the query
// tokens of each sequence are cut into tiles of `toks` tokens that never cross
// a sequence, so every tile reads one sequence's pages.
#pragma once

#include "common.cuh"

namespace msa {

struct TileInfo {
  int b;       // sequence
  int t0;      // first query token (global row)
  int t_end;   // one past the last query token of this sequence
  int p0;      // position of t0
};

MSA_DEV int find_sequence(const int32_t* cu_q, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One block: sequences are walked in order and the tiles of each are filled
// in parallel. A sequence that does not fit its page-table row (or has more
// queries than tokens) is reported as a data error and gets no tiles.
static __global__ void plan_tiles_kernel(const int32_t* __restrict__ seq_lens,
                                         const int32_t* __restrict__ cu_q, int B, int toks,
                                         int max_pages, int max_tiles,
                                         TileInfo* __restrict__ tiles, int* __restrict__ n_tiles,
                                         unsigned* err) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  int n = 0;
  for (int b = 0; b < B; ++b) {
    const int q0 = cu_q[b], q1 = cu_q[b + 1], L = seq_lens[b];
    const int qlen = q1 - q0;
    if (qlen < 0 || L < qlen || L > max_pages * 128) {
      if (threadIdx.x == 0) atomicOr(err, MSA_DEVERR_DATA);
      continue;
    }
    const int nt = min((qlen + toks - 1) / toks, max_tiles - n);
    for (int k = threadIdx.x; k < nt; k += blockDim.x)
      tiles[n + k] = TileInfo{b, q0 + k * toks, q1, L - qlen + k * toks};
    n += nt;
  }
  if (threadIdx.x == 0) *n_tiles = n;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace msa

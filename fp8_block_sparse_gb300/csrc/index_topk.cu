// index_topk.cu -- step (b): indexer block scores and the ascending top-k.
//
// What is computed (vLLM PR 45892 page, implementation steps 1-4; sglang PR
// 30971 page, implementation step 2 and review item 2): for index head i and
// query token t at position p with own block o = p / 128,
//   score[i,t,j] = max over the 128 keys of block j < o of idx_q[t,i] . idx_k[key]
// and topk_indices[i,t,:] lists the topk-1 best blocks j < o (ties: lower id)
// in ascending order followed by o; when o + 1 <= topk it lists 0..o and pads
// with -1. The own block is always selected (a reading of this library).
//
// GB300 design:
// * Prefill scoring is a dense FP8 contraction, so it runs on tcgen05: a CTA
//   holds a 128-row tile of (token, index head) queries in shared memory (one
//   TMA load) and streams the 128-key pages of the index-K cache through a
//   3-stage TMA ring. Each page is one M=128 x N=128 x K=D e4m3 MMA into a
//   double-buffered TMEM accumulator; four epilogue warps read their rows out
//   of TMEM and reduce the 128 columns to the block maximum. Scores of a
//   64-block chunk are staged in shared memory; a full tile's go out by TMA
//   (boxes of [Hidx][tokens][32 blocks]), a ragged tile's by its threads.
// * Decode (one query token per sequence) is a stream over the index-K pages;
//   it runs the same MMA with the roles swapped (M=128 keys of the page,
//   N=16 query columns of which Hidx are used) so the page is the A operand
//   straight out of the TMA ring and the max runs across TMEM lanes.
// * Selection is one warp per row: a radix select over the bits of the
//   order-preserving fp32 key finds the (topk-1)-th largest score exactly,
//   then ballot/popc writes the chosen ids in ascending order (a row whose
//   threshold has exactly topk-1 keys at or above it needs no tie pass).
#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

#include <cstring>

namespace msa {
namespace {

constexpr int kChunk = 64;       // blocks scored per CTA (64 measured 7% faster than 32 and 48)
constexpr int kStages = 3;       // TMA ring depth (3 keeps two CTAs per SM with 64-block chunks)
constexpr int kScorePitch = kChunk + 1;

// Tiled TMA store of one 3-D box from shared memory (bulk-group completion).
MSA_DEV void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Order-preserving map of fp32 onto uint32 (larger float -> larger key).
MSA_DEV uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0;                        // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MSA_DEV float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ------------------------------------------------------------ prefill scores
template <int D>
struct PrefillSmem {
  static constexpr int kQ = 0;                               // 128 x D
  static constexpr int kK = 16384;                           // kStages x (128 x D)
  // 128 x kScorePitch fp32, or (full tiles, TMA store) two 16 KB boxes of
  // [Hidx][tokens][32 columns] in the 128-byte swizzle
  static constexpr int kScore = kK + kStages * 16384;
  static constexpr int kBytes = kScore + 128 * kScorePitch * 4 + 1024;   // + alignment slack
};

// 128 registers at most: two CTAs per SM put up to four of their warps on
// one sub-partition, whose register file holds 4 x 32 x 128.
template <int D>
__global__ void __maxnreg__(128)
index_score_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_s, int tma_store,
                           const int32_t* __restrict__ page_table,
                           const TileInfo* __restrict__ tiles, const int* __restrict__ n_tiles_p,
                           int T, int Hidx, int toks, int max_pages, int num_pages,
                           int chunks_per_tile, float* __restrict__ scores, unsigned* err) {
  pdl_wait();      // the tile list, queries and cache come from earlier kernels
  constexpr int SWZ = D;                    // 128-byte or 64-byte swizzle rows
  constexpr uint32_t kIdesc = idesc_f32(128, 128);
  using L = PrefillSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_full[kStages], bar_empty[kStages], bar_tfull[2], bar_tempty[2],
      bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  const int n_tiles = *n_tiles_p;
  const int tile_rank = blockIdx.x / chunks_per_tile;
  if (tile_rank >= n_tiles) return;
  const int tile_id = n_tiles - 1 - tile_rank;      // longest (latest) tiles first
  const TileInfo ti = tiles[tile_id];
  const int n_tok = min(toks, ti.t_end - ti.t0);
  const int nb = (ti.p0 + n_tok - 1) / 128;        // blocks 0..nb-1 can be needed
  const int c0 = (blockIdx.x % chunks_per_tile) * kChunk;
  if (c0 >= nb) return;
  const int nblk = min(kChunk, nb - c0);
  // a full tile's rows go out by TMA (ragged tiles must not touch the rows
  // of the next sequence's tokens, which the box would cover)
  const bool via_tma = tma_store && n_tok == toks;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sK = smem + L::kK;
  float* sScore = reinterpret_cast<float*>(smem + L::kScore);

  if (tid == 0) {
    abort_s = initial_abort(err);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_drain, 1);
    for (int s = 0; s < kStages; ++s) { mbar_init(&bar_full[s], 1); mbar_init(&bar_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&bar_tfull[s], 1); mbar_init(&bar_tempty[s], 4); }
    fence_barrier_init();
  }
  if (warp == 1) { tmem_alloc(&tmem_base_s, 256); tmem_relinquish(); }
  __syncthreads();
  pdl_trigger();   // after this block's tensor-memory allocation
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(&bar_q, 128 * D);
      tma_load_2d(sQ, &tm_q, &bar_q, 0, ti.t0 * Hidx);
      const int32_t* prow = page_table + size_t(ti.b) * max_pages;
      int nk = 0;
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kStages;
        if (!mbar_wait_ab(&bar_empty[s], ((j / kStages) & 1) ^ 1, err, &abort_s)) break;
        int page = __ldg(prow + c0 + j);
        if (page < 0 || page >= num_pages) { atomicOr(err, MSA_DEVERR_DATA); page = 0; }
        mbar_arrive_expect_tx(&bar_full[s], 128 * D);
        tma_load_2d(sK + s * 16384, &tm_k, &bar_full[s], 0, page * 128);
        ++nk;
      }
      // exit-path drain (a no-op unless a wait gave up): every copy has landed
      mbar_wait(&bar_q, 0, err);
      mbar_drain_ring(bar_full, kStages, nk, err);
    }
  } else if (warp == 1) {
    if (mbar_wait_warp(&bar_q, 0, err, &abort_s)) {          // whole warp, elected issue
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kStages, buf = j & 1;
        if (!mbar_wait_warp(&bar_full[s], (j / kStages) & 1, err, &abort_s)) break;
        if (!mbar_wait_warp(&bar_tempty[buf], ((j >> 1) & 1) ^ 1, err, &abort_s)) break;
        tc_fence_after();
        const uint32_t aq = smem_addr(sQ), bk = smem_addr(sK + s * 16384);
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_e4m3_w(tmem + buf * 128, sdesc_kmajor(aq + 32 * k, SWZ), sdesc_kmajor(bk + 32 * k, SWZ),
                     kIdesc, k > 0);
        mma_commit_w(&bar_empty[s]);
        mma_commit_w(&bar_tfull[buf]);
      }
    }
    mma_drain_w(&bar_drain, err);            // no MMA in flight once TMEM is freed
  } else {
    // epilogue: warps 2..5 own TMEM lanes 32*(warp%4) .. +31
    const int row = (warp & 3) * 32 + lane;
    const int hshift = __ffs(Hidx) - 1;      // Hidx is a power of two
    // box row of this TMEM row (token-major -> head-major) and its 16-byte
    // chunk swizzle
    const int brow = (row & (Hidx - 1)) * toks + (row >> hshift);
    float* bdst = sScore + brow * 32;
    for (int j = 0; j < nblk; ++j) {
      const int buf = j & 1;
      if (!mbar_wait_warp(&bar_tfull[buf], (j >> 1) & 1, err, &abort_s)) break;   // uniform
      tc_fence_after();
      // the row's 128 scores in two TMEM round trips of 64 (128 live values
      // would cost the second CTA per SM its registers), reduced by 3-input
      // maxima in four independent chains (every score is finite)
      float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 64) {
        uint32_t v[64];
        tmem_ld64(tmem_addr(tmem + buf * 128, (warp & 3) * 32, c), v);
#pragma unroll
        for (int x = 0; x < 64; x += 8) {
          a0 = fmax3(a0, __uint_as_float(v[x]), __uint_as_float(v[x + 1]));
          a1 = fmax3(a1, __uint_as_float(v[x + 2]), __uint_as_float(v[x + 3]));
          a2 = fmax3(a2, __uint_as_float(v[x + 4]), __uint_as_float(v[x + 5]));
          a3 = fmax3(a3, __uint_as_float(v[x + 6]), __uint_as_float(v[x + 7]));
        }
      }
      const float m = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tempty[buf]);
      if (via_tma) {
        const int c = j & 31;
        bdst[(j >> 5) * 4096 + ((((c >> 2) ^ (brow & 7)) << 2) | (c & 3))] = m;
      } else {
        sScore[row * kScorePitch + j] = m;
      }
    }
    if (via_tma) {
      fence_async_shared();                  // score writes -> the TMA store's reads
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (tid == 64) {
        // columns past nblk are blocks no token of the tile selects from
        tma_store_3d(&tm_s, sScore, c0, ti.t0, 0);
        if (nblk > 32) tma_store_3d(&tm_s, sScore + 4096, c0 + 32, ti.t0, 0);
        bulk_commit();
        bulk_wait_read();                    // shared memory stays until read
      }
    } else {
      asm volatile("bar.sync 1, 128;" ::: "memory");
      // rows -> (token, head): warp e takes rows e, e+4, ..., e+124 and lane l
      // writes columns l and l+32 of each, eight rows at a time with all their
      // shared-memory reads issued before the first global store (one row per
      // round trip kept this phase at ~18% of a CTA's life). Hidx is a power
      // of two, so a row's token and head are a shift and a mask.
      static_assert(kChunk == 64, "two score columns per lane");
      const bool col_lo = lane < nblk, col_hi = lane + 32 < nblk;
#pragma unroll 1
      for (int r0 = warp - 2; r0 < 128; r0 += 32) {
        float v_lo[8], v_hi[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float* src = sScore + (r0 + 4 * k) * kScorePitch;
          v_lo[k] = src[lane];
          v_hi[k] = src[lane + 32];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = r0 + 4 * k, tl = r >> hshift;
          if (tl < n_tok) {                                   // rows past the tile's tokens: none
            float* dst = scores + (size_t(r & (Hidx - 1)) * T + ti.t0 + tl) * max_pages + c0;
            if (col_lo) dst[lane] = v_lo[k];
            if (col_hi) dst[lane + 32] = v_hi[k];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------ decode scores
// One CTA per (query token, 64-block chunk). A = index-K page (M = 128 keys),
// B = the token's Hidx query rows (N = 16; extra rows are ignored).
template <int D>
__global__ void __launch_bounds__(192, 1)
index_score_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const int32_t* __restrict__ page_table,
                          const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q,
                          int B, int T, int Hidx, int max_pages, int num_pages,
                          int chunks_per_tok, float* __restrict__ scores, unsigned* err) {
  pdl_wait();      // queries, cache and batch description may come from earlier kernels
  constexpr int SWZ = D;
  constexpr int kBufs = 4;
  constexpr uint32_t kIdesc = idesc_f32(128, 16);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_full[kStages], bar_empty[kStages], bar_tfull[kBufs], bar_tempty[kBufs],
      bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ uint32_t sred[kChunk][16];   // order-preserving keys of the block maxima

  const int t = blockIdx.x / chunks_per_tok;
  const int c0 = (blockIdx.x % chunks_per_tok) * kChunk;
  // one query per sequence (q_len <= 1, T == B) makes token t sequence t
  const int b = (T == B) ? t : find_sequence(cu_q, B, t);
  const int qlen = cu_q[b + 1] - cu_q[b];
  const int p = seq_lens[b] - qlen + (t - cu_q[b]);
  if (p < 0 || p >= max_pages * 128) {
    if (threadIdx.x == 0 && c0 == 0) atomicOr(err, MSA_DEVERR_DATA);
    return;
  }
  const int nb = p / 128;
  if (c0 >= nb) return;
  const int nblk = min(kChunk, nb - c0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* sK = smem;                       // kStages x 16 KB
  uint8_t* sQ = smem + kStages * 16384;     // 16 rows x D

  if (tid == 0) {
    abort_s = initial_abort(err);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_drain, 1);
    for (int s = 0; s < kStages; ++s) { mbar_init(&bar_full[s], 1); mbar_init(&bar_empty[s], 1); }
    for (int s = 0; s < kBufs; ++s) { mbar_init(&bar_tfull[s], 1); mbar_init(&bar_tempty[s], 4); }
    fence_barrier_init();
  }
  if (warp == 1) { tmem_alloc(&tmem_base_s, 64); tmem_relinquish(); }
  __syncthreads();
  pdl_trigger();   // after this block's tensor-memory allocation
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_q, 16 * D);
      tma_load_2d(sQ, &tm_q, &bar_q, 0, t * Hidx);
      const int32_t* prow = page_table + size_t(b) * max_pages;
      int nk = 0;
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kStages;
        if (!mbar_wait_ab(&bar_empty[s], ((j / kStages) & 1) ^ 1, err, &abort_s)) break;
        int page = __ldg(prow + c0 + j);
        if (page < 0 || page >= num_pages) { atomicOr(err, MSA_DEVERR_DATA); page = 0; }
        mbar_arrive_expect_tx(&bar_full[s], 128 * D);
        tma_load_2d(sK + s * 16384, &tm_k, &bar_full[s], 0, page * 128);
        ++nk;
      }
      // exit-path drain (a no-op unless a wait gave up): every copy has landed
      mbar_wait(&bar_q, 0, err);
      mbar_drain_ring(bar_full, kStages, nk, err);
    }
  } else if (warp == 1) {
    if (mbar_wait_warp(&bar_q, 0, err, &abort_s)) {          // whole warp, elected issue
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kStages, buf = j % kBufs;
        if (!mbar_wait_warp(&bar_full[s], (j / kStages) & 1, err, &abort_s)) break;
        if (!mbar_wait_warp(&bar_tempty[buf], ((j / kBufs) & 1) ^ 1, err, &abort_s)) break;
        tc_fence_after();
        const uint32_t ak = smem_addr(sK + s * 16384), bq = smem_addr(sQ);
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_e4m3_w(tmem + buf * 16, sdesc_kmajor(ak + 32 * k, SWZ), sdesc_kmajor(bq + 32 * k, SWZ),
                     kIdesc, k > 0);
        mma_commit_w(&bar_empty[s]);
        mma_commit_w(&bar_tfull[buf]);
      }
    }
    mma_drain_w(&bar_drain, err);            // no MMA in flight once TMEM is freed
  } else {
    const int q4 = warp & 3;
    const int et = tid - 64;
    for (int x = et; x < kChunk * 16; x += 128) (&sred[0][0])[x] = 0u;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int j = 0; j < nblk; ++j) {
      const int buf = j % kBufs;
      if (!mbar_wait_warp(&bar_tfull[buf], (j / kBufs) & 1, err, &abort_s)) break;   // uniform
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(tmem_addr(tmem + buf * 16, q4 * 32, 0), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tempty[buf]);
      // block maximum of each index head (columns past Hidx are padding)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c < Hidx) {                                // uniform across the CTA
          float m = __uint_as_float(v[c]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) atomicMax(&sred[j][c], order_key(m));
        }
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int x = et; x < nblk * Hidx; x += 128) {
      const int c = x / nblk, j = x - c * nblk;
      scores[(size_t(c) * T + t) * max_pages + c0 + j] = key_to_float(sred[j][c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 64);
}

// ------------------------------------------------------------ selection

// The ascending top-(kp) of the `own` candidate blocks 0..own-1 of one row,
// plus the own block, by one warp; NPL = candidate slots per lane
// (32 * NPL >= own), so a short row costs only the slots it needs.
template <int NPL>
MSA_DEV void select_row(const float* __restrict__ s, int own, int kp, int lane, int32_t* __restrict__ o) {
  uint32_t key[NPL];
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const int id = r * 32 + lane;
    key[r] = id < own ? order_key(__ldg(s + id)) : 0u;   // 0 sorts below every score
  }
  // largest tau with #{key >= tau} >= kp: the kp-th largest key. The bits
  // every candidate shares are the same in tau (all candidates lie on one
  // side of each such bit), so the search starts below them; and once
  // exactly kp keys reach tau the selected set cannot change any more.
  uint32_t kand = 0xFFFFFFFFu, kor = 0u;
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    if (r * 32 + lane < own) { kand &= key[r]; kor |= key[r]; }
  }
  kand = __reduce_and_sync(0xffffffffu, kand);
  kor = __reduce_or_sync(0xffffffffu, kor);
  const uint32_t diff = kand ^ kor;
  const int top = diff ? 31 - __clz(diff) : -1;            // highest bit that differs
  uint32_t tau = top < 0 ? kand : (top == 31 ? 0u : (kand & ~((2u << top) - 1u)));
  bool exact = false;
  for (int bit = top; bit >= 0; --bit) {
    const uint32_t tr = tau | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int r = 0; r < NPL; ++r) cnt += key[r] >= tr;
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (cnt >= kp) {
      tau = tr;
      if (cnt == kp) { exact = true; break; }               // uniform: cnt is warp-wide
    }
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (exact) {
    // exactly kp keys reach tau (>= 1, so no empty slot among them): no ties
    // to break, the selection is every key >= tau
    int pos = 0;
#pragma unroll
    for (int r = 0; r < NPL; ++r) {
      const bool sel = key[r] >= tau;
      const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
      if (sel) o[pos + __popc(sel_mask & lt_mask)] = r * 32 + lane;
      pos += __popc(sel_mask);
    }
    if (lane == 0) o[kp] = own;
    return;
  }
  int gt = 0;
#pragma unroll
  for (int r = 0; r < NPL; ++r) gt += key[r] > tau;
  gt = __reduce_add_sync(0xffffffffu, gt);
  const int need_ties = kp - gt;
  int pos = 0, ties_seen = 0;
#pragma unroll
  for (int r = 0; r < NPL; ++r) {
    const int id = r * 32 + lane;
    const bool valid = id < own;
    const bool tie = valid && key[r] == tau;
    const uint32_t tie_mask = __ballot_sync(0xffffffffu, tie);
    const int tie_rank = ties_seen + __popc(tie_mask & lt_mask);
    const bool sel = valid && (key[r] > tau || (tie && tie_rank < need_ties));
    const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
    if (sel) o[pos + __popc(sel_mask & lt_mask)] = id;
    pos += __popc(sel_mask);
    ties_seen += __popc(tie_mask);
  }
  if (lane == 0) o[kp] = own;
}

// One warp per (index head, token) row. NPL = candidate slots per lane for
// the longest row (32 * NPL >= max_pages); each row takes the smallest of
// 2, 4, 8, 16, NPL slots that holds its candidates (warp-uniform choice).
template <int NPL>
__global__ void __launch_bounds__(256)
topk_select_kernel(const float* __restrict__ scores, const int32_t* __restrict__ seq_lens,
                   const int32_t* __restrict__ cu_q, int B, int T, int Hidx, int topk,
                   int max_pages, int decode, int32_t* __restrict__ out, unsigned* err) {
  pdl_wait();      // the scores come from the scoring kernel
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.y;                                  // index head
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const size_t row = size_t(i) * T + t;
  // with one query per sequence (decode: q_len <= 1, T == B) token t is
  // sequence t; otherwise search the query offsets
  const int b = (decode && T == B) ? t : find_sequence(cu_q, B, t);
  const int qlen = cu_q[b + 1] - cu_q[b], L = seq_lens[b];
  const int p = L - qlen + (t - cu_q[b]);
  int32_t* o = out + row * topk;
  // a token outside every sequence, or of a sequence that does not fit its
  // page-table row (the tile plan gives it no scores): a -1 row and a data error
  if (t >= cu_q[b + 1] || qlen < 0 || L < qlen || L > max_pages * 128 || p < 0 ||
      p >= max_pages * 128) {
    for (int j = lane; j < topk; j += 32) o[j] = -1;
    if (lane == 0) atomicOr(err, MSA_DEVERR_DATA);
    return;
  }
  const int own = p / 128;
  if (own + 1 <= topk) {
    for (int j = lane; j < topk; j += 32) o[j] = (j <= own) ? j : -1;
    return;
  }
  const float* s = scores + row * max_pages;
  const int kp = topk - 1;
  if (NPL > 2 && own <= 64) select_row<2>(s, own, kp, lane, o);
  else if (NPL > 4 && own <= 128) select_row<4>(s, own, kp, lane, o);
  else if (NPL > 8 && own <= 256) select_row<(NPL > 8 ? 8 : NPL)>(s, own, kp, lane, o);
  else if (NPL > 16 && own <= 512) select_row<(NPL > 16 ? 16 : NPL)>(s, own, kp, lane, o);
  else select_row<NPL>(s, own, kp, lane, o);
}

}  // namespace

size_t index_workspace_bytes(int T, int Hidx, int max_pages) {
  const size_t scores = align256(size_t(Hidx) * T * max_pages * sizeof(float));
  const size_t toks = Hidx > 0 ? size_t(128 / Hidx > 0 ? 128 / Hidx : 1) : 1;
  const size_t max_tiles = (size_t(T) + toks - 1) / toks + size_t(T) + 1;
  return scores + align256(max_tiles * sizeof(TileInfo)) + 256;
}

cudaError_t launch_index_topk(const IndexArgs& a, cudaStream_t stream, const char** why) {
  const int D = a.D;
  if (a.Hidx > 16 || (a.Hidx & (a.Hidx - 1)) != 0) {
    *why = "Hidx must be a power of two <= 16";
    return cudaErrorNotSupported;
  }
  if (a.max_pages > 2048) {
    *why = "max_pages must be <= 2048";
    return cudaErrorNotSupported;
  }
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.scores);
  float* scores = a.scores;
  const size_t scores_bytes = align256(size_t(a.Hidx) * a.T * a.max_pages * sizeof(float));
  const int toks = 128 / a.Hidx;
  const int max_tiles = (a.T + toks - 1) / toks + a.T + 1;
  TileInfo* tiles = reinterpret_cast<TileInfo*>(ws + scores_bytes);
  int* n_tiles = reinterpret_cast<int*>(ws + scores_bytes + align256(size_t(max_tiles) * sizeof(TileInfo)));

  const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap tm_q, tm_k;
  const bool decode = a.max_q_len == 1;
  {
    const uint64_t dims[2] = {uint64_t(D), uint64_t(a.T) * a.Hidx};
    const uint64_t strides[1] = {uint64_t(D)};
    const uint32_t box[2] = {uint32_t(D), decode ? 16u : 128u};
    if (!encode_tensor_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.idx_q, dims, strides, box, swz, why))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {uint64_t(D), uint64_t(a.num_pages) * 128};
    const uint64_t strides[1] = {uint64_t(D)};
    const uint32_t box[2] = {uint32_t(D), 128u};
    if (!encode_tensor_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.idx_k, dims, strides, box, swz, why))
      return cudaErrorInvalidValue;
  }
  const int chunks = (a.max_pages + kChunk - 1) / kChunk;
  cudaError_t e = cudaSuccess;
  if (decode) {
    const int smem = kStages * 16384 + 16 * 128 + 1024;
    auto kern = D == 128 ? index_score_decode_kernel<128> : index_score_decode_kernel<64>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    profile_mark(stream, 0);
    e = launch_pdl(kern, a.T * chunks, 192, smem, stream, tm_q, tm_k, a.page_table, a.seq_lens,
                   a.cu_q, a.B, a.T, a.Hidx, a.max_pages, a.num_pages, chunks, scores, a.err);
    if (e != cudaSuccess) return e;
  } else {
    e = launch_pdl(plan_tiles_kernel, 1, 256, 0, stream, a.seq_lens, a.cu_q, a.B, toks,
                   a.max_pages, max_tiles, tiles, n_tiles, a.err);
    if (e != cudaSuccess) return e;
    const int smem = D == 128 ? PrefillSmem<128>::kBytes : PrefillSmem<64>::kBytes;
    auto kern = D == 128 ? index_score_prefill_kernel<128> : index_score_prefill_kernel<64>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int n_tiles_max = (a.T + toks - 1) / toks + a.B;
    profile_mark(stream, 0);
    // scores as [Hidx][T][max_pages] fp32 for the TMA store of full tiles
    // (row pitch a multiple of 16 bytes, else every tile stores by threads)
    CUtensorMap tm_s;
    int tma_store = 0;
    if (a.max_pages % 4 == 0) {
      const uint64_t dims[3] = {uint64_t(a.max_pages), uint64_t(a.T), uint64_t(a.Hidx)};
      const uint64_t strides[2] = {uint64_t(a.max_pages) * 4, uint64_t(a.T) * a.max_pages * 4};
      const uint32_t box[3] = {32u, uint32_t(toks), uint32_t(a.Hidx)};
      if (!encode_tensor_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scores, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B, why))
        return cudaErrorInvalidValue;
      tma_store = 1;
    } else {
      std::memset(&tm_s, 0, sizeof(tm_s));
    }
    e = launch_pdl(kern, n_tiles_max * chunks, 192, smem, stream, tm_q, tm_k, tm_s, tma_store,
                   a.page_table, tiles,
                   n_tiles, a.T, a.Hidx, toks, a.max_pages, a.num_pages, chunks, scores, a.err);
    if (e != cudaSuccess) return e;
  }
  // one warp per row, grid (tokens, index heads); few rows (a decode batch)
  // go one warp per CTA so that they spread over every SM instead of
  // queueing eight to a CTA
  const long long rows = (long long)a.Hidx * a.T;
  const int wpc = rows < 8LL * num_sms() ? 1 : 8;
  const dim3 grid(unsigned((a.T + wpc - 1) / wpc), unsigned(a.Hidx));
  auto sel = a.max_pages <= 256 ? topk_select_kernel<8>
            : a.max_pages <= 512 ? topk_select_kernel<16> : topk_select_kernel<64>;
  e = launch_pdl(sel, grid, 32 * wpc, 0, stream, scores, a.seq_lens, a.cu_q, a.B, a.T, a.Hidx, a.topk,
                 a.max_pages, int(decode), a.topk_indices, a.err);
  profile_mark(stream, 1);
  return e;
}

}  // namespace msa

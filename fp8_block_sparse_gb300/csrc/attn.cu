// attn.cu -- step (c): GQA sparse attention over the selected 128-token blocks,
// with online softmax, a per-head sink and per-tensor scales.
//
// What is computed (sglang PR 30971 page, implementation step 3 and the
// executive summary; vLLM PR 45892 page, step 2): query row (t, h) attends to
// the keys of the blocks listed in topk_indices[i(h), t, :] at positions <= its
// own, with l_j = c*k_scale*(q.k_j), sigma = c*sink[h], c = sm_scale*q_scale:
//   O = v_scale * sum_j e^{l_j} v_j / (sum_j e^{l_j} + e^{sigma}),
//   max_logit = max_j l_j,  lse = ln(sum_j e^{l_j} + e^{sigma}).
//
// Prefill kernel (GB300 design). One CTA owns a 128-row query tile: 128/G
// tokens x the G q heads of one kv head, so every K/V page it loads serves all
// rows. Rows of different tokens select different blocks, so the CTA walks the
// ascending UNION of its rows' selections; a row that did not select a block
// (or a key beyond its position) gets p = 0 for it. Per block:
//   S  = Q K^T     tcgen05 kind::f8f6f4 (e4m3 x e4m3 -> fp32), M=N=128, K=128,
//                  into one of two TMEM S buffers (QK of block j+1 overlaps the
//                  softmax of block j);
//   P  = exp2(S*c*log2e - m)   one thread per row (four warps, TMEM lanes),
//                  written as f16 into a swizzled shared-memory A operand;
//   O += P V       tcgen05 kind::f16, B = a V^T f16 image of the block
//                  prepared once per call; O accumulates in TMEM.
// P is kept in f16, not e4m3: rounding P to 3 mantissa bits costs about 2.5%
// relative error on O for flat softmax rows (the pages name fp8 P as the main
// error source and test it at 6e-2..1e-1); f16 P keeps O well inside 1e-2.
// The running max is rescaled lazily: O and l are only rescaled when a row's
// max grows by more than 2^8, so P stays <= 256 and rescales are rare.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;   // log2 units

// shared memory of the prefill kernel (byte offsets from a 1024-aligned base)
constexpr int kStages = 3;
constexpr int kQOff = 0;             // 2 tiles x 128 rows x 128 e4m3        32 KB
constexpr int kKOff = 32768;         // 3 stages x 128 keys x 128 e4m3       48 KB
constexpr int kVOff = 81920;         // 3 stages x V^T f16 image             96 KB
constexpr int kBlistOff = 180224;    // union block list (int16)              4 KB
constexpr int kBitsOff = 184320;     // union bitmap, 2048 bits              256 B
constexpr int kPrefillSmem = 184576 + 1024;
constexpr int kPrefillThreads = 576;   // producer, MMA, 16 softmax warps

constexpr uint32_t kIdescQK = idesc_f32(128, 128);
constexpr uint32_t kIdescPV = idesc_f32(128, 128);

// ------------------------------------------------------------ V^T images
// One CTA per (logical block, sequence, kv head): the 128x128 e4m3 V page
// becomes a 32 KB f16 image of V^T (rows = head dim, K = keys) laid out as
// two swizzled K-major atoms of 64 keys. Keys at positions >= seq_len are
// written as zeros so stale cache bytes can never reach the PV product.
__global__ void __launch_bounds__(256)
vt_convert_kernel(const uint8_t* __restrict__ v_cache, const int32_t* __restrict__ page_table,
                  const int32_t* __restrict__ seq_lens, int Hkv, int max_pages, int num_pages,
                  uint8_t* __restrict__ vt_img, unsigned* err) {
  pdl_wait();      // the V cache and batch description may come from earlier kernels
  pdl_trigger();
  const int blk = blockIdx.x, b = blockIdx.y, g = blockIdx.z;
  const int L = seq_lens[b];
  if (L <= blk * 128 || L > max_pages * 128) return;
  const int page = page_table[size_t(b) * max_pages + blk];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) atomicOr(err, MSA_DEVERR_DATA);
    return;
  }
  __shared__ __align__(16) uint8_t tile[128 * 128];
  const uint4* src = reinterpret_cast<const uint4*>(v_cache + (size_t(page) * Hkv + g) * 16384);
  for (int i = threadIdx.x; i < 1024; i += 256) reinterpret_cast<uint4*>(tile)[i] = __ldg(src + i);
  __syncthreads();
  const int nvalid = min(128, L - blk * 128);
  uint8_t* dst = vt_img + ((size_t(b) * max_pages + blk) * Hkv + g) * 32768;
  for (int x = threadIdx.x; x < 2048; x += 256) {
    const int d = x & 127, c = (x >> 7) & 7, a = x >> 10;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k0 = a * 64 + c * 8 + 2 * e;
      const uint32_t lo = k0 < nvalid ? tile[k0 * 128 + d] : 0u;
      const uint32_t hi = k0 + 1 < nvalid ? tile[(k0 + 1) * 128 + d] : 0u;
      w[e] = e4m3x2_to_f16x2(uint16_t(lo | (hi << 8)));
    }
    *reinterpret_cast<uint4*>(dst + a * 16384 + swz_offset(d, c, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------ prefill
// One CTA = two 128-row tiles (X = 0, 1) of one kv head: 2 x 128/G tokens x
// G heads. Warp roles: 0 producer (TMA), 1 MMA issue, 2-17 softmax: two
// threads per row, one per half of the 128 columns (warp w reads TMEM lanes
// 32*(w%4), so the two threads of a row sit in two warps of the same lane
// quarter; they share the row's running maximum through shared memory). A
// row's softmax of one block is thus two 64-column chains, not one
// 128-column chain, which halves the latency the MMAs wait on. With 18 warps
// a sub-partition holds up to 5 of them, so a thread gets 96 registers: each
// half reads its 64 S columns twice (once for the maximum, once for P), 32 at
// a time, and writes its P (f16 pairs) over the first 32 of its own S
// columns, so the two halves never touch each other's columns. TMEM: S_0 and S_1 at columns 0 and 128, O_0 and O_1 at 256
// and 384. P (f16, two per 32-bit column) overwrites the first 64 columns of
// its tile's S once the softmax has read S, and the PV MMA takes it as the A
// operand straight from TMEM, so P never touches shared memory (which would
// otherwise bound the kernel: a 128x128 f16 MMA with both operands in smem
// reads 128 B/clk). Per block j the MMA issue order is PV_0(j), S_0(j+1),
// PV_1(j), S_1(j+1); tcgen05 MMAs of one thread run in order, so S_X(j+1)
// overwrites P_X(j) only after PV_X(j) has read it, and the commit of S_X(j+1)
// also proves PV_X(j) complete -- the softmax needs no other barrier before
// touching O or writing the next P.
__global__ void __launch_bounds__(kPrefillThreads, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const uint8_t* __restrict__ vt_img, const int32_t* __restrict__ page_table,
                    const TileInfo* __restrict__ tiles, const int* __restrict__ n_tiles_p,
                    const int32_t* __restrict__ topk, const float* __restrict__ sink,
                    float qk_scale2, float sink_scale2, float v_scale, int T, int Hq, int Hkv,
                    int Hidx, int toks, int topk_k, int max_pages, int num_pages,
                    uint16_t* __restrict__ out, float* __restrict__ max_logit,
                    float* __restrict__ lse, unsigned* err) {
  pdl_wait();      // tiles, V images, queries and top-k come from earlier kernels
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_q, bar_kf[kStages], bar_ke[kStages], bar_vf[kStages], bar_ve[kStages],
      bar_sf[2], bar_pf[2], bar_done, bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int n_union_s;
  __shared__ int abort_s;
  __shared__ float xmax_s[2][2][2][128];   // [block parity][tile][half][row]: partial row maxima
  __shared__ float lsum_s[2][2][128];      // [tile][half][row]: partial row sums

  const int n_tiles = *n_tiles_p;
  const int tile_rank = blockIdx.x / Hkv;
  if (tile_rank >= n_tiles) return;
  const int g = blockIdx.x % Hkv;
  const TileInfo ti = tiles[n_tiles - 1 - tile_rank];     // latest (longest) tiles first
  const int G = Hq / Hkv;
  const int n_tok = min(2 * toks, ti.t_end - ti.t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int16_t* sBlist = reinterpret_cast<int16_t*>(smem + kBlistOff);
  uint32_t* sBits = reinterpret_cast<uint32_t*>(smem + kBitsOff);

  if (tid < 64) sBits[tid] = 0u;
  if (tid == 0) {
    abort_s = initial_abort(err);
    mbar_init(&bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_kf[s], 1); mbar_init(&bar_ke[s], 1);
      mbar_init(&bar_vf[s], 1); mbar_init(&bar_ve[s], 1);
    }
    for (int x = 0; x < 2; ++x) { mbar_init(&bar_sf[x], 1); mbar_init(&bar_pf[x], 8); }
    mbar_init(&bar_done, 1);
    mbar_init(&bar_drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) { tmem_alloc(&tmem_base_s, 512); tmem_relinquish(); }
  __syncthreads();
  pdl_trigger();   // after this block's tensor-memory allocation

  // ---- softmax threads: tile X, column half hh, row 128*X + 32*(warp%4) + lane
  const bool is_softmax = warp >= 2;
  const int sw = warp - 2;
  const int X = sw >> 3, hh = (sw >> 2) & 1, quarter = warp & 3;
  const int rq = quarter * 32 + lane;                             // row within the tile
  const int row = X * 128 + rq;
  int own = -1, pos = -1, h = 0, t = 0, next_id = -1, ptr = 0;
  bool row_valid = false;
  const int32_t* src = nullptr;
  if (is_softmax) {
    const int tl = row / G;
    t = ti.t0 + tl;
    h = g * G + row % G;
    row_valid = tl < n_tok;
    if (row_valid) {
      pos = ti.p0 + tl;
      own = pos >> 7;
      src = topk + (size_t(h / (Hq / Hidx)) * T + t) * topk_k;
      next_id = topk_k > 0 ? __ldg(src) : -1;
    }
  }
  {
    // the union of the tile pair's lists: every thread takes entries of the
    // (token, index head) lists in turn, all loads independent of one another.
    // A list must be strictly ascending with its -1 padding at the end (each
    // row walks its own list in union order); an entry that breaks this, or
    // that points past its token's own block, is left out and reported.
    const int hpi = Hq / Hidx;
    const int i_first = (g * G) / hpi;
    const int n_idx = (g * G + G - 1) / hpi - i_first + 1;
    const int per_tok = n_idx * topk_k;
    for (int x = tid; x < n_tok * per_tok; x += kPrefillThreads) {
      const int tl = x / per_tok, r = x - tl * per_tok;
      const int il = r / topk_k, k = r - il * topk_k;
      const int32_t* lst = topk + (size_t(i_first + il) * T + ti.t0 + tl) * topk_k;
      const int id = __ldg(lst + k);
      if (id < 0) continue;                                       // -1 padding
      const int prev = k > 0 ? __ldg(lst + k - 1) : -1;
      if ((k > 0 && (prev < 0 || prev >= id)) || id > ((ti.p0 + tl) >> 7)) {
        atomicOr(err, MSA_DEVERR_DATA);
        continue;
      }
      atomicOr(&sBits[id >> 5], 1u << (id & 31));
    }
  }
  __syncthreads();
  if (warp == 0) {                                               // union -> ascending list
    int base = 0;
    for (int w0 = 0; w0 < 64; w0 += 32) {
      const uint32_t bits = sBits[w0 + lane];
      const int cnt = __popc(bits);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int off = base + incl - cnt;
      uint32_t bb = bits;
      while (bb) {
        const int k = __ffs(bb) - 1;
        bb &= bb - 1;
        sBlist[off++] = int16_t((w0 + lane) * 32 + k);
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_union_s = base;
  }
  __syncthreads();
  tc_fence_after();
  const int nU = n_union_s;
  const uint32_t tmem = tmem_base_s;

  if (warp < 2) {
    if (warp == 0 && lane == 0 && nU > 0) {
      // ---------------- producer: Q of both tiles, then K pages and V^T images
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(&bar_q, 32768);
      tma_load_3d(smem + kQOff, &tm_q, &bar_q, 0, g * G, ti.t0);
      tma_load_3d(smem + kQOff + 16384, &tm_q, &bar_q, 0, g * G, ti.t0 + toks);
      const int32_t* prow = page_table + size_t(ti.b) * max_pages;
      int nk = 0, nv = 0;                                  // copies issued per ring
      for (int j = 0; j < nU; ++j) {
        const int s = j % kStages;
        const uint32_t ph = ((j / kStages) & 1) ^ 1;
        const int blk = sBlist[j];
        int page = __ldg(prow + blk);
        if (page < 0 || page >= num_pages) { atomicOr(err, MSA_DEVERR_DATA); page = 0; }
        if (!mbar_wait_ab(&bar_ke[s], ph, err, &abort_s)) break;
        mbar_arrive_expect_tx(&bar_kf[s], 16384);
        tma_load_2d(smem + kKOff + s * 16384, &tm_k, &bar_kf[s], 0, (page * Hkv + g) * 128);
        ++nk;
        if (!mbar_wait_ab(&bar_ve[s], ph, err, &abort_s)) break;
        mbar_arrive_expect_tx(&bar_vf[s], 32768);
        bulk_load(smem + kVOff + s * 32768,
                  vt_img + ((size_t(ti.b) * max_pages + blk) * Hkv + g) * 32768, 32768, &bar_vf[s]);
        ++nv;
      }
      // exit-path drain (a no-op unless a wait gave up): every copy has landed
      mbar_wait(&bar_q, 0, err);
      mbar_drain_ring(bar_kf, kStages, nk, err);
      mbar_drain_ring(bar_vf, kStages, nv, err);
    } else if (warp == 1 && nU > 0) {
     if (mbar_wait_warp(&bar_q, 0, err, &abort_s)) {
      // ---------------- MMA issue (whole warp, one elected lane per instruction)
      const uint32_t sq = smem_addr(smem + kQOff);
      auto issue_s = [&](int j, int x) -> bool {
        const int s = j % kStages;
        if (x == 0 && !mbar_wait_warp(&bar_kf[s], (j / kStages) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t sk = smem_addr(smem + kKOff + s * 16384);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_e4m3_w(tmem + x * 128, sdesc_kmajor(sq + x * 16384 + 32 * k, 128),
                     sdesc_kmajor(sk + 32 * k, 128), kIdescQK, k > 0);
        mma_commit_w(&bar_sf[x]);
        if (x == 1) mma_commit_w(&bar_ke[s]);
        return true;
      };
      bool ok = issue_s(0, 0) && issue_s(0, 1);
      for (int j = 0; ok && j < nU; ++j) {
        const int s = j % kStages;
        if (!mbar_wait_warp(&bar_vf[s], (j / kStages) & 1, err, &abort_s)) break;
        const uint32_t sv = smem_addr(smem + kVOff + s * 32768);
        for (int x = 0; x < 2; ++x) {
          if (!(ok = mbar_wait_warp(&bar_pf[x], j & 1, err, &abort_s))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16_ts_w(tmem + 256 + x * 128, tmem + x * 128 + 64 * (k >> 2) + 8 * (k & 3),
                         sdesc_kmajor(sv + (k >> 2) * 16384 + (k & 3) * 32, 128), kIdescPV,
                         (j > 0 || k > 0) ? 1u : 0u);
          if (x == 1) mma_commit_w(&bar_ve[s]);
          if (j + 1 < nU && !(ok = issue_s(j + 1, x))) break;
        }
        if (ok && j == nU - 1) mma_commit_w(&bar_done);
      }
     }
      mma_drain_w(&bar_drain, err);          // no MMA in flight once TMEM is freed
    }
  } else {
    // ---------------- softmax of tile X, columns [64 hh, 64 hh + 64) of each row
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t s_col = tmem + lane_off + X * 128 + 64 * hh;        // this half's S, then P
    const uint32_t o_col = tmem + lane_off + 256 + X * 128 + 64 * hh;  // this half's O
    const int bar_id = 1 + X * 4 + quarter;                            // the row pair's barrier
    const uint64_t scale2 = pk2(qk_scale2, qk_scale2);
    float m = -INFINITY, m_true = -INFINITY, l = 0.f;
    for (int j = 0; j < nU; ++j) {
      const int blk = sBlist[j];
      const bool sel = row_valid && next_id == blk;
      if (sel) {
        ++ptr;
        // issued here, consumed a block later (volatile: kept ahead of the waits)
        int nid = -1;
        if (ptr < topk_k)
          asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(nid) : "l"(src + ptr));
        next_id = nid;
      }
      const int ncol = !sel ? 0 : (blk < own ? 128 : pos - blk * 128 + 1);
      const int nc = min(64, max(0, ncol - 64 * hh));                 // valid columns of this half
      // S_X(j) done (and with it PV_X(j-1): O is settled and P may be rewritten).
      // The result is not used to leave the loop: the two warps of a row pair
      // must meet at the same named barriers, so after a timeout both keep
      // walking the blocks (every later wait returns at once) and the outputs
      // are meaningless, which msa_check_errors reports.
      mbar_wait_warp(&bar_sf[X], j & 1, err, &abort_s);               // warp-uniform
      tc_fence_after();
      // pass 1: this half's maximum of the raw scores over its valid columns
      // (scale > 0 commutes), then the row's through the partner thread
      float mr = -INFINITY;
      {
        uint32_t v[64];
        tmem_ld64(s_col, v);                                  // one round trip
        if (nc == 64) {
          // columns 0-3 seed four chains, 4-59 in steps of eight, 60-63 last
          float a0 = __uint_as_float(v[0]), a1 = __uint_as_float(v[1]);
          float a2 = __uint_as_float(v[2]), a3 = __uint_as_float(v[3]);
#pragma unroll
          for (int c = 4; c < 60; c += 8) {
            a0 = fmax3(a0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
            a1 = fmax3(a1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
            a2 = fmax3(a2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
            a3 = fmax3(a3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
          }
          a0 = fmax3(a0, __uint_as_float(v[60]), __uint_as_float(v[61]));
          a1 = fmax3(a1, __uint_as_float(v[62]), __uint_as_float(v[63]));
          mr = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        } else if (nc > 0) {
#pragma unroll
          for (int c = 0; c < 64; ++c) mr = (c < nc) ? fmaxf(mr, __uint_as_float(v[c])) : mr;
        }
      }
      xmax_s[j & 1][X][hh][rq] = mr;
      asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
      mr = fmaxf(mr, xmax_s[j & 1][X][hh ^ 1][rq]);
      const float mx = mr * qk_scale2;
      m_true = fmaxf(m_true, mx);
      const bool grow = mx > m + kRescale;                    // also when m == -inf
      const bool need_rescale = grow && (m > -INFINITY);
      if (__any_sync(0xffffffffu, need_rescale)) {
        const float alpha = need_rescale ? exp2f(m - mx) : 1.0f;
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          uint32_t v[16];
          tmem_ld16(o_col + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st16(o_col + c, v);
        }
        if (need_rescale) l *= alpha;
      }
      if (grow) m = mx;

      // pass 2: P = exp2(S * scale - m) as f16 pairs, 32 columns at a time,
      // each piece stored over S columns this thread has already read (and
      // once the lanes have reconverged: the TMEM store is warp-wide). Three
      // paths so the common full half carries no masking and an unselected
      // row costs no exponentials.
      const uint64_t negm = pk2(-m, -m);
      uint64_t acc0 = pk2(0.f, 0.f), acc1 = acc0;
      uint32_t wp[2][16];                                     // the two P pieces
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        uint32_t v[32];
        tmem_ld32(s_col + 32 * hq, v);
        uint32_t (&w)[16] = wp[hq];
        if (nc == 64) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 y = unpk2(ffma2(pk2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), scale2, negm));
            const float p0 = fast_exp2(y.x), p1 = fast_exp2(y.y);
            if (c & 2) acc1 = fadd2(acc1, pk2(p0, p1)); else acc0 = fadd2(acc0, pk2(p0, p1));
            w[c >> 1] = pack_f16x2(p0, p1);
          }
        } else if (nc > 0) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int cc = 32 * hq + c;
            const float p0 = cc < nc ? fast_exp2(fmaf(__uint_as_float(v[c]), qk_scale2, -m)) : 0.f;
            const float p1 = cc + 1 < nc ? fast_exp2(fmaf(__uint_as_float(v[c + 1]), qk_scale2, -m)) : 0.f;
            acc0 = fadd2(acc0, pk2(p0, p1));
            w[c >> 1] = pack_f16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) w[c] = 0u;
        }
        tmem_st16_async(s_col + 16 * hq, w);
      }
      tmem_wait_st2(wp[0], wp[1]);
      {
        const float2 a2 = unpk2(fadd2(acc0, acc1));
        l += a2.x + a2.y;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pf[X]);
    }

    // ---------------- epilogue: O / (l + sink), lse, max_logit
    if (nU > 0) mbar_wait_ab(&bar_done, 0, err, &abort_s);
    tc_fence_after();
    lsum_s[X][hh][rq] = l;
    asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
    const float lrow = l + lsum_s[X][hh ^ 1][rq];
    const float sig2 = (sink != nullptr && row_valid) ? sink_scale2 * __ldg(sink + h) : -INFINITY;
    const float M = fmaxf(m, sig2);
    const float a = (m == -INFINITY) ? 0.f : exp2f(m - M);
    const float ls = (sig2 == -INFINITY) ? 0.f : exp2f(sig2 - M);
    const float Z = lrow * a + ls;
    const float so = (Z > 0.f && nU > 0) ? (a / Z) * v_scale : 0.f;
    uint16_t* orow = out + (size_t(t) * Hq + h) * 128 + 64 * hh;
#pragma unroll
    for (int c = 0; c < 64; c += 32) {
      uint32_t v[32];
      if (nU > 0) {
        tmem_ld32(o_col + c, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;             // no block: O = 0
      }
      if (row_valid) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 o;
          o.x = pack_bf16x2(__uint_as_float(v[e + 0]) * so, __uint_as_float(v[e + 1]) * so);
          o.y = pack_bf16x2(__uint_as_float(v[e + 2]) * so, __uint_as_float(v[e + 3]) * so);
          o.z = pack_bf16x2(__uint_as_float(v[e + 4]) * so, __uint_as_float(v[e + 5]) * so);
          o.w = pack_bf16x2(__uint_as_float(v[e + 6]) * so, __uint_as_float(v[e + 7]) * so);
          *reinterpret_cast<uint4*>(orow + c + e) = o;
        }
      }
    }
    if (row_valid && hh == 0) {
      max_logit[size_t(t) * Hq + h] = m_true * kLn2;
      lse[size_t(t) * Hq + h] = (Z > 0.f) ? (M + log2f(Z)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ paged decode
// One CTA per (query token, kv head, chunk): the G q heads of the kv head
// share one walk over the ascending union of their index heads' selections;
// the union is cut into at most kDecMaxChunks balanced chunks (flash-decoding
// split) so that enough CTAs stream pages at once. Decode is bound by HBM
// (every selected K and V page is read once per (token, kv head)), so the
// kernel spends no work reshaping pages: per 128-key block
//   S^T = K Q^T       tcgen05 e4m3, A = the K page from TMA (M = 128 keys),
//                     B = the G query rows (N = 16), K = 128;
//   P                 softmax across TMEM lanes, one thread per key. The row
//                     max is lazy: a block only costs one vote and one barrier
//                     unless some score exceeds the running reference by
//                     2^8, when that row's exact block max is reduced;
//   O^T += V^T P^T    tcgen05 e4m3 twice, A = the V page straight from TMA
//                     read as an MN-major operand, B = P split into two e4m3
//                     terms (P rounded, then the rounded remainder): together
//                     they carry P to about 2^-8 of its value, where e4m3 P
//                     alone would cost ~2.5% relative error on O. P is taken
//                     relative to a reference 4 below the running max (so the
//                     key that set it has P = 16 and no P exceeds 2^8 < 448),
//                     which keeps the remainders of the large terms clear of
//                     e4m3's subnormal range. (Emulated on the CPU over 64
//                     sequences of the decode workload, two terms cost no more
//                     max-abs error than three: the bf16 rounding of O
//                     dominates.)
// A chunk leaves its unnormalised O, reference max, row sum and true max in
// the workspace; decode_combine_kernel merges the chunks and applies the sink.
constexpr int kDecChunk = 32;
constexpr int kDecKStages = 3;
// Three V stages: V(j) may only be loaded once PV(j - stages) has read its
// stage, so the V ring depth times a page's HBM latency sets the pace of a
// CTA (with two stages the MMA warp waited ~1k cycles per block for V).
constexpr int kDecVStages = 3;
constexpr int kDecMaxList = 1024;   // union entries kept (<= 16 index heads x 64)
constexpr int kDKOff = 0;           // kDecKStages x 16 KB K pages (SW128)
constexpr int kDVOff = 49152;       // kDecVStages x 16 KB V pages (SW128)
constexpr int kDPOff = 98304;       // 2 x 2 terms x 2 KB: 16 rows x 128 keys e4m3 (SW128)
constexpr int kDBitsOff = 98304;    // setup only: 16 bitmaps x 2048 bits (aliases P)
constexpr int kDUnionOff = 102400;  // setup only: 64 union words (aliases P)
constexpr int kDPreOff = 102656;    // setup only: 64 popcount prefixes (aliases P)
constexpr int kDRowMaskOff = 102912;   // setup only: 16 row masks (aliases P)
constexpr int kDQOff = 106496;      // 16 rows x 128 e4m3
constexpr int kDListOff = 108544;   // union list (int16)
constexpr int kDMaskOff = 110592;   // per-entry row mask (uint16)
constexpr int kDecodeSmem = 112640 + 1024;   // two CTAs per SM
constexpr float kDecLimit = 8.0f;   // log2 of the largest P before the reference moves
constexpr float kDecHead = 4.0f;    // log2 of P at the key that set the reference
constexpr uint32_t kIdescDec = idesc_f32(128, 16);
constexpr uint32_t kIdescDecT = idesc_f32(128, 16) | (1u << 15);   // A MN-major

struct DecodePartial {   // per (token, kv head, chunk, row)
  float m, l, m_true, pad;
};

// The most index heads one kv group's query heads read (a group of G heads
// starting at head g*G spans index heads (g*G)/hpi .. (g*G+G-1)/hpi).
inline int dec_group_index_heads(int Hq, int Hkv, int Hidx) {
  const int G = Hq / Hkv, hpi = Hq / Hidx;
  int n = 1;
  for (int g = 0; g < Hkv; ++g) n = max(n, (g * G + G - 1) / hpi - (g * G) / hpi + 1);
  return n;
}

__host__ __device__ inline int dec_max_chunks(int n_idx_per_group, int topk, int max_pages) {
  const int cap = min(max_pages, n_idx_per_group * topk);
  return max(1, (cap + kDecChunk - 1) / kDecChunk);
}

constexpr int kDecThreads = 320;   // producer, MMA, 8 softmax warps

// RPT = query rows per softmax thread: the 16 MMA columns (query rows) are
// split between the two softmax warps of each TMEM lane quarter, rows
// RPT*rh .. RPT*rh+RPT-1 for warp half rh; RPT = 4 when G <= 8.
template <int RPT>
__global__ void __launch_bounds__(kDecThreads, 2)
attn_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q,
                   const int32_t* __restrict__ topk, float qk_scale2, int B, int T, int Hq,
                   int Hkv, int Hidx, int topk_k, int max_pages, int num_pages, int max_chunks,
                   float* __restrict__ part_o, DecodePartial* __restrict__ part_s,
                   int* __restrict__ n_chunks_out, unsigned* err) {
  pdl_wait();      // queries, caches and top-k may come from earlier kernels
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_q, bar_kf[kDecKStages], bar_ke[kDecKStages], bar_vf[kDecVStages],
      bar_ve[kDecVStages], bar_sf[2], bar_se[2], bar_pf[2], bar_pe[2], bar_pv, bar_done, bar_vt,
      bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int n_union_s;
  __shared__ int abort_s;
  __shared__ uint32_t flags[2][8];
  __shared__ float red[2][4][16];
  __shared__ float mrow[16];

  const int G = Hq / Hkv;
  const int c = blockIdx.x % max_chunks;
  const int g = (blockIdx.x / max_chunks) % Hkv;
  const int t = blockIdx.x / (max_chunks * Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // one query per sequence (the decode launch: q_len <= 1, T == B) makes
  // token t sequence t; otherwise search the query offsets
  const int b = (T == B) ? t : find_sequence(cu_q, B, t);
  const int qlen = cu_q[b + 1] - cu_q[b];
  const int L = seq_lens[b];
  const int pos = L - qlen + (t - cu_q[b]);
  const size_t unit = size_t(t) * Hkv + g;
  if (pos < 0 || pos >= max_pages * 128 || L > max_pages * 128) {
    if (tid == 0 && c == 0) { atomicOr(err, MSA_DEVERR_DATA); n_chunks_out[unit] = 0; }
    return;
  }
  const int own = pos >> 7;
  const int hpi = Hq / Hidx;                       // q heads per index head
  const int i_first = (g * G) / hpi;
  const int n_idx = (g * G + G - 1) / hpi - i_first + 1;

  int16_t* sList = reinterpret_cast<int16_t*>(smem + kDListOff);
  uint16_t* sMask = reinterpret_cast<uint16_t*>(smem + kDMaskOff);
  uint32_t* sBits = reinterpret_cast<uint32_t*>(smem + kDBitsOff);
  uint32_t* sUnion = reinterpret_cast<uint32_t*>(smem + kDUnionOff);
  int* sPre = reinterpret_cast<int*>(smem + kDPreOff);
  uint16_t* sRowMask = reinterpret_cast<uint16_t*>(smem + kDRowMaskOff);
  for (int x = tid; x < n_idx * 64; x += kDecThreads) sBits[x] = 0u;
  if (tid < 16) sRowMask[tid] = 0;
  __syncthreads();
  if (tid == 0)                                    // rows of the group fed by each index head
    for (int r = 0; r < G; ++r) sRowMask[(g * G + r) / hpi - i_first] |= uint16_t(1u << r);
  for (int x = tid; x < n_idx * topk_k; x += kDecThreads) {
    const int il = x / topk_k;
    const int id = __ldg(topk + (size_t(i_first + il) * T + t) * topk_k + (x - il * topk_k));
    if (id < 0) continue;
    if (id > own) { atomicOr(err, MSA_DEVERR_DATA); continue; }
    atomicOr(&sBits[il * 64 + (id >> 5)], 1u << (id & 31));
  }
  __syncthreads();
  if (warp == 0) {     // union words (lane: words 2 lane, 2 lane + 1) and their popcount prefix
    uint32_t u0 = 0, u1 = 0;
    for (int il = 0; il < n_idx; ++il) {
      u0 |= sBits[il * 64 + 2 * lane];
      u1 |= sBits[il * 64 + 2 * lane + 1];
    }
    const int c0 = __popc(u0), c1 = __popc(u1);
    int incl = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    sUnion[2 * lane] = u0;
    sUnion[2 * lane + 1] = u1;
    sPre[2 * lane] = incl - c0 - c1;
    sPre[2 * lane + 1] = incl - c1;
    if (lane == 31) n_union_s = min(incl, kDecMaxList);
  }
  __syncthreads();
  // every thread places the union's blocks: ascending list and per-entry row mask
  for (int x = tid; x < 64 * 32; x += kDecThreads) {
    const int w = x >> 5, k = x & 31;
    const uint32_t u = sUnion[w];
    if (!((u >> k) & 1u)) continue;
    const int off = sPre[w] + __popc(u & ((1u << k) - 1u));
    if (off >= kDecMaxList) continue;
    uint32_t m = 0;
    for (int il = 0; il < n_idx; ++il)
      if ((sBits[il * 64 + w] >> k) & 1u) m |= sRowMask[il];
    sList[off] = int16_t(w * 32 + k);
    sMask[off] = uint16_t(m);
  }
  __syncthreads();                                   // the bitmaps (over P) are dead now
  const int nU = n_union_s;
  const int nch = min(max_chunks, (nU + kDecChunk - 1) / kDecChunk);
  if (c == 0 && tid == 0) n_chunks_out[unit] = nch;
  if (c >= nch) return;
  const int cs = (nU + nch - 1) / nch;
  const int j0 = c * cs, n = min(nU, j0 + cs) - j0;

  if (tid == 0) {
    abort_s = initial_abort(err);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_drain, 1);
    for (int s = 0; s < kDecKStages; ++s) { mbar_init(&bar_kf[s], 1); mbar_init(&bar_ke[s], 1); }
    for (int s = 0; s < kDecVStages; ++s) { mbar_init(&bar_vf[s], 1); mbar_init(&bar_ve[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_sf[s], 1); mbar_init(&bar_se[s], 8);
      mbar_init(&bar_pf[s], 8); mbar_init(&bar_pe[s], 1);
    }
    mbar_init(&bar_pv, 1);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_vt, 1);
    fence_barrier_init();
  }
  if (warp == 1) { tmem_alloc(&tmem_base_s, 64); tmem_relinquish(); }
  __syncthreads();
  pdl_trigger();   // after this block's tensor-memory allocation
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;          // S^T buffers at cols 0, 16; O^T at 32

  if (warp == 0) {
    // Producer. Rows of the last page past seq_len hold whatever the cache
    // pool holds there (possibly e4m3 NaN); PV would turn 0 * NaN into NaN,
    // so that page's V is landed on its own barrier, its tail rows are
    // zeroed by the warp, and only then is it handed to the MMA.
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_q, 16 * 128);
      tma_load_2d(smem + kDQOff, &tm_q, &bar_q, 0, t * Hq + g * G);
    }
    const int32_t* prow = page_table + size_t(b) * max_pages;
    const int tail_blk = (L - 1) >> 7, tail_rows = L - tail_blk * 128;
    int nk = 0, nv = 0, nvt = 0;                    // phases armed per ring (lane 0's copies)
    for (int jj = 0; jj < n; ++jj) {
      const int s = jj % kDecKStages, sv = jj % kDecVStages;
      const uint32_t ph = ((jj / kDecKStages) & 1) ^ 1, phv = ((jj / kDecVStages) & 1) ^ 1;
      const int blk = sList[j0 + jj];
      int page = __ldg(prow + blk);
      if (page < 0 || page >= num_pages) {
        if (lane == 0) atomicOr(err, MSA_DEVERR_DATA);
        page = 0;
      }
      const int row0 = (page * Hkv + g) * 128;
      uint8_t* vs = smem + kDVOff + sv * 16384;
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait_ab(&bar_ke[s], ph, err, &abort_s);
        if (ok) {
          mbar_arrive_expect_tx(&bar_kf[s], 16384);
          tma_load_2d(smem + kDKOff + s * 16384, &tm_k, &bar_kf[s], 0, row0);
          ++nk;
          ok = mbar_wait_ab(&bar_ve[sv], phv, err, &abort_s);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (blk == tail_blk && tail_rows < 128) {   // at most once per CTA
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_vt, 16384);
          tma_load_2d(vs, &tm_v, &bar_vt, 0, row0);
          nvt = 1;
        }
        if (!mbar_wait_warp(&bar_vt, 0, err, &abort_s)) break;
        uint4* rows = reinterpret_cast<uint4*>(vs + tail_rows * 128);   // swizzle stays inside a row
        for (int x = lane; x < (128 - tail_rows) * 8; x += 32) rows[x] = make_uint4(0u, 0u, 0u, 0u);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_vf[sv]);
      } else if (lane == 0) {
        mbar_arrive_expect_tx(&bar_vf[sv], 16384);
        tma_load_2d(vs, &tm_v, &bar_vf[sv], 0, row0);
      }
      ++nv;
    }
    if (lane == 0) {            // exit-path drain (a no-op unless a wait gave up)
      mbar_wait(&bar_q, 0, err);
      mbar_drain_ring(bar_kf, kDecKStages, nk, err);
      mbar_drain_ring(bar_vf, kDecVStages, nv, err);
      if (nvt) mbar_wait(&bar_vt, 0, err);
    }
  } else if (warp == 1) {
    if (mbar_wait_warp(&bar_q, 0, err, &abort_s)) {        // whole warp, elected issue
      const uint32_t sq = smem_addr(smem + kDQOff);
      auto issue_s = [&](int jj) -> bool {
        const int s = jj % kDecKStages, sb = jj & 1;
        if (!mbar_wait_warp(&bar_kf[s], (jj / kDecKStages) & 1, err, &abort_s)) return false;
        if (!mbar_wait_warp(&bar_se[sb], ((jj >> 1) & 1) ^ 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t sk = smem_addr(smem + kDKOff + s * 16384);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_e4m3_w(tmem + sb * 16, sdesc_kmajor(sk + 32 * k, 128), sdesc_kmajor(sq + 32 * k, 128),
                   kIdescDec, k > 0);
        mma_commit_w(&bar_ke[s]);
        mma_commit_w(&bar_sf[sb]);
        return true;
      };
      bool ok = n > 0 && issue_s(0);
      for (int jj = 0; ok && jj < n; ++jj) {
        if (jj + 1 < n && !(ok = issue_s(jj + 1))) break;
        const int s = jj % kDecVStages, sb = jj & 1;
        if (!mbar_wait_warp(&bar_pf[sb], (jj >> 1) & 1, err, &abort_s) ||
            !mbar_wait_warp(&bar_vf[s], (jj / kDecVStages) & 1, err, &abort_s))
          break;
        tc_fence_after();
        const uint32_t sv = smem_addr(smem + kDVOff + s * 16384);
        const uint32_t sp = smem_addr(smem + kDPOff + sb * 4096);
#pragma unroll
        for (int part = 0; part < 2; ++part)          // the two terms of P
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_e4m3_w(tmem + 32, sdesc_kmajor(sv + 4096 * k, 128),
                     sdesc_kmajor(sp + part * 2048 + 32 * k, 128), kIdescDecT,
                     (jj > 0 || part > 0 || k > 0) ? 1u : 0u);
        mma_commit_w(&bar_ve[s]);
        mma_commit_w(&bar_pe[sb]);
        mma_commit_w(&bar_pv);
        if (jj == n - 1) mma_commit_w(&bar_done);
      }
    }
    mma_drain_w(&bar_drain, err);            // no MMA in flight once TMEM is freed
  } else {
    // ---------------- softmax: thread = key lane of S^T and d lane of O^T,
    // query rows r0 .. r0+RPT-1
    const int q4 = warp & 3, rh = (warp - 2) >> 2, wi = warp - 2;
    const int r0 = rh * RPT;
    const int key = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    float m[RPT], mt[RPT], ls[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) { m[i] = -INFINITY; mt[i] = -INFINITY; ls[i] = 0.f; }
    for (int jj = 0; jj < n; ++jj) {
      const int sb = jj & 1;
      const uint32_t ph = (jj >> 1) & 1;
      const int blk = sList[j0 + jj];
      const uint32_t rmask = sMask[j0 + jj];
      const bool kvalid = blk * 128 + key <= pos;
      mbar_wait_ab(&bar_sf[sb], ph, err, &abort_s);
      tc_fence_after();
      uint32_t v[RPT];
      tmem_ldn<RPT>(tmem + lane_off + sb * 16 + r0, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_se[sb]);
      float x[RPT];
      uint32_t over = 0;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = r0 + i;
        x[i] = (r < G && kvalid && ((rmask >> r) & 1u)) ? __uint_as_float(v[i]) * qk_scale2 : -INFINITY;
        mt[i] = fmaxf(mt[i], x[i]);
        over |= (x[i] > m[i] + kDecLimit) ? (1u << r) : 0u;
      }
      over = __reduce_or_sync(0xffffffffu, over);
      if (lane == 0) flags[sb][wi] = over;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      uint32_t E = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) E |= flags[sb][w];
      float alpha[RPT];
      bool need = false;
      if (E != 0) {                                // uniform: some row's reference must move
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          if ((E >> (r0 + i)) & 1u) {
            float mr = x[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
            if (lane == 0) red[sb][q4][r0 + i] = mr;
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const int r = r0 + i;
          alpha[i] = 1.0f;
          if ((E >> r) & 1u) {
            const float bm = fmaxf(fmaxf(red[sb][0][r], red[sb][1][r]), fmaxf(red[sb][2][r], red[sb][3][r])) - kDecHead;
            if (m[i] > -INFINITY) { alpha[i] = exp2f(m[i] - bm); need = true; }
            m[i] = bm;
          }
        }
      }
      // P buffer sb is free once PV_{jj-2} is done (also bounds the pv parity below)
      mbar_wait_ab(&bar_pe[sb], ph ^ 1, err, &abort_s);
      if (__any_sync(0xffffffffu, need)) {         // every thread of the warp holds the same m
        mbar_wait_ab(&bar_pv, (jj - 1) & 1, err, &abort_s);
        tc_fence_after();
        uint32_t o[RPT];
        tmem_ldn<RPT>(tmem + lane_off + 32 + r0, o);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const float al = need ? alpha[i] : 1.0f;
          o[i] = __float_as_uint(__uint_as_float(o[i]) * al);
          ls[i] *= al;
        }
        tmem_stn<RPT>(tmem + lane_off + 32 + r0, o);
        tc_fence_before();
      }
      // P -> two e4m3 terms, into row r, column `key` of each operand
      uint8_t* pbuf = smem + kDPOff + sb * 4096;
      const uint32_t kc = uint32_t(key >> 4), kb = uint32_t(key & 15);
#pragma unroll
      for (int i = 0; i < RPT; i += 2) {
        const int r = r0 + i;
        float p0 = fast_exp2(x[i] - (m[i] == -INFINITY ? 0.f : m[i]));
        float p1 = fast_exp2(x[i + 1] - (m[i + 1] == -INFINITY ? 0.f : m[i + 1]));
        ls[i] += p0;
        ls[i + 1] += p1;
        const uint32_t o0 = swz_offset(uint32_t(r), kc, 128) + kb, o1 = swz_offset(uint32_t(r + 1), kc, 128) + kb;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint16_t e = e4m3x2_from_f32(p0, p1);
          pbuf[part * 2048 + o0] = uint8_t(e & 0xFF);
          pbuf[part * 2048 + o1] = uint8_t(e >> 8);
          if (part < 1) {                          // the remainder is exact in fp32
            const uint32_t eh = e4m3x2_to_f16x2(e);
            const float2 ef = __half22float2(*reinterpret_cast<const __half2*>(&eh));
            p0 -= ef.x;
            p1 -= ef.y;
          }
        }
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pf[sb]);
    }
    // chunk result: O^T columns (rows) for this thread's d lane, and row state
    if (n > 0) mbar_wait_ab(&bar_done, 0, err, &abort_s);
    tc_fence_after();
    uint32_t o[RPT];
    tmem_ldn<RPT>(tmem + lane_off + 32 + r0, o);
    const size_t base = (unit * max_chunks + c) * G;
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      if (r0 + i < G) part_o[(base + r0 + i) * 128 + key] = __uint_as_float(o[i]);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      float sr = ls[i], mr = mt[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sr += __shfl_xor_sync(0xffffffffu, sr, off);
        mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
      }
      if (lane == 0) { red[0][q4][r0 + i] = sr; red[1][q4][r0 + i] = mr; }
      if (lane == 0 && q4 == 0) mrow[r0 + i] = m[i];
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (tid - 64 < G) {
      const int r = tid - 64;
      part_s[base + r] = DecodePartial{mrow[r], red[0][0][r] + red[0][1][r] + red[0][2][r] + red[0][3][r],
                                       fmaxf(fmaxf(red[1][0][r], red[1][1][r]), fmaxf(red[1][2][r], red[1][3][r])),
                                       0.f};
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 64);
}

// Merges the chunks of each (token, kv head) and applies the sink. One
// thread per output element (query row r of the group, column d), one pass
// over the chunks with a running maximum; the chunks' loads do not depend on
// one another, so they are all in flight together.
__global__ void __launch_bounds__(1024)
decode_combine_kernel(const float* __restrict__ part_o, const DecodePartial* __restrict__ part_s,
                      const int* __restrict__ n_chunks, const float* __restrict__ sink,
                      float sink_scale2, float v_scale, int Hq, int Hkv, int max_chunks,
                      uint16_t* __restrict__ out, float* __restrict__ max_logit,
                      float* __restrict__ lse) {
  pdl_wait();      // the chunk partials come from the decode kernel
  pdl_trigger();
  const int t = blockIdx.x / Hkv, g = blockIdx.x % Hkv;
  const int G = Hq / Hkv;
  const size_t unit = size_t(t) * Hkv + g;
  const int nch = n_chunks[unit];
  for (int x = threadIdx.x; x < G * 128; x += blockDim.x) {
    const int r = x >> 7, d = x & 127;
    const int h = g * G + r;
    float M = -INFINITY, mt = -INFINITY, Z = 0.f, acc = 0.f;
#pragma unroll 4
    for (int c = 0; c < nch; ++c) {
      const size_t k = (unit * max_chunks + c) * G + r;
      const DecodePartial ps = part_s[k];
      const float po = part_o[k * 128 + d];
      mt = fmaxf(mt, ps.m_true);
      if (ps.m == -INFINITY) continue;
      const float Mn = fmaxf(M, ps.m);
      const float a0 = (M == -INFINITY) ? 0.f : exp2f(M - Mn), a1 = exp2f(ps.m - Mn);
      Z = Z * a0 + ps.l * a1;
      acc = acc * a0 + po * a1;
      M = Mn;
    }
    const float sig2 = sink != nullptr ? sink_scale2 * __ldg(sink + h) : -INFINITY;
    const float Mz = fmaxf(M, sig2);
    const float aM = (M == -INFINITY) ? 0.f : exp2f(M - Mz);
    Z = Z * aM + ((sig2 == -INFINITY) ? 0.f : exp2f(sig2 - Mz));
    acc *= aM;
    const float o = Z > 0.f ? acc / Z * v_scale : 0.f;
    out[(size_t(t) * Hq + h) * 128 + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
    if (d == 0) {
      max_logit[size_t(t) * Hq + h] = mt * kLn2;
      lse[size_t(t) * Hq + h] = Z > 0.f ? (Mz + log2f(Z)) * kLn2 : -INFINITY;
    }
  }
}

cudaError_t launch_decode(const AttnArgs& a, cudaStream_t stream, const char** why) {
  const int G = a.Hq / a.Hkv;
  const int n_idx = dec_group_index_heads(a.Hq, a.Hkv, a.Hidx);
  const int mc = dec_max_chunks(n_idx, a.topk_k, a.max_pages);
  const size_t units = size_t(a.T) * a.Hkv * mc * G;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  float* part_o = reinterpret_cast<float*>(ws);
  DecodePartial* part_s = reinterpret_cast<DecodePartial*>(ws + align256(units * 128 * sizeof(float)));
  int* n_chunks = reinterpret_cast<int*>(ws + align256(units * 128 * sizeof(float)) +
                                         align256(units * sizeof(DecodePartial)));
  CUtensorMap tm_q, tm_k, tm_v;
  {
    const uint64_t dims[2] = {128, uint64_t(a.T) * a.Hq};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {128, 16};
    if (!encode_tensor_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {128, uint64_t(a.num_pages) * a.Hkv * 128};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {128, 128};
    if (!encode_tensor_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.k_cache, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, why) ||
        !encode_tensor_map(&tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.v_cache, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  auto kern = G <= 8 ? attn_decode_kernel<4> : attn_decode_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeSmem);
  if (e != cudaSuccess) return e;
  profile_mark(stream, 0);
  e = launch_pdl(kern, a.T * a.Hkv * mc, kDecThreads, kDecodeSmem, stream, tm_q, tm_k, tm_v,
                 a.page_table, a.seq_lens, a.cu_q, a.topk, a.c_qk * kLog2e, a.B, a.T, a.Hq, a.Hkv,
                 a.Hidx, a.topk_k, a.max_pages, a.num_pages, mc, part_o, part_s, n_chunks, a.err);
  profile_mark(stream, 1);
  if (e != cudaSuccess) return e;
  const int cthreads = G * 128 < 1024 ? G * 128 : 1024;
  return launch_pdl(decode_combine_kernel, a.T * a.Hkv, cthreads, 0, stream, part_o, part_s, n_chunks,
                    a.sink, a.c_sink * kLog2e, a.v_scale, a.Hq, a.Hkv, mc, a.out, a.max_logit,
                    a.lse);
}

}  // namespace

size_t attn_workspace_bytes(int B, int T, int max_q_len, int Hq, int Hkv, int Hidx, int topk,
                            int max_pages) {
  if (max_q_len <= 1) {
    const int G = Hq / Hkv;
    const int n_idx = dec_group_index_heads(Hq, Hkv, Hidx);   // index heads one kv group reads
    const int mc = dec_max_chunks(n_idx, topk, max_pages);
    const size_t units = size_t(T) * Hkv * mc * G;
    return align256(units * 128 * sizeof(float)) + align256(units * sizeof(DecodePartial)) +
           align256(size_t(T) * Hkv * sizeof(int)) + 256;
  }
  const size_t img = size_t(B) * max_pages * Hkv * 32768;
  return img + align256(size_t(T + B + 1) * sizeof(TileInfo)) + 256;
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream, const char** why) {
  if (a.max_pages > 2048) {
    *why = "max_pages must be <= 2048";
    return cudaErrorNotSupported;
  }
  const int G = a.Hq / a.Hkv;
  if (a.max_q_len == 1) return launch_decode(a, stream, why);
  const int toks = 128 / G;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const size_t img_bytes = size_t(a.B) * a.max_pages * a.Hkv * 32768;
  TileInfo* tiles = reinterpret_cast<TileInfo*>(ws + img_bytes);
  const int max_tiles = a.T + a.B + 1;
  int* n_tiles = reinterpret_cast<int*>(ws + img_bytes + align256(size_t(max_tiles) * sizeof(TileInfo)));

  CUtensorMap tm_q, tm_k;
  {
    const uint64_t dims[3] = {128, uint64_t(a.Hq), uint64_t(a.T)};
    const uint64_t strides[2] = {128, uint64_t(a.Hq) * 128};
    const uint32_t box[3] = {128, uint32_t(G), uint32_t(toks)};
    if (!encode_tensor_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.q, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {128, uint64_t(a.num_pages) * a.Hkv * 128};
    const uint64_t strides[1] = {128};
    const uint32_t box[2] = {128, 128};
    if (!encode_tensor_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.k_cache, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = launch_pdl(plan_tiles_kernel, 1, 256, 0, stream, a.seq_lens, a.cu_q, a.B, 2 * toks,
                             a.max_pages, max_tiles, tiles, n_tiles, a.err);
  if (e != cudaSuccess) return e;
  e = launch_pdl(vt_convert_kernel, dim3(a.max_pages, a.B, a.Hkv), 256, 0, stream, a.v_cache,
                 a.page_table, a.seq_lens, a.Hkv, a.max_pages, a.num_pages, ws, a.err);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefillSmem);
  if (e != cudaSuccess) return e;
  const int grid = ((a.T + 2 * toks - 1) / (2 * toks) + a.B) * a.Hkv;
  profile_mark(stream, 0);
  e = launch_pdl(attn_prefill_kernel, grid, kPrefillThreads, kPrefillSmem, stream, tm_q, tm_k,
                 static_cast<const uint8_t*>(ws), a.page_table, static_cast<const TileInfo*>(tiles),
                 static_cast<const int*>(n_tiles), a.topk, a.sink, a.c_qk * kLog2e,
                 a.c_sink * kLog2e, a.v_scale, a.T, a.Hq, a.Hkv, a.Hidx, toks, a.topk_k,
                 a.max_pages, a.num_pages, a.out, a.max_logit, a.lse, a.err);
  profile_mark(stream, 1);
  return e;
}

}  // namespace msa

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

// shared memory (byte offsets from a 1024-aligned base)
constexpr int kQOff = 0;             // 128 rows x 128 e4m3             16 KB
constexpr int kKOff = 16384;         // 2 stages x 128 keys x 128 e4m3  32 KB
constexpr int kVOff = 49152;         // 2 stages x V^T f16 image        64 KB
constexpr int kPOff = 114688;        // 2 buffers x 128 x 128 f16       64 KB
constexpr int kIdsOff = 180224;      // 128 rows x 64 block ids (int16) 16 KB
constexpr int kBlistOff = 196608;    // union block list (int16)         4 KB
constexpr int kBitsOff = 200704;     // union bitmap, 2048 bits         256 B
constexpr int kPrefillSmem = 200960 + 1024;
constexpr int kMaxIds = 64;

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
__global__ void __launch_bounds__(192, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const uint8_t* __restrict__ vt_img, const int32_t* __restrict__ page_table,
                    const TileInfo* __restrict__ tiles, const int* __restrict__ n_tiles_p,
                    const int32_t* __restrict__ topk, const float* __restrict__ sink,
                    float qk_scale2, float sink_scale2, float v_scale, int T, int Hq, int Hkv,
                    int Hidx, int toks, int topk_k, int max_pages, int num_pages,
                    uint16_t* __restrict__ out, float* __restrict__ max_logit,
                    float* __restrict__ lse, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_q, bar_kf[2], bar_ke[2], bar_vf[2], bar_ve[2], bar_sf[2], bar_se[2],
      bar_pf[2], bar_pe[2], bar_pv;
  __shared__ uint32_t tmem_base_s;
  __shared__ int n_union_s;

  const int n_tiles = *n_tiles_p;
  const int tile_rank = blockIdx.x / Hkv;
  if (tile_rank >= n_tiles) return;
  const int g = blockIdx.x % Hkv;
  const TileInfo ti = tiles[n_tiles - 1 - tile_rank];     // latest (longest) tiles first
  const int G = Hq / Hkv;
  const int n_tok = min(toks, ti.t_end - ti.t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int16_t* sIds = reinterpret_cast<int16_t*>(smem + kIdsOff);
  int16_t* sBlist = reinterpret_cast<int16_t*>(smem + kBlistOff);
  uint32_t* sBits = reinterpret_cast<uint32_t*>(smem + kBitsOff);

  if (tid < 64) sBits[tid] = 0u;
  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_kf[s], 1); mbar_init(&bar_ke[s], 1);
      mbar_init(&bar_vf[s], 1); mbar_init(&bar_ve[s], 1);
      mbar_init(&bar_sf[s], 1); mbar_init(&bar_se[s], 4);
      mbar_init(&bar_pf[s], 4); mbar_init(&bar_pe[s], 1);
    }
    mbar_init(&bar_pv, 1);
    fence_barrier_init();
  }
  if (warp == 1) { tmem_alloc(&tmem_base_s, 512); tmem_relinquish(); }
  __syncthreads();

  // ---- each softmax thread owns one row: (token t0 + row/G, head g*G + row%G)
  const bool is_softmax = warp >= 2;
  const int row = (warp & 3) * 32 + lane;
  int n_ids = 0, own = -1, pos = -1, h = 0, t = 0;
  bool row_valid = false;
  if (is_softmax) {
    const int tl = row / G;
    t = ti.t0 + tl;
    h = g * G + row % G;
    row_valid = tl < n_tok;
    if (row_valid) {
      pos = ti.p0 + tl;
      own = pos >> 7;
      const int32_t* src = topk + (size_t(h / (Hq / Hidx)) * T + t) * topk_k;
      int last = -1;
      for (int k = 0; k < topk_k; ++k) {
        const int id = __ldg(src + k);
        if (id < 0) continue;                                   // -1 padding
        if (id <= last || id > own) { atomicOr(err, MSA_DEVERR_DATA); continue; }
        sIds[row * kMaxIds + n_ids++] = int16_t(id);
        atomicOr(&sBits[id >> 5], 1u << (id & 31));
        last = id;
      }
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

  if (warp == 0) {
    // ---------------- producer: Q once, then K pages (TMA) and V^T images (bulk)
    if (lane == 0 && nU > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(&bar_q, 16384);
      tma_load_3d(smem + kQOff, &tm_q, &bar_q, 0, g * G, ti.t0);
      const int32_t* prow = page_table + size_t(ti.b) * max_pages;
      for (int j = 0; j < nU; ++j) {
        const int s = j & 1;
        const uint32_t ph = ((j >> 1) & 1) ^ 1;
        const int blk = sBlist[j];
        int page = __ldg(prow + blk);
        if (page < 0 || page >= num_pages) { atomicOr(err, MSA_DEVERR_DATA); page = 0; }
        if (!mbar_wait(&bar_ke[s], ph, err)) break;
        mbar_arrive_expect_tx(&bar_kf[s], 16384);
        tma_load_2d(smem + kKOff + s * 16384, &tm_k, &bar_kf[s], 0, (page * Hkv + g) * 128);
        if (!mbar_wait(&bar_ve[s], ph, err)) break;
        mbar_arrive_expect_tx(&bar_vf[s], 32768);
        bulk_load(smem + kVOff + s * 32768,
                  vt_img + ((size_t(ti.b) * max_pages + blk) * Hkv + g) * 32768, 32768, &bar_vf[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue: S_{j+1} is issued before PV_j
    if (lane == 0 && nU > 0 && mbar_wait(&bar_q, 0, err)) {
      const uint32_t sq = smem_addr(smem + kQOff);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&bar_kf[s], ph, err)) return false;
        if (!mbar_wait(&bar_se[s], ph ^ 1, err)) return false;
        tc_fence_after();
        const uint32_t sk = smem_addr(smem + kKOff + s * 16384);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_e4m3(tmem + s * 128, sdesc_kmajor(sq + 32 * k, 128), sdesc_kmajor(sk + 32 * k, 128),
                   kIdescQK, k > 0);
        mma_commit(&bar_ke[s]);
        mma_commit(&bar_sf[s]);
        return true;
      };
      bool ok = issue_s(0);
      for (int j = 0; ok && j < nU; ++j) {
        if (j + 1 < nU && !(ok = issue_s(j + 1))) break;
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&bar_pf[s], ph, err) || !mbar_wait(&bar_vf[s], ph, err)) break;
        tc_fence_after();
        const uint32_t sp = smem_addr(smem + kPOff + s * 32768);
        const uint32_t sv = smem_addr(smem + kVOff + s * 32768);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_f16(tmem + 256, sdesc_kmajor(sp + off, 128), sdesc_kmajor(sv + off, 128), kIdescPV,
                  (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&bar_ve[s]);
        mma_commit(&bar_pe[s]);
        mma_commit(&bar_pv);
      }
    }
  } else {
    // ---------------- softmax: one thread per row (TMEM lane `row`)
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    uint8_t* p_row_base = smem + kPOff;
    float m = -INFINITY, m_true = -INFINITY, l = 0.f;
    int ptr = 0;
    for (int j = 0; j < nU; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      const int blk = sBlist[j];
      const bool sel = ptr < n_ids && sIds[row * kMaxIds + ptr] == blk;
      ptr += sel ? 1 : 0;
      const int ncol = !sel ? 0 : (blk < own ? 128 : pos - blk * 128 + 1);
      if (!mbar_wait(&bar_sf[s], ph, err)) break;
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + s * 128 + c, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_se[s]);

      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        x[c] = (c < ncol) ? x[c] * qk_scale2 : -INFINITY;
        mx = fmaxf(mx, x[c]);
      }
      m_true = fmaxf(m_true, mx);
      const bool grow = mx > m + kRescale;                    // also when m == -inf
      const bool need_rescale = grow && (m > -INFINITY);
      if (__any_sync(0xffffffffu, need_rescale)) {
        // O holds PV_0..PV_{j-1}: wait for the last one, then scale this warp's rows
        if (!mbar_wait(&bar_pv, (j - 1) & 1, err)) break;
        tc_fence_after();
        const float alpha = need_rescale ? exp2f(m - mx) : 1.0f;
#pragma unroll
        for (int c = 0; c < 128; c += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_off + 256 + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st16(tmem + lane_off + 256 + c, v);
        }
        tc_fence_before();
        if (need_rescale) l *= alpha;
      }
      if (grow) m = mx;

      // P row (f16) into the swizzled A operand of buffer s, once PV_{j-2} is done
      if (!mbar_wait(&bar_pe[s], ph ^ 1, err)) break;
      const float mref = (m == -INFINITY) ? 0.f : m;
      uint8_t* pbuf = p_row_base + s * 32768;
      float sum = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = fast_exp2(x[c8 * 8 + 2 * e] - mref);
          const float p1 = fast_exp2(x[c8 * 8 + 2 * e + 1] - mref);
          sum += p0 + p1;
          w[e] = pack_f16x2(p0, p1);
        }
        *reinterpret_cast<uint4*>(pbuf + (c8 >> 3) * 16384 + swz_offset(row, c8 & 7, 128)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      l += sum;
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pf[s]);
    }

    // ---------------- epilogue: O / (l + sink), lse, max_logit
    if (nU > 0) mbar_wait(&bar_pv, (nU - 1) & 1, err);
    tc_fence_after();
    const float sig2 = (sink != nullptr && row_valid) ? sink_scale2 * __ldg(sink + h) : -INFINITY;
    const float M = fmaxf(m, sig2);
    const float a = (m == -INFINITY) ? 0.f : exp2f(m - M);
    const float ls = (sig2 == -INFINITY) ? 0.f : exp2f(sig2 - M);
    const float Z = l * a + ls;
    const float so = (Z > 0.f && nU > 0) ? (a / Z) * v_scale : 0.f;
    uint16_t* orow = out + (size_t(t) * Hq + h) * 128;
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      uint32_t v[32];
      if (nU > 0) {
        tmem_ld32(tmem + lane_off + 256 + c, v);
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
    if (row_valid) {
      max_logit[size_t(t) * Hq + h] = m_true * kLn2;
      lse[size_t(t) * Hq + h] = (Z > 0.f) ? (M + log2f(Z)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t attn_workspace_bytes(int B, int T, int max_q_len, int Hkv, int D, int max_pages) {
  (void)D;
  if (max_q_len <= 1) return 0;
  const size_t img = size_t(B) * max_pages * Hkv * 32768;
  return img + align256(size_t(T + B + 1) * sizeof(TileInfo)) + 256;
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream, const char** why) {
  if (a.max_pages > 2048) {
    *why = "max_pages must be <= 2048";
    return cudaErrorNotSupported;
  }
  if (a.max_q_len == 1) {
    *why = "decode attention not built yet";
    return cudaErrorNotSupported;
  }
  const int G = a.Hq / a.Hkv;
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
  plan_tiles_kernel<<<1, 256, 0, stream>>>(a.seq_lens, a.cu_q, a.B, toks, a.max_pages, max_tiles,
                                           tiles, n_tiles, a.err);
  vt_convert_kernel<<<dim3(a.max_pages, a.B, a.Hkv), 256, 0, stream>>>(
      a.v_cache, a.page_table, a.seq_lens, a.Hkv, a.max_pages, a.num_pages, ws, a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefillSmem);
  if (e != cudaSuccess) return e;
  const int grid = ((a.T + toks - 1) / toks + a.B) * a.Hkv;
  attn_prefill_kernel<<<grid, 192, kPrefillSmem, stream>>>(
      tm_q, tm_k, ws, a.page_table, tiles, n_tiles, a.topk, a.sink, a.c_qk * kLog2e,
      a.c_sink * kLog2e, a.v_scale, a.T, a.Hq, a.Hkv, a.Hidx, toks, a.topk_k, a.max_pages,
      a.num_pages, a.out, a.max_logit, a.lse, a.err);
  return cudaGetLastError();
}

}  // namespace msa

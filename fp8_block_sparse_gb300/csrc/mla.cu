// mla.cu -- step (c), sparse-MLA prefill: MQA of 128 query heads over one
// latent kv head, each query attending to its own list of kv rows.
//
// What is computed (sglang PR 25751 page, key source excerpt of
// sparse_mla_q8kv8_prefill_fwd; scale rules of sglang PR 30971 page,
// implementation step 3): query t attends to kv[indices[t, j]] for
// j < topk_length[t] (negative entries skipped); V is the first 512 columns
// of the same rows; with c = sm_scale * q_scale,
//   l_j = c * kv_scale * (q[t,h] . kv[idx_j])      (576-dim dot)
//   out = kv_scale * sum_j e^{l_j} kv[idx_j, :512] / (sum_j e^{l_j} + e^{c*sink[h]})
//   max_logits = max_j l_j,  lse = ln(sum_j e^{l_j} + e^{c*sink[h]}).
//
// GB300 design. The 128 heads of one query share its index list, so they are
// the M = 128 rows of every MMA. A CTA owns one query token and one half of
// d_v (a 128 x 512 fp32 O alone would fill all 512 TMEM columns), so both
// halves compute S. TMEM: the 512 nope bytes of Q per head (columns 0-127,
// four e4m3 per column: the A operand of QK^T, so the largest operand is not
// read from shared memory once per chunk), two 64-column S buffers, and the
// 256-column O half. Per 64-entry chunk of the index list:
//   gather   four warps copy the 64 kv rows (576 B each; a whole warp per
//            row, 16-byte cp.async, indices loaded one chunk ahead) into a
//            K-major tile: four 128-byte swizzled regions plus one 64-byte
//            swizzled region for the last 64 columns; invalid entries become
//            zero rows (zero-filling copies, and masked); four stages. Each
//            gather thread hangs its copies on the stage's full barrier
//            (an arrival once they land) and goes on to the next chunk, so
//            the gather runs up to four chunks ahead and a chunk is ready
//            the moment its rows have landed;
//   S = Q K^T  tcgen05 e4m3, M=128, N=64: 16 MMAs with A = Q's nope part in
//            TMEM, 2 with A = its rope part in shared memory;
//   P        one thread per head row: online softmax with a lazy reference 4
//            below the running maximum (moved only when a chunk's maximum
//            exceeds it by 2^8, so P <= 2^8 < 448); P is split into two e4m3
//            terms (P rounded, then its rounded remainder), written over the
//            first 32 columns of the chunk's own S buffer;
//   O += P V tcgen05 e4m3, M=128, N=256, K=64 per term: A = the P terms in
//            TMEM, B = this CTA's 256 V columns read straight out of the
//            gathered tile as an MN-major operand (no conversion pass).
// Epilogue: O / Z in bf16 is staged in the freed K stages (128-byte swizzled
// rows) and leaves as four TMA stores of 64 x 128 boxes.
// Two e4m3 terms carry P to about 2^-8 of its value: emulated on the CPU over
// full-size queries they cost no more than f16 P (the bf16 rounding of O
// dominates both), while a single e4m3 term costs ~2% relative error.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLimit = 8.0f;    // log2 of the largest P before the reference moves
constexpr float kHead = 4.0f;     // log2 of P at the key that set the reference
constexpr int kDqk = 576, kDv = 512, kChunkKeys = 64, kStagesM = 4;

// shared memory (byte offsets from a 1024-aligned base)
constexpr int kQOff = 0;            // 128 x 576 e4m3: 4 x 16 KB (SW128) + 8 KB (SW64)
constexpr int kQTail = 65536;
constexpr int kKOff = 73728;        // kStagesM stages x 36 KB: 4 x 8 KB (SW128) + 4 KB (SW64)
constexpr int kKStage = 36864;
constexpr int kKTail = 32768;       // offset of the SW64 region inside a stage
constexpr int kMlaSmem = kKOff + kStagesM * kKStage + 1024;
// TMEM columns: Q nope at 0, S_b at 128 + 64*b (P terms over its first 32), O at 256
constexpr uint32_t kTS = 128, kTO = 256;

constexpr uint32_t kIdescQK = idesc_f32(128, 64);
constexpr uint32_t kIdescPV = idesc_f32(128, 256) | (1u << 16);   // B MN-major

constexpr int kMlaThreads = 288;   // MMA, 4 gather, 4 softmax warps

__global__ void __launch_bounds__(kMlaThreads, 1)
mla_prefill_kernel(const __grid_constant__ CUtensorMap tm_q128, const __grid_constant__ CUtensorMap tm_q64,
                   const __grid_constant__ CUtensorMap tm_o, const uint8_t* __restrict__ kv, const int32_t* __restrict__ indices,
                   const int32_t* __restrict__ topk_length, const float* __restrict__ sink,
                   float qk_scale2, float sink_scale2, float v_scale, int T, int S_kv, int topk,
                   uint16_t* __restrict__ out, float* __restrict__ max_logits,
                   float* __restrict__ lse, unsigned* err) {
  pdl_wait();      // queries, latent cache and indices may come from earlier kernels
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_q, bar_qt, bar_kf[kStagesM], bar_ke[kStagesM], bar_sf[2], bar_pf[2],
      bar_pv, bar_done, bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  const int t = blockIdx.x >> 1, hf = blockIdx.x & 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int len = topk_length != nullptr ? topk_length[t] : topk;
  len = max(0, min(len, topk));
  const int nch = (len + kChunkKeys - 1) / kChunkKeys;
  const int32_t* idx_row = indices + size_t(t) * topk;

  if (tid == 0) {
    abort_s = initial_abort(err);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qt, 4);
    mbar_init(&bar_drain, 1);
    for (int s = 0; s < kStagesM; ++s) { mbar_init(&bar_kf[s], 128); mbar_init(&bar_ke[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&bar_sf[s], 1); mbar_init(&bar_pf[s], 4); }
    mbar_init(&bar_pv, 1);
    mbar_init(&bar_done, 1);
    fence_barrier_init();
  }
  if (warp == 0) { tmem_alloc(&tmem_base_s, 512); tmem_relinquish(); }
  __syncthreads();
  pdl_trigger();   // after this block's tensor-memory allocation
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ---------------- Q (one TMA batch), then MMA issue (whole warp, elected lane)
    if (nch > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_q, 128 * kDqk);
        for (int r = 0; r < 4; ++r) tma_load_2d(smem + kQOff + r * 16384, &tm_q128, &bar_q, r * 128, t * 128);
        tma_load_2d(smem + kQTail, &tm_q64, &bar_q, 512, t * 128);
      }
      __syncwarp();
      // the softmax warps move Q's nope part into TMEM columns 0-127
      if (mbar_wait_warp(&bar_qt, 0, err, &abort_s)) {
        tc_fence_after();
        const uint32_t sq = smem_addr(smem + kQOff);
        auto issue_s = [&](int j) -> bool {
          const int s = j % kStagesM, sb = j & 1;
          if (!mbar_wait_warp(&bar_kf[s], (j / kStagesM) & 1, err, &abort_s)) return false;
          // the rows landed through the generic proxy (cp.async); the MMAs
          // read them through the async proxy
          fence_async_shared();
          tc_fence_after();
          const uint32_t sk = smem_addr(smem + kKOff + s * kKStage);
          const uint32_t d = tmem + kTS + 64 * sb;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            mma_e4m3_ts_w(d, tmem + 8 * k, sdesc_kmajor(sk + (k >> 2) * 8192 + (k & 3) * 32, 128),
                          kIdescQK, k > 0);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_e4m3_w(d, sdesc_kmajor(sq + kQTail + k * 32, 64),
                       sdesc_kmajor(sk + kKTail + k * 32, 64), kIdescQK, 1u);
          mma_commit_w(&bar_sf[sb]);
          return true;
        };
        bool ok = issue_s(0) && (nch < 2 || issue_s(1));
        for (int j = 0; ok && j < nch; ++j) {
          const int s = j % kStagesM, sb = j & 1;
          if (!mbar_wait_warp(&bar_pf[sb], (j >> 1) & 1, err, &abort_s)) break;
          tc_fence_after();
          // this CTA's 256 V columns: regions 2*hf and 2*hf + 1 of the tile
          const uint32_t sv = smem_addr(smem + kKOff + s * kKStage) + uint32_t(hf) * 16384u;
#pragma unroll
          for (int term = 0; term < 2; ++term)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)             // 32 keys per step: 8 P columns, 32 V rows
              mma_e4m3_ts_w(tmem + kTO, tmem + kTS + 64 * sb + 16 * term + 8 * kk,
                            sdesc_mn_sw128(sv + kk * 4096, 8192), kIdescPV,
                            (j > 0 || term > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(&bar_ke[s]);          // PV(j) is the stage's last reader
          mma_commit_w(&bar_pv);
          if (j == nch - 1) mma_commit_w(&bar_done);
          // S buffer sb holds P(j) until PV(j) has read it: MMAs of one thread
          // run in order, so QK(j+2) may be issued into it now
          if (j + 2 < nch && !(ok = issue_s(j + 2))) break;
        }
      }
      // exit-path drain (a no-op unless a wait gave up): no MMA in flight and
      // the Q copies landed once TMEM and shared memory are released
      mma_drain_w(&bar_drain, err);
      if (lane == 0) mbar_wait(&bar_q, 0, err);
    }
  } else if (warp <= 4) {
    // ---------------- gather warps: copy chunk j and move on
    // Warp pw copies rows 16*pw .. 16*pw+15 of the chunk, one row at a time
    // with all 32 lanes (576 bytes = 36 chunks of 16 bytes), so every cp.async
    // instruction reads contiguous bytes of one kv row; then each thread
    // arrives on the chunk's full barrier once its copies have landed.
    const int pt = tid - 32, pw = pt >> 5;
    // lanes 0..15 hold the kv index of row 16*pw + lane, loaded one chunk ahead
    int idx_next = -1;
    if (lane < 16 && pw * 16 + lane < len)
      asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(idx_next) : "l"(idx_row + pw * 16 + lane));
    for (int j = 0; j < nch; ++j) {
      const int s = j % kStagesM;
      int my_idx = idx_next;
      const int key_n = (j + 1) * kChunkKeys + pw * 16 + lane;
      idx_next = -1;
      if (lane < 16 && key_n < len)
        asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(idx_next) : "l"(idx_row + key_n));
      if (lane < 16 && my_idx >= S_kv) { atomicOr(err, MSA_DEVERR_DATA); my_idx = -1; }
      // PV(j-4) done: the stage is free (the result is unused: after a
      // timeout the loop still runs, so every thread's arrivals happen)
      mbar_wait_ab(&bar_ke[s], ((j / kStagesM) & 1) ^ 1, err, &abort_s);
      uint8_t* stage = smem + kKOff + s * kKStage;
#pragma unroll 4
      for (int rr = 0; rr < 16; ++rr) {
        const int r = pw * 16 + rr;
        const int idx = __shfl_sync(0xffffffffu, my_idx, rr);
        const uint8_t* src = kv + size_t(idx < 0 ? 0 : idx) * kDqk;
        cp_async16_zfill(stage + (lane >> 3) * 8192 + swz_offset(r, lane & 7, 128), src + lane * 16,
                         idx >= 0);                          // chunks 0..31: SW128 regions
        if (lane < 4)                                        // chunks 32..35: SW64 tail
          cp_async16_zfill(stage + kKTail + swz_offset(r, lane, 64), src + (32 + lane) * 16, idx >= 0);
      }
      cp_async_arrive(&bar_kf[s]);
    }
    cp_async_wait_all();        // nothing of this thread is in flight at the exit
  } else {
    // ---------------- softmax (warps 5-8): thread = head row (TMEM lane)
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    if (nch > 0) {
      // Q's nope bytes of this head into TMEM columns 0-127, four per column
      // in ascending order (the layout of an 8-bit A operand in TMEM)
      if (mbar_wait_warp(&bar_q, 0, err, &abort_s)) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 q = *reinterpret_cast<const uint4*>(smem + kQOff + r * 16384 +
                                                            swz_offset(uint32_t(row), uint32_t(c), 128));
            v[4 * c] = q.x; v[4 * c + 1] = q.y; v[4 * c + 2] = q.z; v[4 * c + 3] = q.w;
          }
          tmem_st32(tmem + lane_off + 32 * r, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_qt);
    }
    float ref = -INFINITY, m_true = -INFINITY, l = 0.f;
    // validity of the chunk's 64 keys: lane holds keys lane and lane + 32,
    // loaded one chunk ahead and combined with two ballots
    int ia = -1, ib = -1;
    if (lane < len) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(ia) : "l"(idx_row + lane));
    if (lane + 32 < len) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(ib) : "l"(idx_row + lane + 32));
    for (int j = 0; j < nch; ++j) {
      const int sb = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      const uint64_t valid = uint64_t(__ballot_sync(0xffffffffu, ia >= 0 && ia < S_kv)) |
                             (uint64_t(__ballot_sync(0xffffffffu, ib >= 0 && ib < S_kv)) << 32);
      {
        const int k0 = (j + 1) * kChunkKeys + lane;
        ia = -1; ib = -1;
        if (k0 < len) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(ia) : "l"(idx_row + k0));
        if (k0 + 32 < len) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(ib) : "l"(idx_row + k0 + 32));
      }
      mbar_wait_ab(&bar_sf[sb], ph, err, &abort_s);
      tc_fence_after();
      const uint32_t s_col = tmem + lane_off + kTS + 64 * sb;
      float x[64];
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t v[32];
        tmem_ld32(s_col + c, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c + e] = __uint_as_float(v[e]);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        x[c] = ((valid >> c) & 1) ? x[c] * qk_scale2 : -INFINITY;
        mx = fmaxf(mx, x[c]);
      }
      m_true = fmaxf(m_true, mx);
      const bool grow = mx > ref + kLimit;                 // also when ref == -inf
      const bool need = grow && (ref > -INFINITY);
      if (__any_sync(0xffffffffu, need)) {
        mbar_wait_ab(&bar_pv, (j - 1) & 1, err, &abort_s);  // PV(j-1) done: O is settled
        tc_fence_after();
        const float alpha = need ? exp2f(ref - (mx - kHead)) : 1.0f;
#pragma unroll 4
        for (int c = 0; c < 256; c += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_off + kTO + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st16(tmem + lane_off + kTO + c, v);
        }
        if (need) l *= alpha;
      }
      if (grow) ref = mx - kHead;
      const float r0 = (ref == -INFINITY) ? 0.f : ref;
      // P and its two e4m3 terms, four codes per TMEM column in key order:
      // term 0 in columns 0-15 of this S buffer, term 1 in columns 16-31
      uint32_t w[32];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[4 * c + i] - r0);
        sum += (p[0] + p[1]) + (p[2] + p[3]);
        const uint16_t e01 = e4m3x2_from_f32(p[0], p[1]), e23 = e4m3x2_from_f32(p[2], p[3]);
        w[c] = uint32_t(e01) | (uint32_t(e23) << 16);
        const uint32_t h01 = e4m3x2_to_f16x2(e01), h23 = e4m3x2_to_f16x2(e23);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        // the remainders are exact in fp32
        const uint16_t g01 = e4m3x2_from_f32(p[0] - f01.x, p[1] - f01.y);
        const uint16_t g23 = e4m3x2_from_f32(p[2] - f23.x, p[3] - f23.y);
        w[16 + c] = uint32_t(g01) | (uint32_t(g23) << 16);
      }
      tmem_st32(s_col, w);
      l += sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pf[sb]);
    }
    // ---------------- epilogue
    if (nch > 0) mbar_wait_ab(&bar_done, 0, err, &abort_s);
    tc_fence_after();
    const float sig2 = sink != nullptr ? sink_scale2 * __ldg(sink + row) : -INFINITY;
    const float M = fmaxf(ref, sig2);
    const float a = (ref == -INFINITY) ? 0.f : exp2f(ref - M);
    const float ls = (sig2 == -INFINITY) ? 0.f : exp2f(sig2 - M);
    const float Z = l * a + ls;
    const float so = (Z > 0.f && nch > 0) ? (a / Z) * v_scale : 0.f;
    // O / Z in bf16 through shared memory (the K stages, free once PV of
    // the last chunk is done) and four TMA stores of 64-column boxes, so
    // the 64 KB leave as whole lines instead of 16-byte pieces of 32 rows
    // per store instruction. Box b holds columns 64b..64b+63 of this
    // CTA's half, a 128-byte row per head, 16-byte chunks swizzled by row.
    uint8_t* stg = smem + kKOff;
#pragma unroll 2
    for (int c = 0; c < 256; c += 32) {
      uint32_t v[32];
      if (nch > 0) {
        tmem_ld32(tmem + lane_off + kTO + c, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      uint8_t* rowp = stg + (c >> 6) * 16384 + row * 128;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        uint4 o;
        o.x = pack_bf16x2(__uint_as_float(v[e + 0]) * so, __uint_as_float(v[e + 1]) * so);
        o.y = pack_bf16x2(__uint_as_float(v[e + 2]) * so, __uint_as_float(v[e + 3]) * so);
        o.z = pack_bf16x2(__uint_as_float(v[e + 4]) * so, __uint_as_float(v[e + 5]) * so);
        o.w = pack_bf16x2(__uint_as_float(v[e + 6]) * so, __uint_as_float(v[e + 7]) * so);
        const uint32_t chunk = uint32_t(((c & 63) + e) >> 3);
        *reinterpret_cast<uint4*>(rowp + ((chunk ^ uint32_t(row & 7)) << 4)) = o;
      }
    }
    fence_async_shared();
    asm volatile("bar.sync 1, 128;" ::: "memory");            // the four softmax warps
    if (tid == 160) {
#pragma unroll
      for (int b = 0; b < 4; ++b) tma_store_2d(&tm_o, stg + b * 16384, hf * 256 + 64 * b, t * 128);
      bulk_commit();
      bulk_wait_read();            // the staging must stay until the copies have read it
    }
    if (hf == 0) {
      max_logits[size_t(t) * 128 + row] = m_true * kLn2;
      lse[size_t(t) * 128 + row] = (Z > 0.f) ? (M + log2f(Z)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaArgs& a, cudaStream_t stream, const char** why) {
  CUtensorMap tm_q128, tm_q64, tm_o;
  const uint64_t dims[2] = {uint64_t(kDqk), uint64_t(a.T) * 128};
  const uint64_t strides[1] = {uint64_t(kDqk)};
  const uint32_t box128[2] = {128, 128}, box64[2] = {64, 128};
  if (!encode_tensor_map(&tm_q128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q, dims, strides, box128,
                         CU_TENSOR_MAP_SWIZZLE_128B, why) ||
      !encode_tensor_map(&tm_q64, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q, dims, strides, box64,
                         CU_TENSOR_MAP_SWIZZLE_64B, why))
    return cudaErrorInvalidValue;
  {
    const uint64_t odims[2] = {uint64_t(kDv), uint64_t(a.T) * 128};
    const uint64_t ostrides[1] = {uint64_t(kDv) * 2};
    const uint32_t obox[2] = {64, 128};
    if (!encode_tensor_map(&tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, odims, ostrides, obox,
                           CU_TENSOR_MAP_SWIZZLE_128B, why))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(mla_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem);
  if (e != cudaSuccess) return e;
  profile_mark(stream, 0);
  e = launch_pdl(mla_prefill_kernel, a.T * 2, kMlaThreads, kMlaSmem, stream, tm_q128, tm_q64, tm_o, a.kv,
                 a.indices, a.topk_length, a.sink, a.c_qk * kLog2e, a.c_sink * kLog2e, a.v_scale,
                 a.T, a.S_kv, a.topk, a.out, a.max_logits, a.lse, a.err);
  profile_mark(stream, 1);
  return e;
}

}  // namespace msa

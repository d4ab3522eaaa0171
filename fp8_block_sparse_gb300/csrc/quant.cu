// quant.cu -- step (a): per-tensor e4m3 quantisation, out = e4m3(fp32(x) * s_inv),
// the quantised KV-cache store that feeds the path with the same rule, and the
// fused rotary embedding + quantisation of MLA q / kv rows (nope || rope(pe)).
//
// sglang PR 25460 page, key source excerpt of fp8_quantize (widen to fp32,
// multiply by a host-side scale_inv, cast to fp8); sglang PR 30971 page,
// implementation step 3 (_quant_q_fp8 on q and idx_q) and step 4 (the sparse KV
// pool's K / V / index-K stores with per-tensor scales, None = unit scale);
// sglang PR 25460 page, implementation step 2 and the _fused_rope_fp8_quantize
// excerpt (rotary embedding of the pe part, nope and pe written side by side
// as one e4m3 row).
//
// Pure streaming work (2 bytes in, 1 byte out per element), so the kernel is
// built for HBM: each thread moves 16 elements per step as two 16-byte loads
// and one 16-byte store, several steps in flight, over a grid sized to the
// SM count. The multiply is __fmul_rn (never contracted) and the cast is the
// hardware round-to-nearest-even satfinite conversion.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

MSA_DEV uint16_t cvt2(float a, float b) {
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// 8 bf16 / fp16 values packed in a uint4 -> 8 fp32 values.
template <bool BF16>
MSA_DEV void widen8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 p = __half22float2(h);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
}

template <bool BF16>
MSA_DEV uint4 quant16(const uint4& lo, const uint4& hi, float s_inv) {
  float a[8], b[8];
  widen8<BF16>(lo, a);
  widen8<BF16>(hi, b);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    o[i] = uint32_t(cvt2(__fmul_rn(a[4 * i], s_inv), __fmul_rn(a[4 * i + 1], s_inv))) |
           (uint32_t(cvt2(__fmul_rn(a[4 * i + 2], s_inv), __fmul_rn(a[4 * i + 3], s_inv))) << 16);
    o[2 + i] = uint32_t(cvt2(__fmul_rn(b[4 * i], s_inv), __fmul_rn(b[4 * i + 1], s_inv))) |
               (uint32_t(cvt2(__fmul_rn(b[4 * i + 2], s_inv), __fmul_rn(b[4 * i + 3], s_inv))) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Rows of `cols` elements (cols % 16 == 0, 16-byte aligned rows): one chunk
// = 16 consecutive elements of one row. Contiguous tensors pass
// chunks_per_row = total chunks and rows = 1.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_vec_kernel(const uint16_t* __restrict__ x,
                                                        uint32_t rows, uint32_t chunks_per_row,
                                                        int64_t x_stride,
                                                        uint8_t* __restrict__ out,
                                                        int64_t out_stride, float s_inv) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  const uint64_t total = uint64_t(rows) * chunks_per_row;
  const uint64_t step = uint64_t(gridDim.x) * blockDim.x;
  uint64_t c = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  // two chunks per iteration keep 64 bytes of loads in flight per thread
  for (; c + step < total; c += 2 * step) {
    const uint64_t c1 = c + step;
    const uint32_t r0 = uint32_t(c / chunks_per_row), r1 = uint32_t(c1 / chunks_per_row);
    const uint64_t j0 = (c - uint64_t(r0) * chunks_per_row) * 16;
    const uint64_t j1 = (c1 - uint64_t(r1) * chunks_per_row) * 16;
    const uint4* s0 = reinterpret_cast<const uint4*>(x + r0 * x_stride + j0);
    const uint4* s1 = reinterpret_cast<const uint4*>(x + r1 * x_stride + j1);
    const uint4 a0 = __ldcs(s0), b0 = __ldcs(s0 + 1), a1 = __ldcs(s1), b1 = __ldcs(s1 + 1);
    *reinterpret_cast<uint4*>(out + r0 * out_stride + j0) = quant16<BF16>(a0, b0, s_inv);
    *reinterpret_cast<uint4*>(out + r1 * out_stride + j1) = quant16<BF16>(a1, b1, s_inv);
  }
  if (c < total) {
    const uint32_t r0 = uint32_t(c / chunks_per_row);
    const uint64_t j0 = (c - uint64_t(r0) * chunks_per_row) * 16;
    const uint4* s0 = reinterpret_cast<const uint4*>(x + r0 * x_stride + j0);
    *reinterpret_cast<uint4*>(out + r0 * out_stride + j0) =
        quant16<BF16>(__ldcs(s0), __ldcs(s0 + 1), s_inv);
  }
}

// Contiguous tensors: chunk c covers elements 16c .. 16c+15 of both x and
// out, so no index arithmetic beyond the chunk number; four chunks per
// iteration keep 128 bytes of loads in flight per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_contig_kernel(const uint4* __restrict__ x,
                                                           uint64_t chunks,
                                                           uint4* __restrict__ out, float s_inv) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  const uint64_t step = uint64_t(gridDim.x) * blockDim.x;
  uint64_t c = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; c + 3 * step < chunks; c += 4 * step) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = __ldcs(x + 2 * (c + u * step));
      b[u] = __ldcs(x + 2 * (c + u * step) + 1);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) out[c + u * step] = quant16<BF16>(a[u], b[u], s_inv);
  }
  for (; c < chunks; c += step) out[c] = quant16<BF16>(__ldcs(x + 2 * c), __ldcs(x + 2 * c + 1), s_inv);
}

// Several contiguous tensors: block b works on the tensor whose block range
// holds it, striding over that tensor's chunks like quant_contig_kernel.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_multi_kernel(const QuantMulti q) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  int j = 0;
  while (j + 1 < q.n && int(blockIdx.x) >= q.block0[j + 1]) ++j;
  const uint4* __restrict__ x = q.x[j];
  uint4* __restrict__ out = q.out[j];
  const uint64_t chunks = q.chunks[j];
  const float s_inv = q.s_inv[j];
  const uint64_t step = uint64_t(q.block0[j + 1] - q.block0[j]) * blockDim.x;
  uint64_t c = uint64_t(int(blockIdx.x) - q.block0[j]) * blockDim.x + threadIdx.x;
  for (; c + 3 * step < chunks; c += 4 * step) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = __ldcs(x + 2 * (c + u * step));
      b[u] = __ldcs(x + 2 * (c + u * step) + 1);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) out[c + u * step] = quant16<BF16>(a[u], b[u], s_inv);
  }
  for (; c < chunks; c += step) out[c] = quant16<BF16>(__ldcs(x + 2 * c), __ldcs(x + 2 * c + 1), s_inv);
}

// Any shape, stride and alignment: one element per thread step.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_scalar_kernel(const uint16_t* __restrict__ x,
                                                           int64_t rows, int64_t cols,
                                                           int64_t x_stride,
                                                           uint8_t* __restrict__ out,
                                                           int64_t out_stride, float s_inv) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  const int64_t total = rows * cols;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / cols, j = i - r * cols;
    const uint16_t bits = x[r * x_stride + j];
    float v;
    if (BF16) {
      v = __uint_as_float(uint32_t(bits) << 16);
    } else {
      v = __half2float(__ushort_as_half(bits));
    }
    const uint16_t p = cvt2(__fmul_rn(v, s_inv), 0.0f);
    out[r * out_stride + j] = uint8_t(p & 0xFF);
  }
}

// The quantised KV-cache store. One block owns `tpb` consecutive new tokens:
// their threads first resolve each token's (page, slot) from the batch
// description into shared memory, then the block walks the tokens' 16-element
// chunks (K heads, V heads, index K), four chunks in flight per thread. Each
// chunk is two 16-byte streaming loads and one 16-byte store; a (page, head,
// slot) row of D codes is written by D/16 neighbouring threads.
template <bool BF16>
__global__ void __launch_bounds__(256) kv_store_kernel(KvStoreArgs a, int tpb) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  __shared__ int s_page[256];
  __shared__ int s_slot[256];
  const int t0 = blockIdx.x * tpb;
  const int nt = min(tpb, a.T - t0);
  if (int(threadIdx.x) < nt) {
    const int t = t0 + threadIdx.x;
    int lo = 0, hi = a.B - 1;                 // last sequence whose first row is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int q0 = __ldg(a.cu_q + lo), qlen = __ldg(a.cu_q + lo + 1) - q0;
    const int pos = __ldg(a.seq_lens + lo) - qlen + (t - q0);
    int page = -1;
    if (pos >= 0 && t - q0 < qlen && (pos >> 7) < a.max_pages)
      page = __ldg(a.page_table + int64_t(lo) * a.max_pages + (pos >> 7));
    if (page < 0 || page >= a.num_pages) {
      atomicOr(a.err, MSA_DEVERR_DATA);
      page = -1;
    }
    s_page[threadIdx.x] = page;
    s_slot[threadIdx.x] = pos & 127;
  }
  __syncthreads();
  const int cd = a.D / 16;
  const int nk = a.k ? a.Hkv * cd : 0, nv = a.v ? a.Hkv * cd : 0, ni = a.idx_k ? a.d_idx / 16 : 0;
  const int cpt = nk + nv + ni;
  const int total = nt * cpt;
  constexpr int U = 4;
  for (int c0 = threadIdx.x; c0 < total; c0 += U * 256) {
    const uint4* src[U];
    uint4* dst[U];
    float sinv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 256;
      dst[u] = nullptr;
      src[u] = nullptr;
      sinv[u] = 1.0f;
      if (c >= total) continue;
      const int tl = c / cpt;
      int r = c - tl * cpt;
      const int page = s_page[tl];
      if (page < 0) continue;
      const int64_t t = t0 + tl;
      const int slot = s_slot[tl];
      if (r < nk + nv) {
        const bool is_k = r < nk;
        if (!is_k) r -= nk;
        const int h = r / cd, cc = r - h * cd;
        const uint16_t* x = is_k ? a.k + t * a.k_stride : a.v + t * a.v_stride;
        uint8_t* cache = is_k ? a.k_cache : a.v_cache;
        src[u] = reinterpret_cast<const uint4*>(x + r * 16);
        dst[u] = reinterpret_cast<uint4*>(cache + ((int64_t(page) * a.Hkv + h) * 128 + slot) * a.D +
                                          cc * 16);
        sinv[u] = is_k ? a.k_sinv : a.v_sinv;
      } else {
        r -= nk + nv;
        src[u] = reinterpret_cast<const uint4*>(a.idx_k + t * a.idx_stride + r * 16);
        dst[u] = reinterpret_cast<uint4*>(a.idx_cache + (int64_t(page) * 128 + slot) * a.d_idx + r * 16);
        sinv[u] = a.i_sinv;
      }
    }
    uint4 lo[U], hi[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (dst[u]) {
        lo[u] = __ldcs(src[u]);
        hi[u] = __ldcs(src[u] + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u]) *dst[u] = quant16<BF16>(lo[u], hi[u], sinv[u]);
  }
}

// 16 fp32 values * s_inv -> 16 e4m3 codes.
MSA_DEV uint4 quant16f(const float (&v)[16], float s_inv) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = uint32_t(cvt2(__fmul_rn(v[4 * i], s_inv), __fmul_rn(v[4 * i + 1], s_inv))) |
           (uint32_t(cvt2(__fmul_rn(v[4 * i + 2], s_inv), __fmul_rn(v[4 * i + 3], s_inv))) << 16);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

MSA_DEV void load16f(const float* p, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p) + i);
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
}

// One output chunk (16 e4m3 codes of nope || rope(pe)) in two phases: fetch
// issues every global load of the chunk, finish does the arithmetic, so a
// thread keeps several chunks' loads in flight before it waits on any.
struct RopeChunk {
  uint4 lo, hi;     // the chunk's own 16 inputs
  uint4 plo, phi;   // neox: the partner half's 16 inputs
  const float* cs;  // table row of the position (rope chunks)
  uint4* dst;       // null: nothing to write
  int e0;           // first pe element (-1: nope chunk)
  bool bad;         // position outside the table
};

template <bool BF16, bool NEOX>
MSA_DEV void rope_fetch(const RopeQuantArgs& a, int64_t r, int h, int j, uint4* dst, RopeChunk& k) {
  const int nn = a.d_nope / 16;
  k.dst = dst;
  k.bad = false;
  if (j < nn) {
    const uint4* src = reinterpret_cast<const uint4*>(a.nope + r * a.nope_tok_stride +
                                                      h * a.nope_head_stride + j * 16);
    k.e0 = -1;
    k.lo = __ldcs(src);
    k.hi = __ldcs(src + 1);
    return;
  }
  k.e0 = (j - nn) * 16;
  const int pos = __ldg(a.positions + r);
  if (pos < 0 || pos >= a.max_pos) {
    k.bad = true;
    return;
  }
  const int half = a.d_rope / 2;
  const uint16_t* pe = a.pe + r * a.pe_tok_stride + h * a.pe_head_stride;
  k.cs = a.cos_sin + int64_t(pos) * a.d_rope;
  const uint4* src = reinterpret_cast<const uint4*>(pe + k.e0);
  k.lo = __ldg(src);
  k.hi = __ldg(src + 1);
  if (NEOX) {
    const uint4* partner = reinterpret_cast<const uint4*>(pe + (k.e0 < half ? k.e0 + half : k.e0 - half));
    k.plo = __ldg(partner);
    k.phi = __ldg(partner + 1);
  }
}

// The rotation is fp32 with every product and sum rounded on its own
// (__fmul_rn / __fadd_rn / __fsub_rn are never contracted into an FMA).
template <bool BF16, bool NEOX>
MSA_DEV void rope_finish(const RopeQuantArgs& a, const RopeChunk& k) {
  if (k.e0 < 0) {
    *k.dst = quant16<BF16>(k.lo, k.hi, a.s_inv);
    return;
  }
  if (k.bad) {
    atomicOr(a.err, MSA_DEVERR_DATA);
    *k.dst = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int half = a.d_rope / 2;
  float x[16], v[16];
  widen8<BF16>(k.lo, *reinterpret_cast<float(*)[8]>(x));
  widen8<BF16>(k.hi, *reinterpret_cast<float(*)[8]>(x + 8));
  if (NEOX) {
    // halves (x1, x2): out1 = x1 c - x2 s, out2 = x2 c + x1 s, angle = index in the half
    const bool first = k.e0 < half;
    const int i0 = first ? k.e0 : k.e0 - half;
    float y[16], c[16], sn[16];
    widen8<BF16>(k.plo, *reinterpret_cast<float(*)[8]>(y));
    widen8<BF16>(k.phi, *reinterpret_cast<float(*)[8]>(y + 8));
    load16f(k.cs + i0, c);
    load16f(k.cs + half + i0, sn);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      v[i] = first ? __fsub_rn(__fmul_rn(x[i], c[i]), __fmul_rn(y[i], sn[i]))
                   : __fadd_rn(__fmul_rn(x[i], c[i]), __fmul_rn(y[i], sn[i]));
  } else {
    // neighbour pairs (x[2k], x[2k+1]) at angle e0/2 + k
    float c[8], sn[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float4 fc = __ldg(reinterpret_cast<const float4*>(k.cs + k.e0 / 2) + i);
      const float4 fs = __ldg(reinterpret_cast<const float4*>(k.cs + half + k.e0 / 2) + i);
      c[4 * i] = fc.x; c[4 * i + 1] = fc.y; c[4 * i + 2] = fc.z; c[4 * i + 3] = fc.w;
      sn[4 * i] = fs.x; sn[4 * i + 1] = fs.y; sn[4 * i + 2] = fs.z; sn[4 * i + 3] = fs.w;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[2 * q] = __fsub_rn(__fmul_rn(x[2 * q], c[q]), __fmul_rn(x[2 * q + 1], sn[q]));
      v[2 * q + 1] = __fadd_rn(__fmul_rn(x[2 * q + 1], c[q]), __fmul_rn(x[2 * q], sn[q]));
    }
  }
  *k.dst = quant16f(v, a.s_inv);
}

// Two block roles in one launch. Blocks [0, nb_nope) quantise the nope
// chunks: each owns `upb_n` consecutive (row, head) units and streams their
// d_nope/16 chunks with four in flight per thread (a strided copy with a
// cast). The remaining blocks own `upb_r` units each and rotate + quantise
// their d_rope/16 pe chunks, two in flight. Chunk indices inside a block are
// 32-bit; a unit's (row, head) follows from the block's first unit by small
// 32-bit steps.
template <bool BF16, bool NEOX>
__global__ void __launch_bounds__(256) rope_quant_kernel(RopeQuantArgs a, int upb_n, int nb_nope,
                                                         int upb_r) {
  pdl_wait();      // inputs may come from the previous kernel in the stream
  pdl_trigger();
  const int nn = a.d_nope / 16, nr = a.d_rope / 16, cpr = nn + nr;
  const int64_t units = a.rows * int64_t(a.heads);
  const bool nope_role = int(blockIdx.x) < nb_nope;
  const int upb = nope_role ? upb_n : upb_r;
  const int per = nope_role ? nn : nr;
  const int64_t u0 = int64_t(nope_role ? blockIdx.x : blockIdx.x - nb_nope) * upb;
  const int nu = int(units - u0 < upb ? units - u0 : upb);
  const int64_t r0 = u0 / a.heads;
  const int h0 = int(u0 - r0 * a.heads);
  const int total = nu * per;
  uint4* out = reinterpret_cast<uint4*>(a.out) + u0 * cpr;
  if (nope_role) {
    constexpr int U = 4;
    for (int c0 = threadIdx.x; c0 < total; c0 += U * 256) {
      uint4 lo[U], hi[U];
      uint4* dst[U];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int c = c0 + i * 256;
        dst[i] = nullptr;
        if (c < total) {
          const int u = c / nn, j = c - u * nn;
          const int hh = h0 + u, dr = hh / a.heads;
          const uint4* src = reinterpret_cast<const uint4*>(
              a.nope + (r0 + dr) * a.nope_tok_stride + (hh - dr * a.heads) * a.nope_head_stride + j * 16);
          lo[i] = __ldcs(src);
          hi[i] = __ldcs(src + 1);
          dst[i] = out + int64_t(u) * cpr + j;
        }
      }
#pragma unroll
      for (int i = 0; i < U; ++i)
        if (dst[i]) *dst[i] = quant16<BF16>(lo[i], hi[i], a.s_inv);
    }
  } else {
    constexpr int U = 2;
    for (int c0 = threadIdx.x; c0 < total; c0 += U * 256) {
      RopeChunk k[U];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int c = c0 + i * 256;
        k[i].dst = nullptr;
        if (c < total) {
          const int u = c / nr, j = c - u * nr;
          const int hh = h0 + u, dr = hh / a.heads;
          rope_fetch<BF16, NEOX>(a, r0 + dr, hh - dr * a.heads, nn + j, out + int64_t(u) * cpr + nn + j,
                                 k[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < U; ++i)
        if (k[i].dst) rope_finish<BF16, NEOX>(a, k[i]);
    }
  }
}

}  // namespace

cudaError_t launch_rope_quant(const RopeQuantArgs& a, bool bf16, bool neox, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  const int nn = a.d_nope / 16, nr = a.d_rope / 16;
  const int64_t units = a.rows * int64_t(a.heads);
  // about 2048 chunks (8 per thread) per block of either role
  const int upb_n = nn > 0 ? (2048 / nn > 0 ? 2048 / nn : 1) : 1;
  const int upb_r = 2048 / nr > 0 ? 2048 / nr : 1;
  const int64_t nb_nope = nn > 0 ? (units + upb_n - 1) / upb_n : 0;
  const int64_t grid = nb_nope + (units + upb_r - 1) / upb_r;
  if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
  const unsigned g = unsigned(grid);
  const int nb = int(nb_nope);
  if (bf16) {
    if (neox) launch_pdl(rope_quant_kernel<true, true>, g, 256, 0, stream, a, upb_n, nb, upb_r);
    else launch_pdl(rope_quant_kernel<true, false>, g, 256, 0, stream, a, upb_n, nb, upb_r);
  } else {
    if (neox) launch_pdl(rope_quant_kernel<false, true>, g, 256, 0, stream, a, upb_n, nb, upb_r);
    else launch_pdl(rope_quant_kernel<false, false>, g, 256, 0, stream, a, upb_n, nb, upb_r);
  }
  return cudaGetLastError();
}

cudaError_t launch_kv_store(const KvStoreArgs& a, bool bf16, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int cd = a.D / 16;
  const int cpt = (a.k ? a.Hkv * cd : 0) + (a.v ? a.Hkv * cd : 0) + (a.idx_k ? a.d_idx / 16 : 0);
  if (cpt == 0) return cudaSuccess;
  // about 2048 chunks (8 per thread) per block, but at least two blocks per
  // SM when the batch allows it
  int tpb = 2048 / cpt;
  const int spread = (a.T + 2 * num_sms() - 1) / (2 * num_sms());
  tpb = tpb < spread ? tpb : spread;
  tpb = tpb < 1 ? 1 : (tpb > 256 ? 256 : tpb);
  const int grid = (a.T + tpb - 1) / tpb;
  if (bf16)
    launch_pdl(kv_store_kernel<true>, grid, 256, 0, stream, a, tpb);
  else
    launch_pdl(kv_store_kernel<false>, grid, 256, 0, stream, a, tpb);
  return cudaGetLastError();
}

bool quant_multi_eligible(const void* x, const void* out, int64_t rows, int64_t cols,
                          int64_t x_stride, int64_t out_stride) {
  return (x_stride == cols) && (out_stride == cols) && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(out) % 16 == 0 && (rows * cols) % 16 == 0 &&
         (rows * cols) / 16 < (1ll << 32);
}

cudaError_t launch_quant_multi(QuantMulti& q, bool bf16, cudaStream_t stream) {
  if (q.n == 0) return cudaSuccess;
  // the grid of one contiguous launch (<= 8 blocks per SM, 4 chunks per
  // thread), dealt out in proportion to the tensors' chunks, >= 1 each
  const int threads = 256;
  uint64_t total = 0;
  for (int j = 0; j < q.n; ++j) total += q.chunks[j];
  const uint64_t want = (total + 4 * threads - 1) / (4 * threads);
  const uint64_t cap = uint64_t(num_sms()) * 8;
  const int grid = int(want < cap ? want : cap) > q.n ? int(want < cap ? want : cap) : q.n;
  int b = 0;
  uint64_t acc = 0;
  for (int j = 0; j < q.n; ++j) {
    q.block0[j] = b;
    acc += q.chunks[j];
    int next = int((acc * uint64_t(grid) + total - 1) / total);
    if (next < b + 1) next = b + 1;
    if (next > grid - (q.n - 1 - j)) next = grid - (q.n - 1 - j);
    b = next;
  }
  q.block0[q.n] = b;
  if (bf16) return launch_pdl(quant_multi_kernel<true>, b, threads, 0, stream, q);
  return launch_pdl(quant_multi_kernel<false>, b, threads, 0, stream, q);
}

cudaError_t launch_quant(const void* x, bool bf16, int64_t rows, int64_t cols, int64_t x_stride,
                         uint8_t* out, int64_t out_stride, float s_inv, cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  const bool contiguous = (x_stride == cols) && (out_stride == cols);
  const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  const int sms = num_sms();
  const int threads = 256;
  if (aligned && contiguous && (rows * cols) % 16 == 0 && (rows * cols) / 16 < (1ll << 32)) {
    const uint64_t chunks = uint64_t(rows * cols) / 16;
    const uint64_t want = (chunks + 4 * threads - 1) / (4 * threads);
    const int grid = int(want < uint64_t(sms) * 8 ? (want ? want : 1) : uint64_t(sms) * 8);
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint4* ov = reinterpret_cast<uint4*>(out);
    if (bf16)
      launch_pdl(quant_contig_kernel<true>, grid, threads, 0, stream, xv, chunks, ov, s_inv);
    else
      launch_pdl(quant_contig_kernel<false>, grid, threads, 0, stream, xv, chunks, ov, s_inv);
  } else if (aligned && cols % 16 == 0 && x_stride % 8 == 0 && out_stride % 16 == 0 &&
             rows < (1ll << 32) && rows * (cols / 16) < (1ll << 40)) {
    const uint64_t chunks = uint64_t(rows) * uint64_t(cols / 16);
    const uint64_t want = (chunks + 2 * threads - 1) / (2 * threads);
    const int grid = int(want < uint64_t(sms) * 8 ? (want ? want : 1) : uint64_t(sms) * 8);
    if (bf16)
      launch_pdl(quant_vec_kernel<true>, grid, threads, 0, stream, xs, uint32_t(rows),
                 uint32_t(cols / 16), x_stride, out, out_stride, s_inv);
    else
      launch_pdl(quant_vec_kernel<false>, grid, threads, 0, stream, xs, uint32_t(rows),
                 uint32_t(cols / 16), x_stride, out, out_stride, s_inv);
  } else {
    const int64_t total = rows * cols;
    const int64_t want = (total + threads - 1) / threads;
    const int grid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    if (bf16)
      launch_pdl(quant_scalar_kernel<true>, grid, threads, 0, stream, xs, rows, cols, x_stride, out, out_stride, s_inv);
    else
      launch_pdl(quant_scalar_kernel<false>, grid, threads, 0, stream, xs, rows, cols, x_stride, out, out_stride, s_inv);
  }
  return cudaGetLastError();
}

}  // namespace msa

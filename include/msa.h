/*
 * msa.h -- C ABI of libmsa.so: FP8 (e4m3) top-k block-sparse attention on
 * GB300 (sm_103a).
 *
 * The library computes the three steps of the sparse-attention hot path,
 * the quantised KV-cache store that feeds it (msa_kv_store_fp8) and a fused
 * rotary + quantisation producer of the MLA inputs (msa_rope_quant_fp8):
 *   (a) per-tensor e4m3 quantisation of Q and the indexer query
 *       -> msa_quant_fp8
 *   (b) indexer scores reduced per 128-token block, then a strictly
 *       ascending top-k of block ids into topk_indices[Hidx, T, topk]
 *       -> msa_index_topk
 *   (c) GQA sparse attention over the selected blocks with a per-head sink,
 *       prefill and paged decode -> msa_sparse_attn_fwd; and the sparse-MLA
 *       prefill variant over per-query token indices -> msa_sparse_mla_fwd
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named as tensors are DEVICE pointers; scale pointers
 *   (q_scale, k_scale, ...) are HOST pointers to one float, and NULL means
 *   unit scale (the C form of the pages' Optional[float] = None).
 * - Every output buffer and every workspace is owned by the caller and
 *   preallocated; the library never allocates device memory and never
 *   synchronises the stream. Work is enqueued on `stream` (NULL = the legacy
 *   default stream) and runs asynchronously.
 * - Kernels overwrite every element of their outputs, so callers may pass
 *   uninitialised buffers.
 * - Arguments are validated on the host before anything is launched. A
 *   failed check returns a non-zero msa_status and launches nothing;
 *   msa_last_error_string() then describes the failure (thread-local).
 * - Device-side data errors (a page id outside [0, num_pages), a wait that
 *   ran out its iteration limit) never trap: the kernel skips the bad tile,
 *   records a bit in a device error word and returns; msa_check_errors()
 *   reports and clears it.
 * - Layouts are row-major with the last dimension contiguous.
 *   KV page layout: [num_pages][Hkv][128 tokens][D] e4m3; one (page, head)
 *   tile is 16 KB contiguous. Index-K cache: [num_pages][128][d_idx] e4m3,
 *   with no head axis (shared by all index heads).
 * - Batch description: sequence b has seq_lens[b] tokens in its cache; its
 *   query tokens are the LAST q_len_b = cu_q[b+1]-cu_q[b] of them, stored at
 *   rows cu_q[b] .. cu_q[b+1]-1 of the query tensors. Prefill of one
 *   sequence: B = 1, cu_q = {0, T}, seq_lens = {T}. Decode: q_len_b = 1.
 *   max_q_len is the host's bound on q_len_b (1 selects the decode kernels).
 *   A sequence may have q_len_b = 0. With T = 0 every entry point returns
 *   MSA_OK at once, after checking its scalar arguments, without reading
 *   any pointer (max_q_len is not checked then).
 *   page_table[b * max_pages + j] is the physical page of logical block j.
 *
 * Sources: the four web pages this method is described on --
 *   [30971] sglang PR 30971 page, "M3 attention GEMMs fully fp8";
 *   [45892] vLLM PR 45892 page, "SM100 MSA indexer backend for MiniMax M3";
 *   [25751] sglang PR 25751 page, "SM90 Q8KV8 FP8 sparse MLA prefill kernel";
 *   [25460] sglang PR 25460 page, "prefill QKV quantize hook and FP8 Triton
 *           kernel".
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* msa_stream_t;

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,  /* null pointer, bad size or stride, misalignment */
  MSA_ERR_UNSUPPORTED = 2,  /* e5m2, head_dim / topk / page size not built */
  MSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MSA_ERR_TIMEOUT = 4,      /* a device wait ran out its iteration limit */
  MSA_ERR_WORKSPACE = 5,    /* workspace pointer NULL or smaller than required */
  MSA_ERR_DATA = 6          /* device-side data error (page id out of range) */
} msa_status;

typedef enum msa_dtype {
  MSA_BF16 = 0,
  MSA_FP16 = 1,
  MSA_E4M3 = 2,
  MSA_E5M2 = 3   /* never accepted: the e5m2 variant must not enter this path */
} msa_dtype;

/* Library version (major*10000 + minor*100 + patch). */
int msa_version(void);

/* Message describing the last non-OK status returned on this thread. */
const char* msa_last_error_string(void);

/*
 * Instrumentation, not part of the computation. While enabled (enable != 0),
 * every msa_sparse_attn_fwd and msa_sparse_mla_fwd call records a pair of
 * CUDA events on its stream around its main attention kernel (the prefill,
 * decode or MLA kernel; not the small planning, conversion or combine
 * kernels), every msa_index_topk / msa_index_topk_noalloc call from its
 * scoring kernel to the end of its selection kernel, and every
 * msa_quant_fp8_multi call around its one-launch kernel (when some tensor
 * went to it). msa_profile_last_ms waits for the most recent stop event and
 * returns the elapsed milliseconds. Disabled by default; the events belong to
 * the library (one pair per device). Do not enable during graph capture.
 */
msa_status msa_profile_enable(int enable);
msa_status msa_profile_last_ms(float* ms);

/*
 * Synchronises `stream`, then reads and clears the device error word.
 * Returns MSA_OK, MSA_ERR_DATA (bad page id / index seen by a kernel) or
 * MSA_ERR_TIMEOUT (a bounded device wait gave up), or MSA_ERR_CUDA.
 * This is the only entry point that synchronises; call it outside graph
 * capture.
 */
msa_status msa_check_errors(msa_stream_t stream);

/*
 * Debug switch (tests of the failure path; off by default, per device).
 * Every wait inside the library's kernels is bounded: when it runs out, the
 * kernel records MSA_ERR_TIMEOUT in the device error word, every role of the
 * block stops waiting, the block drains the copies and tensor-core
 * operations it already issued (waiting at most 2 s for each), frees its
 * tensor memory and returns. With on != 0, every wait that is not complete
 * at its first test gives up at once, so a test can drive that path without
 * anything hanging; the outputs of such calls are meaningless and the next
 * msa_check_errors returns MSA_ERR_TIMEOUT. Synchronous (copies one word to
 * the current device); call it outside graph capture.
 */
msa_status msa_debug_force_timeouts(int on);

/*
 * Step (a): out[r, c] = e4m3_rn_satfinite( fp32(x[r, c]) * s_inv ),
 * s_inv = 1.0f / *scale computed once in fp32 on the host, or 1 when scale
 * is NULL. [25460] key source excerpt (fp8_quantize: widen, multiply by
 * scale_inv, cast); [30971] implementation step 3 (_quant_q_fp8 on q and
 * idx_q; a missing scale means no division).
 *
 * x:        device, `rows` rows of `cols` bf16 or fp16 elements, row r at
 *           element offset r * x_row_stride (any leading dims flattened into
 *           rows; the last dim must be contiguous).
 * out:      device, e4m3 bytes, row r at byte offset r * out_row_stride.
 * x_dtype:  MSA_BF16 or MSA_FP16; out_dtype must be MSA_E4M3 (MSA_E5M2
 *           returns MSA_ERR_UNSUPPORTED; no silent reinterpretation).
 * rows/cols may be 0 (nothing is launched). Strides are in elements, >= cols.
 * Overflow saturates to +-448; NaN stays NaN.
 */
msa_status msa_quant_fp8(const void* x, msa_dtype x_dtype, int64_t rows, int64_t cols,
                         int64_t x_row_stride, void* out, msa_dtype out_dtype,
                         int64_t out_row_stride, const float* scale, msa_stream_t stream);

/*
 * Several step-(a) quantisations in one launch: each entry of `tensors` is
 * quantised exactly as msa_quant_fp8 would with the same x_dtype and
 * out_dtype (the same rounding, s_inv rule, saturation and NaN handling), so
 * the outputs are identical byte for byte; [30971] implementation step 3
 * quantises q and idx_q with their own scales, which is the use this serves:
 * one launch instead of one per tensor, so the tail of the first never idles
 * the GPU before the second starts.
 *
 * tensors:  host array of n descriptors, 1 <= n <= MSA_QUANT_MULTI_MAX; the
 *           descriptors and their scale pointers are read during the call
 *           only (caller-owned).
 * Contiguous tensors (row strides equal to cols, 16-byte aligned, rows*cols a
 * multiple of 16) share one launch; any other entry is handled as its own
 * msa_quant_fp8 call after it. Validation of every entry happens before any
 * launch; errors as msa_quant_fp8.
 */
#define MSA_QUANT_MULTI_MAX 8
typedef struct msa_quant_tensor {
  const void* x;             /* device, rows x cols of x_dtype, row r at r * x_row_stride */
  int64_t rows, cols, x_row_stride;
  void* out;                 /* device e4m3, row r at byte offset r * out_row_stride */
  int64_t out_row_stride;
  const float* scale;        /* host, NULL = unit scale */
} msa_quant_tensor;
msa_status msa_quant_fp8_multi(const msa_quant_tensor* tensors, int n, msa_dtype x_dtype,
                               msa_dtype out_dtype, msa_stream_t stream);

/*
 * The store before the path: quantise the new tokens' K, V and index-K rows
 * into the paged e4m3 pools. [30971] implementation step 4 (the sparse KV
 * pool's K / V / index-K stores, each with a per-tensor scale whose absence
 * means the unit scale and no division) and step 3 (the store runs before
 * the query quantiser); [45892] implementation step 3 (head-less index-K
 * cache).
 *
 * New token t of sequence b (rows cu_q[b] .. cu_q[b+1]-1, see the batch
 * description above) sits at position p = seq_lens[b] - q_len_b + (t - cu_q[b]),
 * physical page pg = page_table[b * max_pages + p / 128], slot s = p % 128:
 *   k_cache[pg][h][s][:]    = e4m3(fp32(k[t][h][:])  * s_inv_k)
 *   v_cache[pg][h][s][:]    = e4m3(fp32(v[t][h][:])  * s_inv_v)
 *   idx_k_cache[pg][s][:]   = e4m3(fp32(idx_k[t][:]) * s_inv_idx)
 * with the rounding and s_inv rule of msa_quant_fp8. No other byte of the
 * pools is written. Tokens must address distinct slots.
 *
 * k, v:      device, bf16 or fp16 (in_dtype), [T][Hkv][D]; token t at element
 *            offset t * k_token_stride (v_token_stride), [Hkv][D] contiguous
 *            within a token (so a slice of a fused QKV row works).
 * idx_k:     device, [T][d_idx], token stride idx_k_token_stride.
 *            Any of k, v, idx_k may be NULL: that pool is not touched and its
 *            cache pointer may be NULL too.
 * k_cache, v_cache: device, [num_pages][Hkv][128][D] e4m3 (updated in place).
 * idx_k_cache:      device, [num_pages][128][d_idx] e4m3 (updated in place).
 * Requirements (MSA_ERR_INVALID_ARG otherwise): D and d_idx positive
 *   multiples of 16 for the parts given; token strides >= the row and
 *   multiples of 8 elements; every given input and cache 16-byte aligned;
 *   B, max_pages, num_pages >= 1. T = 0 returns MSA_OK after these scalar
 *   checks without reading any pointer.
 * Data errors (a position with no page-table entry, a page id outside
 *   [0, num_pages), q_len_b > seq_lens[b], a row beyond cu_q[B]): that token
 *   is skipped and MSA_ERR_DATA is recorded for msa_check_errors().
 */
msa_status msa_kv_store_fp8(const void* k, const void* v, const void* idx_k, msa_dtype in_dtype,
                            int64_t k_token_stride, int64_t v_token_stride,
                            int64_t idx_k_token_stride, const int32_t* page_table,
                            const int32_t* seq_lens, const int32_t* cu_q, int B, int T,
                            int max_pages, int num_pages, int Hkv, int D, int d_idx,
                            const float* k_scale, const float* v_scale, const float* idx_k_scale,
                            void* k_cache, void* v_cache, void* idx_k_cache, msa_stream_t stream);

/*
 * Fused producer of the sparse-MLA inputs: rotary embedding of the pe part
 * and e4m3 quantisation of nope || rope(pe) as one row. [25460]
 * implementation step 2 and the _fused_rope_fp8_quantize excerpt (nope and
 * rotated pe written side by side, a k_pe shared by all heads broadcast,
 * neox flag, per-tensor quantisation scale); key source excerpt of
 * fp8_quantize (widen to fp32, scale, cast).
 *
 * For row r (a token), head h, with p = positions[r], C = cos_sin_cache[p][0 .. d_rope/2),
 * S = cos_sin_cache[p][d_rope/2 .. d_rope):
 *   is_neox != 0: x1 = pe[.. d_rope/2), x2 = pe[d_rope/2 ..);
 *                 rot = (x1*C - x2*S, x2*C + x1*S)
 *   is_neox == 0: pairs (pe[2i], pe[2i+1]) -> (pe[2i]*C[i] - pe[2i+1]*S[i],
 *                 pe[2i+1]*C[i] + pe[2i]*S[i])
 *   out[r][h][0 .. d_nope)               = e4m3(fp32(nope[r][h][:]) * s_inv)
 *   out[r][h][d_nope .. d_nope + d_rope) = e4m3(rot * s_inv)
 * in fp32 with every product and sum rounded on its own (no FMA), s_inv as in
 * msa_quant_fp8 (NULL scale = no multiply), the same RNE-satfinite cast.
 *
 * nope:  device, bf16/fp16 [rows][heads][d_nope]; element (r, h, i) at
 *        r * nope_token_stride + h * nope_head_stride + i. May be NULL when
 *        d_nope = 0.
 * pe:    device, same dtype, [rows][heads][d_rope] with its own strides;
 *        pe_head_stride = 0 broadcasts one pe row (a shared k_pe) to all heads.
 * cos_sin_cache: device fp32 [max_pos][d_rope]; positions: device int32 [rows].
 * out:   device, e4m3 [rows][heads][d_nope + d_rope], contiguous, written in full.
 * Requirements (MSA_ERR_INVALID_ARG otherwise): d_nope a multiple of 16,
 *   d_rope a positive multiple of 32, strides non-negative multiples of 8,
 *   nope / pe / cos_sin_cache / out 16-byte aligned. rows = 0 returns MSA_OK
 *   after the scalar checks without reading any pointer.
 * A position outside [0, max_pos) writes zeros to that row's rope part and
 *   records MSA_ERR_DATA for msa_check_errors().
 */
msa_status msa_rope_quant_fp8(const void* nope, const void* pe, msa_dtype in_dtype, int64_t rows,
                              int heads, int d_nope, int d_rope, int64_t nope_token_stride,
                              int64_t nope_head_stride, int64_t pe_token_stride,
                              int64_t pe_head_stride, const float* cos_sin_cache, int max_pos,
                              const int32_t* positions, int is_neox, const float* scale, void* out,
                              msa_stream_t stream);

/* Bytes of device workspace msa_index_topk needs for these sizes. */
size_t msa_index_topk_workspace_size(int T, int Hidx, int max_pages);

/*
 * Step (b): block scores and the ascending top-k.
 * For index head i and query token t at position p (own block o = p / 128):
 *   score[i, t, j] = max over the 128 keys k of block j < o of
 *                    dot(idx_q[t, i, :], idx_k[k, :])   (codes, fp32 accum.)
 * topk_indices[i, t, :] = if o + 1 <= topk: 0, 1, ..., o, then -1 padding;
 *   else: the topk-1 highest-scoring blocks j < o (equal scores: lower id
 *   first) in ascending order, followed by o.
 * [45892] implementation steps 1-4 (per-page max score, head-less fp8
 * index cache, shared topk_indices_buffer [index_heads, tokens, topk]);
 * [30971] implementation step 2 and review item 2 (strictly ascending ids,
 * -1 padding when the causal blocks do not exceed topk). Forcing the own
 * block and the tie order are readings of this library.
 *
 * idx_q:        device e4m3 [T][Hidx][D]
 * idx_k_cache:  device e4m3 [num_pages][128][D]
 * page_table:   device int32 [B][max_pages]
 * seq_lens:     device int32 [B];  cu_q: device int32 [B+1]
 * topk_indices: device int32 [Hidx][T][topk] (written in full)
 * workspace:    device, >= msa_index_topk_workspace_size(T, Hidx, max_pages)
 *               bytes, 256-byte aligned; contents on entry are ignored.
 * Supported: D in {64, 128}; 1 <= topk <= 64; Hidx a power of two <= 16;
 * max_pages <= 2048.
 * Data errors (a sequence whose seq_len exceeds max_pages * 128 or is below
 * its query count, a row past cu_q[B], a page id outside [0, num_pages)):
 *   MSA_ERR_DATA is recorded for msa_check_errors(); the rows of tokens that
 *   belong to no valid sequence are written as -1.
 */
msa_status msa_index_topk(const uint8_t* idx_q, const uint8_t* idx_k_cache,
                          const int32_t* page_table, const int32_t* seq_lens,
                          const int32_t* cu_q, int B, int T, int max_q_len, int Hidx, int D,
                          int topk, int num_pages, int max_pages, int32_t* topk_indices,
                          void* workspace, size_t workspace_bytes, msa_stream_t stream);

/*
 * msa_index_topk for callers that cannot allocate device memory. The pages
 * have no counterpart to this entry point; it exists for this library's users.
 *
 * Same arguments, results and errors as msa_index_topk, without the
 * workspace: the scratch lives in one fixed 8 MiB array in the library's
 * device image (held on every GPU that loads the library until exit). Meant
 * for callers that get only their input and output pointers from a host
 * engine with no workspace hook, or that reserve all device memory up front
 * and may not call cudaMalloc afterwards. It calls no allocator.
 * - Sizes whose scratch (msa_index_topk_workspace_size(T, Hidx, max_pages))
 *   exceeds 8 MiB are rejected with MSA_ERR_WORKSPACE before any launch; the
 *   paged-decode workload (128 sequences x 4 index heads x 512 pages, 1 MiB)
 *   and short prefills fit, long prefills need msa_index_topk.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current).
 * - Every call uses the same array and leaves its contents behind; calls
 *   that may run at the same time on the GPU (unordered streams) race on it
 *   and must be serialised by the caller. No contents need to start at zero.
 */
msa_status msa_index_topk_noalloc(const uint8_t* idx_q, const uint8_t* idx_k_cache,
                                  const int32_t* page_table, const int32_t* seq_lens,
                                  const int32_t* cu_q, int B, int T, int max_q_len, int Hidx,
                                  int D, int topk, int num_pages, int max_pages,
                                  int32_t* topk_indices, msa_stream_t stream);

/* Bytes of device workspace msa_sparse_attn_fwd needs for these sizes. */
size_t msa_sparse_attn_workspace_size(int B, int T, int max_q_len, int Hq, int Hkv, int Hidx,
                                      int topk, int max_pages);

/*
 * Step (c): GQA sparse attention over the selected blocks.
 * Query row (t, h) uses index head i = h / (Hq/Hidx) and kv head
 * g = h / (Hq/Hkv); it attends to every key of the blocks listed in
 * topk_indices[i, t, :] (ids < 0 ignored) whose position is <= its own.
 * With c = sm_scale * q_scale:
 *   l_j      = c * k_scale * dot(q[t,h,:], k_j)     (codes)
 *   sigma    = c * sink[h]                          (no k_scale)
 *   out      = v_scale * sum_j e^{l_j} v_j / (sum_j e^{l_j} + e^{sigma})
 *   max_logit = max_j l_j;   lse = ln(sum_j e^{l_j} + e^{sigma})
 * (no sigma terms when sink is NULL). [30971] implementation step 3 and the
 * executive summary: q_scale folded into sm_scale acts on the dot and the
 * sink; k_scale never touches the sink; v_scale scales the output.
 * [45892] step 2: attention reads the topk buffer the indexer wrote.
 *
 * q:            device e4m3 [T][Hq][D]
 * k_cache, v_cache: device e4m3 [num_pages][Hkv][128][D]
 * topk_indices: device int32 [Hidx][T][topk], ascending, -1 padded
 * sink:         device fp32 [Hq] or NULL
 * out:          device bf16 [T][Hq][D];  max_logit, lse: device fp32 [T][Hq]
 * workspace:    device, >= msa_sparse_attn_workspace_size(...) bytes,
 *               256-byte aligned; contents on entry are ignored. Prefill
 *               keeps f16 V^T page images there, decode its per-chunk
 *               partial softmax states.
 * Supported: D == 128; Hq % Hkv == 0, Hq % Hidx == 0, Hq/Hkv a power of two
 * <= 16; 1 <= topk <= 64.
 */
msa_status msa_sparse_attn_fwd(const uint8_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                               const int32_t* page_table, const int32_t* seq_lens,
                               const int32_t* cu_q, const int32_t* topk_indices,
                               const float* sink, float sm_scale, const float* q_scale,
                               const float* k_scale, const float* v_scale, int B, int T,
                               int max_q_len, int Hq, int Hkv, int Hidx, int D, int topk,
                               int num_pages, int max_pages, uint16_t* out, float* max_logit,
                               float* lse, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream);

/*
 * Step (c), sparse-MLA prefill: MQA of H query heads over one latent kv head.
 * Query t attends to kv rows indices[t, j] for j < topk_length[t] (all topk
 * when topk_length is NULL), skipping negative entries; V is the first d_v
 * columns of the same rows. With c = sm_scale * q_scale:
 *   l_j = c * kv_scale * dot(q[t,h,:], kv[idx_j, :]);  sigma = c * sink[h]
 *   out = kv_scale * sum_j e^{l_j} kv[idx_j, :d_v] / (sum_j e^{l_j} + e^{sigma})
 *   max_logits = max_j l_j;  lse = ln(sum_j e^{l_j} + e^{sigma})
 * [25751] key source excerpt (sparse_mla_q8kv8_prefill_fwd: q, kv, indices,
 * sm_scale, q_scale, kv_scale, d_v, attn_sink, topk_length; caller-owned
 * out [s_q, h_q, d_v] bf16, max_logits and lse [s_q, h_q] fp32; d_v other
 * than 512 is rejected).
 *
 * q:   device e4m3 [T][H][d_qk];  kv: device e4m3 [S_kv][d_qk]
 * indices: device int32 [T][topk];  topk_length: device int32 [T] or NULL
 * sink: device fp32 [H] or NULL
 * out: device bf16 [T][H][d_v];  max_logits, lse: device fp32 [T][H]
 * Supported: d_qk == 576, d_v == 512, H == 128, topk a multiple of 64.
 * An index >= S_kv is a data error (recorded, key skipped).
 */
msa_status msa_sparse_mla_fwd(const uint8_t* q, const uint8_t* kv, const int32_t* indices,
                              const int32_t* topk_length, const float* sink, float sm_scale,
                              const float* q_scale, const float* kv_scale, int T, int H,
                              int S_kv, int d_qk, int d_v, int topk, uint16_t* out,
                              float* max_logits, float* lse, msa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */

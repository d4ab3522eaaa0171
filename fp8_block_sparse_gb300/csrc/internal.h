// internal.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "msa.h"

namespace msa {

// Bits of the device error word.
constexpr unsigned MSA_DEVERR_DATA = 1u;     // bad page id / index seen by a kernel
constexpr unsigned MSA_DEVERR_TIMEOUT = 2u;  // a bounded wait gave up

// Per-device state in the library image. Kernels get the address of `err`
// (the first member) and find the rest through it.
struct DeviceState {
  unsigned err;              // MSA_DEVERR_* bits, cleared by msa_check_errors
  unsigned force_timeouts;   // debug: nonzero makes every unfinished wait give up
};

// Sets the message msa_last_error_string() returns on this thread.
void set_last_error(const std::string& msg);

// Device address of this device's error word, the first member of its
// DeviceState (set up once per device).
unsigned* device_error_word();

// Builds a tiled TMA descriptor through the driver entry point. Returns false
// (and fills `why`) when the driver rejects it.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle, const char** why);

int num_sms();

// Launches a kernel with programmatic stream serialisation (programmatic
// dependent launch): its blocks may be scheduled while the previous kernel in
// the stream is still finishing, and wait in griddepcontrol.wait (pdl_wait)
// for that kernel's completion before touching global memory. Every kernel of
// the library begins with that wait, in every block, so a kernel never
// completes before the one it follows and the chain stays ordered; outside a
// chain of such kernels the attribute changes nothing.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Instrumentation: records the start (which = 0) or stop (which = 1) event
// around a main attention kernel when profiling is enabled; no-op otherwise.
void profile_mark(cudaStream_t stream, int which);

// Step (a).
cudaError_t launch_quant(const void* x, bool bf16, int64_t rows, int64_t cols, int64_t x_stride,
                         uint8_t* out, int64_t out_stride, float s_inv, cudaStream_t stream);

// Step (a) over several contiguous tensors in one launch (blocks are dealt
// to the tensors in proportion to their sizes).
struct QuantMulti {
  int n;
  const uint4* x[MSA_QUANT_MULTI_MAX];
  uint4* out[MSA_QUANT_MULTI_MAX];
  uint64_t chunks[MSA_QUANT_MULTI_MAX];    // 16-element chunks of each tensor
  float s_inv[MSA_QUANT_MULTI_MAX];
  int block0[MSA_QUANT_MULTI_MAX + 1];     // first block of each tensor; block0[n] = grid
};
cudaError_t launch_quant_multi(QuantMulti& q, bool bf16, cudaStream_t stream);
// Whether msa_quant_fp8_multi can take this tensor into its single launch.
bool quant_multi_eligible(const void* x, const void* out, int64_t rows, int64_t cols,
                          int64_t x_stride, int64_t out_stride);

// The quantised KV-cache store (before the path). Token strides in elements.
struct KvStoreArgs {
  const uint16_t* k;       // [T][Hkv][D] or null
  const uint16_t* v;       // [T][Hkv][D] or null
  const uint16_t* idx_k;   // [T][d_idx] or null
  int64_t k_stride, v_stride, idx_stride;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int B, T, max_pages, num_pages, Hkv, D, d_idx;
  float k_sinv, v_sinv, i_sinv;
  uint8_t* k_cache;        // [num_pages][Hkv][128][D]
  uint8_t* v_cache;
  uint8_t* idx_cache;      // [num_pages][128][d_idx]
  unsigned* err;
};
cudaError_t launch_kv_store(const KvStoreArgs& a, bool bf16, cudaStream_t stream);

// Fused rotary embedding + quantisation: out[r][h] = e4m3(nope || rope(pe)).
// Strides in elements; pe_head_stride 0 broadcasts one pe row to every head.
struct RopeQuantArgs {
  const uint16_t* nope;
  const uint16_t* pe;
  int64_t nope_tok_stride, nope_head_stride, pe_tok_stride, pe_head_stride;
  const float* cos_sin;      // [max_pos][d_rope]: d_rope/2 cosines, then d_rope/2 sines
  int max_pos;
  const int32_t* positions;  // [rows]
  int64_t rows;
  int heads, d_nope, d_rope;
  float s_inv;
  uint8_t* out;              // [rows][heads][d_nope + d_rope]
  unsigned* err;
};
cudaError_t launch_rope_quant(const RopeQuantArgs& a, bool bf16, bool neox, cudaStream_t stream);

// Step (b). Scores go to `scores` [Hidx][T][max_pages] fp32 (workspace).
struct IndexArgs {
  const uint8_t* idx_q;
  const uint8_t* idx_k;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int B, T, max_q_len, Hidx, D, topk, num_pages, max_pages;
  int32_t* topk_indices;
  float* scores;
  unsigned* err;
};
cudaError_t launch_index_topk(const IndexArgs& a, cudaStream_t stream, const char** why);
// The scalar and support checks of msa_index_topk (every check that needs no
// pointer), in its order; fills the last-error message and returns its status.
msa_status check_index_topk_sizes(const char* fn, int B, int T, int max_q_len, int Hidx, int D,
                                  int topk, int num_pages, int max_pages);
size_t index_workspace_bytes(int T, int Hidx, int max_pages);

// Step (c), GQA.
struct AttnArgs {
  const uint8_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  const int32_t* topk;
  const float* sink;
  float c_qk;      // sm_scale * q_scale * k_scale
  float c_sink;    // sm_scale * q_scale
  float v_scale;
  int B, T, max_q_len, Hq, Hkv, Hidx, D, topk_k, num_pages, max_pages;
  uint16_t* out;
  float* max_logit;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  unsigned* err;
};
cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream, const char** why);
size_t attn_workspace_bytes(int B, int T, int max_q_len, int Hq, int Hkv, int Hidx, int topk,
                            int max_pages);

// Step (c), sparse MLA.
struct MlaArgs {
  const uint8_t* q;
  const uint8_t* kv;
  const int32_t* indices;
  const int32_t* topk_length;
  const float* sink;
  float c_qk, c_sink, v_scale;
  int T, H, S_kv, d_qk, d_v, topk;
  uint16_t* out;
  float* max_logits;
  float* lse;
  unsigned* err;
};
cudaError_t launch_sparse_mla(const MlaArgs& a, cudaStream_t stream, const char** why);

}  // namespace msa

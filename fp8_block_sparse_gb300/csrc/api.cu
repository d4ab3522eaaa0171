// api.cu -- the C ABI of libmsa.so (include/msa.h): argument validation,
// scale folding, workspace checks and dispatch to the kernel launchers.
// Nothing here allocates device memory or synchronises a stream (except
// msa_check_errors, which exists to do exactly that).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "msa.h"
#include "internal.h"

namespace msa {

__device__ DeviceState g_msa_state;

namespace {

thread_local std::string g_last_error;

msa_status fail(msa_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

msa_status cuda_fail(cudaError_t e, const char* where, const char* why = nullptr) {
  std::string m = std::string(where) + ": " + cudaGetErrorString(e);
  if (why) m += std::string(" (") + why + ")";
  g_last_error = m;
  return MSA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_profile = false;
cudaEvent_t g_ev[kMaxDevices][2] = {};

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// A missing scale is the unit scale; a given one must be finite and positive.
bool read_scale(const float* s, float* out, const char* name) {
  if (s == nullptr) {
    *out = 1.0f;
    return true;
  }
  if (!std::isfinite(*s) || !(*s > 0.0f)) {
    g_last_error = std::string(name) + " must be finite and > 0";
    return false;
  }
  *out = *s;
  return true;
}

}  // namespace

void set_last_error(const std::string& msg) { g_last_error = msg; }

unsigned* device_error_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_err_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_msa_state) != cudaSuccess) return nullptr;
    g_err_ptr[d] = &static_cast<DeviceState*>(p)->err;
  }
  return g_err_ptr[d];
}

int num_sms() {
  const int d = current_device();
  if (d < 0) return 148;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_sms[d] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 148;
  }
  return g_sms[d];
}

void profile_mark(cudaStream_t stream, int which) {
  if (!g_profile) return;
  const int d = current_device();
  if (d < 0) return;
  cudaEvent_t ev;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_ev[d][0] == nullptr) {
      if (cudaEventCreate(&g_ev[d][0]) != cudaSuccess || cudaEventCreate(&g_ev[d][1]) != cudaSuccess)
        return;
    }
    ev = g_ev[d][which];
  }
  cudaEventRecord(ev, stream);
}

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle, const char** why) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        *why = "cuTensorMapEncodeTiled entry point unavailable";
        return false;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  std::memset(map, 0, sizeof(*map));
  CUresult r = g_encode(map, dtype, rank, const_cast<void*>(base), d, s, b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled rejected the tensor (alignment or extent)";
    return false;
  }
  return true;
}

msa_status check_index_topk_sizes(const char* fn, int B, int T, int max_q_len, int Hidx, int D,
                                  int topk, int num_pages, int max_pages) {
  if (B < 1 || T < 0 || Hidx < 1 || num_pages < 1 || max_pages < 1)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": bad B/T/Hidx/num_pages/max_pages");
  if (T > 0 && (max_q_len < 1 || max_q_len > T))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": max_q_len must be in [1, T]");
  if (D != 64 && D != 128)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": index head dim must be 64 or 128");
  if (topk < 1 || topk > 64)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": topk must be in [1, 64]");
  if (Hidx > 16 || (Hidx & (Hidx - 1)) != 0)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": Hidx must be a power of two <= 16");
  if (max_pages > 2048)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": max_pages must be <= 2048");
  return MSA_OK;
}

}  // namespace msa

using namespace msa;

extern "C" {

int msa_version(void) { return 100; }

const char* msa_last_error_string(void) { return g_last_error.c_str(); }

msa_status msa_profile_enable(int enable) {
  g_profile = enable != 0;
  return MSA_OK;
}

msa_status msa_profile_last_ms(float* ms) {
  if (ms == nullptr) return fail(MSA_ERR_INVALID_ARG, "msa_profile_last_ms: null pointer");
  const int d = current_device();
  if (d < 0 || g_ev[d][0] == nullptr)
    return fail(MSA_ERR_INVALID_ARG, "msa_profile_last_ms: nothing was profiled on this device");
  cudaError_t e = cudaEventSynchronize(g_ev[d][1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, g_ev[d][0], g_ev[d][1]);
  if (e != cudaSuccess) return cuda_fail(e, "msa_profile_last_ms");
  return MSA_OK;
}

msa_status msa_check_errors(msa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "msa_check_errors");
  unsigned* p = device_error_word();
  if (p == nullptr) return fail(MSA_ERR_CUDA, "msa_check_errors: no device error word");
  unsigned word = 0;
  e = cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "msa_check_errors");
  e = cudaMemset(p, 0, sizeof(unsigned));
  if (e != cudaSuccess) return cuda_fail(e, "msa_check_errors");
  if (word & MSA_DEVERR_TIMEOUT) return fail(MSA_ERR_TIMEOUT, "a device wait ran out its limit");
  if (word & MSA_DEVERR_DATA)
    return fail(MSA_ERR_DATA, "a kernel saw a page id or index outside its valid range");
  return MSA_OK;
}

msa_status msa_debug_force_timeouts(int on) {
  unsigned* p = device_error_word();
  if (p == nullptr) return fail(MSA_ERR_CUDA, "msa_debug_force_timeouts: no device state");
  const unsigned v = on ? 1u : 0u;
  DeviceState* st = reinterpret_cast<DeviceState*>(p);
  const cudaError_t e = cudaMemcpy(&st->force_timeouts, &v, sizeof(v), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "msa_debug_force_timeouts");
  return MSA_OK;
}

msa_status msa_quant_fp8(const void* x, msa_dtype x_dtype, int64_t rows, int64_t cols,
                         int64_t x_row_stride, void* out, msa_dtype out_dtype,
                         int64_t out_row_stride, const float* scale, msa_stream_t stream) {
  if (out_dtype == MSA_E5M2)
    return fail(MSA_ERR_UNSUPPORTED, "msa_quant_fp8: e5m2 output is not supported (e4m3 only)");
  if (out_dtype != MSA_E4M3) return fail(MSA_ERR_INVALID_ARG, "msa_quant_fp8: out_dtype must be MSA_E4M3");
  if (x_dtype != MSA_BF16 && x_dtype != MSA_FP16)
    return fail(MSA_ERR_INVALID_ARG, "msa_quant_fp8: x_dtype must be MSA_BF16 or MSA_FP16");
  if (rows < 0 || cols < 0) return fail(MSA_ERR_INVALID_ARG, "msa_quant_fp8: negative size");
  float s = 1.0f;
  if (!read_scale(scale, &s, "msa_quant_fp8: scale")) return MSA_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MSA_OK;
  if (x == nullptr || out == nullptr) return fail(MSA_ERR_INVALID_ARG, "msa_quant_fp8: null pointer");
  if (x_row_stride < cols || out_row_stride < cols)
    return fail(MSA_ERR_INVALID_ARG, "msa_quant_fp8: row stride smaller than cols");
  if (!aligned(x, 2)) return fail(MSA_ERR_INVALID_ARG, "msa_quant_fp8: x not 2-byte aligned");
  const float s_inv = (scale == nullptr) ? 1.0f : 1.0f / s;
  cudaError_t e = launch_quant(x, x_dtype == MSA_BF16, rows, cols, x_row_stride,
                               static_cast<uint8_t*>(out), out_row_stride, s_inv,
                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "msa_quant_fp8");
  return MSA_OK;
}

msa_status msa_quant_fp8_multi(const msa_quant_tensor* tensors, int n, msa_dtype x_dtype,
                               msa_dtype out_dtype, msa_stream_t stream) {
  const char* fn = "msa_quant_fp8_multi";
  if (out_dtype == MSA_E5M2)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": e5m2 output is not supported (e4m3 only)");
  if (out_dtype != MSA_E4M3) return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": out_dtype must be MSA_E4M3");
  if (x_dtype != MSA_BF16 && x_dtype != MSA_FP16)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": x_dtype must be MSA_BF16 or MSA_FP16");
  if (tensors == nullptr || n < 1 || n > MSA_QUANT_MULTI_MAX)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": need 1 <= n <= MSA_QUANT_MULTI_MAX tensors");
  float s_inv[MSA_QUANT_MULTI_MAX];
  for (int i = 0; i < n; ++i) {            // every entry is validated before any launch
    const msa_quant_tensor& t = tensors[i];
    const std::string at = std::string(fn) + ": tensor " + std::to_string(i);
    if (t.rows < 0 || t.cols < 0) return fail(MSA_ERR_INVALID_ARG, at + ": negative size");
    float sc = 1.0f;
    if (!read_scale(t.scale, &sc, (at + ": scale").c_str())) return MSA_ERR_INVALID_ARG;
    s_inv[i] = t.scale == nullptr ? 1.0f : 1.0f / sc;
    if (t.rows == 0 || t.cols == 0) continue;
    if (t.x == nullptr || t.out == nullptr) return fail(MSA_ERR_INVALID_ARG, at + ": null pointer");
    if (t.x_row_stride < t.cols || t.out_row_stride < t.cols)
      return fail(MSA_ERR_INVALID_ARG, at + ": row stride smaller than cols");
    if (!aligned(t.x, 2)) return fail(MSA_ERR_INVALID_ARG, at + ": x not 2-byte aligned");
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  QuantMulti q{};
  for (int i = 0; i < n; ++i) {
    const msa_quant_tensor& t = tensors[i];
    if (t.rows == 0 || t.cols == 0) continue;
    if (!quant_multi_eligible(t.x, t.out, t.rows, t.cols, t.x_row_stride, t.out_row_stride)) continue;
    q.x[q.n] = static_cast<const uint4*>(t.x);
    q.out[q.n] = static_cast<uint4*>(t.out);
    q.chunks[q.n] = uint64_t(t.rows * t.cols) / 16;
    q.s_inv[q.n] = s_inv[i];
    ++q.n;
  }
  if (q.n > 0) profile_mark(st, 0);
  cudaError_t e = launch_quant_multi(q, x_dtype == MSA_BF16, st);
  if (q.n > 0) profile_mark(st, 1);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  for (int i = 0; i < n; ++i) {            // the rest, one launch each
    const msa_quant_tensor& t = tensors[i];
    if (t.rows == 0 || t.cols == 0) continue;
    if (quant_multi_eligible(t.x, t.out, t.rows, t.cols, t.x_row_stride, t.out_row_stride)) continue;
    e = launch_quant(t.x, x_dtype == MSA_BF16, t.rows, t.cols, t.x_row_stride,
                     static_cast<uint8_t*>(t.out), t.out_row_stride, s_inv[i], st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
  }
  return MSA_OK;
}

msa_status msa_kv_store_fp8(const void* k, const void* v, const void* idx_k, msa_dtype in_dtype,
                            int64_t k_token_stride, int64_t v_token_stride,
                            int64_t idx_k_token_stride, const int32_t* page_table,
                            const int32_t* seq_lens, const int32_t* cu_q, int B, int T,
                            int max_pages, int num_pages, int Hkv, int D, int d_idx,
                            const float* k_scale, const float* v_scale, const float* idx_k_scale,
                            void* k_cache, void* v_cache, void* idx_k_cache, msa_stream_t stream) {
  const char* fn = "msa_kv_store_fp8";
  if (in_dtype != MSA_BF16 && in_dtype != MSA_FP16)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": in_dtype must be MSA_BF16 or MSA_FP16");
  if (B < 1 || T < 0 || max_pages < 1 || num_pages < 1)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": need B >= 1, T >= 0, max_pages >= 1, num_pages >= 1");
  const bool has_kv = k != nullptr || v != nullptr;
  if (has_kv && (Hkv < 1 || D < 16 || D % 16 != 0 || int64_t(Hkv) * D > (1 << 20)))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": need Hkv >= 1 and D a positive multiple of 16");
  if (idx_k != nullptr && (d_idx < 16 || d_idx % 16 != 0 || d_idx > (1 << 20)))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": d_idx must be a positive multiple of 16");
  float ks = 1.0f, vs = 1.0f, is = 1.0f;
  if (!read_scale(k_scale, &ks, "msa_kv_store_fp8: k_scale") ||
      !read_scale(v_scale, &vs, "msa_kv_store_fp8: v_scale") ||
      !read_scale(idx_k_scale, &is, "msa_kv_store_fp8: idx_k_scale"))
    return MSA_ERR_INVALID_ARG;
  if (T == 0 || (!has_kv && idx_k == nullptr)) return MSA_OK;
  if (page_table == nullptr || seq_lens == nullptr || cu_q == nullptr)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": null batch description");
  const struct { const void* x; void* cache; int64_t stride, row; const char* name; } parts[3] = {
      {k, k_cache, k_token_stride, int64_t(Hkv) * D, "k"},
      {v, v_cache, v_token_stride, int64_t(Hkv) * D, "v"},
      {idx_k, idx_k_cache, idx_k_token_stride, int64_t(d_idx), "idx_k"}};
  for (const auto& p : parts) {
    if (p.x == nullptr) continue;
    if (p.cache == nullptr)
      return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": " + p.name + " given without its cache");
    if (p.stride < p.row || p.stride % 8 != 0)
      return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": " + p.name +
                                           " token stride must be >= its row and a multiple of 8");
    if (!aligned(p.x, 16) || !aligned(p.cache, 16))
      return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": " + p.name + " and its cache must be 16-byte aligned");
  }
  KvStoreArgs a;
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.idx_k = static_cast<const uint16_t*>(idx_k);
  a.k_stride = k_token_stride;
  a.v_stride = v_token_stride;
  a.idx_stride = idx_k_token_stride;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.cu_q = cu_q;
  a.B = B;
  a.T = T;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.Hkv = has_kv ? Hkv : 0;
  a.D = has_kv ? D : 16;
  a.d_idx = idx_k ? d_idx : 16;
  a.k_sinv = k_scale ? 1.0f / ks : 1.0f;
  a.v_sinv = v_scale ? 1.0f / vs : 1.0f;
  a.i_sinv = idx_k_scale ? 1.0f / is : 1.0f;
  a.k_cache = static_cast<uint8_t*>(k_cache);
  a.v_cache = static_cast<uint8_t*>(v_cache);
  a.idx_cache = static_cast<uint8_t*>(idx_k_cache);
  a.err = device_error_word();
  if (a.err == nullptr) return fail(MSA_ERR_CUDA, std::string(fn) + ": no device error word");
  cudaError_t e = launch_kv_store(a, in_dtype == MSA_BF16, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return MSA_OK;
}

msa_status msa_rope_quant_fp8(const void* nope, const void* pe, msa_dtype in_dtype, int64_t rows,
                              int heads, int d_nope, int d_rope, int64_t nope_token_stride,
                              int64_t nope_head_stride, int64_t pe_token_stride,
                              int64_t pe_head_stride, const float* cos_sin_cache, int max_pos,
                              const int32_t* positions, int is_neox, const float* scale, void* out,
                              msa_stream_t stream) {
  const std::string fn = "msa_rope_quant_fp8";
  if (in_dtype != MSA_BF16 && in_dtype != MSA_FP16)
    return fail(MSA_ERR_INVALID_ARG, fn + ": in_dtype must be MSA_BF16 or MSA_FP16");
  if (rows < 0 || heads < 1 || max_pos < 1)
    return fail(MSA_ERR_INVALID_ARG, fn + ": need rows >= 0, heads >= 1, max_pos >= 1");
  if (d_nope < 0 || d_nope % 16 != 0 || d_rope < 32 || d_rope % 32 != 0 || d_nope + d_rope > (1 << 16))
    return fail(MSA_ERR_INVALID_ARG, fn + ": d_nope must be a multiple of 16 and d_rope a positive multiple of 32");
  float sc = 1.0f;
  if (!read_scale(scale, &sc, "msa_rope_quant_fp8: scale")) return MSA_ERR_INVALID_ARG;
  if (rows == 0) return MSA_OK;
  if (pe == nullptr || cos_sin_cache == nullptr || positions == nullptr || out == nullptr ||
      (d_nope > 0 && nope == nullptr))
    return fail(MSA_ERR_INVALID_ARG, fn + ": null pointer");
  const bool strides_ok = nope_token_stride >= 0 && nope_head_stride >= 0 && pe_token_stride >= 0 &&
                          pe_head_stride >= 0 && nope_token_stride % 8 == 0 &&
                          nope_head_stride % 8 == 0 && pe_token_stride % 8 == 0 &&
                          pe_head_stride % 8 == 0;
  if (!strides_ok) return fail(MSA_ERR_INVALID_ARG, fn + ": strides must be non-negative multiples of 8 elements");
  if ((d_nope > 0 && !aligned(nope, 16)) || !aligned(pe, 16) || !aligned(cos_sin_cache, 16) ||
      !aligned(out, 16))
    return fail(MSA_ERR_INVALID_ARG, fn + ": nope, pe, cos_sin_cache and out must be 16-byte aligned");
  RopeQuantArgs a;
  a.nope = static_cast<const uint16_t*>(nope);
  a.pe = static_cast<const uint16_t*>(pe);
  a.nope_tok_stride = nope_token_stride;
  a.nope_head_stride = nope_head_stride;
  a.pe_tok_stride = pe_token_stride;
  a.pe_head_stride = pe_head_stride;
  a.cos_sin = cos_sin_cache;
  a.max_pos = max_pos;
  a.positions = positions;
  a.rows = rows;
  a.heads = heads;
  a.d_nope = d_nope;
  a.d_rope = d_rope;
  a.s_inv = scale ? 1.0f / sc : 1.0f;
  a.out = static_cast<uint8_t*>(out);
  a.err = device_error_word();
  if (a.err == nullptr) return fail(MSA_ERR_CUDA, fn + ": no device error word");
  cudaError_t e = launch_rope_quant(a, in_dtype == MSA_BF16, is_neox != 0,
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn.c_str());
  return MSA_OK;
}

size_t msa_index_topk_workspace_size(int T, int Hidx, int max_pages) {
  if (T < 0 || Hidx < 0 || max_pages < 0) return 0;
  return index_workspace_bytes(T, Hidx, max_pages);
}

msa_status msa_index_topk(const uint8_t* idx_q, const uint8_t* idx_k_cache,
                          const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q,
                          int B, int T, int max_q_len, int Hidx, int D, int topk, int num_pages,
                          int max_pages, int32_t* topk_indices, void* workspace,
                          size_t workspace_bytes, msa_stream_t stream) {
  const char* fn = "msa_index_topk";
  const msa_status st = check_index_topk_sizes(fn, B, T, max_q_len, Hidx, D, topk, num_pages, max_pages);
  if (st != MSA_OK) return st;
  if (T == 0) return MSA_OK;
  if (!idx_q || !idx_k_cache || !page_table || !seq_lens || !cu_q || !topk_indices)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
  if (!aligned(idx_q, 16) || !aligned(idx_k_cache, 16))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": idx_q / idx_k_cache must be 16-byte aligned");
  const size_t need = index_workspace_bytes(T, Hidx, max_pages);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return fail(MSA_ERR_WORKSPACE, std::string(fn) + ": workspace missing, too small or not 256-byte aligned (need " +
                                       std::to_string(need) + " bytes)");
  IndexArgs a{};
  a.idx_q = idx_q;
  a.idx_k = idx_k_cache;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.cu_q = cu_q;
  a.B = B;
  a.T = T;
  a.max_q_len = max_q_len;
  a.Hidx = Hidx;
  a.D = D;
  a.topk = topk;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.topk_indices = topk_indices;
  a.scores = static_cast<float*>(workspace);
  a.err = device_error_word();
  if (a.err == nullptr) return fail(MSA_ERR_CUDA, std::string(fn) + ": no device error word");
  const char* why = nullptr;
  cudaError_t e = launch_index_topk(a, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return MSA_OK;
}

size_t msa_sparse_attn_workspace_size(int B, int T, int max_q_len, int Hq, int Hkv, int Hidx,
                                      int topk, int max_pages) {
  if (B < 0 || T < 0 || max_q_len < 0 || Hq < 1 || Hkv < 1 || Hidx < 1 || topk < 0 ||
      max_pages < 0 || Hq % Hkv != 0 || Hq % Hidx != 0)
    return 0;
  return attn_workspace_bytes(B, T, max_q_len, Hq, Hkv, Hidx, topk, max_pages);
}

msa_status msa_sparse_attn_fwd(const uint8_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                               const int32_t* page_table, const int32_t* seq_lens,
                               const int32_t* cu_q, const int32_t* topk_indices, const float* sink,
                               float sm_scale, const float* q_scale, const float* k_scale,
                               const float* v_scale, int B, int T, int max_q_len, int Hq, int Hkv,
                               int Hidx, int D, int topk, int num_pages, int max_pages,
                               uint16_t* out, float* max_logit, float* lse, void* workspace,
                               size_t workspace_bytes, msa_stream_t stream) {
  const char* fn = "msa_sparse_attn_fwd";
  if (B < 1 || T < 0 || Hq < 1 || Hkv < 1 || Hidx < 1 || num_pages < 1 || max_pages < 1)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": bad sizes");
  if (T > 0 && (max_q_len < 1 || max_q_len > T))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": max_q_len must be in [1, T]");
  if (Hq % Hkv != 0 || Hq % Hidx != 0)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": Hq must be a multiple of Hkv and of Hidx");
  const int group = Hq / Hkv;
  if (group > 16 || (group & (group - 1)) != 0)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": Hq/Hkv must be a power of two <= 16");
  if (D != 128) return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": head_dim must be 128");
  if (topk < 1 || topk > 64) return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": topk must be in [1, 64]");
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.0f))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": sm_scale must be finite and > 0");
  float qs, ks, vs;
  if (!read_scale(q_scale, &qs, "q_scale") || !read_scale(k_scale, &ks, "k_scale") ||
      !read_scale(v_scale, &vs, "v_scale"))
    return MSA_ERR_INVALID_ARG;
  if (T == 0) return MSA_OK;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !cu_q || !topk_indices || !out ||
      !max_logit || !lse)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": q/k/v/out must be 16-byte aligned");
  const size_t need = attn_workspace_bytes(B, T, max_q_len, Hq, Hkv, Hidx, topk, max_pages);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return fail(MSA_ERR_WORKSPACE, std::string(fn) + ": workspace missing, too small or not 256-byte aligned (need " +
                                       std::to_string(need) + " bytes)");
  AttnArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.cu_q = cu_q;
  a.topk = topk_indices;
  a.sink = sink;
  a.c_sink = sm_scale * qs;   // q_scale folded into sm_scale: acts on the dot and the sink
  a.c_qk = a.c_sink * ks;     // k_scale on the dot only
  a.v_scale = vs;
  a.B = B;
  a.T = T;
  a.max_q_len = max_q_len;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Hidx = Hidx;
  a.D = D;
  a.topk_k = topk;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.out = out;
  a.max_logit = max_logit;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = device_error_word();
  if (a.err == nullptr) return fail(MSA_ERR_CUDA, std::string(fn) + ": no device error word");
  const char* why = nullptr;
  cudaError_t e = launch_sparse_attn(a, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return MSA_OK;
}

msa_status msa_sparse_mla_fwd(const uint8_t* q, const uint8_t* kv, const int32_t* indices,
                              const int32_t* topk_length, const float* sink, float sm_scale,
                              const float* q_scale, const float* kv_scale, int T, int H, int S_kv,
                              int d_qk, int d_v, int topk, uint16_t* out, float* max_logits,
                              float* lse, msa_stream_t stream) {
  const char* fn = "msa_sparse_mla_fwd";
  if (d_v != 512) return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": d_v must be 512");
  if (d_qk != 576) return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": d_qk must be 576");
  if (H != 128) return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": H must be 128");
  if (T < 0 || S_kv < 1) return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": bad T / S_kv");
  if (topk < 64 || topk % 64 != 0)
    return fail(MSA_ERR_UNSUPPORTED, std::string(fn) + ": topk must be a positive multiple of 64");
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.0f))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": sm_scale must be finite and > 0");
  float qs, kvs;
  if (!read_scale(q_scale, &qs, "q_scale") || !read_scale(kv_scale, &kvs, "kv_scale"))
    return MSA_ERR_INVALID_ARG;
  if (T == 0) return MSA_OK;
  if (!q || !kv || !indices || !out || !max_logits || !lse)
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || !aligned(indices, 16))
    return fail(MSA_ERR_INVALID_ARG, std::string(fn) + ": q/kv/indices/out must be 16-byte aligned");
  MlaArgs a{};
  a.q = q;
  a.kv = kv;
  a.indices = indices;
  a.topk_length = topk_length;
  a.sink = sink;
  a.c_sink = sm_scale * qs;
  a.c_qk = a.c_sink * kvs;
  a.v_scale = kvs;
  a.T = T;
  a.H = H;
  a.S_kv = S_kv;
  a.d_qk = d_qk;
  a.d_v = d_v;
  a.topk = topk;
  a.out = out;
  a.max_logits = max_logits;
  a.lse = lse;
  a.err = device_error_word();
  if (a.err == nullptr) return fail(MSA_ERR_CUDA, std::string(fn) + ": no device error word");
  const char* why = nullptr;
  cudaError_t e = launch_sparse_mla(a, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return MSA_OK;
}

}  // extern "C"

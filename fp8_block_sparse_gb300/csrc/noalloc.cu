// noalloc.cu -- msa_index_topk_noalloc: the index top-k step for callers that
// cannot allocate device memory.
//
// msa_index_topk needs a scratch workspace (per-block scores and a tile list)
// that the caller allocates. Some callers have no way to do that: a plugin
// that is handed only its input and output pointers by a host engine with no
// workspace hook, or a serving process that reserves all device memory at
// start-up and treats any later cudaMalloc as an error (cudaMalloc can also
// synchronise the device and stall every other stream). This entry point
// takes the same inputs and outputs and keeps its scratch in a fixed array
// that is part of the library's device image instead.
//
// The array is a file-scope static __device__ buffer of kNoAllocScratchBytes
// (8 MiB). Every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device. All calls share the one array and it keeps
// the last call's contents; calls whose work overlaps on the GPU (different
// streams without ordering between them) race on it and must be serialised
// by the caller.
// Nothing in it needs to start at zero: every entry a call reads was written
// earlier by the same call.
#include <mutex>
#include <string>

#include "msa.h"
#include "internal.h"

namespace msa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_na_mutex;
void* g_na_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device). Returns nullptr and fills `why` on failure.
void* scratch_address(std::string* why) {
  int d = -1;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess || d < 0 || d >= kMaxDevices) {
    *why = std::string("no current CUDA device (") + cudaGetErrorString(e) + ")";
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (g_na_ptr[d] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *why = std::string("cudaGetSymbolAddress failed: ") + cudaGetErrorString(e);
      return nullptr;
    }
    g_na_ptr[d] = p;
  }
  return g_na_ptr[d];
}

}  // namespace
}  // namespace msa

extern "C" msa_status msa_index_topk_noalloc(const uint8_t* idx_q, const uint8_t* idx_k_cache,
                                             const int32_t* page_table, const int32_t* seq_lens,
                                             const int32_t* cu_q, int B, int T, int max_q_len,
                                             int Hidx, int D, int topk, int num_pages,
                                             int max_pages, int32_t* topk_indices,
                                             msa_stream_t stream) {
  // msa_index_topk's own argument checks come first, so an invalid or
  // unsupported call reports that and not the size of the fixed scratch
  const msa_status st = msa::check_index_topk_sizes("msa_index_topk_noalloc", B, T, max_q_len, Hidx,
                                                    D, topk, num_pages, max_pages);
  if (st != MSA_OK) return st;
  if (T == 0) return MSA_OK;
  const size_t need = msa_index_topk_workspace_size(T, Hidx, max_pages);
  if (need > msa::kNoAllocScratchBytes) {
    msa::set_last_error("msa_index_topk_noalloc: these sizes need " + std::to_string(need) +
                        " bytes of scratch but the library's fixed scratch holds " +
                        std::to_string(msa::kNoAllocScratchBytes) +
                        " bytes; use msa_index_topk with a caller-owned workspace");
    return MSA_ERR_WORKSPACE;
  }
  std::string why;
  void* scratch = msa::scratch_address(&why);
  if (scratch == nullptr) {
    msa::set_last_error("msa_index_topk_noalloc: " + why);
    return MSA_ERR_CUDA;
  }
  return msa_index_topk(idx_q, idx_k_cache, page_table, seq_lens, cu_q, B, T, max_q_len, Hidx, D,
                        topk, num_pages, max_pages, topk_indices, scratch,
                        msa::kNoAllocScratchBytes, stream);
}

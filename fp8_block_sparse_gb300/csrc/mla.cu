#include "internal.h"
namespace msa {
cudaError_t launch_sparse_mla(const MlaArgs&, cudaStream_t, const char** why) {
  *why = "not built yet";
  return cudaErrorNotSupported;
}
}  // namespace msa

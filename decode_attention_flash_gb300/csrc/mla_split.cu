// mla_split.cu -- MLA latent decode kernel (placeholder until the tcgen05 kernel lands).
#include "internal.h"

namespace da {
int mla_smem_bytes() { return 200 * 1024; }
int mla_threads() { return 256; }
cudaError_t mla_prepare(int) { return cudaSuccess; }
cudaError_t launch_mla(const CUtensorMap &, const CUtensorMap &, const MlaParams &, dim3,
                       cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace da

// testing.cu -- the test hooks of include/decode_attn_testing.h: a kernel that
// fills shared memory with a pattern, and the stall of a context's next run.
#include "decode_attn_testing.h"
#include "internal.h"

namespace da {
void ctx_set_test_stall(da_ctx *ctx, uint32_t ns);
bool ctx_is_mla(const da_ctx *ctx);
}  // namespace da

namespace {

// The largest dynamic shared memory of one block on sm_100-class GPUs (227 KB).
constexpr int kFillBytes = 227 * 1024;

__global__ void __launch_bounds__(256) fill_smem_kernel(uint32_t word) {
  extern __shared__ uint4 smem4[];
  const uint4 v = make_uint4(word, word, word, word);
  for (int i = threadIdx.x; i < kFillBytes / 16; i += blockDim.x) smem4[i] = v;
  // keep the stores: a block that ends right after them is fine, the pattern
  // stays in the SM's shared memory for the next block placed there
  __syncthreads();
}

}  // namespace

extern "C" da_status decode_attn_test_fill_smem(uint32_t word, int32_t blocks_per_sm,
                                                da_stream_t stream) {
  if (blocks_per_sm < 1 || blocks_per_sm > 16) return DA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DA_ERR_CUDA;
  if (cudaFuncSetAttribute(fill_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kFillBytes) != cudaSuccess)
    return DA_ERR_CUDA;
  fill_smem_kernel<<<sms * blocks_per_sm, 256, kFillBytes, reinterpret_cast<cudaStream_t>(stream)>>>(
      word);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

extern "C" da_status decode_attn_test_set_stall(da_ctx *ctx, uint32_t stall_ns) {
  if (!ctx || da::ctx_is_mla(ctx)) return DA_ERR_INVALID_ARG;
  if (stall_ns < 1 || stall_ns > 1000000000u) return DA_ERR_INVALID_ARG;
  da::ctx_set_test_stall(ctx, stall_ns);
  return DA_OK;
}

// static_scratch.cu -- decode_attn_run_noalloc: decode_attn_run without a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// Some callers of a decode kernel are not allowed to call cudaMalloc at the
// moment they decode: code running inside a caching allocator's own hooks,
// plugins of inference servers that own every device allocation themselves,
// or host code that must not risk an out-of-memory failure (or the device-wide
// synchronisation cudaFree may cause) in the middle of a step. For them the
// scratch that the split kernel needs -- the device error word, the per-unit
// counters and the per-split partial outputs -- lives in one file-scope
// __device__ array of kNoAllocScratchBytes bytes, which every GPU that loads
// this library holds until the process exits.
//
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current; the first call on each device does this set-up (and a
// synchronous clear of the array), so make that first call before any stream
// capture begins. Every call on a device shares the array and finds there what
// the previous call left; calls whose kernels overlap on the GPU race on it.
#include <mutex>

#include "internal.h"

namespace da {
// The device a context was created for (defined beside the context in api.cpp).
int ctx_device(const da_ctx *ctx);
}  // namespace da

namespace {

// The largest workspace a plan may need to use this entry point (the header's
// DA_NOALLOC_SCRATCH_BYTES).
constexpr size_t kNoAllocScratchBytes = DA_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes == (32ull << 20), "the header documents 32 MiB");

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
da_status scratch_address(int device, void **addr) {
  if (device < 0 || device >= kMaxDevices) return DA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_setup_lock);
  if (!g_scratch_addr[device]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return DA_ERR_CUDA;
    if (cudaMemset(ptr, 0, kNoAllocScratchBytes) != cudaSuccess) return DA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DA_ERR_CUDA;
    g_scratch_addr[device] = ptr;
  }
  *addr = g_scratch_addr[device];
  return DA_OK;
}

}  // namespace

extern "C" da_status decode_attn_run_noalloc(da_ctx *ctx, const da_args *args,
                                             da_stream_t stream) {
  if (!ctx || !args) return DA_ERR_INVALID_ARG;
  da_plan_info plan;
  da_status st = decode_attn_get_plan(ctx, &plan);
  if (st != DA_OK) return st;
  // a plan that needs more scratch than the static array holds is refused
  if (plan.workspace_bytes > (int64_t)kNoAllocScratchBytes) return DA_ERR_WORKSPACE;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return DA_ERR_CUDA;
  // the context's device must be current: the array's address is per device
  if (device != da::ctx_device(ctx)) return DA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if ((st = scratch_address(device, &scratch)) != DA_OK) return st;
  // A call starts from a zero error word and zero counters, whatever the
  // previous call on this device left behind (an aborted call may leave its
  // counters non-zero): everything before the partial outputs is cleared (the
  // counter region holds more than one word per unit: MLA counts per row and
  // value half, GQA adds the group counters of its two-level merge). The clear
  // is an ordinary memset node on `stream`.
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, (size_t)plan.partial_o_offset, s) != cudaSuccess)
    return DA_ERR_CUDA;
  return decode_attn_run(ctx, args, scratch, kNoAllocScratchBytes, stream);
}

extern "C" da_status decode_attn_get_error_noalloc(da_ctx *ctx, da_stream_t stream, uint32_t *flags) {
  if (!ctx || !flags) return DA_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return DA_ERR_CUDA;
  if (device != da::ctx_device(ctx)) return DA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  da_status st = scratch_address(device, &scratch);
  if (st != DA_OK) return st;
  return decode_attn_get_error(ctx, scratch, stream, flags);
}

/*
 * decode_attn_testing.h -- hooks of libdecode_attn.so for its own tests.
 *
 * Neither call computes any part of the attention, and the decode path never
 * uses them; they let a test put the kernels in situations that ordinary
 * inputs do not produce. The pages have no counterpart: the decode kernels
 * they print (the TorchInductor flex_decode.py.jinja template, the split-K
 * Triton kernel of mslk splitk_kernels.py, FlashInfer mla.cuh, TensorRT-LLM
 * xqa/mha.cu) define only the result, and these hooks only check that the
 * result does not depend on what shared memory held before a launch, and that
 * a pipeline wait that runs out is reported and leaves the context usable.
 */
#ifndef DECODE_ATTN_TESTING_H_
#define DECODE_ATTN_TESTING_H_

#include <stdint.h>

#include "decode_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Enqueues on `stream` (current device) a kernel whose blocks each take the
 * largest dynamic shared memory a block may have and fill all of it with the
 * 32-bit `word` (e.g. 0x7FC00000, a float NaN, or 0xFFFFFFFF); `blocks_per_sm`
 * (1..16) blocks per SM are launched so that every SM runs at least one. A
 * decode launched next on the same stream then starts on shared memory that
 * holds that pattern wherever it was not written in the launch itself.
 * Errors: INVALID_ARG (blocks_per_sm out of range), CUDA.
 */
da_status decode_attn_test_fill_smem(uint32_t word, int32_t blocks_per_sm, da_stream_t stream);

/*
 * Arms a stall for the context's next GQA decode_attn_run only: in every CTA,
 * the first pipeline wait of the first consumer warp is replaced by a wait on
 * a barrier that nothing arrives on, given up after `stall_ns` nanoseconds
 * (1 .. 10^9). The kernel's timeout handling then runs exactly as after a real
 * stuck wait: the other warps give up their own bounded waits, every copy in
 * flight is waited for, DA_DEVERR_TIMEOUT is set in the workspace error word
 * and the call's outputs are incomplete. The stall is disarmed when that run
 * is enqueued. Errors: INVALID_ARG (null context, MLA problem, stall_ns out of
 * range).
 */
da_status decode_attn_test_set_stall(da_ctx *ctx, uint32_t stall_ns);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_TESTING_H_ */

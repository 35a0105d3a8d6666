/*
 * decode_attn.h -- C ABI of the GB300 split-KV decode-attention library.
 *
 * The operation (per batch row b and query head hq, with kv head h = hq / G,
 * G = num_q_heads / num_kv_heads):
 *
 *     out[b][hq] = softmax(scale * q[b][hq] . K^T over P(b,h)) V
 *     lse[b][hq] = ln sum_{n in P(b,h)} exp(scale * q[b][hq] . k_n)
 *
 * where P(b,h) is the row's valid KV positions: 0 .. seq_lens[b]-1, or, for
 * block-sparse decode, the listed blocks kv_idx[b][h][0 .. kv_num_blks[b][h]-1]
 * (each block of sparse_block_size positions, clipped to seq_lens[b]). An empty
 * P gives out = 0 and lse = -inf.
 *
 * Several query tokens per row (q_len = Q > 1, speculative decoding; GQA and
 * MLA): the row's new tokens are its last Q positions, already in the
 * cache, and query token t < Q attends to the positions n <= seq_lens[b] - Q + t
 * of P(b,h) -- the causal mask of the split-K decode kernel (mslk
 * splitk_kernels.py, `_fwd_kernel_splitK` with IS_CAUSAL). q, out and lse then
 * carry a [Q] axis after the head axis (the flex_decode.py.jinja query layout
 * [.., head, M, D]).
 *
 * Sources of the operation:
 *  - GQA packing and the block-sparse KV_NUM_BLKS / KV_IDX tables (indexed by
 *    kv head): the TorchInductor flex_decode.py.jinja template (header comment
 *    and the "normal blocks" traversal);
 *  - paged translation page = block_table[b][n / page_size]: the split-K
 *    decode kernel of mslk splitk_kernels.py (`_fwd_kernel_splitK`, paged
 *    branch) and the KV page list of TensorRT-LLM xqa/mha.cu (`launchMHA`);
 *  - per-split normalised O plus natural-log LSE and their LSE-weighted merge:
 *    splitk_kernels.py (`_fwd_kernel_splitK` "write back O", `_splitK_reduce`);
 *  - MLA latent decode (scores over [ckv ; kpe], values ckv): FlashInfer
 *    include/flashinfer/attention/mla.cuh (`BatchMLAPagedAttentionKernel`);
 *  - fp8 KV: e4m3 (`float8e4nv` in splitk_kernels.py) times a per-kv-head
 *    fp32 scale (the single K/V cache scale of xqa/mha.cu, kept per head).
 *
 * Conventions for every entry point:
 *  - All tensors are row-major, last index fastest, in device memory owned by
 *    the caller; the library never allocates device memory and never frees a
 *    caller pointer. The only library-owned object is the host-side context.
 *  - Every function returns a da_status; no C++ exception or abort crosses
 *    the ABI. A failed call leaves the outputs unspecified.
 *  - decode_attn_run and decode_attn_merge only enqueue work on the given
 *    stream (no allocation, no synchronisation).
 */
#ifndef DECODE_ATTN_H_
#define DECODE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same type as cudaStream_t / CUstream). */
typedef struct CUstream_st *da_stream_t;

typedef enum {
  DA_OK = 0,
  DA_ERR_INVALID_ARG = 1,  /* null pointer, bad dimension, bad override   */
  DA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. D != 128)   */
  DA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed           */
  DA_ERR_WORKSPACE = 4,    /* workspace missing, misaligned or too small  */
  DA_ERR_NOT_PLANNED = 5,  /* decode_attn_run before decode_attn_plan     */
  DA_ERR_DEVICE = 6        /* the device error word is non-zero           */
} da_status;

typedef enum { DA_KV_CONTIGUOUS = 0, DA_KV_PAGED = 1 } da_kv_layout;
/* KV element types: bf16; e4m3 with one fp32 scale per kv head (k_scale /
 * v_scale); e4m3 with a per-token fp16 scale and shift (k_scale_shift /
 * v_scale_shift: value = e4m3 * scale + shift, the fp8 scale_shift words of
 * the split-K decode page, mslk splitk_kernels.py `dequantize`); or int4
 * group-wise rows, the same page's PACKED_PER_VAL = 8 layout: each cache row
 * of k / v is int32 words, first kv_groups coefficient words (fp16 scale in
 * the low half, fp16 shift in the high half), then D / 8 words of eight
 * unsigned 4-bit codes, element 8w + i in bits 4i..4i+3 of data word w;
 * element d has value code * scale + shift of group d / (D / kv_groups). */
typedef enum {
  DA_DTYPE_BF16 = 0,
  DA_DTYPE_FP8_E4M3 = 1,
  DA_DTYPE_FP8_E4M3_TOKEN_SCALE = 2,
  DA_DTYPE_INT4_GROUPS = 3
} da_dtype;

/* Bits of the device error word (sticky until decode_attn_get_error clears it). */
enum {
  DA_DEVERR_PAGE_INDEX = 1u,   /* block_table entry outside [0, num_pages): page skipped   */
  DA_DEVERR_SPARSE_INDEX = 2u, /* kv_idx outside the cache or kv_num_blks outside
                                  [0, max_sparse_blocks]: block skipped / count clamped   */
  DA_DEVERR_SEQ_LEN = 4u,      /* seq_lens[b] < 0 or over the cache capacity: clamped      */
  DA_DEVERR_TIMEOUT = 8u       /* a pipeline wait gave up after its time limit             */
};

/*
 * Problem description, fixed at create time.
 *
 *   GQA: head_dim_qk = head_dim_v = 128, num_q_heads % num_kv_heads == 0,
 *        G = num_q_heads / num_kv_heads in 1..16.
 *   MLA: is_mla = 1, num_kv_heads = 1, ckv_dim = 512, kpe_dim = 64,
 *        head_dim_qk = 576, head_dim_v = 512, kv_layout = DA_KV_PAGED.
 *   Paged: page_size a multiple of 16 that divides 64 or is a multiple of 64
 *        (MLA: 64); max_pages_per_seq table columns; num_pages pool size.
 *   Contiguous: max_seq_len is the cache length L of [B][HKV][L][D].
 *   Sparse (GQA, contiguous only): sparse_block_size a multiple of 64,
 *        max_sparse_blocks columns of kv_idx; 0 = dense. sparse_batch and
 *        sparse_heads (SZ, SH; 0 = B and HKV) are the block tables' first two
 *        extents: row b and kv head h read table row (b % SZ, h % SH), the
 *        broadcast of the flex decode template (SPARSE_Z, SPARSE_HQ).
 *   q_len: query tokens per row, 0 or 1 = one. GQA: G * Q <= 16 (the G*Q rows
 *        of a kv head share one pass); block-sparse tables apply to every query
 *        token, the causal or tree mask on top of them. MLA: Q <= 16, each query
 *        token a row of its own over the shared latent cache (its pages come
 *        from L2 for the row's other tokens).
 */
typedef struct {
  int32_t batch, num_q_heads, num_kv_heads;
  int32_t head_dim_qk, head_dim_v;
  int32_t is_mla, ckv_dim, kpe_dim;
  da_kv_layout kv_layout;
  int32_t page_size;
  int32_t max_seq_len;        /* contiguous: L; paged: at most max_pages_per_seq * page_size */
  int32_t max_pages_per_seq;
  int32_t num_pages;
  da_dtype q_dtype;           /* DA_DTYPE_BF16 only */
  da_dtype kv_dtype;          /* bf16, or (GQA) e4m3 with per-head or per-token scales */
  int32_t sparse_block_size;
  int32_t max_sparse_blocks;
  int32_t q_len;              /* query tokens per row; 0 or 1 = one */
  int32_t sparse_batch;       /* sparse: block tables' batch extent SZ (0 = batch) */
  int32_t sparse_heads;       /* sparse: block tables' head extent SH (0 = num_kv_heads) */
  int32_t kv_groups;          /* DA_DTYPE_INT4_GROUPS: groups per row, 4 or 8 (rows of 1 or
                                 2 groups are not a multiple of 16 bytes: unsupported);
                                 contiguous caches need max_seq_len a multiple of 8 (4
                                 groups) or 4 (8 groups) */
  int32_t fp8_mma;            /* GQA with DA_DTYPE_FP8_E4M3 K/V only, optional: 1 runs QK and PV
                                 on e4m3 tensor cores. Each query row is quantised to e4m3
                                 in fp32 steps (amax = max |q|, code = e4m3(q * (448 / amax)),
                                 round to nearest even, saturating; the row's scale amax /
                                 448 joins the score factor), and the softmax weights that
                                 meet V are scaled by 2^8, rounded to f16 and then to e4m3
                                 (the row sum uses the unrounded weights). The e4m3 QK
                                 products are exact; the weights' rounding (3 mantissa bits)
                                 is the mode's approximation. 0 = f16 arithmetic */
} da_problem;

/*
 * Per-call arguments: device pointers, caller-owned.
 *
 *   q          bf16 [B][HQ][Dqk]   (MLA: q_nope [B][HQ][512]; q_len Q > 1: [B][HQ][Q][Dqk],
 *              MLA [B][HQ][Q][512])
 *   q_pe       MLA only: bf16 [B][HQ][64] (q_len Q > 1: [B][HQ][Q][64]); else NULL
 *   k, v       contiguous [B][HKV][L][D]; paged [num_pages][HKV][page_size][D];
 *              MLA: k = ckv [num_pages][page_size][512], v = kpe [num_pages][page_size][64].
 *              Element type bf16, or e4m3 bytes when kv_dtype is an e4m3 type;
 *              DA_DTYPE_INT4_GROUPS: int32 rows of kv_groups + D / 8 words.
 *              Base addresses 16-byte aligned.
 *   k_scale, v_scale  DA_DTYPE_FP8_E4M3 only: fp32 [HKV]; dequantised value = e4m3 * scale
 *   k_scale_shift, v_scale_shift  DA_DTYPE_FP8_E4M3_TOKEN_SCALE only: int32, one word per
 *              cache row of k / v (contiguous [B][HKV][L], paged [num_pages][HKV][page_size]):
 *              fp16 scale in the low half, fp16 shift in the high half; dequantised
 *              value = e4m3 * scale + shift. Base addresses 16-byte aligned; L a
 *              multiple of 4 (contiguous)
 *   block_table paged: int32 [B][max_pages_per_seq]; entries past a row's
 *              last page are never read
 *   seq_lens   int32 [B]
 *   kv_num_blks, kv_idx  sparse only: int32 [SZ][SH] and [SZ][SH][max_sparse_blocks]
 *              (SZ, SH = sparse_batch, sparse_heads, default B and HKV)
 *   kv_full_num_blks, kv_full_idx  sparse only, optional (both NULL or both set): the
 *              second table pair of the flex block mask (FULL_KV_NUM_BLKS / FULL_KV_IDX,
 *              blocks that need no mask_mod), same shapes; their blocks are attended
 *              after the kv_idx blocks. Pass the two tables' summed counts as the
 *              planner's kv_num_blks_host, or none.
 *   scale      the full softmax scale (e.g. 1/sqrt(128)); applied in fp32
 *   softcap    GQA: 0, or a tanh soft cap c > 0 on the scaled scores, s -> c * tanh(s / c)
 *              (the logit soft-capping of the FlashAttention-3 page); MLA: 0 only
 *   spec_mask  q_len Q > 1, optional: uint32 [B][Q], the draft-token tree mask of
 *              speculative decoding (the packed mask rows of the TensorRT-LLM XQA
 *              kernel, SPEC_DEC, for Q <= 32): every position before the row's Q new
 *              ones is attended, and new position N_b - Q + j by query token t when
 *              bit j of word [b][t] is set. NULL: causal (bits 0..t). Ignored for Q = 1
 *   out        bf16 [B][HQ][Dv]    (q_len Q > 1: [B][HQ][Q][Dv])
 *   lse        fp32 [B][HQ], natural log; may be NULL (q_len Q > 1: [B][HQ][Q])
 *   mask_window, mask_sink  GQA, optional: int32 [HQ] each (mask_sink may be NULL, meaning
 *              0): a mask_mod per query head in the sense of flex attention (which
 *              the flex_decode.py.jinja template applies element-wise, with the query
 *              head, to the blocks of KV_IDX and not to those of FULL_KV_IDX). With
 *              q_pos = seq_lens[b] - Q + t the query token's position, position n is
 *              kept when n < mask_sink[hq], or mask_window[hq] < 0, or
 *              n > q_pos - mask_window[hq] (the last mask_window[hq] positions): a
 *              sliding window with attention sinks, per head. The blocks of
 *              kv_full_idx are not masked. MLA: NULL only (DA_ERR_UNSUPPORTED)
 *   alibi_slopes GQA, optional: fp32 [HQ]: a score_mod adding slope[hq] * (n - q_pos)
 *              to every scaled score (ALiBi), full blocks included. Not with a soft cap
 *              (the two score_mods would need an order: DA_ERR_UNSUPPORTED); MLA: NULL
 */
typedef struct {
  const void *q;
  const void *q_pe;
  const void *k;
  const void *v;
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *kv_num_blks;
  const int32_t *kv_idx;
  float scale;
  void *out;
  float *lse;
  const int32_t *k_scale_shift;
  const int32_t *v_scale_shift;
  const int32_t *kv_full_num_blks;
  const int32_t *kv_full_idx;
  float softcap;
  const uint32_t *spec_mask;
  const int32_t *mask_sink;
  const int32_t *mask_window;
  const float *alibi_slopes;
} da_args;

/* What the planner decided (host-side, informational). */
typedef struct {
  int32_t kv_tile;          /* tokens per pipeline stage                               */
  int32_t chunk_tokens;     /* positions per split (sparse: list entries x block size) */
  int32_t num_splits;       /* S_max: splits per (b, kv head) unit                     */
  int32_t num_units;        /* B x HKV (MLA: B)                                        */
  int32_t rows_per_unit;    /* G x q_len (MLA: HQ)                                     */
  int32_t grid_x, grid_y, grid_z;
  int32_t ctas_per_sm;      /* resident CTAs of the split kernel per SM                */
  int32_t writes_final;     /* 1: one split, the split kernel writes out/lse directly  */
  int64_t counters_offset;  /* byte offsets inside the workspace: per-unit counters,   */
  int64_t partial_o_offset; /* per-split O and per-split LSE                           */
  int64_t partial_lse_offset;
  int64_t workspace_bytes;
} da_plan_info;

typedef struct da_ctx da_ctx;

/*
 * Validates the problem, reads the SM count and shared-memory limit of
 * `device` and returns a new host context in *out. The caller owns the
 * context and releases it with decode_attn_destroy.
 * Errors: INVALID_ARG (null, bad dims), UNSUPPORTED, CUDA (device query).
 */
da_status decode_attn_create(const da_problem *problem, int device, da_ctx **out);

/*
 * Chooses the split size and grid (the XQA-style split count heuristic: enough
 * (b, kv head, split) CTAs to fill every SM, splits a multiple of the KV tile,
 * at least 256 positions each) and reports the workspace size in
 * *workspace_bytes. seq_lens_host (int32 [B], host memory, may be NULL)
 * lets the planner size splits from the real lengths; without it the plan
 * assumes every row is max_seq_len long. num_splits_override > 0 forces that
 * many splits per unit (positions are cut into equal tile-aligned chunks).
 * Host-only; no GPU work. Errors: INVALID_ARG.
 */
da_status decode_attn_plan(da_ctx *ctx, const int32_t *seq_lens_host, int32_t num_splits_override,
                           size_t *workspace_bytes);

/*
 * decode_attn_plan with the block-sparse list lengths too: kv_num_blks_host
 * (int32 [B][HKV], host memory, may be NULL) lets the planner size splits of a
 * block-sparse problem from the real list lengths instead of max_sparse_blocks.
 */
da_status decode_attn_plan_ex(da_ctx *ctx, const int32_t *seq_lens_host,
                              const int32_t *kv_num_blks_host, int32_t num_splits_override,
                              size_t *workspace_bytes);

/* The plan the last decode_attn_plan produced. Errors: INVALID_ARG, NOT_PLANNED. */
da_status decode_attn_get_plan(const da_ctx *ctx, da_plan_info *info);

/*
 * The planner as a pure host function of (problem, SM count): the same
 * decision decode_attn_plan makes on a device with `num_sms` SMs. Needs no GPU.
 */
da_status decode_attn_plan_info(const da_problem *problem, int32_t num_sms,
                                const int32_t *seq_lens_host, int32_t num_splits_override,
                                da_plan_info *info);

/*
 * Enqueues the decode on `stream` as ONE kernel launch: every (b, kv head,
 * split) CTA writes its split's normalised O and LSE into the workspace, and
 * the last CTA of each (b, kv head) to finish -- found with a per-unit atomic
 * counter, without any spinning wait -- merges that unit's splits into `out`
 * and `lse` (a plan with one split writes them directly). `workspace` is
 * device memory of at least the planned size, 256-byte aligned, and must be
 * zero when first used (allocate it zeroed): it holds the sticky device error
 * word and the per-unit counters, which each call leaves at zero again.
 * Calls that share a workspace must not overlap on the GPU. Out-of-range
 * indices found on the device set error bits (DA_DEVERR_*) and are skipped,
 * never read. The context's device must be current.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, NOT_PLANNED, CUDA.
 */
da_status decode_attn_run(da_ctx *ctx, const da_args *args, void *workspace, size_t workspace_bytes,
                          da_stream_t stream);

/*
 * Standalone LSE merge of `num_splits` partial results per row:
 *   o_part   fp32 [rows][num_splits][dv]  (normalised per split)
 *   lse_part fp32 [rows][num_splits]      (natural log; -inf marks an empty split,
 *                                          whose o_part is never read)
 *   out      bf16 [rows][dv];  lse fp32 [rows] (may be NULL)
 * out = sum_s w_s o_s / sum_s w_s, w_s = exp(lse_s - max lse), lse = max + ln sum w;
 * rows whose splits are all empty get out = 0, lse = -inf (`_splitK_reduce` of
 * splitk_kernels.py). dv must be a multiple of 4, at most 1024; pointers 16-byte
 * aligned. `ctx` may be NULL. Errors: INVALID_ARG, CUDA.
 */
da_status decode_attn_merge(da_ctx *ctx, const float *o_part, const float *lse_part,
                            int32_t num_splits, int32_t rows, int32_t dv, void *out, float *lse,
                            da_stream_t stream);

/*
 * Synchronises `stream`, copies the device error word of `workspace` to
 * *flags and clears it; after a DA_DEVERR_TIMEOUT it also re-zeroes the
 * per-unit counters (an aborted call may leave them non-zero). Returns
 * DA_ERR_DEVICE when the word was non-zero. `ctx` may be NULL (then the
 * counters are left as they are).
 */
da_status decode_attn_get_error(da_ctx *ctx, void *workspace, da_stream_t stream, uint32_t *flags);

/*
 * decode_attn_run for callers that cannot allocate device memory (an
 * allocator's own hooks, server plugins that own every device allocation,
 * code that must not risk an out-of-memory error or the synchronisation of
 * cudaFree mid-step). The paper has no counterpart: it is a packaging variant
 * of decode_attn_run. Instead of a caller workspace it uses one file-scope
 * device array of 32 MiB (DA_NOALLOC_SCRATCH_BYTES) in this library, which
 * every GPU that loads the library keeps until the process exits; it calls no
 * cudaMalloc, cudaFree or allocating library routine. The caller still passes
 * the inputs and outputs in `args`, as for decode_attn_run.
 *
 * The first call on a device looks up the array's device address and clears
 * it synchronously, so make it before any stream capture starts. Each call
 * then clears the error word and counters with a memset on `stream` and
 * enqueues the same kernel as decode_attn_run. All calls on a device share
 * the array: calls whose work overlaps on the GPU (other streams, other
 * threads) race on it. Device-side error bits (bad indices are skipped on
 * the device) stay in the array's error word until the next call clears it:
 * decode_attn_get_error_noalloc reads them. A plan whose workspace
 * exceeds the array is refused with DA_ERR_WORKSPACE, and a call made while
 * another device than the context's is current with DA_ERR_INVALID_ARG
 * (before anything is enqueued).
 * Errors: INVALID_ARG, NOT_PLANNED, WORKSPACE, UNSUPPORTED, CUDA.
 */
#define DA_NOALLOC_SCRATCH_BYTES (32u << 20)
da_status decode_attn_run_noalloc(da_ctx *ctx, const da_args *args, da_stream_t stream);

/*
 * decode_attn_get_error for the calls of decode_attn_run_noalloc: the error
 * word of the device's static array (the context's device must be current),
 * read and cleared on `stream` like decode_attn_get_error does (it
 * synchronises the stream; after a DA_DEVERR_TIMEOUT it re-zeroes the
 * counters). *flags = 0 before the first no-alloc call on the device. Returns
 * DA_ERR_DEVICE when the word was non-zero. Errors: INVALID_ARG, UNSUPPORTED,
 * CUDA.
 */
da_status decode_attn_get_error_noalloc(da_ctx *ctx, da_stream_t stream, uint32_t *flags);

/* Releases the context (NULL is allowed). */
void decode_attn_destroy(da_ctx *ctx);

/* A static, human-readable name for a status code. */
const char *decode_attn_status_string(da_status status);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H_ */

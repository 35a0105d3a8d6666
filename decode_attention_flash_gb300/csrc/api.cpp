// api.cpp -- the C ABI (include/decode_attn.h): argument checks, the host
// context, TMA descriptors and kernel launches. No device allocation happens
// here; every device buffer is the caller's.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"

struct da_ctx {
  da_problem prob;
  int device;
  int num_sms;
  int smem_per_sm;
  bool planned;
  da_plan_info plan;
  // tensor maps are re-encoded only when the cache base pointers change
  const void *map_k_base;
  const void *map_v_base;
  CUtensorMap kmap;
  CUtensorMap vmap;
  // MLA also maps the two query tensors
  const void *map_q_base;
  const void *map_qpe_base;
  CUtensorMap qmap;
  CUtensorMap qpemap;
  // per-token scale words of e4m3 K/V (DA_DTYPE_FP8_E4M3_TOKEN_SCALE)
  const void *map_kss_base;
  const void *map_vss_base;
  CUtensorMap kssmap;
  CUtensorMap vssmap;
  // tests of the timeout path (decode_attn_testing.h): the stall of the next run
  uint32_t test_stall_ns;
};

namespace da {
// The device a context was created for (its calls must run with it current).
int ctx_device(const da_ctx *ctx) { return ctx->device; }
// Arms the test stall of the context's next GQA run (decode_attn_testing.h).
void ctx_set_test_stall(da_ctx *ctx, uint32_t ns) { ctx->test_stall_ns = ns; }
bool ctx_is_mla(const da_ctx *ctx) { return ctx->prob.is_mla != 0; }
}  // namespace da

namespace {

using da::kWorkspaceHeader;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A 2-D map over `rows` rows of `row_bytes` bytes, 128B-swizzled boxes of
// `box_rows` rows; elements are bf16 (row_bytes = 128: a half head row) or bytes.
da_status encode_rows(CUtensorMap *map, const void *base, bool bf16, uint64_t rows,
                      uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[2] = {bf16 ? 64u : 128u, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {bf16 ? 64u : 128u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// A 2-D bf16 map over `rows` rows of `row_elems` elements (row pitch = row_elems * 2
// bytes), 128B-swizzled boxes of 64 elements x `box_rows` rows.
da_status encode_bf16_rows(CUtensorMap *map, const void *base, uint64_t row_elems, uint64_t rows,
                           uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {row_elems * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// Rows of `row_elems` bf16 read 32 columns at a time (64 bytes, 64B-swizzled):
// the per-rank halves of the MLA rope part.
da_status encode_bf16_rows_sw64(CUtensorMap *map, const void *base, uint64_t row_elems, uint64_t rows,
                                uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {row_elems * 2};
  const cuuint32_t box[2] = {32u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// The MLA rope queries [B*HQ][Q][64] as a 3-D tensor (64 elements, token, head
// row): one box copies 32 columns of query token t for `box_rows` head rows,
// 64B-swizzled, and lands as [row][32].
da_status encode_qpe_tokens(CUtensorMap *map, const void *base, uint64_t head_rows, uint32_t Q,
                            uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[3] = {64, Q, head_rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)Q * 128};
  const cuuint32_t box[3] = {32u, 1u, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// A bf16 cache of rows of 128 elements as a 3-D tensor (64 elements, row, half)
// with the half stride (128 B) below the row stride (256 B): one box copies
// `box_rows` rows and lands as [half][row][64], 128B-swizzled.
da_status encode_bf16_halves(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[3] = {64, rows, 2};
  const cuuint64_t strides[2] = {256, 128};
  const cuuint32_t box[3] = {64u, box_rows, 2u};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// int4 group-wise rows (W = groups + 16 words each) viewed as 128-byte lines:
// a box of `box_rows` consecutive rows is box_rows * W / 32 whole lines,
// aligned, and lands as the rows are in the cache (unswizzled). The caller
// keeps every box's first row a multiple of 32 / gcd(W, 32) rows.
da_status encode_int4_lines(CUtensorMap *map, const void *base, uint64_t rows, uint32_t W,
                            uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[2] = {32, rows * W / 32};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {32u, box_rows * W / 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// Per-token scale words: one int32 per cache row, viewed as [rows / 4][4] so a
// box of `box_rows` rows is 4 words wide (16 bytes); rows past the end read 0.
da_status encode_scale_words(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[2] = {4, rows / 4};
  const cuuint64_t strides[1] = {16};
  const cuuint32_t box[2] = {4u, box_rows / 4};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// Query map: [rows][128] bf16, unswizzled boxes of 128 elements x `box_rows` rows.
da_status encode_q_rows(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

da_status check_workspace(const da_ctx *ctx, const void *ws, size_t bytes) {
  if (!ws || !aligned(ws, 256)) return DA_ERR_WORKSPACE;
  if ((int64_t)bytes < ctx->plan.workspace_bytes) return DA_ERR_WORKSPACE;
  return DA_OK;
}

da_status run_gqa(da_ctx *ctx, const da_args *a, uint8_t *ws, cudaStream_t stream) {
  const da_problem &p = ctx->prob;
  const bool fp8 = p.kv_dtype != DA_DTYPE_BF16;
  const bool token_scale = p.kv_dtype == DA_DTYPE_FP8_E4M3_TOKEN_SCALE;
  const bool int4 = p.kv_dtype == DA_DTYPE_INT4_GROUPS;  // takes the f16 (fp8) kernel path
  const bool paged = p.kv_layout == DA_KV_PAGED;
  const bool sparse = p.sparse_block_size > 0;
  if (!a->q || !a->k || !a->v || !a->seq_lens || !a->out) return DA_ERR_INVALID_ARG;
  if (paged && !a->block_table) return DA_ERR_INVALID_ARG;
  if (sparse && (!a->kv_num_blks || !a->kv_idx)) return DA_ERR_INVALID_ARG;
  if ((a->kv_full_num_blks != nullptr) != (a->kv_full_idx != nullptr)) return DA_ERR_INVALID_ARG;
  if (a->kv_full_num_blks && !sparse) return DA_ERR_INVALID_ARG;
  if (fp8 && !token_scale && !int4 && (!a->k_scale || !a->v_scale)) return DA_ERR_INVALID_ARG;
  if (token_scale && (!a->k_scale_shift || !a->v_scale_shift || !aligned(a->k_scale_shift, 16) ||
                      !aligned(a->v_scale_shift, 16)))
    return DA_ERR_INVALID_ARG;
  if (!aligned(a->k, 128) || !aligned(a->v, 128) || !aligned(a->q, 128) || !aligned(a->out, 8))
    return DA_ERR_INVALID_ARG;

  const uint64_t rows = paged ? (uint64_t)p.num_pages * p.num_kv_heads * p.page_size
                              : (uint64_t)p.batch * p.num_kv_heads * p.max_seq_len;
  const uint32_t box_tokens = (uint32_t)da::gqa_box_tokens(p);
  // the G query heads of a kv head, each with Q query tokens, are the unit's
  // R = G x Q consecutive rows of q viewed as [B * HQ * Q][D]
  const int Q = p.q_len > 1 ? p.q_len : 1;
  const int R = p.num_q_heads / p.num_kv_heads * Q;
  if (ctx->map_k_base != a->k || ctx->map_v_base != a->v || ctx->map_q_base != a->q) {
    ctx->map_k_base = ctx->map_v_base = ctx->map_q_base = nullptr;
    da_status st;
    if (int4) {
      const uint32_t W = (uint32_t)p.kv_groups + 16u;
      if ((st = encode_int4_lines(&ctx->kmap, a->k, rows, W, box_tokens)) != DA_OK) return st;
      if ((st = encode_int4_lines(&ctx->vmap, a->v, rows, W, box_tokens)) != DA_OK) return st;
    } else if (fp8) {
      // one 128-byte row per token
      if ((st = encode_rows(&ctx->kmap, a->k, false, rows, box_tokens)) != DA_OK) return st;
      if ((st = encode_rows(&ctx->vmap, a->v, false, rows, box_tokens)) != DA_OK) return st;
    } else {
      // rows of 128 bf16, viewed as (64 elements, row, half): a box of `box_tokens`
      // rows lands half-major in shared memory
      if ((st = encode_bf16_halves(&ctx->kmap, a->k, rows, box_tokens)) != DA_OK) return st;
      if ((st = encode_bf16_halves(&ctx->vmap, a->v, rows, box_tokens)) != DA_OK) return st;
    }
    if ((st = encode_q_rows(&ctx->qmap, a->q, (uint64_t)p.batch * p.num_q_heads * Q, (uint32_t)R)) !=
        DA_OK)
      return st;
    ctx->map_k_base = a->k;
    ctx->map_v_base = a->v;
    ctx->map_q_base = a->q;
  }
  if (token_scale && (ctx->map_kss_base != a->k_scale_shift || ctx->map_vss_base != a->v_scale_shift)) {
    ctx->map_kss_base = ctx->map_vss_base = nullptr;
    da_status st;
    if ((st = encode_scale_words(&ctx->kssmap, a->k_scale_shift, rows, box_tokens)) != DA_OK) return st;
    if ((st = encode_scale_words(&ctx->vssmap, a->v_scale_shift, rows, box_tokens)) != DA_OK) return st;
    ctx->map_kss_base = a->k_scale_shift;
    ctx->map_vss_base = a->v_scale_shift;
  }

  const da_plan_info &pl = ctx->plan;
  da::GqaParams gp;
  std::memset(&gp, 0, sizeof gp);
  gp.q = reinterpret_cast<const __nv_bfloat16 *>(a->q);
  gp.block_table = a->block_table;
  gp.seq_lens = a->seq_lens;
  gp.kv_num_blks = a->kv_num_blks;
  gp.kv_idx = a->kv_idx;
  gp.kv_full_num_blks = a->kv_full_num_blks;
  gp.kv_full_idx = a->kv_full_idx;
  gp.spec_mask = Q > 1 ? a->spec_mask : nullptr;
  if (a->mask_sink && !a->mask_window) return DA_ERR_INVALID_ARG;
  if (a->alibi_slopes && a->softcap != 0.f) return DA_ERR_UNSUPPORTED;  // two score_mods, no order
  gp.mask_sink = a->mask_sink;
  gp.mask_window = a->mask_window;
  gp.alibi_slopes = a->alibi_slopes;
  gp.k_scale = a->k_scale;
  gp.v_scale = a->v_scale;
  gp.o_part = reinterpret_cast<float *>(ws + pl.partial_o_offset);
  gp.lse_part = reinterpret_cast<float *>(ws + pl.partial_lse_offset);
  gp.out = reinterpret_cast<__nv_bfloat16 *>(a->out);
  gp.lse = a->lse;
  gp.err = reinterpret_cast<uint32_t *>(ws);
  gp.counters = reinterpret_cast<uint32_t *>(ws + pl.counters_offset);
  gp.score_scale = a->scale * 1.4426950408889634f;
  if (!(a->softcap >= 0.f)) return DA_ERR_INVALID_ARG;  // negative or NaN
  gp.softcap_l2 = a->softcap * 1.4426950408889634f;
  gp.softcap_k = a->softcap > 0.f ? 2.f / a->softcap : 0.f;
  gp.batch = p.batch;
  gp.num_q_heads = p.num_q_heads * Q;  // rows of q / out / lse per batch row
  gp.num_kv_heads = p.num_kv_heads;
  gp.group = R;
  gp.q_len = Q;
  gp.token_scale = token_scale ? 1 : 0;
  gp.kv_groups = int4 ? p.kv_groups : 0;
  gp.paged = paged ? 1 : 0;
  gp.page_size = p.page_size;
  gp.cache_len = paged ? 0 : p.max_seq_len;
  gp.max_pages = p.max_pages_per_seq;
  gp.num_pages = p.num_pages;
  gp.capacity = paged ? p.max_pages_per_seq * p.page_size : p.max_seq_len;
  gp.sparse_block_size = p.sparse_block_size;
  gp.max_sparse_blocks = p.max_sparse_blocks;
  gp.sparse_batch = p.sparse_batch > 0 ? p.sparse_batch : std::max(p.batch, 1);
  gp.sparse_heads = p.sparse_heads > 0 ? p.sparse_heads : p.num_kv_heads;
  gp.fp8_mma = p.fp8_mma;
  gp.test_stall_ns = ctx->test_stall_ns;
  ctx->test_stall_ns = 0;  // one call only
  if (da::launch_gqa(fp8, gp.group, ctx->kmap, ctx->vmap, ctx->qmap,
                     token_scale ? ctx->kssmap : ctx->kmap, token_scale ? ctx->vssmap : ctx->vmap,
                     gp, pl.grid_x, stream) !=
      cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}

da_status run_mla(da_ctx *ctx, const da_args *a, uint8_t *ws, cudaStream_t stream) {
  const da_problem &p = ctx->prob;
  if (!a->q || !a->q_pe || !a->k || !a->v || !a->seq_lens || !a->out || !a->block_table)
    return DA_ERR_INVALID_ARG;
  // no score or mask modification in the MLA kernel
  if (a->softcap != 0.f || a->mask_window || a->mask_sink || a->alibi_slopes) return DA_ERR_UNSUPPORTED;
  if (!aligned(a->k, 128) || !aligned(a->v, 128) || !aligned(a->q, 128) || !aligned(a->q_pe, 128) ||
      !aligned(a->out, 16))
    return DA_ERR_INVALID_ARG;
  if (ctx->map_k_base != a->k || ctx->map_v_base != a->v || ctx->map_q_base != a->q ||
      ctx->map_qpe_base != a->q_pe) {
    const uint64_t tokens = (uint64_t)p.num_pages * p.page_size;
    const uint64_t qrows = (uint64_t)p.batch * p.num_q_heads;
    ctx->map_k_base = ctx->map_v_base = ctx->map_q_base = ctx->map_qpe_base = nullptr;
    da_status st;
    if ((st = encode_bf16_rows(&ctx->kmap, a->k, 512, tokens, 64)) != DA_OK) return st;
    if ((st = encode_bf16_rows_sw64(&ctx->vmap, a->v, 64, tokens, 64)) != DA_OK) return st;
    st = p.q_len > 1 ? encode_qpe_tokens(&ctx->qpemap, a->q_pe, qrows, (uint32_t)p.q_len, 128)
                     : encode_bf16_rows_sw64(&ctx->qpemap, a->q_pe, 64, qrows, 128);
    if (st != DA_OK) return st;
    ctx->map_k_base = a->k;
    ctx->map_v_base = a->v;
    ctx->map_q_base = a->q;
    ctx->map_qpe_base = a->q_pe;
  }
  const da_plan_info &pl = ctx->plan;
  da::MlaParams mp;
  std::memset(&mp, 0, sizeof mp);
  mp.q_nope = reinterpret_cast<const __nv_bfloat16 *>(a->q);
  mp.q_pe = reinterpret_cast<const __nv_bfloat16 *>(a->q_pe);
  mp.block_table = a->block_table;
  mp.seq_lens = a->seq_lens;
  mp.q_len = p.q_len > 1 ? p.q_len : 1;
  mp.spec_mask = mp.q_len > 1 ? a->spec_mask : nullptr;
  mp.o_part = reinterpret_cast<float *>(ws + pl.partial_o_offset);
  mp.lse_part = reinterpret_cast<float *>(ws + pl.partial_lse_offset);
  mp.out = reinterpret_cast<__nv_bfloat16 *>(a->out);
  mp.lse = a->lse;
  mp.err = reinterpret_cast<uint32_t *>(ws);
  mp.counters = reinterpret_cast<uint32_t *>(ws + pl.counters_offset);
  // a zero scale (uniform weights) becomes 2^-100: every finite score then
  // weighs exactly 1 against the maximum, while a padded (masked) score times
  // the factor stays -inf, so the kernel needs no per-token select
  mp.score_scale = a->scale == 0.f ? 0x1p-100f : a->scale * 1.4426950408889634f;
  mp.batch = p.batch;
  mp.max_pages = p.max_pages_per_seq;
  mp.num_pages = p.num_pages;
  mp.capacity = p.max_pages_per_seq * p.page_size;
  const dim3 grid(pl.grid_x, 1, 1);
  cudaError_t e = da::launch_mla(ctx->qpemap, ctx->kmap, ctx->vmap, mp, grid, stream);
  if (e == cudaErrorNotSupported) return DA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

}  // namespace

extern "C" {

da_status decode_attn_create(const da_problem *problem, int device, da_ctx **out) {
  if (!out) return DA_ERR_INVALID_ARG;
  *out = nullptr;
  da_status st = da::validate_problem(problem);
  if (st != DA_OK) return st;
  int sms = 0, smem = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return DA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) !=
      cudaSuccess)
    return DA_ERR_CUDA;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return DA_ERR_CUDA;
  cudaError_t e = problem->is_mla ? da::mla_prepare(device) : da::gqa_prepare(device);
  cudaSetDevice(prev);
  if (e != cudaSuccess && e != cudaErrorNotSupported) return DA_ERR_CUDA;
  da_ctx *ctx = new (std::nothrow) da_ctx;
  if (!ctx) return DA_ERR_INVALID_ARG;
  std::memset(ctx, 0, sizeof *ctx);
  ctx->prob = *problem;
  ctx->device = device;
  ctx->num_sms = sms;
  ctx->smem_per_sm = smem;
  *out = ctx;
  return DA_OK;
}

da_status decode_attn_plan_ex(da_ctx *ctx, const int32_t *seq_lens_host,
                              const int32_t *kv_num_blks_host, int32_t num_splits_override,
                              size_t *workspace_bytes) {
  if (!ctx) return DA_ERR_INVALID_ARG;
  da_plan_info info;
  da_status st = da::plan_compute(&ctx->prob, ctx->num_sms, ctx->smem_per_sm, seq_lens_host,
                                  kv_num_blks_host, num_splits_override, &info);
  if (st != DA_OK) return st;
  ctx->plan = info;
  ctx->planned = true;
  if (workspace_bytes) *workspace_bytes = (size_t)info.workspace_bytes;
  return DA_OK;
}

da_status decode_attn_plan(da_ctx *ctx, const int32_t *seq_lens_host, int32_t num_splits_override,
                           size_t *workspace_bytes) {
  return decode_attn_plan_ex(ctx, seq_lens_host, nullptr, num_splits_override, workspace_bytes);
}

da_status decode_attn_get_plan(const da_ctx *ctx, da_plan_info *info) {
  if (!ctx || !info) return DA_ERR_INVALID_ARG;
  if (!ctx->planned) return DA_ERR_NOT_PLANNED;
  *info = ctx->plan;
  return DA_OK;
}

da_status decode_attn_plan_info(const da_problem *problem, int32_t num_sms,
                                const int32_t *seq_lens_host, int32_t num_splits_override,
                                da_plan_info *info) {
  // GB300: 228 KB of shared memory per SM
  return da::plan_compute(problem, num_sms, 233472, seq_lens_host, nullptr, num_splits_override,
                          info);
}

da_status decode_attn_run(da_ctx *ctx, const da_args *args, void *workspace, size_t workspace_bytes,
                          da_stream_t stream) {
  if (!ctx || !args) return DA_ERR_INVALID_ARG;
  if (!ctx->planned) return DA_ERR_NOT_PLANNED;
  da_status st = check_workspace(ctx, workspace, workspace_bytes);
  if (st != DA_OK) return st;
  if (!(args->scale == args->scale)) return DA_ERR_INVALID_ARG;  // NaN scale
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DA_ERR_CUDA;
  if (dev != ctx->device) return DA_ERR_INVALID_ARG;  // the context's device must be current
  auto *ws = reinterpret_cast<uint8_t *>(workspace);
  auto s = reinterpret_cast<cudaStream_t>(stream);
  return ctx->prob.is_mla ? run_mla(ctx, args, ws, s) : run_gqa(ctx, args, ws, s);
}

da_status decode_attn_merge(da_ctx *ctx, const float *o_part, const float *lse_part,
                            int32_t num_splits, int32_t rows, int32_t dv, void *out, float *lse,
                            da_stream_t stream) {
  (void)ctx;
  if (!o_part || !lse_part || !out) return DA_ERR_INVALID_ARG;
  if (num_splits <= 0 || rows < 0 || dv <= 0 || dv % 4 != 0 || dv > 1024) return DA_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(out, 8)) return DA_ERR_INVALID_ARG;
  da::MergeParams m;
  m.o_part = o_part;
  m.lse_part = lse_part;
  m.out = reinterpret_cast<__nv_bfloat16 *>(out);
  m.lse = lse;
  m.rows = rows;
  m.num_splits = num_splits;
  m.rows_per_unit = 1;
  m.dv = dv;
  return da::launch_merge(m, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DA_OK
                                                                                      : DA_ERR_CUDA;
}

da_status decode_attn_get_error(da_ctx *ctx, void *workspace, da_stream_t stream, uint32_t *flags) {
  (void)ctx;
  if (!workspace || !flags) return DA_ERR_INVALID_ARG;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DA_ERR_CUDA;
  if (word) {
    if (cudaMemsetAsync(workspace, 0, sizeof word, s) != cudaSuccess) return DA_ERR_CUDA;
    if ((word & DA_DEVERR_TIMEOUT) && ctx && ctx->planned) {
      auto *ws = reinterpret_cast<uint8_t *>(workspace);
      // every counter (the region between the counters and the partials)
      const size_t nbytes = (size_t)(ctx->plan.partial_o_offset - ctx->plan.counters_offset);
      if (cudaMemsetAsync(ws + ctx->plan.counters_offset, 0, nbytes, s) != cudaSuccess)
        return DA_ERR_CUDA;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return DA_ERR_CUDA;
  }
  *flags = word;
  return word ? DA_ERR_DEVICE : DA_OK;
}

void decode_attn_destroy(da_ctx *ctx) { delete ctx; }

const char *decode_attn_status_string(da_status status) {
  switch (status) {
    case DA_OK: return "ok";
    case DA_ERR_INVALID_ARG: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported problem";
    case DA_ERR_CUDA: return "CUDA error";
    case DA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DA_ERR_NOT_PLANNED: return "decode_attn_plan has not been called";
    case DA_ERR_DEVICE: return "device reported an error (see the DA_DEVERR_* bits)";
  }
  return "unknown status";
}

}  // extern "C"

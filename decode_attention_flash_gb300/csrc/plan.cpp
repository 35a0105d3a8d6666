// plan.cpp -- host planner: the grid and the workspace layout of the split
// kernels. Pure host code.
//
// Both kernels are persistent: the host sizes one wave of resident CTAs (GQA)
// or CTA pairs (MLA clusters), never more than there are KV tiles, and the
// device cuts the concatenated tiles of all (row, kv head) units into one equal
// range per CTA or cluster. How a unit is split therefore follows from where
// the range boundaries fall: the split-KV decomposition of the flash-decoding
// method with the split lengths chosen for an even load rather than a fixed
// count (the XQA launcher, TensorRT-LLM xqa/mha.cu `launchMHA`, and the
// flex-decode template, flex_decode.py.jinja, both fix a split count per unit).
#include <algorithm>
#include <cstring>
#include <vector>

#include "internal.h"

namespace da {

namespace {
constexpr int kGqaTile = 64;
constexpr int kMlaTile = 64;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
int64_t align256(int64_t a) { return round_up(a, 256); }
}  // namespace

da_status validate_problem(const da_problem *p) {
  if (!p) return DA_ERR_INVALID_ARG;
  if (p->batch <= 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0) return DA_ERR_INVALID_ARG;
  if (p->q_dtype != DA_DTYPE_BF16) return DA_ERR_UNSUPPORTED;
  if (p->fp8_mma != 0 && p->fp8_mma != 1) return DA_ERR_INVALID_ARG;
  // e4m3 tensor-core arithmetic: e4m3 K/V with per-kv-head scales, GQA
  if (p->fp8_mma && (p->is_mla || p->kv_dtype != DA_DTYPE_FP8_E4M3)) return DA_ERR_UNSUPPORTED;
  if (p->kv_layout != DA_KV_CONTIGUOUS && p->kv_layout != DA_KV_PAGED) return DA_ERR_INVALID_ARG;
  if (p->kv_dtype != DA_DTYPE_BF16 && p->kv_dtype != DA_DTYPE_FP8_E4M3 &&
      p->kv_dtype != DA_DTYPE_FP8_E4M3_TOKEN_SCALE && p->kv_dtype != DA_DTYPE_INT4_GROUPS)
    return DA_ERR_INVALID_ARG;
  if (p->kv_dtype == DA_DTYPE_INT4_GROUPS) {
    if (!(p->kv_groups == 1 || p->kv_groups == 2 || p->kv_groups == 4 || p->kv_groups == 8))
      return DA_ERR_INVALID_ARG;
    // rows of groups + 16 words: TMA strides them only when a multiple of 16 bytes
    if (p->kv_groups < 4) return DA_ERR_UNSUPPORTED;
    // they travel as 128-byte lines: every tile's first row starts a line
    // (80-byte rows: cache lengths a multiple of 8; 96-byte rows: of 4)
    if (p->kv_layout == DA_KV_CONTIGUOUS && p->max_seq_len % (p->kv_groups == 4 ? 8 : 4) != 0)
      return DA_ERR_UNSUPPORTED;
  }
  if (p->max_seq_len < 0 || p->q_len < 0) return DA_ERR_INVALID_ARG;
  const int Q = p->q_len > 1 ? p->q_len : 1;  // query tokens per row
  if (p->kv_layout == DA_KV_PAGED) {
    if (p->page_size <= 0 || p->max_pages_per_seq <= 0 || p->num_pages <= 0)
      return DA_ERR_INVALID_ARG;
    if ((int64_t)p->max_seq_len > (int64_t)p->max_pages_per_seq * p->page_size)
      return DA_ERR_INVALID_ARG;
  }
  if (p->is_mla) {
    if (Q > 16) return DA_ERR_UNSUPPORTED;  // the draft-tree mask is one word per query token
    if (p->num_kv_heads != 1 || p->ckv_dim != 512 || p->kpe_dim != 64 || p->head_dim_qk != 576 ||
        p->head_dim_v != 512 || p->num_q_heads != 128)
      return DA_ERR_UNSUPPORTED;
    if (p->kv_layout != DA_KV_PAGED || p->page_size != 64) return DA_ERR_UNSUPPORTED;
    if (p->kv_dtype != DA_DTYPE_BF16 || p->sparse_block_size != 0) return DA_ERR_UNSUPPORTED;
    if ((int64_t)p->num_pages * p->page_size * 8 >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    return DA_OK;
  }
  if (p->num_q_heads % p->num_kv_heads) return DA_ERR_INVALID_ARG;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G * Q > 16) return DA_ERR_UNSUPPORTED;  // the G x Q rows of a kv head: two n-tiles at most
  if (p->head_dim_qk != 128 || p->head_dim_v != 128) return DA_ERR_UNSUPPORTED;
  if (p->kv_layout == DA_KV_PAGED) {
    const int P = p->page_size;
    if (P % 16 != 0 || !(kGqaTile % P == 0 || P % kGqaTile == 0)) return DA_ERR_UNSUPPORTED;
  }
  if (p->sparse_block_size < 0 || p->max_sparse_blocks < 0) return DA_ERR_INVALID_ARG;
  if (p->sparse_batch < 0 || p->sparse_heads < 0) return DA_ERR_INVALID_ARG;
  // per-token scale words are fetched by TMA in rows of four: cache rows per
  // (b, kv head) a multiple of 4
  if (p->kv_dtype == DA_DTYPE_FP8_E4M3_TOKEN_SCALE && p->kv_layout == DA_KV_CONTIGUOUS &&
      p->max_seq_len % 4 != 0)
    return DA_ERR_UNSUPPORTED;
  if (p->sparse_block_size > 0) {
    if (p->sparse_block_size % kGqaTile != 0) return DA_ERR_UNSUPPORTED;
    if (p->kv_layout != DA_KV_CONTIGUOUS) return DA_ERR_UNSUPPORTED;
    if (p->max_sparse_blocks <= 0) return DA_ERR_INVALID_ARG;
  }
  // TMA row coordinates are 32-bit: (cache rows) x (rows per token) must fit
  const int64_t rows = p->kv_layout == DA_KV_PAGED
                           ? (int64_t)p->num_pages * p->num_kv_heads * p->page_size
                           : (int64_t)p->batch * p->num_kv_heads * p->max_seq_len;
  if (rows * 2 + kGqaTile * 2 >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

// Resident CTAs of the split kernel per SM, from its shared-memory footprint.
static int ctas_per_sm(const da_problem *p, int32_t smem_per_sm) {
  const bool mla = p->is_mla != 0;
  const int per_cta = (mla ? mla_smem_bytes()
                           : gqa_smem_bytes(p->kv_dtype != DA_DTYPE_BF16,
                                            p->num_q_heads / p->num_kv_heads *
                                                (p->q_len > 1 ? p->q_len : 1),
                                            p->kv_dtype == DA_DTYPE_FP8_E4M3_TOKEN_SCALE,
                                            p->kv_dtype == DA_DTYPE_INT4_GROUPS)) +
                      1024;  // the runtime reserves 1 KB per CTA
  const int threads = mla ? mla_threads() : gqa_threads();
  return std::max(1, std::min(smem_per_sm / per_cta, 2048 / threads));
}

da_status plan_compute(const da_problem *p, int32_t num_sms, int32_t smem_per_sm,
                       const int32_t *seq_lens_host, const int32_t *kv_num_blks_host,
                       int32_t num_splits_override, da_plan_info *info) {
  da_status st = validate_problem(p);
  if (st != DA_OK) return st;
  if (!info || num_sms <= 0 || num_splits_override < 0) return DA_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof *info);

  const bool mla = p->is_mla != 0;
  const bool sparse = !mla && p->sparse_block_size > 0;
  const bool paged = p->kv_layout == DA_KV_PAGED;
  const int tile = mla ? kMlaTile : kGqaTile;
  const int align = sparse ? p->sparse_block_size : tile;
  // units: GQA (row, kv head); MLA (row, query token), whose heads share the latent cache
  const int Q = p->q_len > 1 ? p->q_len : 1;
  const int heads = mla ? Q : p->num_kv_heads;
  const int64_t units = (int64_t)p->batch * heads;
  const int64_t capacity =
      paged ? (int64_t)p->max_pages_per_seq * p->page_size : (int64_t)p->max_seq_len;
  // rows per unit: the G query heads (times the query tokens) of a kv head; MLA: all heads
  const int rows = mla ? p->num_q_heads : p->num_q_heads / p->num_kv_heads * Q;
  const int dv = p->head_dim_v;

  // positions per unit the split kernel walks (sparse: the compacted list)
  std::vector<int64_t> unit_len((size_t)units);
  for (int b = 0; b < p->batch; ++b) {
    for (int h = 0; h < heads; ++h) {
      int64_t len;
      if (sparse) {
        // the tables' row for (b, h): broadcast over rows / heads by modulo
        const int64_t sz = p->sparse_batch > 0 ? p->sparse_batch : p->batch;
        const int64_t sh = p->sparse_heads > 0 ? p->sparse_heads : heads;
        int64_t nblk = p->max_sparse_blocks;
        if (kv_num_blks_host)
          nblk = std::min<int64_t>(std::max<int32_t>(kv_num_blks_host[(b % sz) * sh + h % sh], 0),
                                   p->max_sparse_blocks);
        len = nblk * p->sparse_block_size;
      } else {
        len = seq_lens_host ? std::min<int64_t>(std::max<int32_t>(seq_lens_host[b], 0), capacity)
                            : std::min<int64_t>(p->max_seq_len, capacity);
        // MLA query token h of Q sees the positions n <= seq_len - Q + h
        if (mla) len = std::max<int64_t>(0, len - (Q - 1 - h));
      }
      unit_len[(size_t)((int64_t)b * heads + h)] = len;
    }
  }

  const int cps = ctas_per_sm(p, smem_per_sm);
  if (!mla) {
    // Persistent GQA grid: the tiles of all units are cut into equal ranges, one
    // per CTA, on the device; the host only sizes the grid (one wave of the
    // resident CTA slots, never more CTAs than tiles).
    int64_t tiles = 0;
    for (int64_t len : unit_len) tiles += ceil_div(len, tile);
    tiles = std::max<int64_t>(tiles, 1);
    int64_t ctas = (int64_t)num_sms * cps;
    if (num_splits_override > 0) ctas = (int64_t)num_splits_override * units;
    ctas = std::max<int64_t>(1, std::min<int64_t>(ctas, tiles));
    ctas = std::min<int64_t>(ctas, 65535);
    info->kv_tile = tile;
    info->chunk_tokens = (int32_t)(ceil_div(tiles, ctas) * tile);
    info->num_splits = (int32_t)ceil_div(ctas, units);
    info->num_units = (int32_t)units;
    info->rows_per_unit = rows;
    info->grid_x = (int32_t)ctas;
    info->grid_y = 1;
    info->grid_z = 1;
    info->ctas_per_sm = cps;
    info->writes_final = 0;  // decided per unit on the device
    int64_t off = kWorkspaceHeader;
    info->counters_offset = off;  // per unit: its counter, then its merge-group counters
    off = align256(off + units * (1 + max_merge_groups((int)ctas)) * 4);
    info->partial_o_offset = off;  // slots unit + cta
    off = align256(off + (units + ctas) * rows * (int64_t)dv * 4);
    info->partial_lse_offset = off;
    off = align256(off + (units + ctas) * rows * 4);
    info->workspace_bytes = off;
    return DA_OK;
  }

  // Persistent MLA grid: one cluster of two CTAs (one per value half) per pair
  // of SMs, never more clusters than tiles.
  int64_t tiles = 0;
  for (int64_t len : unit_len) tiles += ceil_div(len, tile);
  tiles = std::max<int64_t>(tiles, 1);
  int64_t clusters = std::max<int64_t>(1, (int64_t)num_sms * cps / 2);
  if (num_splits_override > 0) clusters = (int64_t)num_splits_override * units;
  clusters = std::max<int64_t>(1, std::min<int64_t>(clusters, tiles));
  clusters = std::min<int64_t>(clusters, 32767);
  info->kv_tile = tile;
  info->chunk_tokens = (int32_t)(ceil_div(tiles, clusters) * tile);
  info->num_splits = (int32_t)ceil_div(clusters, units);
  info->num_units = (int32_t)units;
  info->rows_per_unit = rows;
  info->grid_x = (int32_t)(2 * clusters);
  info->grid_y = 1;
  info->grid_z = 1;
  info->ctas_per_sm = cps;
  info->writes_final = 0;  // decided per row on the device
  int64_t off = kWorkspaceHeader;
  info->counters_offset = off;
  off = align256(off + units * 2 * 4);
  info->partial_o_offset = off;  // slots row + cluster
  off = align256(off + (units + clusters) * rows * (int64_t)dv * 4);
  info->partial_lse_offset = off;
  off = align256(off + (units + clusters) * rows * 2 * 4);
  info->workspace_bytes = off;
  return DA_OK;
}

}  // namespace da

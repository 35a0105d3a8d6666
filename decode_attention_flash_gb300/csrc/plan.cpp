// plan.cpp -- host planner: how many KV splits per (batch row, kv head) unit,
// the grid, and the workspace layout. Pure host integer code.
//
// The split count follows the idea of the XQA launcher (TensorRT-LLM
// xqa/mha.cu, `launchMHA`: sub-sequences per sequence = SMs / (B x HKV),
// capped by the sequence length in CTA tiles) and the tile-aligned split
// length of the flex-decode template (flex_decode.py.jinja:
// TILE_KV = cdiv(cdiv(KV_LEN, SPLIT_KV), BLOCK_N) * BLOCK_N): the planner
// sizes one split length (a multiple of the KV tile; of the sparse block for
// block-sparse decode) so that the CTAs of all units fill every SM a few
// times over, with at least kMinChunk positions per split so the per-split
// fixed cost (Q load, pipeline fill, partial write) stays small.
#include <algorithm>
#include <cstring>

#include "internal.h"

namespace da {

namespace {
constexpr int kGqaTile = 64;
constexpr int kMlaTile = 64;
constexpr int kMinChunk = 256;
constexpr int kWaves = 2;  // CTA waves per SM the planner aims for

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
int64_t align256(int64_t a) { return round_up(a, 256); }
}  // namespace

da_status validate_problem(const da_problem *p) {
  if (!p) return DA_ERR_INVALID_ARG;
  if (p->batch <= 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0) return DA_ERR_INVALID_ARG;
  if (p->q_dtype != DA_DTYPE_BF16) return DA_ERR_UNSUPPORTED;
  if (p->kv_layout != DA_KV_CONTIGUOUS && p->kv_layout != DA_KV_PAGED) return DA_ERR_INVALID_ARG;
  if (p->kv_dtype != DA_DTYPE_BF16 && p->kv_dtype != DA_DTYPE_FP8_E4M3) return DA_ERR_INVALID_ARG;
  if (p->max_seq_len < 0) return DA_ERR_INVALID_ARG;
  if (p->kv_layout == DA_KV_PAGED) {
    if (p->page_size <= 0 || p->max_pages_per_seq <= 0 || p->num_pages <= 0)
      return DA_ERR_INVALID_ARG;
    if ((int64_t)p->max_seq_len > (int64_t)p->max_pages_per_seq * p->page_size)
      return DA_ERR_INVALID_ARG;
  }
  if (p->is_mla) {
    if (p->num_kv_heads != 1 || p->ckv_dim != 512 || p->kpe_dim != 64 || p->head_dim_qk != 576 ||
        p->head_dim_v != 512 || p->num_q_heads != 128)
      return DA_ERR_UNSUPPORTED;
    if (p->kv_layout != DA_KV_PAGED || p->page_size != 64) return DA_ERR_UNSUPPORTED;
    if (p->kv_dtype != DA_DTYPE_BF16 || p->sparse_block_size != 0) return DA_ERR_UNSUPPORTED;
    if ((int64_t)p->num_pages * p->page_size * 2 >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    return DA_OK;
  }
  if (p->num_q_heads % p->num_kv_heads) return DA_ERR_INVALID_ARG;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G > 16) return DA_ERR_UNSUPPORTED;
  if (p->head_dim_qk != 128 || p->head_dim_v != 128) return DA_ERR_UNSUPPORTED;
  if (p->kv_layout == DA_KV_PAGED) {
    const int P = p->page_size;
    if (P % 16 != 0 || !(kGqaTile % P == 0 || P % kGqaTile == 0)) return DA_ERR_UNSUPPORTED;
  }
  if (p->sparse_block_size < 0 || p->max_sparse_blocks < 0) return DA_ERR_INVALID_ARG;
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
  const int per_cta = (p->is_mla ? mla_smem_bytes() : gqa_smem_bytes(p->kv_dtype == DA_DTYPE_FP8_E4M3)) +
                      1024;  // the runtime reserves 1 KB per CTA
  return std::max(1, std::min(smem_per_sm / per_cta, 2048 / (p->is_mla ? mla_threads() : gqa_threads())));
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
  const int tile = mla ? kMlaTile : kGqaTile;
  const int align = sparse ? p->sparse_block_size : tile;
  const int heads = mla ? 1 : p->num_kv_heads;
  const int64_t units = (int64_t)p->batch * heads;
  const int64_t capacity = p->kv_layout == DA_KV_PAGED
                               ? (int64_t)p->max_pages_per_seq * p->page_size
                               : (int64_t)p->max_seq_len;

  // positions per unit the split kernel walks (sparse: the compacted list)
  int64_t max_len = 0, total = 0;
  for (int b = 0; b < p->batch; ++b) {
    for (int h = 0; h < heads; ++h) {
      int64_t len;
      if (sparse) {
        int64_t nblk = p->max_sparse_blocks;
        if (kv_num_blks_host) {
          nblk = std::min<int64_t>(std::max<int32_t>(kv_num_blks_host[(int64_t)b * heads + h], 0),
                                   p->max_sparse_blocks);
        }
        len = nblk * p->sparse_block_size;
      } else {
        len = seq_lens_host ? std::min<int64_t>(std::max<int32_t>(seq_lens_host[b], 0), capacity)
                            : std::min<int64_t>(p->max_seq_len, capacity);
      }
      max_len = std::max(max_len, len);
      total += len;
    }
  }
  const int cps = ctas_per_sm(p, smem_per_sm);
  int64_t chunk;
  if (num_splits_override > 0) {
    chunk = round_up(std::max<int64_t>(ceil_div(std::max<int64_t>(max_len, 1), num_splits_override), 1),
                     align);
  } else {
    const int64_t target = (int64_t)num_sms * cps * kWaves;
    chunk = round_up(std::max<int64_t>(ceil_div(total, target), 1), align);
    chunk = std::max<int64_t>(chunk, round_up(kMinChunk, align));
  }
  chunk = std::min<int64_t>(chunk, round_up(std::max<int64_t>(max_len, 1), align));
  if (chunk > (1ll << 30)) return DA_ERR_UNSUPPORTED;
  const int64_t splits = std::max<int64_t>(1, ceil_div(max_len, chunk));
  if (splits > 65535) return DA_ERR_UNSUPPORTED;

  const int rows = mla ? p->num_q_heads : p->num_q_heads / p->num_kv_heads;
  const int dv = p->head_dim_v;
  info->kv_tile = tile;
  info->chunk_tokens = (int32_t)chunk;
  info->num_splits = (int32_t)splits;
  info->num_units = (int32_t)units;
  info->rows_per_unit = rows;
  info->grid_x = (int32_t)splits;
  info->grid_y = heads;
  info->grid_z = p->batch;
  info->ctas_per_sm = cps;
  info->writes_final = splits == 1 ? 1 : 0;
  int64_t off = kWorkspaceHeader;
  if (!info->writes_final) {
    info->partial_o_offset = off;
    off = align256(off + units * splits * rows * (int64_t)dv * 4);
    info->partial_lse_offset = off;
    off = align256(off + units * splits * rows * 4);
  }
  info->workspace_bytes = off;
  return DA_OK;
}

}  // namespace da

// internal.h -- host/device structures shared by the C ABI and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_attn.h"

namespace da {

// Time limit of every pipeline wait inside a kernel (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1500ull * 1000ull * 1000ull;

// Workspace: [error word | pad to 256 B][unit counters u32][partial O fp32][partial LSE fp32]
constexpr int64_t kWorkspaceHeader = 256;
// Page / block ids one split CTA stages in shared memory (caps the split length).
constexpr int kGqaMaxIds = 512;
// Splits per unit the fused merge handles (its weights live in shared memory).
constexpr int kMaxSplits = 256;

struct GqaParams {
  const __nv_bfloat16 *q;      // [B][HQ][128]
  const int32_t *block_table;  // paged: [B][max_pages]
  const int32_t *seq_lens;     // [B]
  const int32_t *kv_num_blks;  // sparse: [B][HKV]
  const int32_t *kv_idx;       // sparse: [B][HKV][max_sparse_blocks]
  const int32_t *kv_full_num_blks;  // sparse, optional: the full-block table, [B][HKV]
  const int32_t *kv_full_idx;       // and [B][HKV][max_sparse_blocks] (attended after kv_idx)
  const uint32_t *spec_mask;   // q_len > 1, optional: [B][q_len] draft-tree mask words
  const int32_t *mask_sink;    // optional [HQ] (with mask_window): positions below are kept
  const int32_t *mask_window;  // optional [HQ]: the sink/window mask_mod (< 0: no window)
  const float *alibi_slopes;   // optional [HQ]: the ALiBi score_mod, slope * (n - q_pos)
  const float *k_scale;        // fp8: [HKV]
  const float *v_scale;        // fp8: [HKV]
  float *o_part;               // [units + ctas][G][128] partial slots (slot = unit + cta)
  float *lse_part;             // [units + ctas][G]
  __nv_bfloat16 *out;          // [B][HQ][128]
  float *lse;                  // [B][HQ] or null
  uint32_t *err;               // device error word
  uint32_t *counters;          // [units] finished-split counters (self-resetting)
  float score_scale;           // scale * log2(e)
  float softcap_l2;            // 0, or the soft cap c times log2(e): x -> c2 * tanh(x / c2)
  float softcap_k;             // 2 / c: exp(2 x / c2) = exp2(x * softcap_k)
  int32_t batch, num_q_heads, num_kv_heads, group;  // num_q_heads, group: rows (heads x q_len)
  int32_t token_scale;         // e4m3 K/V with per-token scale words (maps kss / vss)
  int32_t kv_groups;           // int4 group-wise K/V: groups per row (whole rows of
                               // groups + 16 words by maps k / v); 0 otherwise
  int32_t q_len;               // query tokens per row: token t of a unit row g * q_len + t
                               // sees the positions n <= seq_len - q_len + t
  int32_t paged, page_size, cache_len, max_pages, num_pages;
  int32_t capacity;            // max positions per row
  int32_t sparse_block_size, max_sparse_blocks;
  int32_t sparse_batch, sparse_heads;  // block tables' extents (row (b % SZ, h % SH))
  int32_t fp8_mma;             // e4m3 tensor-core QK / PV (the e4m3_mma instantiations)
  uint32_t test_stall_ns;      // 0; else (tests of the timeout path only) the first
                               // pipeline wait of consumer warp 0 is one on a barrier
                               // that nothing arrives on, given up after this long
};

// Group counters per GQA unit for the two-level merge of a unit cut into many
// pieces (groups of ceil(sqrt(pieces)) pieces; pieces <= CTAs): shared by the
// planner, which sizes the workspace, and the kernel.
__host__ __device__ inline int ceil_sqrt(int n) {
  int k = 1;
  while (k * k < n) ++k;
  return k;
}
__host__ __device__ inline int max_merge_groups(int ctas) { return ceil_sqrt(ctas) + 1; }

struct MergeParams {
  const float *o_part;   // element (u, s, g, d) at ((u*S + s)*R + g)*dv + d
  const float *lse_part; // element (u, s, g) at (u*S + s)*R + g
  __nv_bfloat16 *out;    // [rows][dv], row = u*R + g
  float *lse;            // [rows] or null
  int32_t rows, num_splits, rows_per_unit, dv;
};

// MLA rows are (b, t) pairs, v = b * Q + t for the Q query tokens of batch
// row b: token t attends to the positions n <= seq_lens[b] - Q + t (or those
// its draft-tree mask word selects among the last Q).
struct MlaParams {
  const __nv_bfloat16 *q_nope;  // [B][128][Q][512]
  const __nv_bfloat16 *q_pe;    // [B][128][Q][64]
  const int32_t *block_table;
  const int32_t *seq_lens;
  const uint32_t *spec_mask;    // Q > 1, optional: [B][Q] draft-tree mask words
  float *o_part;                // [B*Q + clusters][128][512]: slot v + cluster of a row segment
                                // (rank r writes columns 256r..256r+255)
  float *lse_part;              // [B*Q + clusters][2][128] (one copy per rank)
  __nv_bfloat16 *out;           // [B][128][Q][512]
  float *lse;                   // [B][128][Q]
  uint32_t *err;
  uint32_t *counters;           // [B*Q][2]: finished segments per (row, rank)
  float score_scale;
  int32_t batch, max_pages, num_pages, capacity;
  int32_t q_len;                // Q >= 1
};

// Kernel launchers (return the launch error).
cudaError_t gqa_prepare(int device);  // sets shared-memory attributes once per device
int gqa_smem_bytes(bool fp8, int group, bool token_scale, bool int4);
int gqa_threads();
cudaError_t launch_gqa(bool fp8, int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                       const CUtensorMap &qmap, const CUtensorMap &kssmap,
                       const CUtensorMap &vssmap, const GqaParams &p, int ctas,
                       cudaStream_t stream);
int gqa_box_tokens(const da_problem &p);

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream);

cudaError_t mla_prepare(int device);
int mla_smem_bytes();
int mla_threads();
cudaError_t launch_mla(const CUtensorMap &qp_map, const CUtensorMap &ckv_map,
                       const CUtensorMap &kpe_map, const MlaParams &p, dim3 grid,
                       cudaStream_t stream);

// Planner (pure host code).
da_status plan_compute(const da_problem *p, int32_t num_sms, int32_t smem_per_sm,
                       const int32_t *seq_lens_host, const int32_t *kv_num_blks_host,
                       int32_t num_splits_override, da_plan_info *info);
da_status validate_problem(const da_problem *p);

}  // namespace da

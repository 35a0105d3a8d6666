// gqa_split.cu -- split-KV GQA decode kernel for sm_103a.
//
// One CTA per (split s, kv head h, batch row b). It owns the contiguous slice
// of the row's valid positions [s*chunk, (s+1)*chunk) (block-sparse: that
// slice of the row's compacted block list), loads the whole GQA group of G
// query heads once (the row packing of the TorchInductor flex_decode.py.jinja
// template, hq = h*G + g), streams K/V tiles of 64 tokens by TMA into a
// multi-stage shared-memory ring guarded by mbarriers, and runs
//   S^T = K Q^T  and  O^T += V^T P^T
// on the tensor cores (bf16 or, for e4m3 KV, f16 operands, fp32 accumulate).
// The GQA group is the MMA's N dimension (8 per n-tile) and the tokens / the
// head dimension are its M dimension, so no MMA rows are spent on padding the
// 4-8 query heads up to 16.
//
// Online softmax follows the exp2 form of the split-K Triton kernel page
// (mslk splitk_kernels.py, `_fwd_kernel_splitK`: m_new = max(m, rowmax),
// alpha = 2^(m - m_new), p = 2^(s - m_new), l = alpha*l + sum p), with the
// scale*log2(e) factor folded into the scores (the PRESCALE_QK idea of
// flex_decode.py.jinja) and the guards for a fully masked row. Each of the
// four consumer warps keeps its own running (m, l, acc) over its 16 tokens of
// every tile; the warps are merged once at the end through shared memory.
//
// Split epilogue (`_fwd_kernel_splitK` "write back O"): O_part = acc / l (0
// when l = 0) and lse = ln(l) + m*ln 2 (-inf when l = 0); a plan with a single
// split writes the final bf16 output and LSE directly.
//
// Warp roles: warps 0-3 consume (16 tokens of each tile each), warp 4 lane 0
// produces (page-table / sparse-list lookups, bounds checks, TMA issue).
#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kTile = 64;             // tokens per pipeline stage
constexpr int kConsumerWarps = 4;     // 16 tokens of each tile per warp
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kD = 128;               // head dimension
constexpr int kRedStride = kD + 4;    // padded row of the end-of-split reduction buffer

template <bool FP8>
struct Traits {
  static constexpr int kBytesPerTok = FP8 ? kD : 2 * kD;
  static constexpr int kTileBytes = kTile * kBytesPerTok;  // one of K or V
  static constexpr int kStages = FP8 ? 6 : 3;
  static constexpr int kRingBytes = kStages * 2 * kTileBytes;
};

struct __align__(8) StageMeta {
  uint64_t valid;  // bit j: token j of the tile is a valid position
};

template <bool FP8>
struct Smem {
  // ring: stage s holds K at [s][0] and V at [s][1], each kTileBytes, 1024-aligned
  static constexpr int kRing = 0;
  static constexpr int kFull = Traits<FP8>::kRingBytes;
  static constexpr int kEmpty = kFull + 8 * Traits<FP8>::kStages;
  static constexpr int kMeta = kEmpty + 8 * Traits<FP8>::kStages;
  static constexpr int kFlags = kMeta + 8 * Traits<FP8>::kStages;  // abort, last-CTA
  static constexpr int kStats = kFlags + 16;              // m, l per (warp, g): 2*4*16 floats
  static constexpr int kIds = kStats + 2 * kConsumerWarps * 16 * 4;  // page / block ids
  static constexpr int kTotal = kIds + kGqaMaxIds * 4 + 1024;        // + align slack
};

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// ------------------------------------------------------------------ producer

// Fills tile `i` of this CTA into stage `st`: takes the pages / sparse block
// from the ids staged in shared memory (already range-checked; -1 marks an
// invalid one, which is skipped), records which tokens are valid and issues
// the TMA boxes.
template <bool FP8>
__device__ __forceinline__ void produce_tile(const GqaParams &p, const CUtensorMap *kmap,
                                             const CUtensorMap *vmap, uint8_t *ring,
                                             uint64_t *full, StageMeta *meta, const int *ids,
                                             int st, int i, int b, int h, int n_valid,
                                             int range_lo, int range_hi, uint64_t policy) {
  using T = Traits<FP8>;
  uint8_t *kdst = ring + (size_t)st * 2 * T::kTileBytes;
  uint8_t *vdst = kdst + T::kTileBytes;
  const int row_mult = FP8 ? 1 : 2;  // bf16 rows are split into two 128-byte TMA rows
  uint64_t valid = 0;
  int64_t row0 = -1;  // first cache row of a single-box tile

  if (p.sparse_block_size > 0) {
    const int tiles_per_block = p.sparse_block_size / kTile;
    const int blk = ids[i / tiles_per_block];
    if (blk >= 0) {
      const int tok_base = blk * p.sparse_block_size + (i % tiles_per_block) * kTile;
      int lim = min(n_valid - tok_base, kTile);
      lim = min(lim, p.cache_len - tok_base);
      if (lim > 0) {
        valid = lim >= 64 ? ~0ull : ((1ull << lim) - 1ull);
        row0 = ((int64_t)b * p.num_kv_heads + h) * p.cache_len + tok_base;
      }
    }
  } else {
    const int tok_base = range_lo + i * kTile;
    const int lim = min(range_hi - tok_base, kTile);
    if (!p.paged) {
      if (lim > 0) {
        valid = lim >= 64 ? ~0ull : ((1ull << lim) - 1ull);
        row0 = ((int64_t)b * p.num_kv_heads + h) * p.cache_len + tok_base;
      }
    } else if (p.page_size >= kTile) {
      const int page = ids[tok_base / p.page_size - range_lo / p.page_size];
      if (page >= 0 && lim > 0) {
        valid = lim >= 64 ? ~0ull : ((1ull << lim) - 1ull);
        row0 = ((int64_t)page * p.num_kv_heads + h) * p.page_size + tok_base % p.page_size;
      }
    } else {
      // several pages per tile: one box per page
      const int P = p.page_size;
      const int first = tok_base / P - range_lo / P;
      int nbox = 0;
      for (int j = 0; j < kTile / P; ++j) {
        const int t0 = tok_base + j * P;
        if (t0 >= range_hi) break;
        if (ids[first + j] < 0) continue;
        const int cnt = min(range_hi - t0, P);
        valid |= ((cnt >= 64 ? ~0ull : ((1ull << cnt) - 1ull)) << (j * P));
        ++nbox;
      }
      meta[st].valid = valid;
      // the transaction count is set before any copy is issued
      mbar_arrive_expect_tx(&full[st], 2u * (uint32_t)(nbox * P * T::kBytesPerTok));
      for (int j = 0; j < kTile / P; ++j) {
        if (tok_base + j * P >= range_hi) break;
        const int page = ids[first + j];
        if (page < 0) continue;
        const int y = (int)(((int64_t)page * p.num_kv_heads + h) * P * row_mult);
        const int off = j * P * T::kBytesPerTok;
        tma_load_2d(kdst + off, kmap, &full[st], 0, y, policy);
        tma_load_2d(vdst + off, vmap, &full[st], 0, y, policy);
      }
      return;
    }
  }
  meta[st].valid = valid;
  if (row0 >= 0) {
    const int y = (int)(row0 * row_mult);
    mbar_arrive_expect_tx(&full[st], 2u * (uint32_t)T::kTileBytes);
    tma_load_2d(kdst, kmap, &full[st], 0, y, policy);
    tma_load_2d(vdst, vmap, &full[st], 0, y, policy);
  } else {
    mbar_arrive_expect_tx(&full[st], 0);
  }
}

// Stages the page ids (paged) or listed block ids (sparse) of this CTA's range
// into shared memory with the producer warp's 32 lanes, checking every one:
// an id outside the pool / cache becomes -1 and sets an error bit.
__device__ __forceinline__ uint32_t stage_ids(const GqaParams &p, int *ids, int b, int h,
                                              int range_lo, int range_hi, int lane) {
  uint32_t err = 0;
  if (p.sparse_block_size > 0) {
    const int32_t *list = p.kv_idx + ((int64_t)b * p.num_kv_heads + h) * p.max_sparse_blocks;
    for (int j = lane; j < range_hi - range_lo; j += 32) {
      int blk = list[range_lo + j];
      if (blk < 0 || (int64_t)blk * p.sparse_block_size >= p.cache_len) {
        err |= DA_DEVERR_SPARSE_INDEX;
        blk = -1;
      }
      ids[j] = blk;
    }
  } else if (p.paged) {
    const int first = range_lo / p.page_size;
    const int count = (range_hi - 1) / p.page_size - first + 1;
    const int32_t *row = p.block_table + (int64_t)b * p.max_pages + first;
    for (int j = lane; j < count; j += 32) {
      int page = row[j];
      if (page < 0 || page >= p.num_pages) {
        err |= DA_DEVERR_PAGE_INDEX;
        page = -1;
      }
      ids[j] = page;
    }
  }
  return err;
}

// The last CTA of a (b, kv head) unit to finish merges the unit's per-split
// results (LSE-weighted, as `_splitK_reduce` of splitk_kernels.py) into the
// final bf16 output and LSE -- the multi-block merge of TensorRT-LLM
// xqa/mha.cu, found with an atomic counter per unit and no spinning wait. The
// counter is reset by the merging CTA, so it is zero again for the next call.
__device__ __forceinline__ void merge_if_last(const GqaParams &p, int b, int h, int G,
                                              float *scratch, volatile int *last_flag) {
  const int64_t unit = (int64_t)b * p.num_kv_heads + h;
  const int S = p.num_splits;
  __threadfence();  // this CTA's partial results are visible before the count
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(p.counters + unit, 1u);
    *last_flag = (prev == (unsigned)(S - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!*last_flag) return;
  __threadfence();
  float *w = scratch;           // [S][16] weights (lse first)
  float *stat = w + S * 16;     // [16] 1/sum, [16] lse
  const float *lse_part = p.lse_part + unit * S * G;
  for (int i = threadIdx.x; i < S * G; i += blockDim.x)
    w[(i / G) * 16 + (i % G)] = __ldcg(lse_part + i);
  __syncthreads();
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float M = neg_inf();
    for (int s = 0; s < S; ++s) M = fmaxf(M, w[s * 16 + g]);
    float sum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float l = w[s * 16 + g];
      const float e = (M == neg_inf() || l == neg_inf()) ? 0.f : ex2((l - M) * 1.4426950408889634f);
      w[s * 16 + g] = e;
      sum += e;
    }
    stat[g] = sum > 0.f ? 1.f / sum : 0.f;
    stat[16 + g] = sum > 0.f ? M + __log2f(sum) * 0.69314718055994531f : neg_inf();
  }
  __syncthreads();
  const float4 *o_part = reinterpret_cast<const float4 *>(p.o_part + unit * S * G * kD);
  for (int i = threadIdx.x; i < G * (kD / 4); i += blockDim.x) {
    const int g = i / (kD / 4), c = i % (kD / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = 0; s < S; ++s) {
      const float e = w[s * 16 + g];
      if (e != 0.f) {
        const float4 v = __ldcg(o_part + ((int64_t)s * G + g) * (kD / 4) + c);
        acc.x += e * v.x;
        acc.y += e * v.y;
        acc.z += e * v.z;
        acc.w += e * v.w;
      }
    }
    const float inv = stat[g];
    __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
        p.out + ((int64_t)b * p.num_q_heads + h * G + g) * kD + 4 * c);
    dst[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    dst[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  }
  if (threadIdx.x < G && p.lse) p.lse[(int64_t)b * p.num_q_heads + h * G + threadIdx.x] = stat[16 + threadIdx.x];
  if (threadIdx.x == 0) p.counters[unit] = 0u;
}

// ------------------------------------------------------------------ consumer helpers

// Address of the 16-byte chunk `c` (0..15 for bf16 rows of 256 bytes, 0..7 for
// fp8 rows of 128 bytes) of token `t` in a 128B-swizzled tile.
template <bool FP8>
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int t, int c) {
  if (FP8) {
    return base + t * 128 + (((c ^ t) & 7) << 4);
  } else {
    const int r = 2 * t + (c >> 3);
    return base + r * 128 + ((((c & 7) ^ r) & 7) << 4);
  }
}

__device__ __forceinline__ uint32_t lo16_mask(bool a, bool b) {
  return (a ? 0x0000FFFFu : 0u) | (b ? 0xFFFF0000u : 0u);
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&x);
  float2 f = __bfloat1622float2(v);
  return pack_f16(f.x, f.y);
}

// ------------------------------------------------------------------ kernel

template <bool FP8, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_split_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const GqaParams p) {
  using T = Traits<FP8>;
  using S = Smem<FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem + S::kRing;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kFull);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + S::kEmpty);
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + S::kMeta);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kFlags);
  volatile int *last_flag = abort_flag + 1;
  int *ids = reinterpret_cast<int *>(smem + S::kIds);
  float *stat_m = reinterpret_cast<float *>(smem + S::kStats);
  float *stat_l = stat_m + kConsumerWarps * 16;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;

  // ---- this CTA's slice of the row
  int n_valid = p.seq_lens[b];
  uint32_t dev_err = 0;
  if (n_valid < 0 || n_valid > p.capacity) {
    dev_err |= DA_DEVERR_SEQ_LEN;
    n_valid = n_valid < 0 ? 0 : p.capacity;
  }
  int range_lo, range_hi, num_tiles;
  if (p.sparse_block_size > 0) {
    int nblk = p.kv_num_blks[(int64_t)b * p.num_kv_heads + h];
    if (nblk < 0 || nblk > p.max_sparse_blocks) {
      dev_err |= DA_DEVERR_SPARSE_INDEX;
      nblk = nblk < 0 ? 0 : p.max_sparse_blocks;
    }
    const int per_split = p.chunk / p.sparse_block_size;  // list entries per split
    range_lo = split * per_split;
    range_hi = min(range_lo + per_split, nblk);
    num_tiles = range_hi > range_lo ? (range_hi - range_lo) * (p.sparse_block_size / kTile) : 0;
  } else {
    range_lo = split * p.chunk;
    range_hi = min(range_lo + p.chunk, n_valid);
    num_tiles = range_hi > range_lo ? (range_hi - range_lo + kTile - 1) / kTile : 0;
  }

  const int64_t unit = (int64_t)b * p.num_kv_heads + h;
  const int64_t slot = unit * p.num_splits + split;

  if (num_tiles == 0) {
    // empty split: O = 0, LSE = -inf (its O slot is never read by the merge)
    if (threadIdx.x == 0 && dev_err) atomicOr(p.err, dev_err);
    if (threadIdx.x < G) {
      if (p.write_final) {
        const int64_t row = (int64_t)b * p.num_q_heads + h * G + threadIdx.x;
        if (p.lse) p.lse[row] = neg_inf();
      } else {
        p.lse_part[slot * G + threadIdx.x] = neg_inf();
      }
    }
    if (p.write_final) {
      for (int e = threadIdx.x; e < G * kD; e += blockDim.x)
        p.out[((int64_t)b * p.num_q_heads + h * G) * kD + e] = __float2bfloat16(0.f);
      return;
    }
    merge_if_last(p, b, h, G, reinterpret_cast<float *>(ring), last_flag);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < T::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // consumer state (per thread): O^T accumulators and the running softmax state
  float oacc[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[nt][mt][e] = 0.f;
  float m_run[NT][2], l_part[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = neg_inf();
    l_part[nt][0] = l_part[nt][1] = 0.f;
  }

  if (warp == kConsumerWarps) {
    // ================= producer =================
    dev_err |= stage_ids(p, ids, b, h, range_lo, range_hi, lane);
    __syncwarp();
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      const uint64_t policy = l2_policy_evict_first();
      for (int i = 0; i < num_tiles; ++i) {
        const int st = i % T::kStages;
        if (i >= T::kStages) {
          const uint32_t par = ((i / T::kStages) & 1) ^ 1;
          if (!mbar_wait_bounded(&empty[st], par, kWaitLimitNs)) {
            dev_err |= DA_DEVERR_TIMEOUT;
            *abort_flag = 1;
            break;
          }
        }
        produce_tile<FP8>(p, &kmap, &vmap, ring, full, meta, ids, st, i, b, h, n_valid,
                          range_lo, range_hi, policy);
      }
    }
  } else {
    // ================= consumers =================
    const int q4 = lane & 3;      // quad index: owns g = nt*8 + 2*q4 + {0,1}
    const int r8 = lane >> 2;     // row inside an 8-row group
    // Q^T as the B operand (k = head dim, n = query head of the group)
    uint32_t qf[NT][8][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = nt * 8 + r8;
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          p.q + ((int64_t)b * p.num_q_heads + h * G + (g < G ? g : 0)) * kD);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (!FP8) {
          // b0: d = 16ks + 2q4 (+1), b1: d = 16ks + 8 + 2q4 (+1)
          qf[nt][ks][0] = g < G ? qrow[(16 * ks + 2 * q4) / 2] : 0u;
          qf[nt][ks][1] = g < G ? qrow[(16 * ks + 8 + 2 * q4) / 2] : 0u;
        } else {
          // k-step ks = 2pp + e covers bytes 32pp + 16e + 4q4 .. +3 of each key row:
          // logical k (2q4, 2q4+1) -> d +0,+1 ; (2q4+8, 2q4+9) -> d +2,+3
          const int pp = ks >> 1, e = ks & 1;
          const int d0 = 32 * pp + 16 * e + 4 * q4;
          qf[nt][ks][0] = g < G ? bf16x2_to_f16x2(qrow[d0 / 2]) : 0u;
          qf[nt][ks][1] = g < G ? bf16x2_to_f16x2(qrow[d0 / 2 + 1]) : 0u;
        }
      }
    }
    float sscale = p.score_scale;
    if (FP8) sscale *= p.k_scale[h];


    const int tok_lane = 16 * warp + (lane & 7);  // ldmatrix row supplied by this lane
    const int mi = lane >> 3;                      // which 8x8 matrix this lane addresses

    for (int i = 0; i < num_tiles; ++i) {
      const int st = i % T::kStages;
      const uint32_t par = (i / T::kStages) & 1;
      if (!mbar_wait_bounded(&full[st], par, kWaitLimitNs)) {
        dev_err |= DA_DEVERR_TIMEOUT;
        *abort_flag = 1;
        break;
      }
      const uint32_t vbits = (uint32_t)(meta[st].valid >> (16 * warp)) & 0xFFFFu;
      if (vbits != 0) {
        const uint32_t kbase = smem_u32(ring + (size_t)st * 2 * T::kTileBytes);
        const uint32_t vbase = kbase + T::kTileBytes;
        // ---------------- S^T = K Q^T (16 tokens x 8*NT heads)
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
        if (!FP8) {
          const int t = tok_lane + (mi & 1) * 8;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(chunk_addr<false>(kbase, t, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16_16816(sacc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
          }
        } else {
          const int t = tok_lane + (mi & 1) * 8;
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(chunk_addr<true>(kbase, t, 2 * pp + (mi >> 1)), r0, r1, r2, r3);
            const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(r0 & 0xFFFF));
            const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(r0 >> 16));
            const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(r1 & 0xFFFF));
            const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(r1 >> 16));
            const uint32_t c0 = e4m3x2_to_f16x2((uint16_t)(r2 & 0xFFFF));
            const uint32_t c2 = e4m3x2_to_f16x2((uint16_t)(r2 >> 16));
            const uint32_t c1 = e4m3x2_to_f16x2((uint16_t)(r3 & 0xFFFF));
            const uint32_t c3 = e4m3x2_to_f16x2((uint16_t)(r3 >> 16));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_f16_16816(sacc[nt], a0, a1, a2, a3, qf[nt][2 * pp][0], qf[nt][2 * pp][1]);
              mma_f16_16816(sacc[nt], c0, c1, c2, c3, qf[nt][2 * pp + 1][0],
                            qf[nt][2 * pp + 1][1]);
            }
          }
        }
        // ---------------- mask, online softmax (exp2), P^T fragments
        const bool ok_r = (vbits >> r8) & 1u, ok_r8 = (vbits >> (r8 + 8)) & 1u;
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float alpha[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float x0 = ok_r ? sacc[nt][e] * sscale : neg_inf();
            const float x1 = ok_r8 ? sacc[nt][2 + e] * sscale : neg_inf();
            float tmax = fmaxf(x0, x1);
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
            const float m_new = fmaxf(m_run[nt][e], tmax);
            float p0 = 0.f, p1 = 0.f, a = 1.f;
            if (m_new != neg_inf()) {
              a = ex2(m_run[nt][e] - m_new);
              p0 = ex2(x0 - m_new);
              p1 = ex2(x1 - m_new);
            }
            l_part[nt][e] = l_part[nt][e] * a + (p0 + p1);
            m_run[nt][e] = m_new;
            sacc[nt][e] = p0;
            sacc[nt][2 + e] = p1;
            alpha[e] = a;
          }
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            oacc[nt][mt][0] *= alpha[0];
            oacc[nt][mt][1] *= alpha[1];
            oacc[nt][mt][2] *= alpha[0];
            oacc[nt][mt][3] *= alpha[1];
          }
          // P^T as the B operand: transpose the (token x head) 8x8 blocks
          const uint32_t x0 = FP8 ? pack_f16(sacc[nt][0], sacc[nt][1])
                                  : pack_bf16(sacc[nt][0], sacc[nt][1]);
          const uint32_t x1 = FP8 ? pack_f16(sacc[nt][2], sacc[nt][3])
                                  : pack_bf16(sacc[nt][2], sacc[nt][3]);
          pb[nt][0] = movmatrix_trans(x0);
          pb[nt][1] = movmatrix_trans(x1);
        }
        // ---------------- O^T += V^T P^T
        // tokens of this lane in the A fragment: 2q4, 2q4+1 (a0, a1) and +8 (a2, a3)
        const bool full16 = vbits == 0xFFFFu;
        const uint32_t m01 = lo16_mask((vbits >> (2 * q4)) & 1u, (vbits >> (2 * q4 + 1)) & 1u);
        const uint32_t m89 =
            lo16_mask((vbits >> (2 * q4 + 8)) & 1u, (vbits >> (2 * q4 + 9)) & 1u);
        if (!FP8) {
          const int t = tok_lane + (mi >> 1) * 8;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(chunk_addr<false>(vbase, t, 2 * mt + (mi & 1)), a0, a1, a2, a3);
            if (!full16) {
              a0 &= m01;
              a1 &= m01;
              a2 &= m89;
              a3 &= m89;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16_16816(oacc[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
          }
        } else {
          const int t = tok_lane + (mi & 1) * 8;
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(chunk_addr<true>(vbase, t, 2 * pp + (mi >> 1)), r0, r1, r2, r3);
            // r = [V[2q][2c], V[2q][2c+1], V[2q+1][2c], V[2q+1][2c+1]] -> token pairs per d
            const uint32_t s0 = prmt(r0, 0, 0x3120), s1 = prmt(r1, 0, 0x3120);
            const uint32_t s2 = prmt(r2, 0, 0x3120), s3 = prmt(r3, 0, 0x3120);
            uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(s0 & 0xFFFF));  // d 2c,   tokens 2q..
            uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(s0 >> 16));     // d 2c+1, tokens 2q..
            uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(s1 & 0xFFFF));  // d 2c,   tokens 2q+8..
            uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(s1 >> 16));
            uint32_t c0 = e4m3x2_to_f16x2((uint16_t)(s2 & 0xFFFF));
            uint32_t c1 = e4m3x2_to_f16x2((uint16_t)(s2 >> 16));
            uint32_t c2 = e4m3x2_to_f16x2((uint16_t)(s3 & 0xFFFF));
            uint32_t c3 = e4m3x2_to_f16x2((uint16_t)(s3 >> 16));
            if (!full16) {
              a0 &= m01;
              a1 &= m01;
              a2 &= m89;
              a3 &= m89;
              c0 &= m01;
              c1 &= m01;
              c2 &= m89;
              c3 &= m89;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_f16_16816(oacc[nt][2 * pp], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
              mma_f16_16816(oacc[nt][2 * pp + 1], c0, c1, c2, c3, pb[nt][0], pb[nt][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---------------- merge the four warps' partial softmax states
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = l_part[nt][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_part[nt][e] = l;
        if (r8 == 0) {
          const int g = nt * 8 + 2 * q4 + e;
          stat_m[warp * 16 + g] = m_run[nt][e];
          stat_l[warp * 16 + g] = l;
        }
      }
  }

  __syncthreads();  // all loops done: every issued TMA box has been consumed

  if (*abort_flag) {
    // a wait gave up: drain copies still in flight (bounded), report, leave
    if (threadIdx.x == kConsumerWarps * 32) {
      const int last = num_tiles - 1;
      for (int st = 0; st < T::kStages && st <= last; ++st) {
        const int i_last = last - ((last - st) % T::kStages);
        mbar_wait_bounded(&full[st], (i_last / T::kStages) & 1, kWaitLimitNs);
      }
    }
    if (lane == 0 || dev_err) atomicOr(p.err, dev_err | DA_DEVERR_TIMEOUT);
    return;
  }

  // Reduction buffer (reuses the ring): red[warp][g][kRedStride] fp32
  float *red = reinterpret_cast<float *>(ring);
  if (warp < kConsumerWarps) {
    const int q4 = lane & 3, r8 = lane >> 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int g = nt * 8 + 2 * q4 + e;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stat_m[w * 16 + g]);
        const float wscale = (M == neg_inf()) ? 0.f : ex2(m_run[nt][e] - M);
        float *dst = red + ((size_t)warp * 16 + g) * kRedStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          int d0, d1;
          if (!FP8) {
            d0 = 16 * mt + r8;
            d1 = d0 + 8;
          } else {
            d0 = 16 * mt + 2 * r8;
            d1 = d0 + 1;
          }
          dst[d0] = oacc[nt][mt][e] * wscale;
          dst[d1] = oacc[nt][mt][2 + e] * wscale;
        }
      }
  }
  __syncthreads();

  // thread tid < 128 owns head-dim element d = tid for every g of the group
  if (threadIdx.x < kD) {
    const int d = threadIdx.x;
    const float vmul = FP8 ? p.v_scale[h] : 1.f;
    for (int g = 0; g < G; ++g) {
      float M = neg_inf();
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stat_m[w * 16 + g]);
      float L = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = stat_m[w * 16 + g];
        const float sw = (M == neg_inf()) ? 0.f : ex2(mw - M);
        L += stat_l[w * 16 + g] * sw;
        acc += red[((size_t)w * 16 + g) * kRedStride + d];
      }
      const float o = (L > 0.f) ? acc * vmul / L : 0.f;
      // natural-log LSE: (m + log2 l) * ln 2
      const float lse = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : neg_inf();
      if (p.write_final) {
        const int64_t row = (int64_t)b * p.num_q_heads + h * G + g;
        p.out[row * kD + d] = __float2bfloat16(o);
        if (d == 0 && p.lse) p.lse[row] = lse;
      } else {
        p.o_part[(slot * G + g) * kD + d] = o;
        if (d == 0) p.lse_part[slot * G + g] = lse;
      }
    }
  }
  if (dev_err) atomicOr(p.err, dev_err);
  if (!p.write_final) merge_if_last(p, b, h, G, red, last_flag);
}

template <bool FP8, int NT>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gqa_split_kernel<FP8, NT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<FP8>::kTotal);
}

}  // namespace

int gqa_smem_bytes(bool fp8) { return fp8 ? Smem<true>::kTotal : Smem<false>::kTotal; }
int gqa_threads() { return kThreads; }

int gqa_box_tokens(const da_problem &p) {
  if (p.kv_layout == DA_KV_PAGED && p.page_size < kTile) return p.page_size;
  return kTile;
}

cudaError_t gqa_prepare(int /*device*/) {
  cudaError_t e;
  if ((e = set_attr<false, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<false, 2>()) != cudaSuccess) return e;
  if ((e = set_attr<true, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<true, 2>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_gqa(bool fp8, int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                       const GqaParams &p, dim3 grid, cudaStream_t stream) {
  const dim3 block(kThreads);
  if (!fp8) {
    if (group <= 8)
      gqa_split_kernel<false, 1><<<grid, block, Smem<false>::kTotal, stream>>>(kmap, vmap, p);
    else
      gqa_split_kernel<false, 2><<<grid, block, Smem<false>::kTotal, stream>>>(kmap, vmap, p);
  } else {
    if (group <= 8)
      gqa_split_kernel<true, 1><<<grid, block, Smem<true>::kTotal, stream>>>(kmap, vmap, p);
    else
      gqa_split_kernel<true, 2><<<grid, block, Smem<true>::kTotal, stream>>>(kmap, vmap, p);
  }
  return cudaGetLastError();
}

}  // namespace da

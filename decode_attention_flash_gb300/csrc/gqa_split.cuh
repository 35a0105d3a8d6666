// gqa_split.cuh -- persistent split-KV GQA decode kernel for sm_103a.
//
// What it computes: for every batch row b and query head hq = h*G + g (the
// GQA row packing of the TorchInductor flex_decode.py.jinja template), the
// softmax attention of q[b][hq] over the valid KV positions of kv head h --
// contiguous, paged through a block table, or the listed blocks of a
// block-sparse row (KV_NUM_BLKS / KV_IDX, indexed by kv head) -- with K/V in
// bf16 or in e4m3 with a per-kv-head scale.
//
// How. Every (b, kv head) pair is a "unit" of ceil(len / 64) KV tiles. The
// tiles of all units, laid end to end, are cut into gridDim.x equal ranges,
// one per CTA (a persistent grid sized to the resident CTA slots): every CTA
// streams the same number of 64-token tiles, wherever the unit boundaries
// fall, so all SMs stay busy to the end. A CTA's range covers pieces
// ("segments") of one or more units; a unit cut into several segments is the
// split-KV decomposition of the flex-decode / split-K pages. The range is
// computed on the device from seq_lens (and kv_num_blks), so the schedule
// follows the lengths the kernel actually reads.
//
// Per CTA: warp 4 produces -- it walks the tiles, looks up page / block ids one
// tile ahead, checks them, and streams K/V (and the segment's query group) by
// TMA into a multi-stage shared-memory ring guarded by mbarriers -- and warps
// 0-3 consume: each owns 16 tokens of every tile and runs
//   S^T = K Q^T  and  O^T += V^T P^T
// on the tensor cores (mma.sync m16n8k16, bf16 or -- for e4m3 KV, decoded
// exactly in registers -- f16 operands, fp32 accumulate). The GQA group is the
// MMA's N dimension (8 per n-tile), so no MMA rows are spent padding 4-8 query
// heads up to 16. The online softmax follows the exp2 form of the split-K
// Triton kernel page (mslk splitk_kernels.py, `_fwd_kernel_splitK`), with
// scale*log2(e) folded into the scores (flex's PRESCALE_QK idea) and guards
// for fully masked rows.
//
// Segment epilogue (`_fwd_kernel_splitK` "write back O"): the four warps'
// (m, l, O) are merged in shared memory; a unit held by one segment writes
// the final bf16 output and natural-log LSE, otherwise the segment writes its
// normalised O and LSE to a partial slot and the last segment of the unit to
// finish (an atomic counter, the multi-block merge of TensorRT-LLM
// xqa/mha.cu) merges the unit's segments LSE-weighted (`_splitK_reduce`).
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kTile = 64;             // tokens per pipeline stage
constexpr int kIdAhead = 4;           // tiles whose page / block ids are fetched ahead (ids <= 32)
constexpr int kConsumerWarps = 4;     // 16 tokens of each tile per warp
// A sixth warp takes the row-counter atomics of partial segments off the
// consumers and merges small units while they stream.
template <int NT>
constexpr bool has_helper() { return true; }
template <int NT>
constexpr int threads_for() { return (kConsumerWarps + 1 + (has_helper<NT>() ? 1 : 0)) * 32; }
constexpr int kMaxThreads = (kConsumerWarps + 2) * 32;
constexpr int kD = 128;               // head dimension
constexpr int kRedStride = kD + 4;    // padded row of the epilogue reduction buffer
constexpr uint32_t kConsumerBar = 1;  // named barrier of the 128 consumer threads

// int4 group-wise rows: a token's groups coefficient words, then its 16 data
// words (64 bytes); at most 8 groups. The rows land in shared memory as they
// are in the cache (row pitch (groups + 16) * 4 bytes).
constexpr int kI4MaxGroups = 8;

template <bool FP8, int NT, bool TOK = false, bool I4 = false>
struct Cfg {
  static constexpr int kBytesPerTok = I4 ? (kI4MaxGroups + kD / 8) * 4 : (FP8 ? kD : 2 * kD);
  static constexpr int kTileBytes = kTile * kBytesPerTok;  // one of K or V
  static constexpr int kStages = I4 ? 6 : (FP8 ? (NT == 1 ? 5 : 4) : 3);
  static constexpr int kQSlot = NT * 8 * kD * 2;             // the query group (bf16 rows)
  // shared-memory layout (byte offsets from a 1024-aligned base)
  static constexpr int oRing = 0;                            // [stage][K|V][tile]
  static constexpr int oQ = oRing + kStages * 2 * kTileBytes;
  // The segment epilogue reduces the four warps' partial O^T through the
  // segment's consumed stage: rows padded to kRedStride floats when that fits,
  // else plain 128-float rows with an XOR swizzle of the column (both free of
  // bank conflicts); a separate buffer only when neither fits (e4m3 stages).
  static constexpr bool kScrPadded = kConsumerWarps * 8 * NT * kRedStride * 4 <= 2 * kTileBytes;
  static constexpr bool kScrSwizzled = !kScrPadded && kConsumerWarps * 8 * NT * kD * 4 <= 2 * kTileBytes;
  static constexpr bool kStageScratch = kScrPadded || kScrSwizzled;
  static constexpr int kScrStride = kScrPadded ? kRedStride : kD;
  // (the separate buffer also serves the rare staged merge; two n-tiles of
  // bf16 drop it for a third KV stage and use the query slots there instead)
  static constexpr int kRedBytes = (kStageScratch && NT == 2) ? 0 : 8 * NT * kRedStride * 4;
  static constexpr int oRed = oQ + kStages * kQSlot;          // [8*NT][kRedStride] fp32, or nothing
  static constexpr int oFull = oRed + kRedBytes;
  static constexpr int oEmpty = oFull + 8 * kStages;
  static constexpr int oMeta = oEmpty + 8 * kStages;
  // m, l per (warp, g), two copies: segment k's epilogue uses copy k & 1, so a
  // warp that has finished segment k and reaches segment k + 1's epilogue never
  // overwrites what another warp still reads for segment k (a warp with no
  // valid token in a short segment gets there quickly)
  static constexpr int kStatFloats = 2 * kConsumerWarps * 16;
  static constexpr int oStats = oMeta + 32 * kStages;
  static constexpr int oScan = oStats + 2 * kStatFloats * 4;
  static constexpr int oFlags = oScan + 16 * 4;              // 40 ints (see the kernel)
  static constexpr int oIds = oFlags + 40 * 4;               // page / block id queue (32 ints)
  static constexpr int oMergeBar = oIds + 32 * 4;            // mbarriers: 2 of the merge staging,
                                                             // 2 partial-segment, 1 epilogue,
                                                             // 1 never arrived on (test stall)
  // e4m3 with per-token scales: [stage][K|V][kSSWords] scale words (TMA
  // destinations: 128-byte aligned, each box at a multiple of 128 bytes, so a
  // 16-token page box takes 32 words), and the per-warp sums of p * shift of
  // the value rows ([warp][16])
  static constexpr int kSSWords = 2 * kTile;
  static constexpr int oSS = (oMergeBar + 6 * 8 + 127) & ~127;
  static constexpr int kSSBytes = TOK ? kStages * 2 * kSSWords * 4 : 0;
  static constexpr int oStatZ = oSS + kSSBytes;                // [2 copies][warp][16]
  static constexpr int kTotal = oStatZ + (TOK ? 2 * kConsumerWarps * 16 * 4 : 0) + 1024;  // + slack
  static_assert(oSS % 128 == 0 && (2 * kSSWords * 4) % 128 == 0, "TMA destinations need 128 B");
  static_assert(oQ % 128 == 0 && kQSlot % 128 == 0 && kTileBytes % 128 == 0, "TMA destinations");
  static_assert(!I4 || (FP8 && !TOK), "int4 rows take the f16 operand path and their own scales");
};

// What the producer tells the consumers about the tile in a stage.
struct __align__(8) StageMeta {
  uint64_t valid;   // bit t: token t of the tile is a valid position
  int32_t unit;     // b * HKV + h
  int32_t flags;    // kFirst: first tile of a segment (query group in the stage); kLast
  int32_t c_first;  // first CTA holding a segment of this unit
  int32_t n_seg;    // segments of this unit
  int32_t nval;     // the row's length minus the tile's first position
  int32_t pos0;     // the tile's first position in the row (a kept block's for sparse)
};
static_assert(sizeof(StageMeta) == 32, "the shared-memory layout keeps 32 bytes per stage");

// Word of token t of a tile in a stage's scale words: boxes of `box_rows` tokens
// start every max(box_rows, 32) words (128-byte aligned TMA destinations).
__device__ __forceinline__ int ss_word(int t, int box_rows) {
  return box_rows >= 32 ? t : t + (t / box_rows) * (32 - box_rows);
}
// kFull: a tile of the full-block table (flex's FULL_KV_IDX: no mask_mod there)
constexpr int32_t kFirst = 1, kLast = 2, kFull = 4;

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Soft cap of a score x in log2 units: c2 * tanh(x / c2), from the identity
// tanh(u) = 1 - 2 / (exp(2u) + 1) with exp(2u) = exp2(x * k), k = 2 log2(e) / c2.
// Both ends saturate: exp2 -> inf gives c2, exp2 -> 0 gives -c2. The error is
// absolute, a few ulp of c2, which is what the softmax weight exp2(x - m) sees.
__device__ __forceinline__ float cap_tanh(float x, float c2, float k) {
  return c2 - __fdividef(2.f * c2, ex2(x * k) + 1.f);
}

__device__ __forceinline__ uint64_t low_bits(int n) {
  return n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1ull));
}

// Warp-uniform outcome of a bounded wait (every lane then takes the same path).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, limit_ns));
}

// Barrier of the consumer warps on an mbarrier of kConsumerWarps * 32 arrivals:
// each consumer thread arrives and waits, bounded, for the phase (release /
// acquire at CTA scope, like bar.sync for shared memory). A warp whose wait
// runs out returns false instead of waiting forever for a warp that left the
// stream after a failed wait of its own.
__device__ __forceinline__ bool consumer_sync(uint64_t *bar, uint32_t &phase) {
  mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase, kWaitLimitNs);
  phase ^= 1u;
  return ok;
}

// ------------------------------------------------------------------ units and the schedule

struct UnitInfo {
  int b, h, n_valid, tiles;
  int nbp;   // sparse: blocks of the first table (the full table's follow them)
  int trow;  // sparse: the block tables' row, (b % SZ) * SH + h % SH
};

// Length (checked against the cache) and tile count of unit u.
__device__ __forceinline__ UnitInfo unit_info(const GqaParams &p, int u, uint32_t &err) {
  UnitInfo x;
  x.b = u / p.num_kv_heads;
  x.h = u - x.b * p.num_kv_heads;
  int n = p.seq_lens[x.b];
  if (n < 0 || n > p.capacity) {
    err |= DA_DEVERR_SEQ_LEN;
    n = n < 0 ? 0 : p.capacity;
  }
  x.n_valid = n;
  x.trow = 0;
  if (p.sparse_block_size > 0) {
    // block masks broadcast over rows and heads (flex's SPARSE_Z / SPARSE_HQ)
    x.trow = (x.b % p.sparse_batch) * p.sparse_heads + x.h % p.sparse_heads;
    int nb = p.kv_num_blks[x.trow];
    if (nb < 0 || nb > p.max_sparse_blocks) {
      err |= DA_DEVERR_SPARSE_INDEX;
      nb = nb < 0 ? 0 : p.max_sparse_blocks;
    }
    int nf = p.kv_full_num_blks ? p.kv_full_num_blks[x.trow] : 0;  // the flex FULL_KV table
    if (nf < 0 || nf > p.max_sparse_blocks) {
      err |= DA_DEVERR_SPARSE_INDEX;
      nf = nf < 0 ? 0 : p.max_sparse_blocks;
    }
    x.nbp = nb;
    x.tiles = (nb + nf) * (p.sparse_block_size / kTile);
  } else {
    x.nbp = 0;
    x.tiles = (n + kTile - 1) / kTile;
  }
  return x;
}

// CTA whose tile range [floor(c*T/C), floor((c+1)*T/C)) contains global tile t
// (a 32-bit division whenever the operands fit, as they do below 2^32 / C tiles).
__device__ __forceinline__ int cta_of(int64_t t, int64_t T, int C) {
  const uint64_t num = (uint64_t)(t + 1) * (uint64_t)C - 1u;
  if ((num >> 32) == 0 && ((uint64_t)T >> 32) == 0) return (int)((uint32_t)num / (uint32_t)T);
  return (int)(num / (uint64_t)T);
}

// This CTA's share (1 / gridDim.x) of a table of `bytes` bytes prefetched into L2:
// the whole 16-byte chunks inside [base, base + bytes), cut into equal pieces.
__device__ __forceinline__ void prefetch_share_l2(const void *base, int64_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(base);
  const uint64_t lo = (a + 15) & ~uint64_t(15), hi = (a + (uint64_t)bytes) & ~uint64_t(15);
  if (base == nullptr || bytes <= 0 || hi <= lo) return;
  const uint64_t n16 = (hi - lo) / 16, per = (n16 + gridDim.x - 1) / gridDim.x;
  const uint64_t s = (uint64_t)blockIdx.x * per, e = s + per < n16 ? s + per : n16;
  if (e > s) prefetch_l2(reinterpret_cast<const void *>(lo + s * 16), (uint32_t)((e - s) * 16));
}

// Inclusive scan over the block's threads; returns the block total in *total.
__device__ __forceinline__ int block_inclusive_scan(int v, int *scratch, int *total) {
  const int nwarps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int before = 0, sum = 0;
  for (int w = 0; w < nwarps; ++w) {
    const int t = scratch[w];
    if (w < warp) before += t;
    sum += t;
  }
  __syncthreads();
  *total = sum;
  return v + before;
}

struct TileDesc {
  int unit, b, h, n_valid, j, tiles, nbp;  // unit, its row / head, length, tile index, tile count
  int trow;                                // sparse: the block tables' row
  int64_t P;                          // global index of the unit's first tile
  int c_first, n_seg;                 // CTAs holding the unit's segments
  int wi;                             // position in this CTA's processing order
};

// ------------------------------------------------------------------ consumer helpers

// Byte offset of token t inside a K or V tile of shared memory. A tile is
// filled by boxes of `br` tokens (one page, or the whole 64-token tile). fp8:
// one 128-byte row per token. bf16: each box holds its rows' two 64-element
// halves in two regions of `br` 128-byte rows ([box][half][row]), so eight
// consecutive tokens of one 16-byte chunk fall on eight different swizzle
// phases (no bank conflicts); the half stride is br * 128 bytes.
template <bool FP8>
__device__ __forceinline__ uint32_t token_offset(int t, int br_shift) {
  if (FP8) return (uint32_t)t * 128;
  const int br = 1 << br_shift;
  return (uint32_t)((t >> br_shift) * (2 * br * 128) + (t & (br - 1)) * 128);
}

// Address of 16-byte chunk c (bf16: 0..15, fp8: 0..7) of the token at
// `tok_off` (token t) in the 128B-swizzled tile at `base`.
template <bool FP8>
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, uint32_t tok_off, int t, int c,
                                               int br_shift) {
  if (FP8) return base + tok_off + (((c ^ t) & 7) << 4);
  return base + tok_off + (uint32_t)(c >> 3) * (128u << br_shift) + ((((c & 7) ^ t) & 7) << 4);
}

__device__ __forceinline__ uint32_t lo16_mask(bool a, bool b) {
  return (a ? 0x0000FFFFu : 0u) | (b ? 0xFFFF0000u : 0u);
}

// int4 tiles: the cache rows as they are, `row_bytes` = (groups + 16) * 4
// apart (80 or 96 bytes: 16-byte aligned); 16-byte data chunk c of row t
// follows its groups coefficient words. With 80-byte rows the eight rows an
// ldmatrix reads fall in eight different bank groups.
__device__ __forceinline__ uint32_t i4_addr(uint32_t base, int t, int c, int row_bytes, int ng) {
  return base + (uint32_t)(t * row_bytes + ng * 4 + c * 16);
}

// The two 4-bit codes in bits 4j.. of each 16-bit half of x, as an f16 pair
// 1024 + code (an f16 whose unit in the last place is 1).
__device__ __forceinline__ uint32_t i4_codes(uint32_t x, int j) {
  return ((x >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
}

// code * scale + shift on f16 pairs: the 1024 is subtracted exactly first.
__device__ __forceinline__ uint32_t i4_dequant(uint32_t codes, uint32_t scale2, uint32_t shift2) {
  const uint32_t bias = 0x64006400u;
  const __half2 n = __hsub2(*reinterpret_cast<const __half2 *>(&codes),
                            *reinterpret_cast<const __half2 *>(&bias));
  const __half2 r = __hfma2(n, *reinterpret_cast<const __half2 *>(&scale2),
                            *reinterpret_cast<const __half2 *>(&shift2));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// A bf16 pair times the power of two `s` (exact), rounded to an f16 pair.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, float s) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&x);
  float2 f = __bfloat1622float2(v);
  return pack_f16(f.x * s, f.y * s);
}

// 2^e as a float, for -126 <= e <= 127.
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// max|q| over this lane's quarter of a query row (the four lanes of a quad
// share the row; each reads 16 of its 64 words, rotated by the row so that the
// eight rows' reads fall in different banks).
__device__ __forceinline__ float q_row_amax(const uint32_t *qrow, int q4, int r8) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t w = qrow[q4 * 16 + ((j + r8) & 15)];
    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xFFFF0000u))));
  }
  return amax;
}

// Exponent e of the power of two that puts `amax` in [2^14, 2^15) (0 for zero),
// at most 100 (an all-but-zero query stays far below f16's largest value).
__device__ __forceinline__ int q_exponent(float amax) {
  const int lg = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;  // floor(log2), normal amax
  return amax > 0.f ? min(14 - lg, 100) : 0;
}

// Merge of one unit's segments (slots unit + c_first .. unit + c_first + n_seg
// - 1) into the final output, run by the CTA that finished the unit's last
// segment once its own range is done (so its K/V ring is free). The partial O
// blocks are staged into the two halves of the ring by bulk copies, each half
// refilled while the other is summed, and the first copies start before the
// LSEs are read; the weighted sum goes into shared-memory accumulators. The
// loops are kept compact on purpose: this code runs once per unit, so its
// instructions are usually not cached when it starts. Returns false if a
// staging wait gave up.
__device__ __noinline__ bool merge_unit(const GqaParams &p, int unit, int c_first, int n_seg,
                                        int G, uint8_t *stage, int stage_bytes, float *buf,
                                        int cap, float *acc, uint64_t *bars, uint32_t *phase) {
  const int b = unit / p.num_kv_heads, h = unit - b * p.num_kv_heads;
  const int tid = threadIdx.x;  // 0..127 (consumer threads)
  const int nthr = kConsumerWarps * 32;
  const int blk = G * kD * 4;                // bytes of one segment's partial O
  float *stat = buf;                         // [16] max, [16] sum of weights
  float *w = buf + 32;                       // LSE, then weights, [s][g]
  const int wcap = cap - 32;
  const int half = stage_bytes / 2;
  const int seg_chunk = max(1, half / blk);  // segments per staging half
  const int nchunks = (n_seg + seg_chunk - 1) / seg_chunk;
  const bool all_lse = n_seg * G <= wcap;    // every LSE fits at once (the usual case)
  const float *lse_base = p.lse_part + ((int64_t)unit + c_first) * G;
  const float *o_base = p.o_part + ((int64_t)unit + c_first) * G * kD;

  auto issue = [&](int k) {  // chunk k -> half k & 1, completion on bars[k & 1]
    // the unit's slots are consecutive: one copy per chunk
    const int s0 = k * seg_chunk, ns = min(seg_chunk, n_seg - s0);
    mbar_arrive_expect_tx(&bars[k & 1], (uint32_t)(ns * blk));
    bulk_copy_g2s(stage + (k & 1) * half, o_base + (int64_t)s0 * G * kD, (uint32_t)(ns * blk),
                  &bars[k & 1]);
  };
  if (tid == 0) {
    fence_proxy_async_shared();  // earlier reads of the ring before the copies
    fence_proxy_async_global();  // the partials other CTAs wrote, for the copies
    issue(0);
  }
  for (int e = tid; e < G * kD; e += nthr) acc[e] = 0.f;
  // ---- LSEs: maximum, weights and their sum per head
  if (tid < 16) {
    stat[tid] = neg_inf();
    stat[16 + tid] = 0.f;
  }
  named_barrier_sync(kConsumerBar, nthr);
  const int lchunk = all_lse ? n_seg : max(1, wcap / G);
#pragma unroll 1
  for (int pass = 0; pass < (all_lse ? 1 : 2); ++pass) {
#pragma unroll 1
    for (int s0 = 0; s0 < n_seg; s0 += lchunk) {
      const int ns = min(lchunk, n_seg - s0);
#pragma unroll 1
      for (int i = tid; i < ns * G; i += nthr) w[i] = __ldcg(lse_base + (int64_t)s0 * G + i);
      named_barrier_sync(kConsumerBar, nthr);
      if (tid < 32) {  // warp 0: lane = (segment group, head); groups of 32/Gp lanes per head
        const int Gp = G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : (G <= 8 ? 8 : 16)));
        const int g = tid & (Gp - 1), lanes = 32 / Gp;
        float M = neg_inf();
        if (g < G)
#pragma unroll 1
          for (int s = tid / Gp; s < ns; s += lanes) M = fmaxf(M, w[s * G + g]);
        for (int o = Gp; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if (tid < G) stat[tid] = fmaxf(stat[tid], M);
      }
      named_barrier_sync(kConsumerBar, nthr);
    }
  }
  if (all_lse) {  // turn the LSEs (still in w) into weights
#pragma unroll 1
    for (int i = tid; i < n_seg * G; i += nthr) {
      const float l = w[i], Mg = stat[i % G];
      w[i] = l == neg_inf() ? 0.f : ex2((l - Mg) * 1.4426950408889634f);
    }
    named_barrier_sync(kConsumerBar, nthr);
    if (tid < 32) {
      const int Gp = G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : (G <= 8 ? 8 : 16)));
      const int g = tid & (Gp - 1), lanes = 32 / Gp;
      float sum = 0.f;
      if (g < G)
#pragma unroll 1
        for (int s = tid / Gp; s < n_seg; s += lanes) sum += w[s * G + g];
      for (int o = Gp; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (tid < G) stat[16 + tid] = sum;
    }
  }
  // ---- weighted sum of the staged partial O blocks, two halves in flight
  bool ok = true;
#pragma unroll 1
  for (int k = 0; k < nchunks; ++k) {
    const int s0 = k * seg_chunk, ns = min(seg_chunk, n_seg - s0);
    if (tid == 0 && k + 1 < nchunks) issue(k + 1);  // its half was freed by chunk k - 1
    float *wk = w + (all_lse ? s0 * G : 0);
    if (!all_lse) {  // weights of this chunk only (the rare long case)
#pragma unroll 1
      for (int i = tid; i < ns * G; i += nthr) {
        const float l = __ldcg(lse_base + (int64_t)s0 * G + i), Mg = stat[i % G];
        w[i] = l == neg_inf() ? 0.f : ex2((l - Mg) * 1.4426950408889634f);
      }
      named_barrier_sync(kConsumerBar, nthr);
      if (tid < G) {
        float sum = stat[16 + tid];
#pragma unroll 1
        for (int s = 0; s < ns; ++s) sum += w[s * G + tid];
        stat[16 + tid] = sum;
      }
    }
    if (!mbar_wait_bounded(&bars[k & 1], phase[k & 1], kWaitLimitNs)) ok = false;
    phase[k & 1] ^= 1u;
    const float *sf = reinterpret_cast<const float *>(stage + (k & 1) * half);
    // four independent accumulation chains per thread (G * kD is a multiple of 4 * nthr)
#pragma unroll 1
    for (int e0 = tid; e0 < G * kD; e0 += 4 * nthr) {
      float a[4];
      int gi[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = e0 + q * nthr;
        gi[q] = e < G * kD ? e / kD : 0;
        a[q] = e < G * kD ? acc[e] : 0.f;
      }
#pragma unroll 2
      for (int s = 0; s < ns; ++s) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = e0 + q * nthr;
          if (e < G * kD) a[q] += wk[s * G + gi[q]] * sf[(size_t)s * G * kD + e];
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = e0 + q * nthr;
        if (e < G * kD) acc[e] = a[q];
      }
    }
    named_barrier_sync(kConsumerBar, nthr);
  }
  // ---- output rows b, h*G .. h*G+G-1 are contiguous
  __nv_bfloat16 *out = p.out + ((int64_t)b * p.num_q_heads + h * G) * kD;
#pragma unroll 1
  for (int e = tid; e < G * kD; e += nthr) {
    const float sum = stat[16 + e / kD];
    out[e] = __float2bfloat16(sum == 0.f ? 0.f : acc[e] / sum);
  }
  if (tid < G && p.lse) {
    const float sum = stat[16 + tid];
    p.lse[(int64_t)b * p.num_q_heads + h * G + tid] =
        sum == 0.f ? neg_inf() : stat[tid] + __log2f(sum) * 0.69314718055994531f;
  }
  if (tid == 0) p.counters[unit] = 0u;  // ready for the next call
  named_barrier_sync(kConsumerBar, nthr);
  return ok;
}

// ------------------------------------------------------------------ kernel

// Units held by more than kOneLevelSegs pieces are merged in two levels, so
// that no merge reads more than about sqrt(n_seg) pieces: consecutive groups of
// K = ceil(sqrt(n_seg)) pieces, each merged (in place, into the slot of its
// first piece) by the piece that completes the group's counter, then the
// group results merged by the group that completes the unit's counter. No
// CTA ever waits for another.
constexpr int kOneLevelSegs = 8;
constexpr int kWarpMergeSegs = 4;  // a unit of at most this many pieces: merged by one warp
__host__ __device__ inline int merge_group_size(int n_seg) { return ceil_sqrt(n_seg); }

// All threads of the CTA merge n pieces of `unit`, slots slot0 + s * stride
// (after the stream, shared memory free): the LSEs in one load round, per head
// the maximum, weights exp(lse_s - max) and their sum in one warp, then the
// weighted sum of the pieces' normalised O in work items of (output float4, 16
// pieces), each with its 16 loads in flight, added into shared memory. The
// result goes to the final output or, as a normalised piece, to slot `dst`.
// Needs merge_cta_floats(n, G) floats of scratch.
__host__ __device__ constexpr int merge_cta_floats(int n, int G) {
  return ((n * G + 2 * G + 3) & ~3) + G * kD;
}
__device__ __noinline__ void merge_slots_cta(const GqaParams &p, int unit, int G, int64_t slot0,
                                             int stride, int n_seg, bool final_out, int64_t dst,
                                             float *scratch) {
  const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = nthr >> 5;
  const int b = unit / p.num_kv_heads, h = unit - b * p.num_kv_heads;
  const int nout = G * (kD / 4);                    // float4 outputs of the unit
  float *w = scratch;                               // [n_seg][G]: LSE, then weights
  float *mx = w + n_seg * G, *sum = mx + G;         // [G] each
  float4 *acc = reinterpret_cast<float4 *>(scratch + ((n_seg * G + 2 * G + 3) & ~3));  // [nout]
  for (int i = tid; i < n_seg * G; i += nthr)
    w[i] = __ldcg(p.lse_part + (slot0 + (int64_t)(i / G) * stride) * G + i % G);
  for (int i = tid; i < nout; i += nthr) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  for (int g = warp; g < G; g += nwarps) {
    float M = neg_inf();
    for (int s = lane; s < n_seg; s += 32) M = fmaxf(M, w[s * G + g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float ssum = 0.f;
    for (int s = lane; s < n_seg; s += 32) {
      const float l = w[s * G + g];
      const float e = l == neg_inf() ? 0.f : ex2((l - M) * 1.4426950408889634f);
      w[s * G + g] = e;
      ssum += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (lane == 0) {
      mx[g] = M;
      sum[g] = ssum;
    }
  }
  __syncthreads();
  constexpr int kChunk = 16;
  const int nch = (n_seg + kChunk - 1) / kChunk;
  const float4 *src = reinterpret_cast<const float4 *>(p.o_part + slot0 * G * kD);
  for (int item = tid; item < nout * nch; item += nthr) {
    const int o = item % nout, s0 = (item / nout) * kChunk, g = o / (kD / 4);
    float4 v[kChunk];
#pragma unroll
    for (int k = 0; k < kChunk; ++k)
      v[k] = s0 + k < n_seg ? __ldcg(src + (int64_t)(s0 + k) * stride * nout + o)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      const float e = s0 + k < n_seg ? w[(s0 + k) * G + g] : 0.f;
      if (e != 0.f) {  // a piece of weight 0 may hold anything
        a.x += e * v[k].x;
        a.y += e * v[k].y;
        a.z += e * v[k].z;
        a.w += e * v[k].w;
      }
    }
    if (nch == 1) {
      acc[o] = a;
    } else {
      atomicAdd(&acc[o].x, a.x);
      atomicAdd(&acc[o].y, a.y);
      atomicAdd(&acc[o].z, a.z);
      atomicAdd(&acc[o].w, a.w);
    }
  }
  __syncthreads();  // every piece has been read: `dst` may be one of them
  if (final_out) {
    __nv_bfloat16 *out = p.out + ((int64_t)b * p.num_q_heads + h * G) * kD;
    for (int o = tid; o < nout; o += nthr) {
      const int g = o / (kD / 4);
      const float inv = sum[g] == 0.f ? 0.f : 1.f / sum[g];
      const float4 a = acc[o];
      *reinterpret_cast<uint2 *>(out + 4 * o) =
          make_uint2(pack_bf16(a.x * inv, a.y * inv), pack_bf16(a.z * inv, a.w * inv));
    }
  } else {
    float4 *out = reinterpret_cast<float4 *>(p.o_part + dst * G * kD);
    for (int o = tid; o < nout; o += nthr) {
      const int g = o / (kD / 4);
      const float inv = sum[g] == 0.f ? 0.f : 1.f / sum[g];
      const float4 a = acc[o];
      out[o] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    }
  }
  if (tid < G) {
    const float lse = sum[tid] == 0.f ? neg_inf() : mx[tid] + __log2f(sum[tid]) * 0.69314718055994531f;
    if (!final_out) p.lse_part[dst * G + tid] = lse;
    else if (p.lse) p.lse[(int64_t)b * p.num_q_heads + h * G + tid] = lse;
  }
  __syncthreads();
}

// The same for n <= kSmallMerge pieces in one round of loads: each thread
// issues, for its (at most two) output float4s, the loads of every piece's O
// and of the pieces' LSEs of its head together, then weights, sums and
// writes. One barrier keeps an in-place result's LSE write behind every
// thread's reads. Needs G floats of scratch.
constexpr int kSmallMerge = 8;
__device__ __noinline__ void merge_slots_small(const GqaParams &p, int unit, int G, int64_t slot0,
                                               int stride, int n, bool final_out, int64_t dst,
                                               float *scratch) {
  const int nthr = blockDim.x, tid = threadIdx.x;
  const int b = unit / p.num_kv_heads, h = unit - b * p.num_kv_heads;
  const int nout = G * (kD / 4);
  const float4 *src = reinterpret_cast<const float4 *>(p.o_part + slot0 * G * kD);
  float4 v[2][kSmallMerge];
  float l[2][kSmallMerge];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int o = tid + u * nthr, g = o / (kD / 4);
#pragma unroll
    for (int k = 0; k < kSmallMerge; ++k) {
      const bool on = o < nout && k < n;
      v[u][k] = on ? __ldcg(src + (int64_t)k * stride * nout + o) : make_float4(0.f, 0.f, 0.f, 0.f);
      l[u][k] = on ? __ldcg(p.lse_part + (slot0 + (int64_t)k * stride) * G + g) : neg_inf();
    }
  }
  float lse_out[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int o = tid + u * nthr;
    float M = neg_inf();
#pragma unroll
    for (int k = 0; k < kSmallMerge; ++k) M = fmaxf(M, l[u][k]);
    float sum = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kSmallMerge; ++k) {
      const float e = l[u][k] == neg_inf() ? 0.f : ex2((l[u][k] - M) * 1.4426950408889634f);
      if (e != 0.f) {  // a piece of weight 0 may hold anything
        sum += e;
        a.x += e * v[u][k].x;
        a.y += e * v[u][k].y;
        a.z += e * v[u][k].z;
        a.w += e * v[u][k].w;
      }
    }
    lse_out[u] = sum == 0.f ? neg_inf() : M + __log2f(sum) * 0.69314718055994531f;
    if (o < nout) {
      const float inv = sum == 0.f ? 0.f : 1.f / sum;
      if (final_out) {
        __nv_bfloat16 *out = p.out + ((int64_t)b * p.num_q_heads + h * G) * kD;
        *reinterpret_cast<uint2 *>(out + 4 * o) =
            make_uint2(pack_bf16(a.x * inv, a.y * inv), pack_bf16(a.z * inv, a.w * inv));
      } else {
        reinterpret_cast<float4 *>(p.o_part + dst * G * kD)[o] =
            make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
      }
    }
  }
  // the head's LSE (every thread of a head computed the same value)
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int o = tid + u * nthr;
    if (o < nout && o % (kD / 4) == 0) scratch[o / (kD / 4)] = lse_out[u];
  }
  __syncthreads();  // every thread has read the pieces' LSEs
  if (tid < G) {
    if (!final_out) p.lse_part[dst * G + tid] = scratch[tid];
    else if (p.lse) p.lse[(int64_t)b * p.num_q_heads + h * G + tid] = scratch[tid];
  }
  __syncthreads();
}

// One warp merges a unit held by at most kWarpMergeSegs pieces whose LSEs fit
// in its lanes (pieces x rows <= 32): lane l owns head dims 4l..4l+3 of each
// row in turn; per row the pieces' LSE give weights
// exp(lse_s - max) and the output is the weighted mean of their normalised O.
__device__ __noinline__ void merge_unit_warp(const GqaParams &p, int unit, int c_first, int n_seg,
                                             int G) {
  const int lane = threadIdx.x & 31;
  const int b = unit / p.num_kv_heads, h = unit - b * p.num_kv_heads;
  const int64_t slot0 = (int64_t)unit + c_first;
  const float my_lse = lane < n_seg * G ? __ldcg(p.lse_part + slot0 * G + lane) : neg_inf();
  const float4 *o_base = reinterpret_cast<const float4 *>(p.o_part + slot0 * G * kD);
  __nv_bfloat16 *out = p.out + ((int64_t)b * p.num_q_heads + h * G) * kD;
  // rows in rounds of four, every load of a round issued before any use
  constexpr int kRows = 4;
#pragma unroll 1
  for (int g0 = 0; g0 < G; g0 += kRows) {
    float4 v[kRows][kWarpMergeSegs];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int s = 0; s < kWarpMergeSegs; ++s)
        v[r][s] = (g0 + r < G && s < n_seg)
                      ? __ldcg(o_base + ((int64_t)s * G + g0 + r) * (kD / 4) + lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int g = g0 + r;
      float l[kWarpMergeSegs], M = neg_inf();
#pragma unroll
      for (int s = 0; s < kWarpMergeSegs; ++s) {
        l[s] = __shfl_sync(0xffffffffu, my_lse, min(s * G + g, 31));
        if (s < n_seg) M = fmaxf(M, l[s]);
      }
      if (g >= G) continue;
      float sum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < kWarpMergeSegs; ++s) {
        const float w = (s < n_seg && l[s] != neg_inf())
                            ? ex2((l[s] - M) * 1.4426950408889634f)
                            : 0.f;
        if (w != 0.f) {  // a piece of weight 0 may hold anything
          sum += w;
          acc.x += w * v[r][s].x;
          acc.y += w * v[r][s].y;
          acc.z += w * v[r][s].z;
          acc.w += w * v[r][s].w;
        }
      }
      const float inv = sum == 0.f ? 0.f : 1.f / sum;
      *reinterpret_cast<uint2 *>(out + (int64_t)g * kD + 4 * lane) =
          make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
      if (lane == 0 && p.lse)
        p.lse[(int64_t)b * p.num_q_heads + h * G + g] =
            sum == 0.f ? neg_inf() : M + __log2f(sum) * 0.69314718055994531f;
    }
  }
  if (lane == 0) p.counters[unit] = 0u;  // ready for the next call
}

// Counts one finished partial segment of `unit` (release: its writes are
// visible before the count); the segment that completes the count records the
// unit's merge for this CTA (at most two: a range holds at most two partial
// segments, its first and its last).
__device__ __forceinline__ bool count_segment(const GqaParams &p, int unit, int n_seg) {
  return atomic_add_acq_rel_gpu(p.counters + unit, 1u) == (unsigned)(n_seg - 1);
}
// Merges this CTA owes after its stream (at most two: a range holds at most two
// partial segments): (unit, c_first, n_seg, group), group -1 for a one-level merge.
__device__ __forceinline__ void record_merge(volatile int *flags, int unit, int c_first, int n_seg,
                                             int group) {
  if (flags[12] < 2) {
    const int k = flags[12];
    flags[24 + 4 * k] = unit;
    flags[25 + 4 * k] = c_first;
    flags[26 + 4 * k] = n_seg;
    flags[27 + 4 * k] = group;
    flags[12] = k + 1;
  }
}
// Counts this CTA's finished piece of a unit of n_seg > 1 pieces. Returns true
// when it completes a unit of at most kWarpMergeSegs pieces that the caller
// merges right away (warp_merge); otherwise records the merge this CTA owes.
__device__ __forceinline__ bool count_piece(const GqaParams &p, volatile int *flags, int unit,
                                            int c_first, int n_seg, bool warp_merge) {
  if (n_seg <= kOneLevelSegs) {
    if (!count_segment(p, unit, n_seg)) return false;
    if (warp_merge && n_seg <= kWarpMergeSegs && n_seg * p.group <= 32) return true;
    record_merge(flags, unit, c_first, n_seg, -1);
    return false;
  }
  const int K = merge_group_size(n_seg), q = ((int)blockIdx.x - c_first) / K;
  const int gs = min(K, n_seg - q * K);
  uint32_t *gc = p.counters + p.batch * p.num_kv_heads +
                 (int64_t)unit * max_merge_groups(gridDim.x) + q;
  if (atomic_add_acq_rel_gpu(gc, 1u) == (unsigned)(gs - 1)) record_merge(flags, unit, c_first, n_seg, q);
  return false;
}

// TOK: e4m3 K/V with per-token scale and shift words (FP8 only).
// MOD: 0 -- the plain decode, whose softmax keeps only the length mask; 1 --
// score modifications are possible (several query tokens with their mask
// words, a soft cap); 2 -- the flex-style mods too (the sink/window mask_mod and
// the ALiBi score_mod, per query head), in an instantiation of their own so
// that the other two keep their registers.
template <bool FP8, int NT, bool TOK, bool I4, int MOD, bool Q8>
__global__ void __launch_bounds__(threads_for<NT>(), 2)
    gqa_split_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kssmap,
                     const __grid_constant__ CUtensorMap vssmap, const GqaParams p) {
  using C = Cfg<FP8, NT, TOK, I4>;
  static_assert(!TOK || FP8, "per-token scales are an e4m3 format");
  static_assert(!Q8 || (FP8 && !TOK && !I4), "e4m3 tensor-core arithmetic: per-head e4m3 K/V");
  constexpr int kThreads = threads_for<NT>();
  constexpr bool kHelper = has_helper<NT>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem + C::oRing;
  uint8_t *qslots = smem + C::oQ;
  float *red = reinterpret_cast<float *>(smem + C::oRed);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::oFull);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + C::oEmpty);
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + C::oMeta);
  float *stats = reinterpret_cast<float *>(smem + C::oStats);  // [2 copies][m | l][warp][16]
  int *scan = reinterpret_cast<int *>(smem + C::oScan);
  int *idq = reinterpret_cast<int *>(smem + C::oIds);
  volatile int *flags = reinterpret_cast<volatile int *>(smem + C::oFlags);
  // flags: [0] abort, [1] tiles the producer issued, [2] start unit, [3] start
  //        tile, [4..5] start P (int64), [6..9] the start unit's n_valid, tiles,
  //        nbp, trow (UnitInfo, so the producer starts without a table load),
  //        [12] merges owed after the stream, [13] scratch, [24..31] those merges
  //        (unit, c_first, n_seg, group),
  //        [14..19] the range's partial segments (unit, c_first, n_seg) handed to
  //        the helper warp, [20] unit holding the range's last tile, [21] whether
  //        its segment here is partial, [22..23] its first tile (int64), [32..35]
  //        its UnitInfo as [6..9]
  uint64_t *merge_bar = reinterpret_cast<uint64_t *>(smem + C::oMergeBar);
  uint64_t *part_bar = merge_bar + 2;  // [2] a partial segment is in global memory
  uint64_t *epi_bar = merge_bar + 4;   // the consumer warps' segment-epilogue barrier
  uint64_t *stall_bar = merge_bar + 5; // nothing arrives on it (the test stall of GqaParams)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int U = p.batch * p.num_kv_heads;
  const int cta = blockIdx.x;
  uint32_t dev_err = 0;

  // The producer's first page / block id loads depend on the schedule below (a
  // scan of every unit's length), so the id tables are fetched into L2 now, by
  // all CTAs together, and the first ids then come from L2 instead of DRAM.
  if (threadIdx.x == kConsumerWarps * 32) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
    if (p.paged) prefetch_share_l2(p.block_table, (int64_t)p.batch * p.max_pages * 4);
    if (p.sparse_block_size > 0) {
      const int64_t tb = (int64_t)p.sparse_batch * p.sparse_heads * p.max_sparse_blocks * 4;
      prefetch_share_l2(p.kv_idx, tb);
      prefetch_share_l2(p.kv_full_idx, tb);
    }
  }

  // ---- the schedule: this CTA's range of the global tile sequence. Thread t
  // takes the consecutive units [t*per, t*per + per): one scan gives each
  // thread the first tile of its block, and a second walk over its own units
  // (their lengths now in L1) finds the range's first and last unit.
  if (threadIdx.x == 0) {
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = -1;
    flags[12] = 0;
  }
  const int per = (U + kThreads - 1) / kThreads;
  const int u_beg = min(U, (int)threadIdx.x * per), u_end = min(U, u_beg + per);
  int local = 0;
  for (int u = u_beg; u < u_end; ++u) local += unit_info(p, u, dev_err).tiles;
  int T32 = 0;
  const int incl = block_inclusive_scan(local, scan, &T32);
  const int64_t T = T32;
  // Never more ranges than tiles, so every working CTA holds at least one tile
  // and a unit's segments come from consecutive CTAs c_first..c_last.
  const int CTAS = (int)(T < (int64_t)gridDim.x ? T : (int64_t)gridDim.x);
  const int64_t lo = cta < CTAS ? (int64_t)cta * T / CTAS : 0;
  const int64_t hi = cta < CTAS ? (int64_t)(cta + 1) * T / CTAS : 0;
  const int owner_of_tail = CTAS > 0 ? CTAS - 1 : 0;  // writes empty units past the last tile
  {
    int64_t Pu = incl - local;
    uint32_t ignored = 0;
    for (int u = u_beg; u < u_end; ++u) {
      const UnitInfo x = unit_info(p, u, ignored);
      const int t_u = x.tiles;
      if (t_u > 0 && Pu <= lo && lo < Pu + t_u) {
        flags[2] = u;
        flags[3] = (int)(lo - Pu);
        *reinterpret_cast<volatile int64_t *>(flags + 4) = Pu;
        flags[6] = x.n_valid;
        flags[7] = x.tiles;
        flags[8] = x.nbp;
        flags[9] = x.trow;
      }
      if (t_u > 0 && Pu < hi && hi <= Pu + t_u) {
        // the unit holding the last tile: its segment here is partial when
        // the unit goes on past this range or started before it
        flags[20] = u;
        flags[21] = (Pu + t_u > hi || Pu < lo) ? 1 : 0;
        *reinterpret_cast<volatile int64_t *>(flags + 22) = Pu;
        flags[32] = x.n_valid;
        flags[33] = x.tiles;
        flags[34] = x.nbp;
        flags[35] = x.trow;
      }
      // a unit without tiles is written here by the CTA whose range holds its start
      if (t_u == 0 && ((Pu >= lo && Pu < hi) || (Pu >= T && cta == owner_of_tail))) {
        const int64_t row0 = (int64_t)x.b * p.num_q_heads + x.h * G;
        for (int e = 0; e < G * kD; ++e) p.out[row0 * kD + e] = __float2bfloat16(0.f);
        if (p.lse)
          for (int g = 0; g < G; ++g) p.lse[row0 + g] = neg_inf();
      }
      Pu += t_u;
    }
  }
  const int ntiles = (int)(hi - lo);
  if (ntiles <= 0) {
    if (dev_err) atomicOr(p.err, dev_err);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&merge_bar[0], 1);
    mbar_init(&merge_bar[1], 1);
    mbar_init(&part_bar[0], kConsumerWarps * 32);
    mbar_init(&part_bar[1], kConsumerWarps * 32);
    mbar_init(epi_bar, kConsumerWarps * 32);
    mbar_init(stall_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int start_u = flags[2], start_j = flags[3];
  const int64_t start_P = *reinterpret_cast<volatile int64_t *>(flags + 4);

  if (warp == kConsumerWarps) {
    // ======================================================= producer
    const uint64_t policy = l2_policy_evict_first();
    const uint64_t q_policy = l2_policy_evict_last();
    const int P = p.page_size;
    const int pages_per_tile = p.paged ? (P >= kTile ? 1 : kTile / P) : 1;
    const bool multi_box = (!FP8 || I4) && pages_per_tile > 1;  // several page boxes per tile

    // Walker over (unit, tile) in processing order. When the range ends in the
    // head of a unit that goes on into the next CTA, that segment is streamed
    // first and the walk then jumps back to lo: both pieces of such a unit are
    // then finished early in their CTAs, so its merge (by the helper warp)
    // overlaps streaming instead of trailing the range.
    // (u, j, P0) with the unit's UnitInfo as the schedule staged it in flags[f..f+3]
    auto set_at = [&](TileDesc &d, int u, int j, int64_t P0, int f) {
      UnitInfo x;
      x.b = u / p.num_kv_heads;
      x.h = u - x.b * p.num_kv_heads;
      x.n_valid = flags[f];
      x.tiles = flags[f + 1];
      x.nbp = flags[f + 2];
      x.trow = flags[f + 3];
      d.unit = u;
      d.b = x.b;
      d.h = x.h;
      d.n_valid = x.n_valid;
      d.tiles = x.tiles;
      d.nbp = x.nbp;
      d.trow = x.trow;
      d.j = j;
      d.P = P0;
      d.c_first = cta_of(d.P, T, CTAS);
      d.n_seg = cta_of(d.P + d.tiles - 1, T, CTAS) - d.c_first + 1;
    };
    const int last_u = flags[20];
    const int64_t last_P = *reinterpret_cast<volatile int64_t *>(flags + 22);
    const bool reorder = kHelper && last_u != start_u && flags[21];
    const int i_jump = reorder ? (int)(hi - last_P) : ntiles;  // position of the jump back to lo
    TileDesc cur;
    if (reorder) set_at(cur, last_u, 0, last_P, 32);
    else set_at(cur, start_u, start_j, start_P, 6);
    cur.wi = 0;
    // Page (paged) or block (sparse) id number k of a tile: where it sits in
    // the tables (null when the tile has no such page), and its check when it
    // is used (-1 when absent or invalid; an invalid one also sets its error
    // bit and is skipped; a slot whose copy was never issued is never used).
    auto id_src = [&](const TileDesc &d, int k) -> const int32_t * {
      if (p.sparse_block_size > 0) {
        const int e = d.j / (p.sparse_block_size / kTile);
        // list entry e: the first table's, then the full table's
        return e < d.nbp ? p.kv_idx + (int64_t)d.trow * p.max_sparse_blocks + e
                         : p.kv_full_idx + (int64_t)d.trow * p.max_sparse_blocks + e - d.nbp;
      }
      const int tok0 = d.j * kTile + k * (P >= kTile ? 0 : P);
      if (tok0 >= d.n_valid) return nullptr;
      return p.block_table + (int64_t)d.b * p.max_pages + tok0 / P;
    };
    auto check_id = [&](const TileDesc &d, int k, const int *slot) -> int {
      if (p.sparse_block_size > 0) {
        const int raw = *slot;
        const bool bad = raw < 0 || (int64_t)raw * p.sparse_block_size >= p.cache_len;
        dev_err |= bad ? DA_DEVERR_SPARSE_INDEX : 0u;
        return bad ? -1 : raw;
      }
      const int tok0 = d.j * kTile + k * (P >= kTile ? 0 : P);
      if (tok0 >= d.n_valid) return -1;
      const int raw = *slot;
      const bool bad = raw < 0 || raw >= p.num_pages;
      dev_err |= bad ? DA_DEVERR_PAGE_INDEX : 0u;
      return bad ? -1 : raw;
    };
    auto advance = [&](TileDesc &d) {
      if (++d.wi == i_jump) {
        set_at(d, start_u, start_j, start_P, 6);
        return;
      }
      if (++d.j < d.tiles) return;
      d.P += d.tiles;
      int u = d.unit;
      UnitInfo x;
      do {  // units without tiles were written in the prologue
        ++u;
        x = unit_info(p, u < U ? u : U - 1, dev_err);
      } while (u < U && x.tiles == 0);
      d.unit = u;
      d.b = x.b;
      d.h = x.h;
      d.n_valid = x.n_valid;
      d.tiles = x.tiles;
      d.nbp = x.nbp;
      d.trow = x.trow;
      d.j = 0;
      d.c_first = cta_of(d.P, T, CTAS);
      d.n_seg = cta_of(d.P + d.tiles - 1, T, CTAS) - d.c_first + 1;
    };

    // Ids are fetched kIdAhead tiles before they are used, by 4-byte cp.async
    // into a queue in shared memory (slot t % kIdAhead holds the L ids of tile
    // t; L ids per tile: the pages of a tile, or one block / page): no register
    // waits on a table load in flight, so one tile's lookup never holds up the
    // next tile's issue. Lanes 0 .. L-1 copy, one commit group per tile.
    const bool needs_ids = p.paged || p.sparse_block_size > 0;
    const int L = pages_per_tile;
    TileDesc ahead = cur;
    if (needs_ids) {
      for (int k = 0; k < kIdAhead; ++k) {
        if (k < ntiles && lane < L) {
          const int32_t *src = id_src(ahead, lane);
          if (src) cp_async_4(idq + k * L + lane, src);
        }
        cp_async_commit();
        if (k + 1 < ntiles) advance(ahead);
      }
    }
    int issued = 0;  // tiles whose copies are issued (the drain after a timeout waits for them)
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % C::kStages;
      bool ok = true;
      if (lane == 0 && i >= C::kStages)
        ok = mbar_wait_bounded(&empty[st], ((i / C::kStages) & 1) ^ 1, kWaitLimitNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        dev_err |= DA_DEVERR_TIMEOUT;
        if (lane == 0) flags[0] = 1;
        break;
      }
      const int *ids = idq + (i % kIdAhead) * L;  // this tile's ids
      if (needs_ids) {
        cp_async_wait_group<kIdAhead - 1>();  // this lane's copies for tile i have landed
        __syncwarp();                         // and so have the other lanes'
      }
      // ---- this tile's boxes (y = first cache row of the box)
      uint64_t valid = 0;
      int nbox = 0;
      int ys[kTile / 16];
      const int tok_base = cur.j * kTile;
      int pos0 = tok_base;  // the tile's first position in the row
      if (p.sparse_block_size > 0) {
        const int blk = check_id(cur, 0, ids);
        if (blk >= 0) {
          const int tb = blk * p.sparse_block_size + (cur.j % (p.sparse_block_size / kTile)) * kTile;
          pos0 = tb;
          const int lim = min(min(cur.n_valid - tb, kTile), p.cache_len - tb);
          valid = low_bits(lim);
          if (lim > 0) {
            ys[0] = (int)(((int64_t)cur.unit * p.cache_len + tb) );
            nbox = 1;
          }
        }
      } else if (!p.paged) {
        const int lim = min(cur.n_valid - tok_base, kTile);
        valid = low_bits(lim);
        ys[0] = (int)(((int64_t)cur.unit * p.cache_len + tok_base) );
        nbox = 1;
      } else if (P >= kTile) {
        const int page = check_id(cur, 0, ids);
        if (page >= 0) {
          valid = low_bits(min(cur.n_valid - tok_base, kTile));
          ys[0] = (int)((((int64_t)page * p.num_kv_heads + cur.h) * P + tok_base % P) );
          nbox = 1;
        }
      } else {
        for (int k = 0; k < kTile / P; ++k) {
          const int page = check_id(cur, k, ids + k);
          ys[k] = -1;
          if (page >= 0) {
            valid |= low_bits(min(cur.n_valid - (tok_base + k * P), P)) << (k * P);
            ys[k] = (int)(((int64_t)page * p.num_kv_heads + cur.h) * P );
            ++nbox;
          }
        }
      }
      if (lane == 0) {
        const bool first = (i == 0) || (i == i_jump) || (cur.j == 0);
        const bool last = (i + 1 == ntiles) || (i + 1 == i_jump) || (cur.j + 1 == cur.tiles);
        StageMeta m;
        m.valid = valid;
        m.unit = cur.unit;
        const bool full_blk =
            p.sparse_block_size > 0 && cur.j / (p.sparse_block_size / kTile) >= cur.nbp;
        m.flags = (first ? kFirst : 0) | (last ? kLast : 0) | (full_blk ? kFull : 0);
        m.c_first = cur.c_first;
        m.n_seg = cur.n_seg;
        m.nval = cur.n_valid - pos0;
        m.pos0 = pos0;
        meta[st] = m;
        const uint32_t box_tokens = (p.paged && P < kTile) ? (uint32_t)P : (uint32_t)kTile;
        const uint32_t row_bytes = I4 ? (uint32_t)(p.kv_groups + kD / 8) * 4u : (uint32_t)C::kBytesPerTok;
        uint32_t bytes = 2u * (uint32_t)nbox * box_tokens * row_bytes;
        if (TOK) bytes += 2u * (uint32_t)nbox * box_tokens * 4;  // scale words
        if (first) bytes += (uint32_t)G * kD * 2;
        mbar_arrive_expect_tx(&full[st], bytes);
        if (!multi_box) {
          uint8_t *kdst = ring + (size_t)st * 2 * C::kTileBytes;
          uint8_t *vdst = kdst + C::kTileBytes;
          if (first)
            tma_load_2d(qslots + st * C::kQSlot, &qmap, &full[st], 0,
                        (int)((int64_t)cur.b * p.num_q_heads + cur.h * G), q_policy);
          const int nb = (p.paged && P < kTile) ? kTile / P : (nbox ? 1 : 0);
          const int box_rows = (p.paged && P < kTile) ? P : kTile;
          for (int k = 0; k < nb; ++k) {
            if (ys[k] < 0) continue;
            const int off = k * box_rows * (int)row_bytes;  // box k of a multi-page tile
            if (I4) {
              // whole int4 rows, as the 128-byte lines they fill
              const int yl = (int)((int64_t)ys[k] * (p.kv_groups + kD / 8) / 32);
              tma_load_2d(kdst + off, &kmap, &full[st], 0, yl, policy);
              tma_load_2d(vdst + off, &vmap, &full[st], 0, yl, policy);
            } else if (FP8) {
              tma_load_2d(kdst + off, &kmap, &full[st], 0, ys[k], policy);
              tma_load_2d(vdst + off, &vmap, &full[st], 0, ys[k], policy);
              if (TOK) {
                // the boxes' per-token scale words ([K|V][kTile] per stage; the
                // rows of a box start at a multiple of 4)
                int32_t *ss = reinterpret_cast<int32_t *>(smem + C::oSS) + st * 2 * C::kSSWords +
                              ss_word(k * box_rows, box_rows);
                tma_load_2d(ss, &kssmap, &full[st], 0, ys[k] / 4, policy);
                tma_load_2d(ss + C::kSSWords, &vssmap, &full[st], 0, ys[k] / 4, policy);
              }
            } else {
              // one 3-D box: both 64-element halves of box_rows rows, half-major
              tma_load_3d(kdst + off, &kmap, &full[st], 0, ys[k], 0, policy);
              tma_load_3d(vdst + off, &vmap, &full[st], 0, ys[k], 0, policy);
            }
          }
        }
      }
      if (multi_box) {
        // the page boxes of the tile are issued by several lanes at once (lane
        // k: K box k, lane 8 + k: V box k, lane 16: the query group) once lane
        // 0 has set the stage's byte count: one lane issuing them in turn
        // limits the rate at which a CTA streams small pages
        __syncwarp();
        const bool first = (i == 0) || (i == i_jump) || (cur.j == 0);
        const int k = lane & 7;
        int y = -1;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          if (kk == k) y = ys[kk];
        if (lane < 16 && k < kTile / P && y >= 0) {
          const bool isv = lane >= 8;
          const int row_bytes = I4 ? (p.kv_groups + kD / 8) * 4 : C::kBytesPerTok;
          uint8_t *dst = ring + (size_t)st * 2 * C::kTileBytes + (isv ? C::kTileBytes : 0) +
                         k * P * row_bytes;
          if (I4) {
            tma_load_2d(dst, isv ? &vmap : &kmap, &full[st], 0,
                        (int)((int64_t)y * (p.kv_groups + kD / 8) / 32), policy);
          } else {
            tma_load_3d(dst, isv ? &vmap : &kmap, &full[st], 0, y, 0, policy);
          }
        }
        if (first && lane == 16)
          tma_load_2d(qslots + st * C::kQSlot, &qmap, &full[st], 0,
                      (int)((int64_t)cur.b * p.num_q_heads + cur.h * G), q_policy);
      }
      // fetch the ids of tile i + kIdAhead into the slot just read
      if (needs_ids) {
        __syncwarp();  // every lane has read this tile's ids
        if (i + kIdAhead < ntiles) {
          if (lane < L) {
            const int32_t *src = id_src(ahead, lane);
            if (src) cp_async_4(idq + (i % kIdAhead) * L + lane, src);
          }
          if (i + kIdAhead + 1 < ntiles) advance(ahead);
        }
        cp_async_commit();
      }
      issued = i + 1;
      if (i + 1 < ntiles) advance(cur);
    }
    if (needs_ids) cp_async_wait_group<0>();  // no copy outlives the loop (a timeout leaves early)
    if (lane == 0) flags[1] = issued;
  } else if (warp > kConsumerWarps) {
    // ======================================================= helper (kHelper only)
    // Counts this range's partial segments as the consumers finish them and,
    // when one completes a unit of at most kWarpMergeSegs pieces, merges the
    // unit right away (larger merges are left to the consumers' end).
    // Partial segments: the first (its unit started before lo, or goes on past
    // hi when the range holds a single unit) and the last.
    const int n_partial = flags[20] == start_u ? flags[21] : (start_j > 0 ? 1 : 0) + flags[21];
    bool ok = true;
    for (int k = 0; k < n_partial; ++k) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(&part_bar[k & 1], (k >> 1) & 1, kWaitLimitNs))))
        break;
      const int unit = flags[14 + 3 * k], c_first = flags[15 + 3 * k], n_seg = flags[16 + 3 * k];
      const bool merge_now = __shfl_sync(
          0xffffffffu, lane == 0 ? count_piece(p, flags, unit, c_first, n_seg, true) : false, 0);
      __syncwarp();  // lane 0's acquire covers the whole warp's reads of the pieces
      if (merge_now) merge_unit_warp(p, unit, c_first, n_seg, G);
    }
    if (!ok) {
      dev_err |= DA_DEVERR_TIMEOUT;
      if (lane == 0) flags[0] = 1;
    }
  } else {
    // ======================================================= consumers
    const int q4 = lane & 3;   // owns heads g = nt*8 + 2*q4 + {0,1}
    const int r8 = lane >> 2;  // row inside an 8-row group
    const int tok_lane = 16 * warp + (lane & 7);
    const int mi = lane >> 3;  // which 8x8 matrix this lane addresses
    const int br_shift = (p.paged && p.page_size < kTile) ? __ffs(p.page_size) - 1 : 6;
    // this lane's ldmatrix row tokens: (mi & 1) selects +8 for QK / fp8 V, (mi >> 1) for bf16 V
    const uint32_t toff_a = token_offset<FP8>(tok_lane + (mi & 1) * 8, br_shift);
    const uint32_t toff_b = token_offset<FP8>(tok_lane + (mi >> 1) * 8, br_shift);
    uint32_t qf[NT][8][2];
    // fp8_mma (Q8): e4m3 query fragments (B operand of the k32 MMAs: dims
    // 32pp + 16j + 4q4 .. +3 of row r8) and the score factor of the thread's
    // rows nt * 8 + 2 * q4 + e, which holds each row's e4m3 scale
    uint32_t qf8[NT][4][2];
    float rq[NT][2];
    float oacc[NT][8][4];
    float m_run[NT][2], l_part[NT][2];
    float sscale = p.score_scale, vmul = 1.f;
    const bool softcap = MOD >= 1 && p.softcap_l2 > 0.f;
    // e4m3 with per-token scale and shift (value = e4m3 * sc + sh): the score
    // of a key is sc * (q . e4m3) + sh * sum(q), so the MMA runs on the codes
    // and qsum holds sum(q) of the thread's two query rows; a value's scale
    // multiplies its row in the PV operand, and its shift adds p * sh to every
    // output element of the query row (zacc, rescaled like l).
    constexpr bool tok_scale = TOK;
    const int32_t *ssw = reinterpret_cast<const int32_t *>(smem + C::oSS);
    const int ss_rows = (p.paged && p.page_size < kTile) ? p.page_size : kTile;  // rows per box
    float qsum[NT][2], zacc[NT][2];
    // Query row g * q_len + t (several query tokens per row): the row's last
    // q_len positions are its new tokens, new token j at seq_len - q_len + j.
    // Token t sees every older position and the new tokens set in its mask
    // word: bits 0..t (causal) unless a draft-tree mask gives the word.
    int trow[NT][2];
    uint32_t mword[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        trow[nt][e] = (nt * 8 + 2 * q4 + e) % p.q_len;
        mword[nt][e] = (2u << trow[nt][e]) - 1u;
      }
    // The flex-style mods (the sink/window mask_mod, the ALiBi score_mod) are
    // per query head: row g * Q + t of a unit of kv head h belongs to query
    // head h * (rows / Q) + g; their arrays are read per tile (L1 hits).
    const bool mods = MOD == 2 && (p.mask_window != nullptr || p.alibi_slopes != nullptr);
    auto reset = [&]() {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) oacc[nt][mt][e] = 0.f;
        m_run[nt][0] = m_run[nt][1] = neg_inf();
        l_part[nt][0] = l_part[nt][1] = 0.f;
        zacc[nt][0] = zacc[nt][1] = 0.f;
        qsum[nt][0] = qsum[nt][1] = 0.f;
      }
    };
    reset();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) qf[nt][ks][0] = qf[nt][ks][1] = 0u;
    bool ok = true;
    int npart = 0;  // partial segments written so far
    int nseg = 0;   // segments finished so far (their parity picks the stats copy)
    uint32_t epi_phase = 0;

    // (the test stall of GqaParams: warp 0 waits on a barrier that nothing
    // arrives on, with the stall's limit, instead of its first pipeline wait;
    // the timeout path then runs as it would after a real failure)
    if (p.test_stall_ns != 0 && warp == 0) ok = warp_wait(stall_bar, 0u, p.test_stall_ns);
    for (int i = 0; ok && i < ntiles; ++i) {
      const int st = i % C::kStages;
      if (!warp_wait(&full[st], (i / C::kStages) & 1, kWaitLimitNs)) {
        ok = false;
        break;
      }
      const StageMeta m = meta[st];
      const int unit = m.unit;
      if (m.flags & kFirst) {
        // the segment's query group: Q^T fragments (B operand), read once per segment
        const int h = unit % p.num_kv_heads;
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(qslots + st * C::kQSlot);
        // e4m3 / int4 keys meet Q in f16. The segment's query rows are scaled by
        // an exact power of two 2^e that puts their largest |q| in [2^14, 2^15),
        // so every finite bf16 q lands in f16's range (an element more than 2^28
        // below that largest one becomes an f16 subnormal: an error under 2^-28
        // of the largest product), and 2^-e joins the score factor.
        int qexp = 0;
        if (FP8 && !Q8) {
          float amax = 0.f;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int g = nt * 8 + r8;
            amax = fmaxf(amax, q_row_amax(qs + (g < G ? g : 0) * (kD / 2), q4, r8));
          }
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          qexp = q_exponent(amax);
        }
        const float q2 = pow2f(qexp);
        float qsq[NT];  // Q8: the e4m3 scale of the lane's row r8
        if (Q8) {
          // e4m3 queries in fp32 steps: amax = max |q| of the row, inv = 448 /
          // amax, code = e4m3(q * inv) to nearest even, saturating; the row's
          // scale amax / 448 goes into its score factor (rows with amax below
          // 2^-100 are zero)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int g = nt * 8 + r8;
            const uint32_t *qrow = qs + (g < G ? g : 0) * (kD / 2);
            float amax = q_row_amax(qrow, q4, r8);
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const bool tiny = !(amax >= 0x1p-100f);
            const float inv = tiny ? 0.f : __fdiv_rn(448.f, amax);
            qsq[nt] = tiny ? 0.f : __fdiv_rn(amax, 448.f);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int d0 = 32 * pp + 16 * j + 4 * q4;  // four consecutive dims
                const uint32_t w0 = qrow[d0 / 2], w1 = qrow[d0 / 2 + 1];
                const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(__uint_as_float(w0 << 16), inv),
                                                    __fmul_rn(__uint_as_float(w0 & 0xFFFF0000u), inv));
                const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(__uint_as_float(w1 << 16), inv),
                                                    __fmul_rn(__uint_as_float(w1 & 0xFFFF0000u), inv));
                qf8[nt][pp][j] = g < G ? (lo | (hi << 16)) : 0u;
              }
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int g = nt * 8 + r8;
          const uint32_t *qrow = qs + (g < G ? g : 0) * (kD / 2);
#pragma unroll
          for (int ks = 0; ks < 8 && !Q8; ++ks) {
            if (I4) {
              // k-step 2c+s pairs the elements one int4 data word gives a lane:
              // 32c + 8q4 + 2s + {0, 4} (b0) and 32c + 8q4 + 2s + 1 + {0, 4} (b1)
              const __nv_bfloat16 *qh = reinterpret_cast<const __nv_bfloat16 *>(qrow);
              const int d0 = 32 * (ks >> 1) + 8 * q4 + 2 * (ks & 1);
              qf[nt][ks][0] =
                  g < G ? pack_f16(__bfloat162float(qh[d0]) * q2, __bfloat162float(qh[d0 + 4]) * q2) : 0u;
              qf[nt][ks][1] =
                  g < G ? pack_f16(__bfloat162float(qh[d0 + 1]) * q2, __bfloat162float(qh[d0 + 5]) * q2)
                        : 0u;
            } else if (!FP8) {
              qf[nt][ks][0] = g < G ? qrow[(16 * ks + 2 * q4) / 2] : 0u;
              qf[nt][ks][1] = g < G ? qrow[(16 * ks + 8 + 2 * q4) / 2] : 0u;
            } else {
              // k-step 2pp+e covers bytes 32pp + 16e + 4q4 .. +3 of each fp8 key row
              const int pp = ks >> 1, e = ks & 1;
              const int d0 = 32 * pp + 16 * e + 4 * q4;
              qf[nt][ks][0] = g < G ? bf16x2_to_f16x2(qrow[d0 / 2], q2) : 0u;
              qf[nt][ks][1] = g < G ? bf16x2_to_f16x2(qrow[d0 / 2 + 1], q2) : 0u;
            }
          }
        }
        if (tok_scale) {
          sscale = p.score_scale;
          vmul = 1.f;
          // sum of each query row's values as the MMA sees them (f16): this
          // thread holds 32 of row r8's elements; the quad's four threads hold all
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float part = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&qf[nt][ks][j]));
                part += f.x + f.y;
              }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            qsum[nt][0] = __shfl_sync(0xffffffffu, part, 4 * (2 * q4));
            qsum[nt][1] = __shfl_sync(0xffffffffu, part, 4 * (2 * q4 + 1));
          }
        } else if (FP8 && !I4) {
          sscale = p.score_scale * p.k_scale[h];
          vmul = p.v_scale[h];
          if (Q8) vmul *= 0.00390625f;  // the weights met V scaled by 2^8
        } else {
          sscale = p.score_scale;
        }
        if (FP8) sscale *= pow2f(-qexp);
        if (Q8) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) rq[nt][e] = sscale * __shfl_sync(0xffffffffu, qsq[nt], 4 * (2 * q4 + e));
        }
        if (MOD >= 1 && p.spec_mask != nullptr) {
          const uint32_t *mrow = p.spec_mask + (size_t)(unit / p.num_kv_heads) * p.q_len;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) mword[nt][e] = mrow[trow[nt][e]];
        }
      }
      const uint32_t vbits = (uint32_t)(m.valid >> (16 * warp)) & 0xFFFFu;
      if (vbits != 0) {
        const uint32_t kbase = smem_u32(ring + (size_t)st * 2 * C::kTileBytes);
        const uint32_t vbase = kbase + C::kTileBytes;
        // ---------------- S^T = K Q^T (16 tokens x 8*NT heads)
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
        {
          const int t = tok_lane + (mi & 1) * 8;
          if (I4) {
            // int4 K: each lane's ldmatrix word is 8 codes of one token row;
            // its pairs (j, j + 4) are the A fragments of two k-steps, scaled
            // by the row's group coefficients
            const int ng = p.kv_groups, rw = ng + kD / 8;  // row words
            const int32_t *cfk = reinterpret_cast<const int32_t *>(ring + (size_t)st * 2 * C::kTileBytes);
            const int tA = 16 * warp + r8, tB = tA + 8;
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
              uint32_t r[4];
              ldsm_x4(i4_addr(kbase, t, 2 * cp + (mi >> 1), rw * 4, ng), r[0], r[1], r[2], r[3]);
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {  // chunk 2cp + h2: words r[2h2] (row tA), r[2h2+1] (tB)
                const int cc = 2 * cp + h2;
                const int gi = ng == 4 ? cc : 2 * cc + (q4 >> 1);
                const uint32_t wA = (uint32_t)cfk[tA * rw + gi], wB = (uint32_t)cfk[tB * rw + gi];
                const uint32_t sA = prmt(wA, 0, 0x1010), hA = prmt(wA, 0, 0x3232);
                const uint32_t sB = prmt(wB, 0, 0x1010), hB = prmt(wB, 0, 0x3232);
#pragma unroll
                for (int sidx = 0; sidx < 2; ++sidx) {
                  const uint32_t a0 = i4_dequant(i4_codes(r[2 * h2], 2 * sidx), sA, hA);
                  const uint32_t a2 = i4_dequant(i4_codes(r[2 * h2], 2 * sidx + 1), sA, hA);
                  const uint32_t a1 = i4_dequant(i4_codes(r[2 * h2 + 1], 2 * sidx), sB, hB);
                  const uint32_t a3 = i4_dequant(i4_codes(r[2 * h2 + 1], 2 * sidx + 1), sB, hB);
                  const int ks = 2 * cc + sidx;
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma_f16_16816(sacc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
                }
              }
            }
          } else if (!FP8) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(chunk_addr<false>(kbase, toff_a, t, 2 * ks + (mi >> 1), br_shift), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_bf16_16816(sacc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
            }
          } else if (Q8) {
            // e4m3 K straight from ldmatrix: the four 8x16-byte matrices (rows 0-7
            // and 8-15, bytes 32pp..+15 and +16..+31) are the k32 A fragment
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
              uint32_t r0, r1, r2, r3;
              ldsm_x4(chunk_addr<true>(kbase, toff_a, t, 2 * pp + (mi >> 1), br_shift), r0, r1, r2, r3);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_e4m3_16832(sacc[nt], r0, r1, r2, r3, qf8[nt][pp][0], qf8[nt][pp][1]);
            }
          } else {
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
              uint32_t r0, r1, r2, r3;
              ldsm_x4(chunk_addr<true>(kbase, toff_a, t, 2 * pp + (mi >> 1), br_shift), r0, r1, r2, r3);
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
        }
        // ---------------- mask, online softmax (exp2), P^T fragments
        const bool ok_r = (vbits >> r8) & 1u, ok_r8 = (vbits >> (r8 + 8)) & 1u;
        float vsh0 = 0.f, vsh1 = 0.f;  // value shifts of the thread's two tokens
        if (tok_scale) {
          const int32_t *ssk = ssw + st * 2 * C::kSSWords;
          const int w0 = ss_word(16 * warp + r8, ss_rows), w1 = ss_word(16 * warp + r8 + 8, ss_rows);
          const uint32_t k0 = (uint32_t)ssk[w0], k1 = (uint32_t)ssk[w1];
          const uint32_t v0 = (uint32_t)ssk[C::kSSWords + w0], v1 = (uint32_t)ssk[C::kSSWords + w1];
          const float2 kf0 = __half22float2(*reinterpret_cast<const __half2 *>(&k0));
          const float2 kf1 = __half22float2(*reinterpret_cast<const __half2 *>(&k1));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              sacc[nt][e] = fmaf(sacc[nt][e], kf0.x, kf0.y * qsum[nt][e]);
              sacc[nt][2 + e] = fmaf(sacc[nt][2 + e], kf1.x, kf1.y * qsum[nt][e]);
            }
          // a token past the row's end may hold any word: its shift must not
          // meet its zero weight (0 * inf)
          vsh0 = ok_r ? __half2float(__ushort_as_half((unsigned short)(v0 >> 16))) : 0.f;
          vsh1 = ok_r8 ? __half2float(__ushort_as_half((unsigned short)(v1 >> 16))) : 0.f;
        }
        // new-token index of this thread's first token (negative: an older position)
        const int jnew = 16 * warp + r8 - (m.nval - p.q_len);
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float alpha[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            // the query token's mask over the new tokens (the tile's valid bits
            // already stop at the row's length; one query token keeps all)
            bool ok0 = ok_r && (MOD == 0 || jnew < 0 || ((mword[nt][e] >> min(jnew, 31)) & 1u));
            bool ok1 =
                ok_r8 && (MOD == 0 || jnew + 8 < 0 || ((mword[nt][e] >> min(jnew + 8, 31)) & 1u));
            const float f = Q8 ? rq[nt][e] : sscale;
            float x0 = sacc[nt][e] * f, x1 = sacc[nt][2 + e] * f;
            if (softcap) {  // c * tanh(s / c), in log2 units: c2 * tanh(x / c2)
              x0 = cap_tanh(x0, p.softcap_l2, p.softcap_k);
              x1 = cap_tanh(x1, p.softcap_l2, p.softcap_k);
            }
            if (mods) {
              const int row = min(nt * 8 + 2 * q4 + e, G - 1);
              const int hq = (unit % p.num_kv_heads) * (G / p.q_len) + row / p.q_len;
              // positions of the thread's two tokens and of the row's query token
              const int kv0 = m.pos0 + 16 * warp + r8, kv1 = kv0 + 8;
              const int qpos = m.nval + m.pos0 - p.q_len + trow[nt][e];
              if (p.mask_window && !(m.flags & kFull)) {  // the mask_mod skips full blocks
                const int w = __ldg(p.mask_window + hq), sk = p.mask_sink ? __ldg(p.mask_sink + hq) : 0;
                ok0 = ok0 && (kv0 < sk || w < 0 || kv0 > qpos - w);
                ok1 = ok1 && (kv1 < sk || w < 0 || kv1 > qpos - w);
              }
              if (p.alibi_slopes) {  // in log2 units, like the scores
                const float sl = __ldg(p.alibi_slopes + hq) * 1.4426950408889634f;
                x0 += sl * (float)(kv0 - qpos);
                x1 += sl * (float)(kv1 - qpos);
              }
            }
            x0 = ok0 ? x0 : neg_inf();
            x1 = ok1 ? x1 : neg_inf();
            float tmax = fmaxf(x0, x1);
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
            const float m_new = fmaxf(m_run[nt][e], tmax);
            // while no score of the row is valid the reference is 0: masked
            // scores weigh 0, NaN scores (a NaN query or key) weigh NaN
            const float m_use = m_new == neg_inf() ? 0.f : m_new;
            const float a = ex2(m_run[nt][e] - m_use);
            const float p0 = ex2(x0 - m_use), p1 = ex2(x1 - m_use);
            l_part[nt][e] = l_part[nt][e] * a + (p0 + p1);
            if (tok_scale) zacc[nt][e] = zacc[nt][e] * a + (p0 * vsh0 + p1 * vsh1);
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
          if (Q8) {
            // the weights times 2^8 as f16, transposed (lane (g, t): tokens 2t,
            // 2t+1 and 8+2t, 9+2t of head g), then rounded to e4m3: bytes in the
            // token order (2t, 2t+1, 8+2t, 9+2t) of k 4t..4t+3 (tokens 16-31 of
            // the k32 step are absent: 0)
            const uint32_t y0 = movmatrix_trans(pack_f16(256.f * sacc[nt][0], 256.f * sacc[nt][1]));
            const uint32_t y1 = movmatrix_trans(pack_f16(256.f * sacc[nt][2], 256.f * sacc[nt][3]));
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&y0));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&y1));
            pb[nt][0] = f32x2_to_e4m3x2(f0.x, f0.y) | (f32x2_to_e4m3x2(f1.x, f1.y) << 16);
            pb[nt][1] = 0u;
          } else {
            const uint32_t x0 = FP8 ? pack_f16(sacc[nt][0], sacc[nt][1])
                                    : pack_bf16(sacc[nt][0], sacc[nt][1]);
            const uint32_t x1 = FP8 ? pack_f16(sacc[nt][2], sacc[nt][3])
                                    : pack_bf16(sacc[nt][2], sacc[nt][3]);
            pb[nt][0] = movmatrix_trans(x0);
            pb[nt][1] = movmatrix_trans(x1);
          }
        }
        // ---------------- O^T += V^T P^T (masked tokens' V zeroed in registers)
        const bool full16 = vbits == 0xFFFFu;
        const uint32_t m01 = lo16_mask((vbits >> (2 * q4)) & 1u, (vbits >> (2 * q4 + 1)) & 1u);
        const uint32_t m89 =
            lo16_mask((vbits >> (2 * q4 + 8)) & 1u, (vbits >> (2 * q4 + 9)) & 1u);
        if (I4) {
          // int4 V through ldmatrix.trans: a lane's word holds four codes of each
          // of two tokens (2q4, 2q4+1 or +8, +9) for elements 32c + 4r8 + 0..3;
          // code j of chunks 2cp / 2cp + 1 gives rows r8 / r8 + 8 of the
          // O^T tile 4cp + j (elements 64cp + 4r8 + j and + 32)
          const int ng = p.kv_groups, rw = ng + kD / 8;  // row words
          const int32_t *cfv =
              reinterpret_cast<const int32_t *>(ring + (size_t)st * 2 * C::kTileBytes + C::kTileBytes);
          const int t0 = 16 * warp + 2 * q4;
          const int t = tok_lane + (mi & 1) * 8;
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {
            uint32_t r[4];
            ldsm_x4_trans(i4_addr(vbase, t, 2 * cp + (mi >> 1), rw * 4, ng), r[0], r[1], r[2], r[3]);
            // coefficient pairs (scale, shift) of the token pairs, per chunk
            uint32_t sc[2][2], sh[2][2];  // [chunk 2cp + h2][lo pair | hi pair]
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int cc = 2 * cp + h2;
              const int gi = ng == 4 ? cc : 2 * cc + (r8 >> 2);
#pragma unroll
              for (int hp = 0; hp < 2; ++hp) {
                const int ta = t0 + 8 * hp;
                const uint32_t w0 = (uint32_t)cfv[ta * rw + gi], w1 = (uint32_t)cfv[(ta + 1) * rw + gi];
                sc[h2][hp] = prmt(w0, w1, 0x5410);
                sh[h2][hp] = prmt(w0, w1, 0x7632);
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t a0 = i4_dequant(i4_codes(r[0], j), sc[0][0], sh[0][0]);
              uint32_t a2 = i4_dequant(i4_codes(r[1], j), sc[0][1], sh[0][1]);
              uint32_t a1 = i4_dequant(i4_codes(r[2], j), sc[1][0], sh[1][0]);
              uint32_t a3 = i4_dequant(i4_codes(r[3], j), sc[1][1], sh[1][1]);
              if (!full16) {  // tokens past the row's end: zero values (their rows may hold anything)
                a0 &= m01;
                a1 &= m01;
                a2 &= m89;
                a3 &= m89;
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_f16_16816(oacc[nt][4 * cp + j], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
          }
        } else if (!FP8) {
          const int t = tok_lane + (mi >> 1) * 8;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(chunk_addr<false>(vbase, toff_b, t, 2 * mt + (mi & 1), br_shift), a0, a1, a2, a3);
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
        } else if (Q8) {
          // e4m3 V^T (k32 A fragment, tokens in the order (2t, 2t+1, 8+2t, 9+2t) of
          // the weights): ldmatrix.trans on byte pairs gives lane (g, t) tokens
          // 2t, 2t+1 (r0: 0-7, r1: 8-15) x dims 2g, 2g+1 of a 16-dim chunk; a byte
          // permutation splits the two dims into rows g (dim 2g) and g + 8 (dim
          // 2g + 1) of the m-tile (the dim order the epilogue undoes)
          const int t = tok_lane + (mi & 1) * 8;
          const uint32_t tmask = full16 ? 0xFFFFFFFFu
                                        : (((vbits >> (2 * q4)) & 1u) ? 0x000000FFu : 0u) |
                                              (((vbits >> (2 * q4 + 1)) & 1u) ? 0x0000FF00u : 0u) |
                                              (((vbits >> (2 * q4 + 8)) & 1u) ? 0x00FF0000u : 0u) |
                                              (((vbits >> (2 * q4 + 9)) & 1u) ? 0xFF000000u : 0u);
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(chunk_addr<true>(vbase, toff_a, t, 2 * pp + (mi >> 1), br_shift), r0, r1, r2, r3);
            // tokens past the row's end may hold anything (NaN): zero their bytes
            const uint32_t a0 = prmt(r0, r1, 0x6420) & tmask, a1 = prmt(r0, r1, 0x7531) & tmask;
            const uint32_t c0 = prmt(r2, r3, 0x6420) & tmask, c1 = prmt(r2, r3, 0x7531) & tmask;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_e4m3_16832(oacc[nt][2 * pp], a0, a1, 0u, 0u, pb[nt][0], 0u);
              mma_e4m3_16832(oacc[nt][2 * pp + 1], c0, c1, 0u, 0u, pb[nt][0], 0u);
            }
          }
        } else {
          const int t = tok_lane + (mi & 1) * 8;
          // per-token value scales of the fragment's token pairs (2q4, 2q4+1) and
          // (2q4+8, 2q4+9), f16x2, zero past the row's end
          uint32_t s01 = 0u, s89 = 0u;
          if (tok_scale) {
            const int32_t *ssv = ssw + st * 2 * C::kSSWords + C::kSSWords;
            const int t0 = 16 * warp + 2 * q4;
            s01 = (((uint32_t)ssv[ss_word(t0, ss_rows)] & 0xFFFFu) |
                   ((uint32_t)ssv[ss_word(t0 + 1, ss_rows)] << 16)) & m01;
            s89 = (((uint32_t)ssv[ss_word(t0 + 8, ss_rows)] & 0xFFFFu) |
                   ((uint32_t)ssv[ss_word(t0 + 9, ss_rows)] << 16)) & m89;
          }
          auto hmul2 = [](uint32_t x, uint32_t y) {
            const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&x),
                                      *reinterpret_cast<const __half2 *>(&y));
            return *reinterpret_cast<const uint32_t *>(&r);
          };
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(chunk_addr<true>(vbase, toff_a, t, 2 * pp + (mi >> 1), br_shift), r0, r1, r2, r3);
            // r = [V[2q][2c], V[2q][2c+1], V[2q+1][2c], V[2q+1][2c+1]] -> token pairs per d
            const uint32_t s0 = prmt(r0, 0, 0x3120), s1 = prmt(r1, 0, 0x3120);
            const uint32_t s2 = prmt(r2, 0, 0x3120), s3 = prmt(r3, 0, 0x3120);
            uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(s0 & 0xFFFF));
            uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(s0 >> 16));
            uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(s1 & 0xFFFF));
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
            if (tok_scale) {
              a0 = hmul2(a0, s01);
              a1 = hmul2(a1, s01);
              a2 = hmul2(a2, s89);
              a3 = hmul2(a3, s89);
              c0 = hmul2(c0, s01);
              c1 = hmul2(c1, s01);
              c2 = hmul2(c2, s89);
              c3 = hmul2(c3, s89);
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
      if (!(m.flags & kLast)) {
        if (lane == 0) mbar_arrive(&empty[st]);
        continue;
      }
      // ======================= segment epilogue (consumer threads only)
      // (the segment's last stage is released at its end: it may serve as scratch)
      const int b = unit / p.num_kv_heads, h = unit - b * p.num_kv_heads;
      float *stat_m = stats + (nseg & 1) * C::kStatFloats;  // this segment's copy
      float *stat_l = stat_m + kConsumerWarps * 16;
      float *stat_z = reinterpret_cast<float *>(smem + C::oStatZ) + (nseg & 1) * kConsumerWarps * 16;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float l = l_part[nt][e];
          l += __shfl_xor_sync(0xffffffffu, l, 4);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          l_part[nt][e] = l;
          float z = 0.f;
          if (tok_scale) {
            z = zacc[nt][e];
            z += __shfl_xor_sync(0xffffffffu, z, 4);
            z += __shfl_xor_sync(0xffffffffu, z, 8);
            z += __shfl_xor_sync(0xffffffffu, z, 16);
          }
          if (r8 == 0) {
            const int g = nt * 8 + 2 * q4 + e;
            stat_m[warp * 16 + g] = m_run[nt][e];
            stat_l[warp * 16 + g] = l;
            if (tok_scale) stat_z[warp * 16 + g] = z;
          }
        }
      if (!consumer_sync(epi_bar, epi_phase)) {
        ok = false;
        break;
      }
      // each warp's O^T rescaled to the group maximum: into its own region of the
      // consumed stage when it fits (one barrier), else added into one buffer
      // one warp at a time
      float *scr = reinterpret_cast<float *>(ring + (size_t)st * 2 * C::kTileBytes);
      constexpr int kWarpScr = 8 * NT * C::kScrStride;
      // column of element (g, d) in a warp's region (swizzled 128-float rows)
      auto col = [](int g, int d) { return C::kScrSwizzled ? d ^ ((g & 7) << 2) : d; };
      // this warp's O^T rescaled to the group maximum, to dst (row stride
      // `stride`, column d at d ^ x); `add` accumulates into the shared buffer
      auto put = [&](float *dst_base, bool add) {
        constexpr int stride = C::kStageScratch ? C::kScrStride : kRedStride;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int g = nt * 8 + 2 * q4 + e;
            float M = neg_inf();
#pragma unroll
            for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, stat_m[ww * 16 + g]);
            const float wscale = (M == neg_inf()) ? 0.f : ex2(m_run[nt][e] - M);
            float *dst = dst_base + (size_t)g * stride;
            const int x = C::kScrSwizzled ? (g & 7) << 2 : 0;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int d0 = I4 ? 64 * (mt >> 2) + 4 * r8 + (mt & 3)
                                : (FP8 ? 16 * mt + 2 * r8 : 16 * mt + r8);
              const int d1 = I4 ? d0 + 32 : (FP8 ? d0 + 1 : d0 + 8);
              const float v0 = oacc[nt][mt][e] * wscale, v1 = oacc[nt][mt][2 + e] * wscale;
              if (!add) {
                dst[d0 ^ x] = v0;
                dst[d1 ^ x] = v1;
              } else {
                dst[d0] += v0;
                dst[d1] += v1;
              }
            }
          }
      };
      if (C::kStageScratch) {
        put(scr + warp * kWarpScr, false);
        ok = consumer_sync(epi_bar, epi_phase);
      } else {
        for (int w = 0; w < kConsumerWarps && ok; ++w) {
          if (warp == w) put(red, w > 0);
          ok = consumer_sync(epi_bar, epi_phase);
        }
      }
      if (!ok) break;
      // thread tid (< 128) owns head-dim element d = tid for every g of the group
      const int d = threadIdx.x;
      const bool whole = m.n_seg == 1;
      const int64_t slot = (int64_t)unit + cta;
      for (int g = 0; g < G; ++g) {
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stat_m[w * 16 + g]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
          L += (stat_l[w * 16 + g] == 0.f) ? 0.f : stat_l[w * 16 + g] * ex2(stat_m[w * 16 + g] - M);
        float acc;
        if (C::kStageScratch) {
          acc = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w)
            acc += scr[w * kWarpScr + (size_t)g * C::kScrStride + col(g, d)];
        } else {
          acc = red[(size_t)g * kRedStride + d];
        }
        if (tok_scale) {  // the value shifts: the same term for every element of the row
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w)
            acc += (M == neg_inf()) ? 0.f : stat_z[w * 16 + g] * ex2(stat_m[w * 16 + g] - M);
        }
        // no valid token: 0 and -inf; a NaN among the weights reaches both
        const float o = (L == 0.f) ? 0.f : acc * vmul / L;
        const float lse = (L == 0.f) ? neg_inf() : (M + __log2f(L)) * 0.69314718055994531f;
        if (whole) {
          const int64_t row = (int64_t)b * p.num_q_heads + h * G + g;
          p.out[row * kD + d] = __float2bfloat16(o);
          if (d == 0 && p.lse) p.lse[row] = lse;
        } else {
          p.o_part[(slot * G + g) * kD + d] = o;
          if (d == 0) p.lse_part[slot * G + g] = lse;
        }
      }
      // the stage was read through the generic proxy: order that before the
      // next TMA write into it, then release it
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (!whole) {
        // the helper warp counts the segment (its writes are released by the arrivals)
        if (threadIdx.x == 0) {
          flags[14 + 3 * npart] = unit;
          flags[15 + 3 * npart] = m.c_first;
          flags[16 + 3 * npart] = m.n_seg;
        }
        mbar_arrive(&part_bar[npart & 1]);
        ++npart;
      }
      ++nseg;
      reset();
    }
    if (!ok) {
      dev_err |= DA_DEVERR_TIMEOUT;
      flags[0] = 1;
    }
  }

  // every issued TMA box has been consumed (or a wait gave up), and the helper
  // has recorded every merge this CTA owes
  __syncthreads();
  if (flags[0]) {
    // a wait gave up: before leaving, wait (bounded) for the copies of every
    // tile the producer issued -- the last one of each stage (a stage's earlier
    // uses completed before it was refilled). Tiles never issued are not waited
    // for: their phase was never armed.
    if (threadIdx.x == kConsumerWarps * 32) {
      const int issued = flags[1];
      for (int st = 0; st < C::kStages && st < issued; ++st) {
        const int i_last = (issued - 1) - ((issued - 1 - st) % C::kStages);
        mbar_wait_bounded(&full[st], (i_last / C::kStages) & 1, kWaitLimitNs);
      }
    }
    dev_err |= DA_DEVERR_TIMEOUT;
  } else {
    // ---- the merges this CTA owes, by all its threads (the ring is free now)
    const int npending = flags[12];
    float *scr = reinterpret_cast<float *>(ring);
    const int scr_floats = C::kStages * 2 * C::kTileBytes / 4;
    volatile int *last_group = flags + 13;
    for (int k = 0; k < npending; ++k) {
      const int unit = flags[24 + 4 * k], c_first = flags[25 + 4 * k], n_seg = flags[26 + 4 * k];
      const int q = flags[27 + 4 * k];
      const int64_t slot0 = (int64_t)unit + c_first;
      if (q < 0) {
        if (n_seg <= kSmallMerge && 2 * kThreads >= G * (kD / 4)) {
          merge_slots_small(p, unit, G, slot0, 1, n_seg, true, 0, scr);
        } else if (merge_cta_floats(n_seg, G) <= scr_floats) {
          merge_slots_cta(p, unit, G, slot0, 1, n_seg, true, 0, scr);
        } else if (warp < kConsumerWarps) {
          // more pieces than the ring holds at once: the staged merge of the consumers
          uint32_t merge_phase[2] = {0u, 0u};
          // scratch: the epilogue buffer, else the query slots past the accumulators
          float *buf = red;
          int cap = 8 * NT * kRedStride;
          if constexpr (C::kRedBytes == 0) {
            buf = reinterpret_cast<float *>(qslots) + G * kD;
            cap = C::kStages * C::kQSlot / 4 - G * kD;
          }
          if (!merge_unit(p, unit, c_first, n_seg, G, ring, C::kStages * 2 * C::kTileBytes, buf,
                          cap, reinterpret_cast<float *>(qslots), merge_bar, merge_phase))
            dev_err |= DA_DEVERR_TIMEOUT;
        }
        __syncthreads();
        if (threadIdx.x == 0) p.counters[unit] = 0u;  // ready for the next call
        continue;
      }
      // two levels: this CTA completed group q; merge it in place into its first slot
      const int K = merge_group_size(n_seg), ng = (n_seg + K - 1) / K;
      const int gs = min(K, n_seg - q * K);
      const bool small = 2 * kThreads >= G * (kD / 4);
      if (small && gs <= kSmallMerge)
        merge_slots_small(p, unit, G, slot0 + (int64_t)q * K, 1, gs, false, slot0 + (int64_t)q * K, scr);
      else
        merge_slots_cta(p, unit, G, slot0 + (int64_t)q * K, 1, gs, false, slot0 + (int64_t)q * K, scr);
      if (threadIdx.x == 0)  // the group result is written (barrier above): count the group
        *last_group = atomic_add_acq_rel_gpu(p.counters + unit, 1u) == (unsigned)(ng - 1) ? 1 : 0;
      __syncthreads();
      if (*last_group) {
        if (small && ng <= kSmallMerge) merge_slots_small(p, unit, G, slot0, K, ng, true, 0, scr);
        else merge_slots_cta(p, unit, G, slot0, K, ng, true, 0, scr);
        // ready for the next call: the unit's counter and its group counters
        uint32_t *gc = p.counters + p.batch * p.num_kv_heads +
                       (int64_t)unit * max_merge_groups(gridDim.x);
        for (int i = threadIdx.x; i < ng; i += kThreads) gc[i] = 0u;
        if (threadIdx.x == 0) p.counters[unit] = 0u;
      }
      __syncthreads();
    }
  }
  if (dev_err) atomicOr(p.err, dev_err);
}

template <bool FP8, int NT, bool TOK, bool I4, int MOD, bool Q8>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gqa_split_kernel<FP8, NT, TOK, I4, MOD, Q8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<FP8, NT, TOK, I4>::kTotal);
}

template <bool FP8, int NT, bool TOK, bool I4, int MOD, bool Q8>
void launch(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
            const CUtensorMap &kssmap, const CUtensorMap &vssmap, const GqaParams &p, int ctas,
            cudaStream_t stream) {
  gqa_split_kernel<FP8, NT, TOK, I4, MOD, Q8>
      <<<ctas, threads_for<NT>(), Cfg<FP8, NT, TOK, I4>::kTotal, stream>>>(kmap, vmap, qmap, kssmap,
                                                                           vssmap, p);
}

// The six instantiations of one element kind (one or two n-tiles; no, some or
// all score modifications), set up and launched from that kind's own
// translation unit.
template <bool FP8, bool TOK, bool I4, bool Q8 = false>
cudaError_t prepare_kind() {
  cudaError_t e;
  if ((e = set_attr<FP8, 1, TOK, I4, 0, Q8>()) != cudaSuccess) return e;
  if ((e = set_attr<FP8, 2, TOK, I4, 0, Q8>()) != cudaSuccess) return e;
  if ((e = set_attr<FP8, 1, TOK, I4, 1, Q8>()) != cudaSuccess) return e;
  if ((e = set_attr<FP8, 2, TOK, I4, 1, Q8>()) != cudaSuccess) return e;
  if ((e = set_attr<FP8, 1, TOK, I4, 2, Q8>()) != cudaSuccess) return e;
  return set_attr<FP8, 2, TOK, I4, 2, Q8>();
}

template <bool FP8, bool TOK, bool I4, bool Q8 = false>
cudaError_t launch_kind(bool two, int mod, const CUtensorMap &kmap, const CUtensorMap &vmap,
                        const CUtensorMap &qmap, const CUtensorMap &kssmap,
                        const CUtensorMap &vssmap, const GqaParams &p, int ctas,
                        cudaStream_t stream) {
#define DA_LAUNCH(NT, M) \
  launch<FP8, NT, TOK, I4, M, Q8>(kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream)
  if (mod == 0) two ? DA_LAUNCH(2, 0) : DA_LAUNCH(1, 0);
  else if (mod == 1) two ? DA_LAUNCH(2, 1) : DA_LAUNCH(1, 1);
  else two ? DA_LAUNCH(2, 2) : DA_LAUNCH(1, 2);
#undef DA_LAUNCH
  return cudaGetLastError();
}

}  // namespace

// Each element kind's instantiations (bf16; e4m3 with a scale per kv head;
// e4m3 with a scale and shift per token; int4 group-wise rows) live in their
// own translation unit, gqa_kind_<kind>.cu.
#define DA_GQA_KIND_DECL(name)                                                                 \
  cudaError_t gqa_prepare_kind_##name();                                                       \
  cudaError_t gqa_launch_kind_##name(bool two, int mod, const CUtensorMap &kmap,               \
                                     const CUtensorMap &vmap, const CUtensorMap &qmap,         \
                                     const CUtensorMap &kssmap, const CUtensorMap &vssmap,     \
                                     const GqaParams &p, int ctas, cudaStream_t stream);
DA_GQA_KIND_DECL(bf16)
DA_GQA_KIND_DECL(e4m3)
DA_GQA_KIND_DECL(e4m3_token)
DA_GQA_KIND_DECL(e4m3_mma)
DA_GQA_KIND_DECL(int4)
#undef DA_GQA_KIND_DECL

}  // namespace da

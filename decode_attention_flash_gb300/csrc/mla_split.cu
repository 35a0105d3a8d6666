// mla_split.cu -- split-KV MLA latent decode on 5th-generation tensor cores.
//
// The computation is the MLA decode of FlashInfer
// include/flashinfer/attention/mla.cuh (`BatchMLAPagedAttentionKernel`):
// for every batch row b and each of the 128 query heads,
//   s_n = scale * ([q_nope ; q_pe] . [ckv_n ; kpe_n]),  out = softmax(s) . ckv
// over the row's tokens, read through the block table from a paged latent
// cache (64 tokens per page), split along the tokens with a per-split
// normalised O plus LSE and an LSE-weighted merge (as the GQA kernels do).
//
// GB300 design. A 128-head x 512-wide fp32 output accumulator fills all 512
// columns of one SM's tensor memory, so the work is done by CLUSTERS OF TWO
// CTAs, each owning half of the value dimension (256 TMEM columns of O):
//   * rank r holds q_nope[:, 256r:256r+256] and q_pe[:, 32r:32r+32], and streams
//     ckv[:, 256r:256r+256] and kpe[:, 32r:32r+32] of every page (288 of the 576
//     contraction elements each, so the two score MMAs take equal time).
// Each CTA computes a partial score tile S_r = Q_r K_r^T (128 heads x 64 tokens,
// tcgen05.mma, fp32 in TMEM) over its part of the 576-long contraction, the two
// partials are exchanged through distributed shared memory and added (both
// CTAs then hold the same scores and make the same softmax decisions), and
// each CTA accumulates O_r += P V_r with V_r = the ckv half it already holds in
// shared memory (MN-major operand). Every KV byte is read from HBM once, no
// tensor-core work is repeated, and nothing is multicast.
//
// Persistent schedule: the tiles (pages) of all rows, concatenated, are cut
// into one equal range per cluster (computed on the device from seq_lens), so
// the split of a row is decided by where the cluster boundaries fall. A
// cluster streams its range without draining between rows: at a row boundary
// the new q_nope is written into TMEM once the previous scores are complete,
// and the first PV of the new row overwrites O once the previous row's
// epilogue has read it. A row wholly inside one range is written directly;
// the pieces of a row cut by range boundaries are written as normalised
// partials (O, LSE) to slot row + cluster, and the last piece to finish (a
// per-row counter) merges them after its cluster's stream.
//
// Tensor memory per CTA: O half in columns 0-255, the CTA's 256 q_nope values
// per head in 256-383 (the A operand of the score MMAs), the score tile in
// 384-447 (the next tile's scores are issued as soon as a softmax group has
// read it), and two P tiles (bf16, the A operand of the PV MMAs) in 448-479
// and 480-511, one per softmax group. The kpe part is a shared-memory MMA on
// 64-byte-swizzled tiles (q_pe is a TMA tile).
//
// Warp roles per CTA (352 threads): warp 0 = TMA producer (four KV stages),
// warp 1 = MMA issuer (and TMEM owner), warp 2 = exchange helper, warps 3-10 =
// softmax in two groups of four warps (one warp per TMEM lane quadrant, one
// thread per head row). Group g takes the tiles j = g (mod 2) of the range
// with their own score and exchange buffers, so one group's exchange and
// exponentials overlap the other's; between consecutive tiles each row's
// running maximum and running sum are handed over through shared memory. The
// score exchange uses st.async, whose bytes complete on the receiver's
// mbarrier, so the sender never waits for the remote stores; the helper warp
// returns each buffer to the peer (a cluster-scope release) off the softmax
// warps' path. The online softmax rescales O lazily: only when a row's maximum
// grows by more than 2^8 is the TMEM accumulator rescaled (exact: O is always
// relative to the running maximum, and so is every P tile).
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kTok = 64;          // tokens per tile (= page)
constexpr int kHeads = 128;
constexpr int kSoftmaxWarps = 8;                       // two groups of four
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kGroupThreads = kSoftmaxThreads / 2;      // one thread per head row
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kPvWarp = kFirstSoftmaxWarp + kSoftmaxWarps;  // issues the PV MMAs
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr int kStages = 4;                // KV ring depth
constexpr int kKvBlock = kTok * 128;      // 8 KB: 64 tokens x 64 bf16
constexpr int kKpeBlock = kTok * 64;     // 4 KB: 64 tokens x 32 bf16, 64B-swizzled
constexpr int kKvStage = 4 * kKvBlock + kKpeBlock;  // 4 ckv blocks + the kpe half
constexpr int kQpeBlock = kHeads * 64;   // 8 KB: 128 rows x 32 bf16, 64B-swizzled
constexpr int kXBytes = kHeads * kTok * 3;  // one exchange buffer: 128 x 64 scores, 24 bits each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O half: columns 0..255
constexpr uint32_t kTmemQ = 256;   // q_nope half, two bf16 per column: 256..383
constexpr uint32_t kTmemS = 384;   // score tile: 384..447
constexpr uint32_t kTmemP = 448;   // P tiles of the two groups: 448..479, 480..511
constexpr float kRescaleThreshold = 8.f;
// The schedule weighs a row's start like this many tiles: a row change costs
// a CTA pair ~5 tiles' time (the row's epilogue in one softmax group, which
// holds up the running maximum's hand-off, and the next row's queries into
// TMEM), so equal ranges of tiles alone leave the pairs with more rows behind.
constexpr int kRowCost = 4;

// What the producer tells the other roles about the tile in a KV stage.
struct TileMeta {
  int32_t b, k, nval, flags;  // row, tile of the row, valid tokens, kFirst | kLast | kFullRow
  int32_t c_first, n_seg;     // clusters holding the row's pieces
  int32_t draft0;             // position of the batch row's first new token (seq_len - Q)
  uint32_t tree;              // the query token's draft-tree mask word (all ones: none)
};
enum { kFirst = 1, kLast = 2, kFullRow = 4 };

struct Ctrl {
  uint32_t tmem_base;
  int abort;
  int start_b, start_k;
  long long start_P;
  int npend, nempty, ntiles;
  int pend[4][3];  // rows this CTA merges: b, c_first, n_seg
};

struct Lay {
  static constexpr int QPE = 0;                              // 8 KB
  static constexpr int KV = QPE + kQpeBlock;                 // kStages x 36 KB
  static constexpr int X = KV + kStages * kKvStage;          // 2 x [12][128] uint4
  static constexpr int MR = X + 2 * kXBytes;                 // [2][128] running maximum
  static constexpr int LR = MR + 2 * kHeads * 4;             // [2][128] running sum
  static constexpr int META = LR + 2 * kHeads * 4;           // [kStages] TileMeta
  static constexpr int SCAN = META + kStages * 32;           // [kThreads / 32] + empty rows
  static constexpr int EMPTY = SCAN + 64;                    // [kThreads] rows without tokens
  static constexpr int CTRL = EMPTY + kThreads * 4;
  static constexpr int BAR = CTRL + 128;
  static constexpr int NBAR = 30;
  static constexpr int TOTAL = BAR + NBAR * 8 + 1024;        // + alignment slack
};
enum {
  B_QPE = 0,    // q_pe tile of the current row landed
  B_QT = 1,     // q_nope half of the current row stored in TMEM
  B_KVF = 2,    // [kStages] KV stage full
  B_KVE = 6,    // [kStages] KV stage consumed by the PV MMA
  B_SF = 10,    // [2] score tile of a tile of that parity written (per parity, so
                //     that each group waits on its own tiles' phases only)
  B_SE = 12,    // score tile read (the next one may be written)
  B_PF = 13,    // [2] P of a tile of that parity written (TMEM)
  B_PE = 15,    // [2] PV MMA of a tile of that parity done (its P buffer is free)
  B_XF = 17,    // [2] peer scores landed (local expect_tx + the peer's bytes)
  B_XE = 19,    // [2] the peer has read what this CTA sent into its buffer
  B_XR = 21,    // [2] this CTA's softmax group has read the buffer
  B_MRF = 23,   // [2] group g has published the running maximum of its latest tile
  B_LRF = 25,   // [2] group g has published the running sum of its latest tile
  B_OFREE = 27, // a row's epilogue has read O (the next row may overwrite it)
  B_EPI = 28,   // [2] group g has written a partial (before the row counter counts it)
};

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t mapa_peer(uint32_t smem_addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(rank));
  return d;
}

// Asynchronous store into the peer CTA's shared memory; its 16 bytes are
// counted on the peer's mbarrier (complete_tx), so the sender never waits.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d,
                                            uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          addr),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
      : "memory");
}

__device__ __forceinline__ void st_async_u4(uint32_t addr, uint4 v, uint32_t remote_bar) {
  st_async_v4(addr, __uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
              __uint_as_float(v.w), remote_bar);
}

// Partial scores cross the cluster as the upper three bytes of their fp32
// encoding (sign, exponent, 15 mantissa bits: a relative error below 2^-15,
// far inside the bf16 rounding of the weights they become; NaN and the
// infinities keep their meaning), four scores in three words. DSMEM
// bandwidth limits the exchange; a 16-bit code on per-group steps moved 25 %
// fewer bytes but its encode and decode arithmetic cost more than that saved.
__device__ __forceinline__ void pack24(const float *s, uint32_t *w) {
  const uint32_t a = __float_as_uint(s[0]), b = __float_as_uint(s[1]);
  const uint32_t c = __float_as_uint(s[2]), d = __float_as_uint(s[3]);
  w[0] = prmt(a, b, 0x5321);  // a1 a2 a3 b1
  w[1] = prmt(b, c, 0x6532);  // b2 b3 c1 c2
  w[2] = prmt(c, d, 0x7653);  // c3 d1 d2 d3
}

__device__ __forceinline__ void unpack24_add(const uint32_t *w, float *s) {
  s[0] += __uint_as_float(w[0] << 8);
  s[1] += __uint_as_float(prmt(w[0], w[1], 0x5430) & 0xffffff00u);
  s[2] += __uint_as_float(prmt(w[1], w[2], 0x4320) & 0xffffff00u);
  s[3] += __uint_as_float(w[2] & 0xffffff00u);
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Warp-uniform outcomes of bounded waits (the lanes then stay converged for
// the .sync.aligned tensor-memory instructions that follow).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kWaitLimitNs));
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_cluster_bounded(bar, parity));
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ int cluster_of(int64_t t, int64_t T, int C) {
  return (int)(((t + 1) * C - 1) / T);
}

// Tiles of row b; an out-of-range length is clamped and flagged.
// Batch row of row v = b * Q + t (query token t of batch row b).
__device__ __forceinline__ int batch_of(const MlaParams &p, int v) { return p.q_len == 1 ? v : v / p.q_len; }

// Index of (row v, head h) in the [B][128][Q] layouts of q, out and lse.
__device__ __forceinline__ int64_t head_row(const MlaParams &p, int v, int h) {
  const int b = batch_of(p, v), t = v - b * p.q_len;
  return ((int64_t)b * kHeads + h) * p.q_len + t;
}

// Positions of row v: token t of Q sees n <= seq_lens[b] - Q + t.
__device__ __forceinline__ int row_tiles(const MlaParams &p, int v, int &len, uint32_t &err) {
  const int b = batch_of(p, v);
  int n = p.seq_lens[b];
  if (n < 0 || n > p.capacity) {
    err |= DA_DEVERR_SEQ_LEN;
    n = n < 0 ? 0 : p.capacity;
  }
  n -= p.q_len - 1 - (v - b * p.q_len);
  len = n > 0 ? n : 0;
  return (len + kTok - 1) / kTok;
}

__device__ int block_scan(int v, int *scratch, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int before = 0, sum = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const int t = scratch[w];
    if (w < warp) before += t;
    sum += t;
  }
  __syncthreads();
  *total = sum;
  return v + before;
}

// Merges the n_seg partials of row b (slots b + c_first ..) for value half r:
// LSE-weighted sum of the normalised pieces.
__device__ void mla_merge_row(const MlaParams &p, int b, int r, int c_first, int n_seg,
                              float *scratch) {
  float *w = scratch;                 // [n_seg][128] weights (lse first)
  float *inv = w + n_seg * kHeads;    // [128]
  float *lse_out = inv + kHeads;      // [128]
  const int64_t slot0 = (int64_t)b + c_first;
  for (int i = threadIdx.x; i < n_seg * kHeads; i += blockDim.x) {
    const int s = i / kHeads, h = i % kHeads;
    w[i] = __ldcg(p.lse_part + ((slot0 + s) * 2 + r) * kHeads + h);
  }
  __syncthreads();
  if (threadIdx.x < kHeads) {
    const int h = threadIdx.x;
    float M = neg_inf();
    for (int s = 0; s < n_seg; ++s) M = fmaxf(M, w[s * kHeads + h]);
    float sum = 0.f;
    for (int s = 0; s < n_seg; ++s) {
      const float l = w[s * kHeads + h];
      const float e = l == neg_inf() ? 0.f : ex2((l - M) * 1.4426950408889634f);
      w[s * kHeads + h] = e;
      sum += e;
    }
    inv[h] = sum == 0.f ? 0.f : 1.f / sum;
    lse_out[h] = sum == 0.f ? neg_inf() : M + __log2f(sum) * 0.69314718055994531f;
  }
  __syncthreads();
  // out[b][h][256 r + 4c .. +3] for c < 64: each thread sums 8 float4 outputs
  // at a time, two slots' loads in flight together (the pieces live in L2)
  constexpr int kU = 8;
  const int nthr = blockDim.x;
  for (int base = threadIdx.x; base < kHeads * 64; base += kU * nthr) {
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_seg; s += 2) {
      float4 v0[kU], v1[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = min(base + u * nthr, kHeads * 64 - 1), h = i / 64, c = i % 64;
        const float4 *src = reinterpret_cast<const float4 *>(p.o_part + ((slot0 + s) * kHeads + h) * 512 + r * 256) + c;
        v0[u] = __ldcg(src);
        v1[u] = s + 1 < n_seg ? __ldcg(src + kHeads * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int h = min(base + u * nthr, kHeads * 64 - 1) / 64;
        const float e0 = w[s * kHeads + h], e1 = s + 1 < n_seg ? w[(s + 1) * kHeads + h] : 0.f;
        // a piece with weight 0 (no valid token) may hold anything: skip it
        if (e0 != 0.f) {
          acc[u].x += e0 * v0[u].x;
          acc[u].y += e0 * v0[u].y;
          acc[u].z += e0 * v0[u].z;
          acc[u].w += e0 * v0[u].w;
        }
        if (e1 != 0.f) {
          acc[u].x += e1 * v1[u].x;
          acc[u].y += e1 * v1[u].y;
          acc[u].z += e1 * v1[u].z;
          acc[u].w += e1 * v1[u].w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + u * nthr;
      if (i < kHeads * 64) {
        const int h = i / 64, c = i % 64;
        const float iv = inv[h];
        __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(p.out + head_row(p, b, h) * 512 +
                                                                 r * 256 + 4 * c);
        dst[0] = __floats2bfloat162_rn(acc[u].x * iv, acc[u].y * iv);
        dst[1] = __floats2bfloat162_rn(acc[u].z * iv, acc[u].w * iv);
      }
    }
  }
  if (r == 0 && threadIdx.x < kHeads && p.lse) p.lse[head_row(p, b, threadIdx.x)] = lse_out[threadIdx.x];
  if (threadIdx.x == 0) p.counters[b * 2 + r] = 0u;  // ready for the next call
  __syncthreads();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ CUtensorMap qp_map,
                     const __grid_constant__ CUtensorMap ckv_map,
                     const __grid_constant__ CUtensorMap kpe_map, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Lay::BAR);
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + Lay::CTRL);
  TileMeta *meta = reinterpret_cast<TileMeta *>(smem + Lay::META);
  int *scan = reinterpret_cast<int *>(smem + Lay::SCAN);
  int *empty_rows = reinterpret_cast<int *>(smem + Lay::EMPTY);

  const uint32_t r = cluster_rank();  // 0: value dims 0..255; 1: 256..511 (+ rope part)
  const uint32_t peer = r ^ 1u;
  const int cl = blockIdx.x >> 1, NC = gridDim.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- the cluster's tile range
  uint32_t dev_err = 0;
  // Ranges are cut in cost units: a row with tiles costs kRowCost + its tiles,
  // its tile k sitting at cost position Q_b + kRowCost + k (Q_b the row's
  // start, the prefix of the costs before it); the first kRowCost positions
  // of a row hold no tile. A cluster takes the tiles whose positions fall in
  // its range (possibly none) and the pieces of a row come from the
  // consecutive clusters c_first..c_last.
  int local = 0;
  const int nrows = p.batch * p.q_len;
  for (int b = threadIdx.x; b < nrows; b += kThreads) {
    int len;
    const int t_b = row_tiles(p, b, len, dev_err);
    local += t_b > 0 ? t_b + kRowCost : 0;
  }
  int T32 = 0;
  block_scan(local, scan, &T32);
  const int64_t T = T32;
  const int C = (int)(T < (int64_t)NC ? T : (int64_t)NC);
  const int64_t lo = cl < C ? (int64_t)cl * T / C : 0;
  const int64_t hi = cl < C ? (int64_t)(cl + 1) * T / C : 0;
  const int tail_owner = C > 0 ? C - 1 : 0;  // writes rows without tokens past the last position
  if (threadIdx.x == 0) {
    ctrl->abort = 0;
    ctrl->start_b = -1;
    ctrl->npend = 0;
    ctrl->nempty = 0;
    ctrl->ntiles = 0;
  }
  __syncthreads();
  {
    int64_t base = 0;
    for (int b0 = 0; b0 < nrows; b0 += kThreads) {
      const int b = b0 + threadIdx.x;
      int len = 0;
      uint32_t ignored = 0;
      const int t_b = b < nrows ? row_tiles(p, b, len, ignored) : 0;
      const int c_b = t_b > 0 ? t_b + kRowCost : 0;
      int total = 0;
      const int incl = block_scan(c_b, scan, &total);
      const int64_t Pb = base + incl - c_b;  // the row's start in cost units
      if (b < nrows) {
        if (t_b > 0) {
          if (Pb <= lo && lo < Pb + c_b) {  // the row holding the range's first position
            ctrl->start_b = b;
            ctrl->start_k = lo - Pb > kRowCost ? (int)(lo - Pb - kRowCost) : 0;
            ctrl->start_P = Pb;
          }
          // the row's tiles in this range
          const int64_t t0 = lo > Pb + kRowCost ? lo : Pb + kRowCost, t1 = hi < Pb + c_b ? hi : Pb + c_b;
          if (t1 > t0) atomicAdd(&ctrl->ntiles, (int)(t1 - t0));
        }
        // a row without tokens is written by the cluster whose range holds its start
        if (t_b == 0 && ((Pb >= lo && Pb < hi) || (Pb >= T && cl == tail_owner)))
          empty_rows[atomicAdd(&ctrl->nempty, 1)] = b;
      }
      __syncthreads();
      const int ne = ctrl->nempty;
      for (int e = threadIdx.x; e < ne * kHeads * 32; e += kThreads) {
        // this CTA's value half of the row: zeros; lse = -inf
        const int rb = empty_rows[e / (kHeads * 32)], h = (e / 32) % kHeads, c = e % 32;
        *reinterpret_cast<uint4 *>(p.out + head_row(p, rb, h) * 512 + r * 256 + 8 * c) =
            make_uint4(0, 0, 0, 0);
        if (r == 0 && c == 0 && p.lse) p.lse[head_row(p, rb, h)] = neg_inf();
      }
      __syncthreads();
      if (threadIdx.x == 0) ctrl->nempty = 0;
      base += total;
    }
  }
  __syncthreads();
  const int n = ctrl->ntiles;
  if (cl >= C || n == 0) {  // no tiles for this cluster (both CTAs take this exit)
    if (dev_err) atomicOr(p.err, dev_err);
    return;
  }

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    mbar_init(&bar[B_QPE], 1);
    mbar_init(&bar[B_QT], kGroupThreads);
    mbar_init(&bar[B_OFREE], kGroupThreads);
    mbar_init(&bar[B_SE], kGroupThreads);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar[B_KVF + s], 1);
      mbar_init(&bar[B_KVE + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_PE + s], 1);
      mbar_init(&bar[B_SF + s], 1);
      mbar_init(&bar[B_PF + s], kGroupThreads);
      mbar_init(&bar[B_XF + s], 1);  // the local expect_tx; the bytes come from the peer
      mbar_init(&bar[B_XE + s], 1);  // the peer helper's arrival
      mbar_init(&bar[B_XR + s], kGroupThreads);
      mbar_init(&bar[B_MRF + s], kGroupThreads);
      mbar_init(&bar[B_LRF + s], kGroupThreads);
      mbar_init(&bar[B_EPI + s], kGroupThreads);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  const uint32_t tmem = ctrl->tmem_base;
  volatile int *abort_flag = &ctrl->abort;

  uint8_t *sQpe = smem + Lay::QPE;
  uint8_t *sKV = smem + Lay::KV;
  float *sX = reinterpret_cast<float *>(smem + Lay::X);
  float *sMr = reinterpret_cast<float *>(smem + Lay::MR);
  float *sLr = reinterpret_cast<float *>(smem + Lay::LR);

  int issued_kv = 0, issued_qk = 0, issued_pv = 0, qpe_seg = -1;  // for draining after an abort

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&ckv_map);
      const uint64_t kv_policy = l2_policy_evict_first();
      uint32_t ignored = 0;
      int b = ctrl->start_b, k = ctrl->start_k, len = 0;
      int64_t Pb = ctrl->start_P;
      int t_b = row_tiles(p, b, len, ignored);
      auto row_pieces = [&](int &c_first, int &n_seg, bool &full) {
        c_first = cluster_of(Pb + kRowCost, T, C);
        n_seg = cluster_of(Pb + kRowCost + t_b - 1, T, C) - c_first + 1;
        full = n_seg == 1;
      };
      int c_first, n_seg;
      bool full;
      row_pieces(c_first, n_seg, full);
      // the row's new positions and its query token's tree-mask word (read
      // only when there is a tree mask: the causal cut is the row's length)
      int draft0 = 0;
      uint32_t tree = ~0u;
      auto row_draft = [&] {
        if (!p.spec_mask) return;
        const int bb = batch_of(p, b);
        const int n = min(max(p.seq_lens[bb], 0), p.capacity);
        draft0 = n - p.q_len;
        tree = p.spec_mask[(int64_t)bb * p.q_len + (b - bb * p.q_len)];
      };
      row_draft();
      int page_next = p.block_table[(int64_t)batch_of(p, b) * p.max_pages + k];
      for (int i = 0, st = 0, ph = 0; i < n; ++i) {
        if (i >= kStages && !mbar_wait_bounded(&bar[B_KVE + st], ph ^ 1, kWaitLimitNs)) {
          dev_err |= DA_DEVERR_TIMEOUT;
          *abort_flag = 1;
          break;
        }
        int page = page_next;
        const bool bad = page < 0 || page >= p.num_pages;
        if (bad) dev_err |= DA_DEVERR_PAGE_INDEX;
        TileMeta &m = meta[st];
        m.b = b;
        m.k = k;
        m.nval = bad ? 0 : min(kTok, len - k * kTok);
        m.flags = ((i == 0 || k == 0) ? kFirst : 0) | ((i == n - 1 || k == t_b - 1) ? kLast : 0) |
                  (full ? kFullRow : 0);
        m.c_first = c_first;
        m.n_seg = n_seg;
        m.draft0 = draft0;
        m.tree = tree;
        if (m.flags & kFirst) {
          // the row's queries into L2 ahead of their use at the row's first
          // tile (this CTA's half of q_nope's rows, and its q_pe columns' rows)
          // (all Q tokens' rows of these heads: [64][Q][512] and [64][Q][64])
          const int64_t q0 = ((int64_t)batch_of(p, b) * kHeads + 64 * (int)r) * p.q_len;
          prefetch_l2(p.q_nope + q0 * 512, 64u * p.q_len * 512 * 2);
          prefetch_l2(p.q_pe + q0 * 64, 64u * p.q_len * 64 * 2);
        }
        uint8_t *dst = sKV + st * kKvStage;
        if (bad) {
          // a skipped page: zeros instead of stale data (its scores are masked)
          for (int e = 0; e < kKvStage / 16; ++e)
            reinterpret_cast<uint4 *>(dst)[e] = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&bar[B_KVF + st], 0);
        } else {
          mbar_arrive_expect_tx(&bar[B_KVF + st], (uint32_t)kKvStage);
          for (int c = 0; c < 4; ++c)
            tma_load_2d(dst + c * kKvBlock, &ckv_map, &bar[B_KVF + st], 64 * (4 * (int)r + c),
                        page * kTok, kv_policy);
          tma_load_2d(dst + 4 * kKvBlock, &kpe_map, &bar[B_KVF + st], 32 * (int)r, page * kTok,
                      kv_policy);
        }
        ++issued_kv;
        if (++st == kStages) st = 0, ph ^= 1;
        // the next tile (possibly of the next row with tokens); its page id is
        // fetched now, while this warp waits for a free stage
        if (i + 1 < n) {
          if (++k == t_b) {
            Pb += t_b + kRowCost;
            do {
              ++b;
              t_b = b < nrows ? row_tiles(p, b, len, ignored) : 1;
            } while (t_b == 0);
            k = 0;
            row_pieces(c_first, n_seg, full);
            if (b < nrows) row_draft();
          }
          page_next = b < nrows ? p.block_table[(int64_t)batch_of(p, b) * p.max_pages + k] : -1;
        }
      }
    }
  } else if (warp == 1) {
    // ============================================================ QK issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(128, kTok, false, false);
      const uint64_t q_policy = l2_policy_evict_last();
      // Scores of tile k need its KV stage, the scores of tile k - 1 read out
      // and, on a row's first tile, that row's q (q_nope in TMEM, and q_pe,
      // loaded here once the previous tile's scores -- which read the previous
      // row's q_pe -- are complete). The PV MMAs are issued by their own warp,
      // so a tile's PV never waits behind the next tile's score MMAs.
      int qk_seg = -1;
      bool ok = true;
      for (int k = 0; k < n && ok; ++k) {
        if (*abort_flag) break;
        if (!(ok = mbar_wait_bounded(&bar[B_KVF + k % kStages], (k / kStages) & 1, kWaitLimitNs))) break;
        const TileMeta m = meta[k % kStages];
        const bool first = (m.flags & kFirst) != 0;
        const int seg = first ? qk_seg + 1 : qk_seg;
        if (k >= 1 && !(ok = mbar_wait_bounded(&bar[B_SE], (k - 1) & 1, kWaitLimitNs))) break;
        if (first) {
          if (k >= 1 && !(ok = mbar_wait_bounded(&bar[B_SF + ((k - 1) & 1)], ((k - 1) >> 1) & 1, kWaitLimitNs)))
            break;
          mbar_arrive_expect_tx(&bar[B_QPE], kQpeBlock);
          if (p.q_len == 1) {
            tma_load_2d(sQpe, &qp_map, &bar[B_QPE], 32 * (int)r, m.b * kHeads, q_policy);
          } else {
            const int bb = batch_of(p, m.b);
            tma_load_3d(sQpe, &qp_map, &bar[B_QPE], 32 * (int)r, m.b - bb * p.q_len, bb * kHeads, q_policy);
          }
          qpe_seg = seg;
          if (!(ok = mbar_wait_bounded(&bar[B_QT], seg & 1, kWaitLimitNs))) break;
          if (!(ok = mbar_wait_bounded(&bar[B_QPE], seg & 1, kWaitLimitNs))) break;
        }
        tc_fence_after();
        const uint32_t kv = smem_u32(sKV + (k % kStages) * kKvStage);
        const uint32_t d = tmem + kTmemS;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ts(d, tmem + kTmemQ + 32 * c + 8 * kk,
                         umma_desc_sw128(kv + c * kKvBlock + kk * 32, 16, 1024), idesc_qk,
                         (c | kk) != 0);
        const uint32_t q = smem_u32(sQpe);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          umma_bf16_ss(d, umma_desc_sw64(q + kk * 32), umma_desc_sw64(kv + 4 * kKvBlock + kk * 32),
                       idesc_qk, true);
        umma_commit(&bar[B_SF + (k & 1)]);
        qk_seg = seg;
        ++issued_qk;
      }
      if (!ok) {
        dev_err |= DA_DEVERR_TIMEOUT;
        *abort_flag = 1;
      }
    }
  } else if (warp == kPvWarp) {
    // ============================================================ PV issuer
    // PV of tile j needs its P and, on a row's first tile, the previous row's O
    // read out by that row's epilogue.
    if (lane == 0) {
      const uint32_t idesc_pv = umma_idesc_bf16(128, 256, false, true);
      int pv_seg = -1;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        if (*abort_flag) break;
        if (!(ok = mbar_wait_bounded(&bar[B_PF + (j & 1)], (j >> 1) & 1, kWaitLimitNs))) break;
        const TileMeta m = meta[j % kStages];
        const bool first = (m.flags & kFirst) != 0;
        const int seg = first ? pv_seg + 1 : pv_seg;
        if (first && seg > 0 && !(ok = mbar_wait_bounded(&bar[B_OFREE], (seg - 1) & 1, kWaitLimitNs)))
          break;
        tc_fence_after();
        const int st = j % kStages;
        const uint32_t v = smem_u32(sKV + st * kKvStage);
        const uint32_t pa = tmem + kTmemP + 32 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ts(tmem + kTmemO, pa + 8 * kk, umma_desc_sw128(v + kk * 2048, kKvBlock, 1024),
                       idesc_pv, kk != 0 || !first);
        umma_commit(&bar[B_PE + (j & 1)]);
        umma_commit(&bar[B_KVE + st]);
        pv_seg = seg;
        ++issued_pv;
      }
      if (!ok) {
        dev_err |= DA_DEVERR_TIMEOUT;
        *abort_flag = 1;
      }
    }
  } else if (warp == 2) {
    // ============================================================ exchange helper
    // hands each exchange buffer back to the peer once this CTA has read it
    // (only the buffers the peer still writes into are returned)
    if (lane == 0) {
      const uint32_t peer_xe0 = mapa_peer(smem_u32(&bar[B_XE]), peer);
      for (int j = 0; j + 2 < n; ++j) {
        if (!mbar_wait_bounded(&bar[B_XR + (j & 1)], (j >> 1) & 1, kWaitLimitNs)) {
          dev_err |= DA_DEVERR_TIMEOUT;
          *abort_flag = 1;
          break;
        }
        mbar_arrive_remote(peer_xe0 + 8 * (j & 1));
        if (*abort_flag) break;
      }
    }
  } else {
    // ============================================================ softmax
    const int tid = threadIdx.x - 32 * kFirstSoftmaxWarp;  // 0..255
    const int g = tid >> 7;                                 // group: tiles i = g (mod 2)
    const int quad = warp & 3;                              // TMEM lane quadrant of this warp
    const int h = quad * 32 + lane;                         // head row
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // exchange buffer g: words 4j..4j+3 of head h's 48 packed words sit in the
    // uint4 at [j][h], so one warp-wide store moves 512 contiguous bytes
    const uint32_t peer_x = mapa_peer(smem_u32(sX + g * (kXBytes / 4) + 4 * h), peer);
    const uint32_t peer_xf = mapa_peer(smem_u32(&bar[B_XF + g]), peer);
    const uint4 *my_x = reinterpret_cast<const uint4 *>(sX + g * (kXBytes / 4)) + h;
    const float sscale = p.score_scale;
    bool ok = true;
    int x_next = g;         // first tile of this group whose peer scores have not been waited for
    bool x_posted = false;  // whether its expect_tx has been posted
    int epi = 0;            // partials written by this group (phase of B_EPI + g)
    // q_nope of a row (this CTA's half) into TMEM, the A operand of its score MMAs
    // (two rounds of sixteen 16-byte loads per thread: at the start of a range
    // the row comes from DRAM, and each round is one round trip)
    auto store_q = [&](int b) {
      const uint4 *src =
          reinterpret_cast<const uint4 *>(p.q_nope + head_row(p, b, h) * 512 + 256 * r);
#pragma unroll
      for (int c0 = 0; c0 < 8; c0 += 4) {
        uint4 qv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) qv[e] = __ldg(src + 4 * c0 + e);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[16];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[4 * e] = __uint_as_float(qv[4 * c + e].x);
            v[4 * e + 1] = __uint_as_float(qv[4 * c + e].y);
            v[4 * e + 2] = __uint_as_float(qv[4 * c + e].z);
            v[4 * e + 3] = __uint_as_float(qv[4 * c + e].w);
          }
          tmem_st16(tmem + lane_off + kTmemQ + 16 * (c0 + c), v);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar[B_QT]);
    };
    // the range's first row is known from the schedule: its q goes in at once,
    // while the first KV stage is still in flight
    if (g == 0) store_q(ctrl->start_b);
    for (int i = g; i < n; i += 2) {
      const int ii = i >> 1;  // this group's tile counter (phase of its barriers)
      // the tile's description (its stage cannot be refilled before this tile's PV)
      if (!(ok = warp_wait(&bar[B_KVF + i % kStages], (i / kStages) & 1))) break;
      const TileMeta m = meta[i % kStages];
      const bool first = (m.flags & kFirst) != 0;
      if (first && i > 0) {
        // q_nope of the row into TMEM once the previous tile's scores are complete
        if (!(ok = warp_wait(&bar[B_SF + ((i - 1) & 1)], ((i - 1) >> 1) & 1))) break;
        tc_fence_after();
        store_q(m.b);
      }
      if (!(ok = warp_wait(&bar[B_SF + g], ii & 1))) break;
      tc_fence_after();
      float s[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[16];
        tmem_ld16(tmem + lane_off + kTmemS + 16 * q, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) s[16 * q + e] = v[e];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar[B_SE]);
      // ---- exchange the partial scores with the peer CTA
      if (ii >= 1 && !(ok = warp_wait_cluster(&bar[B_XE + g], (ii - 1) & 1))) break;
      {
        uint32_t w[48];
#pragma unroll
        for (int q = 0; q < 16; ++q) pack24(s + 4 * q, w + 3 * q);
#pragma unroll
        for (int j = 0; j < 12; ++j)
          st_async_u4(peer_x + j * kHeads * 16, make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]),
                      peer_xf);
      }
      // this tile's phase of x_full completes once the peer's 32 KB have landed
      if (tid == kGroupThreads * g) mbar_arrive_expect_tx(&bar[B_XF + g], kXBytes);
      x_posted = true;
      if (!(ok = warp_wait_cluster(&bar[B_XF + g], ii & 1))) break;
      x_next = i + 2;
      x_posted = false;
      {
        uint32_t w[48];
#pragma unroll
        for (int j = 0; j < 12; ++j) {
          const uint4 o = my_x[j * kHeads];
          w[4 * j] = o.x;
          w[4 * j + 1] = o.y;
          w[4 * j + 2] = o.z;
          w[4 * j + 3] = o.w;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) unpack24_add(w + 3 * q, s + 4 * q);
      }
      mbar_arrive(&bar[B_XR + g]);
      // ---- mask and tile maximum
      const int nval = m.nval;
      // the tile's live tokens: the valid ones, less those the query token's
      // draft-tree mask removes among the batch row's last Q positions (a
      // uniform branch: ragged tiles and tiles that reach the new positions)
      const int first_new = kTok * m.k - m.draft0;  // the tile's first token among the new ones
      const bool tree_tile = p.spec_mask != nullptr && first_new > -kTok;
      const bool masked = nval < kTok || tree_tile;
      uint64_t live = ~0ull;
      const float pad = sscale >= 0.f ? neg_inf() : -neg_inf();
      if (masked) {
        live = nval >= kTok ? ~0ull : (1ull << nval) - 1ull;
        if (tree_tile) {
          const uint64_t w = m.tree;
          live &= first_new >= 0 ? (w >> first_new) : ((w << -first_new) | ((1ull << -first_new) - 1ull));
        }
        // raw scores of the other tokens become a value that never wins the
        // extreme below
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (!((live >> k) & 1ull)) s[k] = pad;
      }
      // the scaled maximum is the raw maximum (minimum for a negative scale)
      // times the scale; four independent chains
      float e4[4] = {s[0], s[1], s[2], s[3]};
      if (sscale >= 0.f) {
#pragma unroll
        for (int k = 4; k < 64; ++k) e4[k & 3] = fmaxf(e4[k & 3], s[k]);
      } else {
#pragma unroll
        for (int k = 4; k < 64; ++k) e4[k & 3] = fminf(e4[k & 3], s[k]);
      }
      const float ext = sscale >= 0.f ? fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]))
                                      : fminf(fminf(e4[0], e4[1]), fminf(e4[2], e4[3]));
      const float mt = live != 0ull && nval > 0 ? ext * sscale : neg_inf();
      // ---- running maximum of the row through tile i - 1 (the other group);
      // the hand-off is waited for on a row's first tile too, which keeps the
      // other group's read of this group's previous value ahead of the overwrite
      float m_prev = neg_inf();
      if (i >= 1) {
        if (!(ok = warp_wait(&bar[B_MRF + ((i - 1) & 1)], ((i - 1) >> 1) & 1))) break;
        if (!first) m_prev = sMr[((i - 1) & 1) * kHeads + h];
      }
      const bool need = mt > m_prev + kRescaleThreshold || (m_prev == neg_inf() && mt != neg_inf());
      const float m_new = need ? mt : m_prev;
      sMr[g * kHeads + h] = m_new;
      mbar_arrive(&bar[B_MRF + g]);
      // p = 2^(scale * s - m_new), 0 past the valid tokens and while no score is valid
      const float neg_m = m_new == neg_inf() ? 0.f : -m_new;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
      // (a masked token's padded score times the scale is -inf: the scale is
      // never 0, see the score factor)
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float p0 = ex2(fmaf(s[k], sscale, neg_m)), p1 = ex2(fmaf(s[k + 1], sscale, neg_m));
        ps4[(k >> 1) & 3] += p0 + p1;
        pk[k / 2] = pack_bf16(p0, p1);
      }
      // ---- running sum of the row through tile i, relative to m_new
      float l_prev = 0.f;
      if (i >= 1) {
        if (!(ok = warp_wait(&bar[B_LRF + ((i - 1) & 1)], ((i - 1) >> 1) & 1))) break;
        if (!first) l_prev = sLr[((i - 1) & 1) * kHeads + h];
      }
      const float l_new = (l_prev != 0.f && m_new != m_prev ? l_prev * ex2(m_prev - m_new) : l_prev) +
                          ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));
      sLr[g * kHeads + h] = l_new;
      mbar_arrive(&bar[B_LRF + g]);
      // ---- P into this group's TMEM buffer (the A operand of the tile's PV),
      // free once the PV of the group's previous tile is done
      if (i >= 2 && !(ok = warp_wait(&bar[B_PE + g], ((i >> 1) - 1) & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(pk[16 * c + e]);
        tmem_st16(tmem + lane_off + kTmemP + 32 * g + 16 * c, v);
      }
      // ---- a grown maximum rescales O, after the PV of the previous tile
      if (!first && __any_sync(0xffffffffu, need)) {
        if (!(ok = warp_wait(&bar[B_PE + ((i - 1) & 1)], ((i - 1) >> 1) & 1))) break;
        tc_fence_after();
        const float alpha = need ? ex2(m_prev - m_new) : 1.f;  // 0 when m_prev is -inf
        for (int c = 0; c < 256; c += 16) {
          float v[16];
          tmem_ld16(tmem + lane_off + kTmemO + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= alpha;
          tmem_st16(tmem + lane_off + kTmemO + c, v);
        }
      }
      tmem_wait_st();
      if (nval < kTok) {
        // value rows past the valid tokens may hold anything: zero them
        uint8_t *kv = sKV + (i % kStages) * kKvStage;
        for (int e = tid - kGroupThreads * g; e < (kTok - nval) * 4 * 8; e += kGroupThreads) {
          const int t = nval + e / 32, blk = (e / 8) % 4, c = e % 8;
          *reinterpret_cast<uint4 *>(kv + blk * kKvBlock + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&bar[B_PF + g]);
      if (m.flags & kLast) {
        // ---- end of the row's piece: O / l of this value half
        if (!(ok = warp_wait(&bar[B_PE + (i & 1)], (i >> 1) & 1))) break;
        tc_fence_after();
        const bool full = (m.flags & kFullRow) != 0;
        // no valid token: 0 and -inf; a NaN among the weights reaches both
        const float inv = l_new == 0.f ? 0.f : 1.f / l_new;
        const float lse = l_new == 0.f ? neg_inf() : (m_new + __log2f(l_new)) * 0.69314718055994531f;
        const int64_t slot = (int64_t)m.b + cl;
        for (int c0 = 0; c0 < 256; c0 += 128) {
          float v[128];  // eight loads per wait
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float t[16];
            tmem_ld16(tmem + lane_off + kTmemO + c0 + 16 * q, t);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[16 * q + e] = t[e];
          }
          tmem_wait_ld();
          if (full) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + head_row(p, m.b, h) * 512 + r * 256 + c0);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              dst[e] = make_uint4(pack_bf16(v[8 * e] * inv, v[8 * e + 1] * inv),
                                  pack_bf16(v[8 * e + 2] * inv, v[8 * e + 3] * inv),
                                  pack_bf16(v[8 * e + 4] * inv, v[8 * e + 5] * inv),
                                  pack_bf16(v[8 * e + 6] * inv, v[8 * e + 7] * inv));
          } else {
            float4 *dst = reinterpret_cast<float4 *>(p.o_part + (slot * kHeads + h) * 512 + r * 256 + c0);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              dst[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
          }
        }
        tc_fence_before();
        mbar_arrive(&bar[B_OFREE]);
        if (full) {
          if (r == 0 && p.lse) p.lse[head_row(p, m.b, h)] = lse;
        } else {
          p.lse_part[(slot * 2 + r) * kHeads + h] = lse;
          // the whole piece is in global memory before the row's counter counts it
          mbar_arrive(&bar[B_EPI + g]);
          if (!(ok = warp_wait(&bar[B_EPI + g], epi & 1))) break;
          ++epi;
          if (tid == kGroupThreads * g) {
            const uint32_t prev = atomic_add_acq_rel_gpu(p.counters + m.b * 2 + r, 1u);
            if (prev == (uint32_t)(m.n_seg - 1)) {
              const int q = atomicAdd(&ctrl->npend, 1);
              ctrl->pend[q][0] = m.b;
              ctrl->pend[q][1] = m.c_first;
              ctrl->pend[q][2] = m.n_seg;
            }
          }
        }
      }
    }
    if (!ok) {
      dev_err |= DA_DEVERR_TIMEOUT;
      *abort_flag = 1;
      // the peer may still be storing the scores of tile x_next into this
      // group's buffer (it cannot start the group's next one): let them land
      if (tid == kGroupThreads * g && x_next < n) {
        if (!x_posted) mbar_arrive_expect_tx(&bar[B_XF + g], kXBytes);
        mbar_wait_cluster_bounded(&bar[B_XF + g], (x_next >> 1) & 1);
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // drain what is still in flight (bounded), so nothing lands after exit
    if (warp == 0 && lane == 0) {
      for (int j = max(0, issued_kv - kStages); j < issued_kv; ++j)
        mbar_wait_bounded(&bar[B_KVF + j % kStages], (j / kStages) & 1, kWaitLimitNs);
    }
    if (warp == 1 && lane == 0) {
      if (issued_qk > 0)
        mbar_wait_bounded(&bar[B_SF + ((issued_qk - 1) & 1)], ((issued_qk - 1) >> 1) & 1, kWaitLimitNs);
      if (qpe_seg >= 0) mbar_wait_bounded(&bar[B_QPE], qpe_seg & 1, kWaitLimitNs);
    }
    if (warp == kPvWarp && lane == 0 && issued_pv > 0)
      mbar_wait_bounded(&bar[B_PE + ((issued_pv - 1) & 1)], ((issued_pv - 1) >> 1) & 1, kWaitLimitNs);
    __syncthreads();
  }
  if (dev_err) atomicOr(p.err, dev_err | (*abort_flag ? DA_DEVERR_TIMEOUT : 0u));
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (*abort_flag) return;
  // ---- rows whose last piece finished here: merge them (this value half)
  const int npend = ctrl->npend;
  for (int q = 0; q < npend; ++q)
    mla_merge_row(p, ctrl->pend[q][0], (int)r, ctrl->pend[q][1], ctrl->pend[q][2],
                  reinterpret_cast<float *>(smem + Lay::KV));
}

}  // namespace

int mla_smem_bytes() { return Lay::TOTAL; }
int mla_threads() { return kThreads; }

cudaError_t mla_prepare(int /*device*/) {
  return cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Lay::TOTAL);
}

cudaError_t launch_mla(const CUtensorMap &qp_map, const CUtensorMap &ckv_map,
                       const CUtensorMap &kpe_map, const MlaParams &p, dim3 grid,
                       cudaStream_t stream) {
  mla_split_kernel<<<grid, kThreads, Lay::TOTAL, stream>>>(qp_map, ckv_map, kpe_map, p);
  return cudaGetLastError();
}

}  // namespace da

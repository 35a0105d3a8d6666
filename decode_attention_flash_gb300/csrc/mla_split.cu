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
// columns of one SM's tensor memory, so one (b, split) is handled by a CLUSTER
// OF TWO CTAs, each owning half of the value dimension (256 TMEM columns of O):
//   * rank 0 holds q_nope[:, 0:256] and streams ckv[:, 0:256] of every page;
//   * rank 1 holds q_nope[:, 256:512] and q_pe, and streams ckv[:, 256:512] and kpe.
// Each CTA computes a partial score tile S_r = Q_r K_r^T (128 heads x 64 tokens,
// tcgen05.mma, fp32 in TMEM) over its part of the 576-long contraction, the two
// partials are exchanged through distributed shared memory and added (both
// CTAs then hold the same scores and make the same softmax decisions), and
// each CTA accumulates O_r += P V_r with V_r = the ckv half it already holds in
// shared memory (MN-major operand). Every KV byte is read from HBM once, no
// tensor-core work is repeated, and nothing is multicast.
//
// Tensor memory per CTA: O half in columns 0-255, the CTA's 256 q_nope values
// per head in 256-383 (the A operand of the score MMAs, read from TMEM so that
// only the 2 KB K slice of each MMA comes from shared memory), two score
// buffers in 384-447 and 448-511. The kpe block of rank 1 is an ordinary
// shared-memory MMA (q_pe is a TMA tile).
//
// Warp roles per CTA (352 threads): warp 0 = TMA producer (three KV stages),
// warp 1 = MMA issuer (and TMEM owner), warp 2 = exchange helper, warps 3-10 =
// softmax in two groups of four warps (one warp per TMEM lane quadrant, one
// thread per head row). Group g takes the tiles j = g (mod 2) with their own
// score buffer and exchange buffer, so one group's exchange and exponentials
// overlap the other's; the only hand-over between consecutive tiles is the
// running maximum of each row (shared memory + mbarrier), and each group keeps
// its part of the row sum relative to the maximum of its own latest tile.
// The score exchange uses st.async, whose bytes complete on the receiver's
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
constexpr int kThreads = 32 * (kFirstSoftmaxWarp + kSoftmaxWarps);
constexpr int kStages = 3;                // KV ring depth
constexpr int kQBlock = kHeads * 128;     // 16 KB: 128 rows x 64 bf16, 128B-swizzled
constexpr int kKvBlock = kTok * 128;      // 8 KB: 64 tokens x 64 bf16
constexpr int kKvStage = 5 * kKvBlock;    // 4 ckv blocks (+ kpe on rank 1)
constexpr int kXBytes = kHeads * kTok * 4;  // one exchange buffer: 128 x 64 fp32
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O half: columns 0..255
constexpr uint32_t kTmemQ = 256;   // q_nope half, two bf16 per column: 256..383
constexpr uint32_t kTmemS = 384;   // two score buffers: 384..447, 448..511
constexpr float kRescaleThreshold = 8.f;
constexpr int kMaxMlaSplits = 32;

struct Lay {
  static constexpr int QPE = 0;                              // 16 KB (rank 1)
  static constexpr int KV = QPE + kQBlock;                   // kStages x 40 KB
  static constexpr int P = KV + kStages * kKvStage;          // 16 KB
  static constexpr int X = P + kQBlock;                      // 2 x [16][128] float4
  static constexpr int MR = X + 2 * kXBytes;                 // [2 groups][128] running max
  static constexpr int FIN = MR + 2 * kHeads * 4;            // [2 groups][l, m][128]
  static constexpr int BAR = FIN + 2 * 2 * kHeads * 4;
  static constexpr int NBAR = 24;
  static constexpr int FLAGS = BAR + NBAR * 8;               // tmem base, abort, last
  static constexpr int IDS = FLAGS + 16;
  static constexpr int TOTAL = IDS + kGqaMaxIds * 4 + 1024;  // + alignment slack
};
enum {
  B_QPE = 0,   // q_pe tile landed (rank 1)
  B_QT = 1,    // q_nope half stored in TMEM (one arrival per softmax thread)
  B_KVF = 2,   // [kStages] KV stage full
  B_KVE = 5,   // [kStages] KV stage consumed by the PV MMA
  B_SF = 8,    // [2] score buffer written
  B_SE = 10,   // [2] score buffer read
  B_PF = 12,   // P tile written
  B_PE = 13,   // PV MMA done
  B_XF = 14,   // [2] peer scores landed (local expect_tx + the peer's bytes)
  B_XE = 16,   // [2] the peer has read what this CTA sent into its buffer
  B_XR = 18,   // [2] this CTA's softmax group has read the buffer
  B_MRF = 20,  // [2] group g has published the running maximum of its latest tile
  B_FIN = 22,  // both groups have published their row sums
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

// Non-blocking check of a phase (the MMA issuer polls several barriers).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
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

// Last CTA of rank r for batch row b merges that row's splits for its value half.
__device__ void mla_merge_if_last(const MlaParams &p, int b, int r, float *scratch,
                                  volatile int *last_flag) {
  const int S = p.num_splits;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(p.counters + b * 2 + r, 1u);
    *last_flag = (prev == (unsigned)(S - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!*last_flag) return;
  __threadfence();
  float *w = scratch;             // [S][128] weights (lse first)
  float *inv = w + S * kHeads;    // [128]
  float *lse_out = inv + kHeads;  // [128]
  for (int i = threadIdx.x; i < S * kHeads; i += blockDim.x) {
    const int s = i / kHeads, h = i % kHeads;
    w[i] = __ldcg(p.lse_part + (((int64_t)b * S + s) * 2 + r) * kHeads + h);
  }
  __syncthreads();
  if (threadIdx.x < kHeads) {
    const int h = threadIdx.x;
    float M = neg_inf();
    for (int s = 0; s < S; ++s) M = fmaxf(M, w[s * kHeads + h]);
    float sum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float l = w[s * kHeads + h];
      const float e = (M == neg_inf() || l == neg_inf()) ? 0.f : ex2((l - M) * 1.4426950408889634f);
      w[s * kHeads + h] = e;
      sum += e;
    }
    inv[h] = sum > 0.f ? 1.f / sum : 0.f;
    lse_out[h] = sum > 0.f ? M + __log2f(sum) * 0.69314718055994531f : neg_inf();
  }
  __syncthreads();
  // out[b][h][256 r + 4c .. +3] for c < 64
  for (int i = threadIdx.x; i < kHeads * 64; i += blockDim.x) {
    const int h = i / 64, c = i % 64;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float e = w[s * kHeads + h];
      if (e != 0.f) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                    p.o_part + (((int64_t)b * S + s) * kHeads + h) * 512 + r * 256) +
                                c);
        acc.x += e * v.x;
        acc.y += e * v.y;
        acc.z += e * v.z;
        acc.w += e * v.w;
      }
    }
    const float iv = inv[h];
    __nv_bfloat162 *dst =
        reinterpret_cast<__nv_bfloat162 *>(p.out + ((int64_t)b * kHeads + h) * 512 + r * 256 + 4 * c);
    dst[0] = __floats2bfloat162_rn(acc.x * iv, acc.y * iv);
    dst[1] = __floats2bfloat162_rn(acc.z * iv, acc.w * iv);
  }
  if (r == 0 && threadIdx.x < kHeads && p.lse) p.lse[(int64_t)b * kHeads + threadIdx.x] = lse_out[threadIdx.x];
  if (threadIdx.x == 0) p.counters[b * 2 + r] = 0u;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ CUtensorMap qp_map,
                     const __grid_constant__ CUtensorMap ckv_map,
                     const __grid_constant__ CUtensorMap kpe_map, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Lay::BAR);
  volatile uint32_t *tmem_base_slot = reinterpret_cast<volatile uint32_t *>(smem + Lay::FLAGS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Lay::FLAGS + 4);
  volatile int *last_flag = reinterpret_cast<volatile int *>(smem + Lay::FLAGS + 8);
  int *ids = reinterpret_cast<int *>(smem + Lay::IDS);

  const uint32_t r = cluster_rank();  // 0: value dims 0..255; 1: 256..511 (+ rope part)
  const uint32_t peer = r ^ 1u;
  const int split = blockIdx.x >> 1, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = r == 0 ? 4 : 5;  // 64-wide KV blocks this CTA streams

  uint32_t dev_err = 0;
  int n_valid = p.seq_lens[b];
  if (n_valid < 0 || n_valid > p.capacity) {
    dev_err |= DA_DEVERR_SEQ_LEN;
    n_valid = n_valid < 0 ? 0 : p.capacity;
  }
  const int range_lo = split * p.chunk;
  const int range_hi = min(range_lo + p.chunk, n_valid);
  const int num_tiles = range_hi > range_lo ? (range_hi - range_lo + kTok - 1) / kTok : 0;
  const int64_t slot = (int64_t)b * p.num_splits + split;

  if (num_tiles == 0) {
    if (threadIdx.x == 0 && dev_err) atomicOr(p.err, dev_err);
    if (p.write_final) {
      for (int e = threadIdx.x; e < kHeads * 256; e += blockDim.x) {
        const int h = e / 256, d = e % 256;
        p.out[((int64_t)b * kHeads + h) * 512 + r * 256 + d] = __float2bfloat16(0.f);
      }
      if (r == 0 && p.lse && threadIdx.x < kHeads) p.lse[(int64_t)b * kHeads + threadIdx.x] = neg_inf();
      return;
    }
    if (threadIdx.x < kHeads) p.lse_part[(slot * 2 + r) * kHeads + threadIdx.x] = neg_inf();
    mla_merge_if_last(p, b, r, reinterpret_cast<float *>(smem + Lay::KV), last_flag);
    return;
  }

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    mbar_init(&bar[B_QPE], 1);
    mbar_init(&bar[B_QT], kSoftmaxThreads);
    mbar_init(&bar[B_FIN], kSoftmaxThreads);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar[B_KVF + s], 1);
      mbar_init(&bar[B_KVE + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_SF + s], 1);
      mbar_init(&bar[B_SE + s], kGroupThreads);
      mbar_init(&bar[B_XF + s], 1);  // the local expect_tx; the bytes come from the peer
      mbar_init(&bar[B_XE + s], 1);  // the peer helper's arrival
      mbar_init(&bar[B_XR + s], kGroupThreads);
      mbar_init(&bar[B_MRF + s], kGroupThreads);
    }
    mbar_init(&bar[B_PF], kGroupThreads);
    mbar_init(&bar[B_PE], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // page ids of this split, checked against the pool
    const int first = range_lo / kTok;
    const int32_t *row = p.block_table + (int64_t)b * p.max_pages + first;
    for (int j = lane; j < num_tiles; j += 32) {
      int page = row[j];
      if (page < 0 || page >= p.num_pages) {
        dev_err |= DA_DEVERR_PAGE_INDEX;
        page = -1;
      }
      ids[j] = page;
    }
  }
  if (warp == 1) {
    tmem_alloc(const_cast<uint32_t *>(tmem_base_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  const uint32_t tmem = *tmem_base_slot;

  uint8_t *sQpe = smem + Lay::QPE;
  uint8_t *sKV = smem + Lay::KV;
  uint8_t *sP = smem + Lay::P;
  float *sX = reinterpret_cast<float *>(smem + Lay::X);
  float *sMr = reinterpret_cast<float *>(smem + Lay::MR);
  float *sFin = reinterpret_cast<float *>(smem + Lay::FIN);

  int issued_kv = 0, issued_qk = 0, issued_pv = 0;  // for draining after an abort

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&ckv_map);
      const uint64_t kv_policy = l2_policy_evict_first();
      if (r == 1) {
        mbar_arrive_expect_tx(&bar[B_QPE], kQBlock);
        tma_load_2d(sQpe, &qp_map, &bar[B_QPE], 0, b * kHeads, l2_policy_evict_last());
      }
      for (int j = 0, st = 0, ph = 0; j < num_tiles; ++j) {
        if (j >= kStages && !mbar_wait_bounded(&bar[B_KVE + st], ph ^ 1, kWaitLimitNs)) {
          dev_err |= DA_DEVERR_TIMEOUT;
          *abort_flag = 1;
          break;
        }
        uint8_t *dst = sKV + st * kKvStage;
        const int page = ids[j];
        if (page < 0) {
          // a skipped page: zeros instead of stale data (its scores are masked)
          for (int i = 0; i < nkb * kKvBlock / 16; ++i)
            reinterpret_cast<uint4 *>(dst)[i] = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&bar[B_KVF + st], 0);
        } else {
          mbar_arrive_expect_tx(&bar[B_KVF + st], (uint32_t)nkb * kKvBlock);
          for (int c = 0; c < 4; ++c)
            tma_load_2d(dst + c * kKvBlock, &ckv_map, &bar[B_KVF + st], 64 * (4 * (int)r + c),
                        page * kTok, kv_policy);
          if (r == 1)
            tma_load_2d(dst + 4 * kKvBlock, &kpe_map, &bar[B_KVF + st], 0, page * kTok, kv_policy);
        }
        ++issued_kv;
        if (++st == kStages) st = 0, ph ^= 1;
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(128, kTok, false, false);
      const uint32_t idesc_pv = umma_idesc_bf16(128, 256, false, true);
      bool ok = mbar_wait_bounded(&bar[B_QT], 0, kWaitLimitNs);
      if (ok && r == 1) ok = mbar_wait_bounded(&bar[B_QPE], 0, kWaitLimitNs);
      // Scores of tile k need its KV stage and the score buffer read back from
      // tile k - 2; PV of tile k needs its P. Neither waits for the other: the
      // issuer polls both and issues what is ready, so the next scores are in
      // flight while a softmax group still works on the previous tile. (No
      // barrier polled here can run a phase ahead of the tile being tested.)
      uint64_t idle_since = 0;
      while (ok && issued_pv < num_tiles) {
        if (*abort_flag) break;
        bool progress = false;
        const int k = issued_qk;
        if (k < num_tiles && mbar_test(&bar[B_KVF + k % kStages], (k / kStages) & 1) &&
            (k < 2 || mbar_test(&bar[B_SE + (k & 1)], ((k >> 1) - 1) & 1))) {
          tc_fence_after();
          const uint32_t kv = smem_u32(sKV + (k % kStages) * kKvStage);
          const uint32_t d = tmem + kTmemS + 64 * (k & 1);
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ts(d, tmem + kTmemQ + 32 * c + 8 * kk,
                           umma_desc_sw128(kv + c * kKvBlock + kk * 32, 16, 1024), idesc_qk,
                           (c | kk) != 0);
          if (r == 1) {
            const uint32_t q = smem_u32(sQpe);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ss(d, umma_desc_sw128(q + kk * 32, 16, 1024),
                           umma_desc_sw128(kv + 4 * kKvBlock + kk * 32, 16, 1024), idesc_qk, true);
          }
          umma_commit(&bar[B_SF + (k & 1)]);
          ++issued_qk;
          progress = true;
        }
        const int j = issued_pv;
        if (j < issued_qk && mbar_test(&bar[B_PF], j & 1)) {
          tc_fence_after();
          const int st = j % kStages;
          const uint32_t v = smem_u32(sKV + st * kKvStage);
          const uint32_t pa = smem_u32(sP);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ss(tmem + kTmemO, umma_desc_sw128(pa + kk * 32, 16, 1024),
                         umma_desc_sw128(v + kk * 2048, kKvBlock, 1024), idesc_pv, (j | kk) != 0);
          umma_commit(&bar[B_PE]);
          umma_commit(&bar[B_KVE + st]);
          ++issued_pv;
          progress = true;
        }
        if (progress) {
          idle_since = 0;
        } else {
          const uint64_t now = global_timer_ns();
          if (idle_since == 0) idle_since = now;
          else if (now - idle_since > kWaitLimitNs) ok = false;
        }
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
      for (int j = 0; j + 2 < num_tiles; ++j) {
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
    const int g = tid >> 7;                                 // group: tiles j = g (mod 2)
    const int quad = warp & 3;                              // TMEM lane quadrant of this warp
    const int h = quad * 32 + lane;                         // head row
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // this CTA's q_nope half of row h into TMEM: group g stores columns
    // kTmemQ + 64 g .. + 63 (values 128 g .. 128 g + 127 of the half)
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(p.q_nope + ((int64_t)b * kHeads + h) * 512 +
                                                         256 * r + 128 * g);
      uint4 qv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) qv[i] = __ldg(src + i);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[4 * i] = __uint_as_float(qv[4 * c + i].x);
          v[4 * i + 1] = __uint_as_float(qv[4 * c + i].y);
          v[4 * i + 2] = __uint_as_float(qv[4 * c + i].z);
          v[4 * i + 3] = __uint_as_float(qv[4 * c + i].w);
        }
        tmem_st16(tmem + lane_off + kTmemQ + 64 * g + 16 * c, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar[B_QT]);
    }
    // exchange buffer g: the float4 holding scores 4q..4q+3 of head h sits at
    // [q][h], so one warp-wide store moves 512 contiguous bytes
    const uint32_t peer_x = mapa_peer(smem_u32(sX + g * (kXBytes / 4) + 4 * h), peer);
    const uint32_t peer_xf = mapa_peer(smem_u32(&bar[B_XF + g]), peer);
    const float4 *my_x = reinterpret_cast<const float4 *>(sX + g * (kXBytes / 4)) + h;
    const float sscale = p.score_scale;
    // m_last: running maximum after this group's latest tile (scaled, log2
    // units); l: this group's part of the row sum, relative to m_last
    float m_last = neg_inf(), l = 0.f;
    bool ok = true;
    int x_next = g;         // first tile of this group whose peer scores have not been waited for
    bool x_posted = false;  // whether its expect_tx has been posted
    for (int j = g; j < num_tiles; j += 2) {
      const int i = j >> 1;  // this group's tile counter (phase of its barriers)
      if (!(ok = warp_wait(&bar[B_SF + g], i & 1))) break;
      tc_fence_after();
      float s[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[16];
        tmem_ld16(tmem + lane_off + kTmemS + 64 * g + 16 * q, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) s[16 * q + e] = v[e];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar[B_SE + g]);
      // ---- exchange the partial scores with the peer CTA
      if (i >= 1 && !(ok = warp_wait_cluster(&bar[B_XE + g], (i - 1) & 1))) break;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        st_async_v4(peer_x + q * kHeads * 16, s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3],
                    peer_xf);
      // this tile's phase of x_full completes once the peer's 32 KB have landed
      if (tid == kGroupThreads * g) mbar_arrive_expect_tx(&bar[B_XF + g], kXBytes);
      x_posted = true;
      if (!(ok = warp_wait_cluster(&bar[B_XF + g], i & 1))) break;
      x_next = j + 2;
      x_posted = false;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 o = my_x[q * kHeads];
        s[4 * q] += o.x;
        s[4 * q + 1] += o.y;
        s[4 * q + 2] += o.z;
        s[4 * q + 3] += o.w;
      }
      mbar_arrive(&bar[B_XR + g]);
      // ---- mask and tile maximum
      const int tok0 = range_lo + j * kTok;
      const int nval = ids[j] < 0 ? 0 : min(kTok, range_hi - tok0);
      // raw scores past the valid tokens become a value that never wins the
      // extreme below (uniform branch: ragged tiles only)
      const float pad = sscale >= 0.f ? neg_inf() : -neg_inf();
      if (nval < kTok) {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= nval) s[k] = pad;
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
      const float mt = nval > 0 ? ext * sscale : neg_inf();
      // ---- running maximum: that of tile j - 1 (the other group) grows lazily
      float m_prev = neg_inf();
      if (j >= 1) {
        const int jp = j - 1;
        if (!(ok = warp_wait(&bar[B_MRF + (jp & 1)], (jp >> 1) & 1))) break;
        m_prev = sMr[(jp & 1) * kHeads + h];
      }
      const bool need = mt > m_prev + kRescaleThreshold || (m_prev == neg_inf() && mt != neg_inf());
      const float m_new = need ? mt : m_prev;
      sMr[g * kHeads + h] = m_new;
      mbar_arrive(&bar[B_MRF + g]);
      // p = 2^(scale * s - m_new), 0 past the valid tokens and while no score is valid
      const float neg_m = m_new == neg_inf() ? 0.f : -m_new;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
      auto exp_pack = [&](auto ragged) {
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          float t0 = fmaf(s[k], sscale, neg_m), t1 = fmaf(s[k + 1], sscale, neg_m);
          if (decltype(ragged)::value) {
            t0 = k < nval ? t0 : neg_inf();
            t1 = k + 1 < nval ? t1 : neg_inf();
          }
          const float p0 = ex2(t0), p1 = ex2(t1);
          ps4[(k >> 1) & 3] += p0 + p1;
          pk[k / 2] = pack_bf16(p0, p1);
        }
      };
      if (nval < kTok) exp_pack(std::true_type{});
      else exp_pack(std::false_type{});
      if (l != 0.f && m_new != m_last) l *= ex2(m_last - m_new);
      l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      m_last = m_new;
      // ---- PV of the previous tile must be done before O or P change
      if (j >= 1 && !(ok = warp_wait(&bar[B_PE], (j - 1) & 1))) break;
      tc_fence_after();
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m_prev - m_new) : 1.f;  // 0 when m_prev is -inf
        for (int c = 0; c < 256; c += 16) {
          float v[16];
          tmem_ld16(tmem + lane_off + kTmemO + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= alpha;
          tmem_st16(tmem + lane_off + kTmemO + c, v);
        }
        tmem_wait_st();
      }
      // P row h (bf16, 64 tokens = 128 bytes), 128B-swizzled K-major A operand
      uint8_t *prow = sP + h * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(prow + ((c ^ (h & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (nval < kTok) {
        // value rows past the valid tokens may hold anything: zero them
        uint8_t *kv = sKV + (j % kStages) * kKvStage;
        for (int e = tid - kGroupThreads * g; e < (kTok - nval) * 4 * 8; e += kGroupThreads) {
          const int t = nval + e / 32, blk = (e / 8) % 4, c = e % 8;
          *reinterpret_cast<uint4 *>(kv + blk * kKvBlock + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar[B_PF]);
    }
    if (!ok) {
      dev_err |= DA_DEVERR_TIMEOUT;
      *abort_flag = 1;
      // the peer may still be storing the scores of tile x_next into this
      // group's buffer (it cannot start the group's next one): let them land
      if (tid == kGroupThreads * g && x_next < num_tiles) {
        if (!x_posted) mbar_arrive_expect_tx(&bar[B_XF + g], kXBytes);
        mbar_wait_cluster_bounded(&bar[B_XF + g], (x_next >> 1) & 1);
      }
    }
    // ---- epilogue: O_r / l for this CTA's value half (group g: columns 128 g ..)
    if (ok && warp_wait(&bar[B_PE], (num_tiles - 1) & 1)) {
      tc_fence_after();
      sFin[g * 2 * kHeads + h] = l;
      sFin[g * 2 * kHeads + kHeads + h] = m_last;
      mbar_arrive(&bar[B_FIN]);
      if (warp_wait(&bar[B_FIN], 0)) {
        // both groups' sums relative to the final maximum, added in one order
        const float l0 = sFin[h], m0 = sFin[kHeads + h];
        const float l1 = sFin[2 * kHeads + h], m1 = sFin[3 * kHeads + h];
        const float mf = fmaxf(m0, m1);
        const float lt = (l0 != 0.f ? l0 * ex2(m0 - mf) : 0.f) + (l1 != 0.f ? l1 * ex2(m1 - mf) : 0.f);
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float lse = lt > 0.f ? (mf + __log2f(lt)) * 0.69314718055994531f : neg_inf();
        for (int c = 0; c < 128; c += 16) {
          float v[16];
          tmem_ld16(tmem + lane_off + kTmemO + 128 * g + c, v);
          tmem_wait_ld();
          const int col = r * 256 + 128 * g + c;
          if (p.write_final) {
            __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
                p.out + ((int64_t)b * kHeads + h) * 512 + col);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = __floats2bfloat162_rn(v[2 * e] * inv, v[2 * e + 1] * inv);
          } else {
            float4 *dst = reinterpret_cast<float4 *>(p.o_part + (slot * kHeads + h) * 512 + col);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
          }
        }
        if (g == 0) {
          if (p.write_final) {
            if (r == 0 && p.lse) p.lse[(int64_t)b * kHeads + h] = lse;
          } else {
            p.lse_part[(slot * 2 + r) * kHeads + h] = lse;
          }
        }
      } else {
        dev_err |= DA_DEVERR_TIMEOUT;
        *abort_flag = 1;
      }
    } else if (ok) {
      dev_err |= DA_DEVERR_TIMEOUT;
      *abort_flag = 1;
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
      if (issued_pv > 0) mbar_wait_bounded(&bar[B_PE], (issued_pv - 1) & 1, kWaitLimitNs);
    }
    __syncthreads();
  }
  if (dev_err) atomicOr(p.err, dev_err | (*abort_flag ? DA_DEVERR_TIMEOUT : 0u));
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (*abort_flag) return;
  if (!p.write_final) mla_merge_if_last(p, b, (int)r, reinterpret_cast<float *>(smem + Lay::KV), last_flag);
}

}  // namespace

int mla_smem_bytes() { return Lay::TOTAL; }
int mla_threads() { return kThreads; }
int mla_max_splits() { return kMaxMlaSplits; }

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

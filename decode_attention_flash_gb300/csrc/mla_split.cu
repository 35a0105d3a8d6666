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
// Warp roles per CTA (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer
// (and TMEM owner), warps 2-5 = softmax (one thread per head row: the TMEM
// lane layout gives each thread a whole score row, so no shuffles). The
// online softmax rescales O lazily: only when a row's maximum grows by more
// than 2^8 is the TMEM accumulator rescaled (exact: O and l always share the
// same reference maximum).
#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kTok = 64;          // tokens per tile (= page)
constexpr int kHeads = 128;
constexpr int kThreads = 192;
constexpr int kQBlock = kHeads * 128;  // 16 KB: 128 rows x 64 bf16, 128B-swizzled
constexpr int kKvBlock = kTok * 128;   // 8 KB: 64 tokens x 64 bf16
constexpr int kXStride = 68;           // floats per row of the score exchange buffer
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;         // O half: columns 0..255
constexpr uint32_t kTmemS = 256;       // two score buffers: 256..319, 320..383
constexpr float kRescaleThreshold = 8.f;
constexpr int kMaxMlaSplits = 32;

struct Lay {
  static constexpr int Q = 0;                                // 5 x 16 KB
  static constexpr int KV = Q + 5 * kQBlock;                 // 2 stages x 5 x 8 KB
  static constexpr int P = KV + 2 * 5 * kKvBlock;            // 16 KB
  static constexpr int X = P + kQBlock;                      // 128 x 68 fp32
  static constexpr int BAR = X + kHeads * kXStride * 4;
  static constexpr int NBAR = 13;
  static constexpr int FLAGS = BAR + NBAR * 8;               // tmem base, abort, last
  static constexpr int IDS = FLAGS + 16;
  static constexpr int TOTAL = IDS + kGqaMaxIds * 4 + 1024;  // + alignment slack
};
enum { B_Q = 0, B_KVF = 1, B_KVE = 3, B_SF = 5, B_SE = 7, B_PF = 9, B_PE = 10, B_XF = 11, B_XE = 12 };

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

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
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
    mla_split_kernel(const __grid_constant__ CUtensorMap qn_map,
                     const __grid_constant__ CUtensorMap qp_map,
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
  const int nkb = r == 0 ? 4 : 5;  // 64-wide contraction blocks this CTA holds

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
    mbar_init(&bar[B_Q], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_KVF + s], 1);
      mbar_init(&bar[B_KVE + s], 1);
      mbar_init(&bar[B_SF + s], 1);
      mbar_init(&bar[B_SE + s], 128);
    }
    mbar_init(&bar[B_PF], 128);
    mbar_init(&bar[B_PE], 1);
    mbar_init(&bar[B_XF], 128);
    mbar_init(&bar[B_XE], 128);
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

  uint8_t *sQ = smem + Lay::Q;
  uint8_t *sKV = smem + Lay::KV;
  uint8_t *sP = smem + Lay::P;
  float *sX = reinterpret_cast<float *>(smem + Lay::X);

  int issued_kv = 0, issued_qk = 0, issued_pv = 0;  // for draining after an abort

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qn_map);
      tma_prefetch_desc(&ckv_map);
      const uint64_t kv_policy = l2_policy_evict_first();
      const uint64_t q_policy = l2_policy_evict_last();
      mbar_arrive_expect_tx(&bar[B_Q], (uint32_t)nkb * kQBlock);
      for (int c = 0; c < 4; ++c)
        tma_load_2d(sQ + c * kQBlock, &qn_map, &bar[B_Q], 64 * (4 * (int)r + c), b * kHeads,
                    q_policy);
      if (r == 1) tma_load_2d(sQ + 4 * kQBlock, &qp_map, &bar[B_Q], 0, b * kHeads, q_policy);
      for (int j = 0; j < num_tiles; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait_bounded(&bar[B_KVE + st], ((j >> 1) - 1) & 1, kWaitLimitNs)) {
          dev_err |= DA_DEVERR_TIMEOUT;
          *abort_flag = 1;
          break;
        }
        uint8_t *dst = sKV + st * 5 * kKvBlock;
        const int page = ids[j];
        if (page < 0) {
          // a skipped page: zeros instead of stale data (its scores are masked)
          for (int i = 0; i < 5 * kKvBlock / 16; ++i)
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
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(128, kTok, false, false);
      const uint32_t idesc_pv = umma_idesc_bf16(128, 256, false, true);
      bool ok = mbar_wait_bounded(&bar[B_Q], 0, kWaitLimitNs);
      auto issue_qk = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait_bounded(&bar[B_KVF + st], (j >> 1) & 1, kWaitLimitNs)) return false;
        if (j >= 2 && !mbar_wait_bounded(&bar[B_SE + st], ((j >> 1) - 1) & 1, kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t kv = smem_u32(sKV + st * 5 * kKvBlock);
        const uint32_t q = smem_u32(sQ);
        for (int c = 0; c < nkb; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ss(tmem + kTmemS + 64 * st,
                         umma_desc_sw128(q + c * kQBlock + kk * 32, 16, 1024),
                         umma_desc_sw128(kv + c * kKvBlock + kk * 32, 16, 1024), idesc_qk,
                         (c | kk) != 0);
        umma_commit(&bar[B_SF + st]);
        ++issued_qk;
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < num_tiles; ++j) {
        if (*abort_flag) break;
        if (j + 1 < num_tiles && !(ok = issue_qk(j + 1))) break;
        if (!(ok = mbar_wait_bounded(&bar[B_PF], j & 1, kWaitLimitNs))) break;
        tc_fence_after();
        const int st = j & 1;
        const uint32_t v = smem_u32(sKV + st * 5 * kKvBlock);
        const uint32_t pa = smem_u32(sP);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ss(tmem + kTmemO, umma_desc_sw128(pa + kk * 32, 16, 1024),
                       umma_desc_sw128(v + kk * 2048, kKvBlock, 1024),
                       idesc_pv, (j | kk) != 0);
        umma_commit(&bar[B_PE]);
        umma_commit(&bar[B_KVE + st]);
        ++issued_pv;
      }
      if (!ok) {
        dev_err |= DA_DEVERR_TIMEOUT;
        *abort_flag = 1;
      }
    }
  } else {
    // ============================================================ softmax (one head row per thread)
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const int h = quad * 32 + lane;             // head row
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t peer_x = mapa_peer(smem_u32(sX + h * kXStride), peer);
    const uint32_t peer_xf = mapa_peer(smem_u32(&bar[B_XF]), peer);
    const uint32_t peer_xe = mapa_peer(smem_u32(&bar[B_XE]), peer);
    const float sscale = p.score_scale;
    float m_ref = neg_inf(), l = 0.f;
    bool ok = true;
    for (int j = 0; j < num_tiles; ++j) {
      const int st = j & 1;
      if (!(ok = mbar_wait_bounded(&bar[B_SF + st], (j >> 1) & 1, kWaitLimitNs))) break;
      tc_fence_after();
      float s[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[16];
        tmem_ld16(tmem + lane_off + kTmemS + 64 * st + 16 * q, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[16 * q + i] = v[i];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar[B_SE + st]);
      // ---- exchange the partial scores with the peer CTA
      if (j >= 1 && !(ok = mbar_wait_cluster_bounded(&bar[B_XE], (j - 1) & 1))) break;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        st_cluster_v4(peer_x + 16 * q, s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
      mbar_arrive_remote(peer_xf);
      if (!(ok = mbar_wait_cluster_bounded(&bar[B_XF], j & 1))) break;
      const float4 *xr = reinterpret_cast<const float4 *>(sX + h * kXStride);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 o = xr[q];
        s[4 * q] += o.x;
        s[4 * q + 1] += o.y;
        s[4 * q + 2] += o.z;
        s[4 * q + 3] += o.w;
      }
      mbar_arrive_remote(peer_xe);
      // ---- mask, lazy-rescaled online softmax (exp2 domain)
      const int tok0 = range_lo + j * kTok;
      const int nval = ids[j] < 0 ? 0 : min(kTok, range_hi - tok0);
      float mt = neg_inf();
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        s[k] = k < nval ? s[k] * sscale : neg_inf();
        mt = fmaxf(mt, s[k]);
      }
      const bool need = mt > m_ref + kRescaleThreshold || (m_ref == neg_inf() && mt != neg_inf());
      const float alpha = need ? ex2(m_ref - mt) : 1.f;
      if (need) m_ref = mt;
      float psum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float p0 = m_ref == neg_inf() ? 0.f : ex2(s[k] - m_ref);
        const float p1 = m_ref == neg_inf() ? 0.f : ex2(s[k + 1] - m_ref);
        psum += p0 + p1;
        pk[k / 2] = pack_bf16(p0, p1);
      }
      l = l * alpha + psum;
      // ---- PV of the previous tile must be done before O or P change
      if (j >= 1 && !(ok = mbar_wait_bounded(&bar[B_PE], (j - 1) & 1, kWaitLimitNs))) break;
      tc_fence_after();
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        for (int c = 0; c < 256; c += 16) {
          float v[16];
          tmem_ld16(tmem + lane_off + kTmemO + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= alpha;
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
        // rows past the valid tokens may hold anything: zero their value part
        uint8_t *kv = sKV + st * 5 * kKvBlock;
        const int t_id = threadIdx.x - 64;  // 0..127
        for (int i = t_id; i < (kTok - nval) * 4 * 8; i += 128) {
          const int t = nval + i / 32, blk = (i / 8) % 4, c = i % 8;
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
    }
    // ---- epilogue: O_r / l for this CTA's value half
    if (ok && mbar_wait_bounded(&bar[B_PE], (num_tiles - 1) & 1, kWaitLimitNs)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : neg_inf();
      for (int c = 0; c < 256; c += 16) {
        float v[16];
        tmem_ld16(tmem + lane_off + kTmemO + c, v);
        tmem_wait_ld();
        if (p.write_final) {
          __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
              p.out + ((int64_t)b * kHeads + h) * 512 + r * 256 + c);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = __floats2bfloat162_rn(v[2 * i] * inv, v[2 * i + 1] * inv);
        } else {
          float4 *dst = reinterpret_cast<float4 *>(p.o_part + (slot * kHeads + h) * 512 + r * 256 + c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
        }
      }
      if (p.write_final) {
        if (r == 0 && p.lse) p.lse[(int64_t)b * kHeads + h] = lse;
      } else {
        p.lse_part[(slot * 2 + r) * kHeads + h] = lse;
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
      for (int j = max(0, issued_kv - 2); j < issued_kv; ++j)
        mbar_wait_bounded(&bar[B_KVF + (j & 1)], (j >> 1) & 1, kWaitLimitNs);
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

cudaError_t launch_mla(const CUtensorMap &qn_map, const CUtensorMap &qp_map,
                       const CUtensorMap &ckv_map, const CUtensorMap &kpe_map,
                       const MlaParams &p, dim3 grid, cudaStream_t stream) {
  mla_split_kernel<<<grid, kThreads, Lay::TOTAL, stream>>>(qn_map, qp_map, ckv_map, kpe_map, p);
  return cudaGetLastError();
}

}  // namespace da

/*
 * oracle.c -- float64 CPU oracle for split-KV decode attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA path shares no
 * code, header, table or helper with it, and it never calls the CUDA path.
 *
 * What it computes (the definition, written out directly; no tiling, no online
 * softmax, no reordering beyond the definition):
 *
 *   for every batch row b and query head hq, with kv head h = hq / G:
 *     P(b,h)  = the valid KV positions of that row (dense: 0..N_b-1; block
 *               sparse: the listed blocks, in list order, clipped to N_b --
 *               the blocks of KV_IDX, then those of FULL_KV_IDX when given)
 *     s_n     = scale * sum_d q[d] * k_n[d]                  (n in P)
 *               (with a soft cap c > 0: s_n = c * tanh(s_n / c))
 *     m       = max_n s_n
 *     l       = sum_n exp(s_n - m)
 *     out[d]  = sum_n exp(s_n - m) * v_n[d] / l
 *     lse     = m + ln(l)                                    (natural log)
 *   and out = 0, lse = -inf when P is empty.
 *
 *   A mask_mod and a score_mod in the sense of flex attention (the
 *   flex_decode.py.jinja template calls them per element, with the query
 *   head, for the blocks of KV_IDX; the blocks of FULL_KV_IDX take the
 *   score_mod only), with q_pos = N_b - Q + t the query token's position:
 *     sink/window mask: position n is kept when n < sink[hq], or window[hq]
 *       < 0, or n > q_pos - window[hq] (the last window[hq] positions);
 *     ALiBi score: s_n += slope[hq] * (n - q_pos).
 *
 *   fp8 tensor-core arithmetic (fp8_mma, with e4m3 K/V and per-kv-head
 *   scales): the query row is quantised to e4m3 as the kernel does it, in
 *   fp32 -- amax = max_d |q_d|, inv = 448 / amax, code_d = e4m3(q_d * inv)
 *   rounded to nearest even and saturated to +-448, and q~_d = code_d * s with
 *   s = amax / 448 (codes 0 and s = 0 when amax < 2^-100) -- and the scores
 *   use q~. The weights that meet V are rounded too: w_n = r8(r16(2^8 p_n)) /
 *   2^8 with p_n = exp(s_n - m), r16 / r8 the round-to-nearest-even into f16
 *   and into e4m3 (saturating); out = sum_n w_n v_n / l with l = sum_n p_n
 *   unrounded. The kernel rounds its weights relative to the running maximum
 *   it holds at each tile, not the row's maximum, so the two differ by up to
 *   twice the rounding bound of every weight, b(p) = (2^-4 + 2^-10) p + 2^-17,
 *   which the oracle reports per output element as sum_n b(p_n) |v_n| / l.
 *
 *   Several query tokens per row (q_len = Q > 1, speculative decoding): the
 *   row's new tokens are its last Q positions, so query token t < Q keeps the
 *   positions of P(b,h) with n <= N_b - Q + t (the causal mask of the split-K
 *   decode kernel, `_fwd_kernel_splitK` with IS_CAUSAL: q_pos = kv_len -
 *   num_queries + t, position kept when q_pos - kv_pos >= 0). Rows are then
 *   (b, hq, t) with t fastest. With a packed tree mask instead (the
 *   speculative-decoding mask of the TensorRT-LLM XQA kernel page, mha.cu,
 *   `applyMaskFromInput` under SPEC_DEC): every position before the Q new
 *   ones is kept, and new position N_b - Q + j is kept for token t when bit
 *   j % 32 of word j / 32 of mask row (b, t) is set.
 *
 * Sources: the per-split output and log-sum-exp of the split-K Triton decode
 * kernel page (mslk splitk_kernels.py, `_fwd_kernel_splitK`, "write back O"
 * and the LSE store), its reduce (`_splitK_reduce`), the GQA packing of the
 * TorchInductor flex_decode.py.jinja template (query head hq reads kv head
 * hq / G), its block-sparse traversal (KV_NUM_BLKS / KV_IDX, tables indexed
 * by kv head), the paged translation of splitk_kernels.py (physical page =
 * block_table[b][n / page_size]) and the MLA latent decode of FlashInfer
 * include/flashinfer/attention/mla.cuh (scores over [ckv; kpe], values = ckv).
 *
 * Every input is converted exactly to float64 before any arithmetic:
 *   - bf16 is the upper half of an IEEE-754 binary32 word;
 *   - fp8 is OCP E4M3FN (the `float8e4nv` type of splitk_kernels.py): sign,
 *     4-bit exponent with bias 7, 3-bit mantissa, subnormals at exponent 0,
 *     no infinities, S.1111.111 is NaN, largest finite value 448; the
 *     dequantised value is e4m3(byte) * scale[kv head], or, with a per-token
 *     scale and shift (the split-K page's fp8 scale_shift words),
 *     e4m3(byte) * scale[row] + shift[row];
 *   - int4 group-wise (the split-K page's PACKED_PER_VAL = 8 rows): a cache
 *     row is int32 words, first N_GROUPS coefficient words (fp16 scale in the
 *     low half, fp16 shift in the high half), then D / 8 words of eight
 *     unsigned 4-bit codes, element 8w + i in bits 4i..4i+3 of data word w;
 *     element d belongs to group d / (D / N_GROUPS) and is code * scale +
 *     shift of its group;
 *   - fp16 (the scales and shifts) is IEEE-754 binary16.
 *
 * Parity pins: see tests/test_oracle_pins.py (closed forms, invariants, brute
 * force with exact decimal arithmetic, all-code decoder checks).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* element decoders                                                   */
/* ------------------------------------------------------------------ */

double oracle_bf16_to_double(uint16_t bits) {
  uint32_t word = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &word, sizeof f);
  return (double)f;
}

/* IEEE-754 binary16: sign, 5-bit exponent with bias 15, 10-bit mantissa. */
double oracle_f16_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 10) & 0x1F;
  int mant = bits & 0x3FF;
  double mag;
  if (expo == 0x1F) return mant ? NAN : (sign ? -INFINITY : INFINITY);
  if (expo == 0)
    mag = ldexp((double)mant / 1024.0, 1 - 15); /* subnormal */
  else
    mag = ldexp(1.0 + (double)mant / 1024.0, expo - 15);
  return sign ? -mag : mag;
}

double oracle_e4m3_to_double(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int expo = (byte >> 3) & 0xF;
  int mant = byte & 0x7;
  double mag;
  if (expo == 0xF && mant == 0x7) return NAN;
  if (expo == 0)
    mag = ldexp((double)mant / 8.0, 1 - 7); /* subnormal: 0.mmm * 2^(1-bias) */
  else
    mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
  return sign ? -mag : mag;
}

/* ------------------------------------------------------------------ */
/* the softmax-attention core over an explicit score list             */
/* ------------------------------------------------------------------ */

/*
 * out[d] = sum_j exp(s_j - m) v_j[d] / sum_j exp(s_j - m);  lse = m + ln(sum).
 * v is row-major [n][dv]. n == 0 gives out = 0 and lse = -inf (the empty-split
 * convention of `_fwd_kernel_splitK`: l == 0 stores zeros, and `_splitK_reduce`
 * keeps lse = -inf for such rows).
 */
void oracle_softmax_attend(int64_t n, const double *s, const double *v, int dv,
                           double *out, double *lse) {
  for (int d = 0; d < dv; ++d) out[d] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j)
    if (s[j] > m) m = s[j];
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
  for (int64_t j = 0; j < n; ++j) {
    double w = exp(s[j] - m);
    for (int d = 0; d < dv; ++d) out[d] += w * v[j * (int64_t)dv + d];
  }
  for (int d = 0; d < dv; ++d) out[d] /= l;
  *lse = m + log(l);
}

/*
 * LSE-weighted merge of per-split results, as `_splitK_reduce` of
 * splitk_kernels.py defines it: M = max_s lse_s; w_s = exp(lse_s - M);
 * out = sum_s w_s o_s / sum_s w_s; lse = M + ln(sum_s w_s). When M = -inf
 * (every split empty) out = 0 and lse = -inf.
 */
void oracle_merge(int num_splits, int dv, const double *o, const double *lse_s,
                  double *out, double *lse) {
  double M = -INFINITY;
  for (int s = 0; s < num_splits; ++s)
    if (lse_s[s] > M) M = lse_s[s];
  for (int d = 0; d < dv; ++d) out[d] = 0.0;
  if (M == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  double wsum = 0.0;
  for (int s = 0; s < num_splits; ++s) wsum += exp(lse_s[s] - M);
  for (int s = 0; s < num_splits; ++s) {
    double w = exp(lse_s[s] - M);
    if (w == 0.0) continue; /* an empty split contributes nothing */
    for (int d = 0; d < dv; ++d) out[d] += w * o[(int64_t)s * dv + d];
  }
  for (int d = 0; d < dv; ++d) out[d] /= wsum;
  *lse = M + log(wsum);
}

/*
 * Round-to-nearest-even of a float into OCP E4M3FN, saturating to +-448 (a
 * value beyond 448 gives 448, NaN gives the NaN code 0x7F): the code byte.
 * From the format: 3 mantissa bits, exponent bias 7, normal exponents -6..8,
 * subnormals k * 2^-9.
 */
uint8_t oracle_e4m3_encode(float x) {
  if (x != x) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  if (a == 0.0) return sign;
  int E;
  frexp(a, &E); /* a = f * 2^E, f in [0.5, 1): floor(log2 a) = E - 1 */
  int e = E - 1;
  if (e < -6) { /* subnormal: multiples of 2^-9 */
    double k = rint(ldexp(a, 9));
    if (k >= 8.0) return sign | 0x08; /* rounds up to 2^-6, the smallest normal */
    return sign | (uint8_t)k;
  }
  double k = rint(ldexp(a, 3 - e)); /* 8 <= k <= 16 */
  if (k >= 16.0) {
    k = 8.0;
    ++e;
  }
  return sign | (uint8_t)((e + 7) << 3) | (uint8_t)(k - 8.0);
}

/* Round-to-nearest-even of a double into IEEE binary16 (the value, as a double;
 * overflow gives inf): 10 mantissa bits, normal exponents -14..15,
 * subnormals k * 2^-24. */
double oracle_f16_round(double x) {
  if (x != x || isinf(x)) return x;
  double a = fabs(x);
  if (a == 0.0) return x;
  int E;
  frexp(a, &E);
  int e = E - 1;
  double r;
  if (e < -14)
    r = ldexp(rint(ldexp(a, 24)), -24);
  else
    r = ldexp(rint(ldexp(a, 10 - e)), e - 10);
  if (r > 65504.0) r = INFINITY;
  return x < 0 ? -r : r;
}

/*
 * Softmax attention with the weights that meet V rounded as the fp8
 * tensor-core path rounds them: w = r8(r16(2^8 p)) / 2^8, p = exp(s - m), out
 * = sum w v / l, l = sum p; bound[d] = sum b(p) |v[d]| / l with b(p) =
 * (2^-4 + 2^-10) p + 2^-17 (the rounding bound of one weight). n == 0 gives
 * out = 0, lse = -inf, bound = 0.
 */
void oracle_softmax_attend_p8(int64_t n, const double *s, const double *v, int dv, double *out,
                              double *lse, double *bound) {
  for (int d = 0; d < dv; ++d) {
    out[d] = 0.0;
    if (bound) bound[d] = 0.0;
  }
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j)
    if (s[j] > m) m = s[j];
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
  for (int64_t j = 0; j < n; ++j) {
    const double p = exp(s[j] - m);
    const double w = oracle_e4m3_to_double(oracle_e4m3_encode((float)oracle_f16_round(256.0 * p))) / 256.0;
    const double b = (0.0625 + 0.0009765625) * p + 7.62939453125e-06;
    for (int d = 0; d < dv; ++d) {
      out[d] += w * v[j * (int64_t)dv + d];
      if (bound) bound[d] += b * fabs(v[j * (int64_t)dv + d]);
    }
  }
  for (int d = 0; d < dv; ++d) {
    out[d] /= l;
    if (bound) bound[d] /= l;
  }
  *lse = m + log(l);
}

/* ------------------------------------------------------------------ */
/* problem description (the oracle's own; not shared with the kernels) */
/* ------------------------------------------------------------------ */

typedef struct {
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;   /* MLA: 1 */
  int32_t head_dim_qk;    /* GQA: D; MLA: ckv_dim + kpe_dim */
  int32_t head_dim_v;     /* GQA: D; MLA: ckv_dim */
  int32_t is_mla;
  int32_t ckv_dim;
  int32_t kpe_dim;
  int32_t paged;          /* 0 contiguous, 1 paged through block_table */
  int32_t page_size;
  int32_t cache_len;      /* contiguous cache length L */
  int32_t max_pages_per_seq;
  int32_t num_pages;
  int32_t kv_fp8;         /* 0: bf16 bits, 1: e4m3 bytes with per-kv-head scale,
                             2: e4m3 bytes with a per-token fp16 scale and shift,
                             3: int4 group-wise rows of int32 words (kv_groups groups) */
  int32_t sparse_block_size; /* 0: dense */
  int32_t max_sparse_blocks;
  int32_t q_len;          /* query tokens per row (0 or 1: one) */
  int32_t sparse_batch;   /* sparse: extents of the tables' batch and head axes, */
  int32_t sparse_heads;   /* 0 = B and HKV; row (b, h) reads table (b % SZ, h % SH) */
  int32_t kv_groups;      /* kv_fp8 == 3: N_GROUPS, 1, 2, 4 or 8 */
  int32_t fp8_mma;        /* 1: e4m3 tensor-core arithmetic (Q and the weights of V
                             rounded as described at the top; kv_fp8 == 1 only) */
} oracle_problem;

typedef struct {
  const uint16_t *q;      /* bf16 [B][HQ][Q][Dq] (MLA: q_nope [B][HQ][Q][ckv]), Q = q_len */
  const uint16_t *q_pe;   /* MLA: bf16 [B][HQ][Q][kpe] */
  const void *k;          /* GQA contiguous [B][HKV][L][D]; paged [pages][HKV][P][D]
                             MLA ckv: contiguous [B][L][ckv]; paged [pages][P][ckv] */
  const void *v;          /* GQA: same layout as k; MLA kpe: [B][L][kpe] / [pages][P][kpe] */
  const float *k_scale;   /* fp8: [HKV] */
  const float *v_scale;   /* fp8: [HKV] */
  const int32_t *block_table; /* paged: [B][max_pages_per_seq] */
  const int32_t *seq_lens;    /* [B] */
  const int32_t *kv_num_blks; /* sparse: [SZ][SH] (SZ, SH = sparse_batch, sparse_heads) */
  const int32_t *kv_idx;      /* sparse: [SZ][SH][max_sparse_blocks] */
  double scale;
  const int32_t *k_scale_shift; /* kv_fp8 == 2: one word per cache row of k: fp16 scale in
                                   the low half, fp16 shift in the high half */
  const int32_t *v_scale_shift; /* the same for v */
  const int32_t *kv_full_num_blks; /* sparse, optional: [SZ][SH] blocks of the full list */
  const int32_t *kv_full_idx;      /* sparse, optional: [SZ][SH][max_sparse_blocks] */
  double softcap;                  /* > 0: scores become softcap * tanh(score / softcap) */
  const uint32_t *spec_mask;       /* Q > 1, optional (else causal): [B][Q][ceil(Q / 32)] words;
                                      bit j of row (b, t) keeps position N_b - Q + j for token t */
  const int32_t *mask_sink;        /* optional, with mask_window: [HQ] sink lengths */
  const int32_t *mask_window;      /* optional: [HQ] windows (< 0: no window) -- the mask_mod */
  const float *alibi_slopes;       /* optional: [HQ] slopes -- the score_mod */
  double *p8_bound;                /* fp8_mma, optional output [rows][Dv]: the weights'
                                      rounding bound (unsplit decode only) */
} oracle_inputs;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_BAD_INDEX = -2, ORACLE_NO_MEM = -3 };

/* ------------------------------------------------------------------ */
/* positions and element fetches                                      */
/* ------------------------------------------------------------------ */

static int64_t max_positions(const oracle_problem *p) {
  int64_t cap = p->paged ? (int64_t)p->max_pages_per_seq * p->page_size : p->cache_len;
  if (p->sparse_block_size > 0) {
    /* both tables of the block mask */
    int64_t sp = 2 * (int64_t)p->max_sparse_blocks * p->sparse_block_size;
    if (sp > cap) cap = sp;
  }
  return cap;
}

/*
 * The valid positions of (b, h), in order. Dense: 0..N_b-1. Sparse (the
 * block-sparse traversal of flex_decode.py.jinja): for each listed block j <
 * KV_NUM_BLKS[b][h], positions KV_IDX[b][h][j] * SBS + t, t < SBS, kept when
 * < N_b. Returns the count, or a negative error code; *n_masked is the number
 * of leading positions a mask_mod applies to (all of them but those of the
 * full-block table).
 */
static int64_t positions(const oracle_problem *p, const oracle_inputs *in, int b, int h,
                         int64_t *pos, int64_t *n_masked) {
  int64_t nb = in->seq_lens[b];
  int64_t capacity = p->paged ? (int64_t)p->max_pages_per_seq * p->page_size : p->cache_len;
  if (nb < 0 || nb > capacity) return ORACLE_BAD_INDEX;
  int64_t count = 0;
  if (p->sparse_block_size == 0) {
    for (int64_t n = 0; n < nb; ++n) pos[count++] = n;
    *n_masked = count;
    return count;
  }
  int64_t sbs = p->sparse_block_size;
  /* the block mask may have fewer batch rows or heads than the problem and is
   * then broadcast: flex_decode.py.jinja reads the tables at (off_z % SPARSE_Z,
   * off_hkv % SPARSE_HQ), the extents of KV_NUM_BLKS' first two axes */
  const int64_t sz = p->sparse_batch > 0 ? p->sparse_batch : p->batch;
  const int64_t sh = p->sparse_heads > 0 ? p->sparse_heads : p->num_kv_heads;
  const int64_t trow = (b % sz) * sh + h % sh;
  int32_t nblk = in->kv_num_blks[trow];
  if (nblk < 0 || nblk > p->max_sparse_blocks) return ORACLE_BAD_INDEX;
  const int32_t *list = in->kv_idx + trow * p->max_sparse_blocks;
  for (int32_t j = 0; j < nblk; ++j) {
    int64_t blk = list[j];
    if (blk < 0 || blk * sbs >= capacity) return ORACLE_BAD_INDEX;
    for (int64_t t = 0; t < sbs; ++t) {
      int64_t n = blk * sbs + t;
      if (n < nb) pos[count++] = n;
    }
  }
  /* the second table of the flex block mask (FULL_KV_NUM_BLKS / FULL_KV_IDX):
   * blocks that need no mask_mod; they are attended like the first table's
   * blocks, after them, with the score_mod but without the mask_mod */
  *n_masked = count;
  if (in->kv_full_num_blks) {
    int32_t nfull = in->kv_full_num_blks[trow];
    if (nfull < 0 || nfull > p->max_sparse_blocks) return ORACLE_BAD_INDEX;
    const int32_t *full = in->kv_full_idx + trow * p->max_sparse_blocks;
    for (int32_t j = 0; j < nfull; ++j) {
      int64_t blk = full[j];
      if (blk < 0 || blk * sbs >= capacity) return ORACLE_BAD_INDEX;
      for (int64_t t = 0; t < sbs; ++t) {
        int64_t n = blk * sbs + t;
        if (n < nb) pos[count++] = n;
      }
    }
  }
  return count;
}

/* Row index of token n of (b, h) in the cache, or -1 when the page is invalid. */
static int64_t cache_row(const oracle_problem *p, const oracle_inputs *in, int b, int h,
                         int64_t n) {
  int64_t heads = p->is_mla ? 1 : p->num_kv_heads;
  if (!p->paged) {
    return ((int64_t)b * heads + h) * p->cache_len + n;
  }
  int64_t page = in->block_table[(int64_t)b * p->max_pages_per_seq + n / p->page_size];
  if (page < 0 || page >= p->num_pages) return -1;
  return (page * heads + h) * p->page_size + n % p->page_size;
}

static double kv_elem(const oracle_problem *p, const void *base, int64_t idx, double scale) {
  if (p->kv_fp8) return oracle_e4m3_to_double(((const uint8_t *)base)[idx]) * scale;
  return oracle_bf16_to_double(((const uint16_t *)base)[idx]);
}

/* Fills key row kr[Dqk] and value row vr[Dv] for token n of (b, h). */
static int fetch_kv(const oracle_problem *p, const oracle_inputs *in, int b, int h, int64_t n,
                    double *kr, double *vr) {
  int64_t row = cache_row(p, in, b, h, n);
  if (row < 0) return ORACLE_BAD_INDEX;
  if (p->is_mla) {
    /* MLA latent cache: key = [ckv ; kpe], value = ckv */
    for (int d = 0; d < p->ckv_dim; ++d) {
      double c = kv_elem(p, in->k, row * p->ckv_dim + d, 1.0);
      kr[d] = c;
      vr[d] = c;
    }
    for (int d = 0; d < p->kpe_dim; ++d)
      kr[p->ckv_dim + d] = kv_elem(p, in->v, row * p->kpe_dim + d, 1.0);
    return ORACLE_OK;
  }
  if (p->kv_fp8 == 3) {
    /* int4 group-wise (the split-K decode page: `dequantize` with
     * PACKED_PER_VAL = 8 splits each data word into eight 4-bit codes, element
     * 8w + i from bits 4i.., and applies its group's fp16 scale and shift) */
    const int ng = p->kv_groups;
    const uint32_t *kw = (const uint32_t *)in->k + row * (ng + p->head_dim_qk / 8);
    const uint32_t *vw = (const uint32_t *)in->v + row * (ng + p->head_dim_v / 8);
    for (int d = 0; d < p->head_dim_qk; ++d) {
      const uint32_t coef = kw[d / (p->head_dim_qk / ng)];
      const uint32_t code = (kw[ng + d / 8] >> (4 * (d % 8))) & 0xFu;
      kr[d] = (double)code * oracle_f16_to_double((uint16_t)(coef & 0xFFFF)) +
              oracle_f16_to_double((uint16_t)(coef >> 16));
    }
    for (int d = 0; d < p->head_dim_v; ++d) {
      const uint32_t coef = vw[d / (p->head_dim_v / ng)];
      const uint32_t code = (vw[ng + d / 8] >> (4 * (d % 8))) & 0xFu;
      vr[d] = (double)code * oracle_f16_to_double((uint16_t)(coef & 0xFFFF)) +
              oracle_f16_to_double((uint16_t)(coef >> 16));
    }
    return ORACLE_OK;
  }
  if (p->kv_fp8 == 2) {
    /* per-token asymmetric e4m3 (the split-K decode page's fp8 K/V with a
     * per-token scale_shift word: `cast_uint32_to_half2` splits it into an
     * fp16 scale (low half) and shift (high half), and `dequantize` gives
     * value = e4m3 * scale + shift) */
    uint32_t kw = (uint32_t)in->k_scale_shift[row], vw = (uint32_t)in->v_scale_shift[row];
    double ksc = oracle_f16_to_double((uint16_t)(kw & 0xFFFF));
    double ksh = oracle_f16_to_double((uint16_t)(kw >> 16));
    double vsc = oracle_f16_to_double((uint16_t)(vw & 0xFFFF));
    double vsh = oracle_f16_to_double((uint16_t)(vw >> 16));
    const uint8_t *kb = (const uint8_t *)in->k, *vb = (const uint8_t *)in->v;
    for (int d = 0; d < p->head_dim_qk; ++d)
      kr[d] = oracle_e4m3_to_double(kb[row * p->head_dim_qk + d]) * ksc + ksh;
    for (int d = 0; d < p->head_dim_v; ++d)
      vr[d] = oracle_e4m3_to_double(vb[row * p->head_dim_v + d]) * vsc + vsh;
    return ORACLE_OK;
  }
  double ks = p->kv_fp8 ? (double)in->k_scale[h] : 1.0;
  double vs = p->kv_fp8 ? (double)in->v_scale[h] : 1.0;
  for (int d = 0; d < p->head_dim_qk; ++d) kr[d] = kv_elem(p, in->k, row * p->head_dim_qk + d, ks);
  for (int d = 0; d < p->head_dim_v; ++d) vr[d] = kv_elem(p, in->v, row * p->head_dim_v + d, vs);
  return ORACLE_OK;
}

static int q_tokens(const oracle_problem *p) { return p->q_len > 1 ? p->q_len : 1; }

/* Query token t of (b, hq). */
static void fetch_q(const oracle_problem *p, const oracle_inputs *in, int b, int hq, int t,
                    double *qr) {
  const int64_t r = ((int64_t)b * p->num_q_heads + hq) * q_tokens(p) + t;
  if (p->is_mla) {
    const uint16_t *qn = in->q + r * p->ckv_dim;
    const uint16_t *qp = in->q_pe + r * p->kpe_dim;
    for (int d = 0; d < p->ckv_dim; ++d) qr[d] = oracle_bf16_to_double(qn[d]);
    for (int d = 0; d < p->kpe_dim; ++d) qr[p->ckv_dim + d] = oracle_bf16_to_double(qp[d]);
    return;
  }
  const uint16_t *qq = in->q + r * p->head_dim_qk;
  for (int d = 0; d < p->head_dim_qk; ++d) qr[d] = oracle_bf16_to_double(qq[d]);
  if (p->fp8_mma) {
    /* the e4m3 query row, in the kernel's fp32 steps (see the top) */
    float amax = 0.0f;
    for (int d = 0; d < p->head_dim_qk; ++d) {
      const float a = fabsf((float)qr[d]);
      if (a > amax) amax = a;
    }
    const int tiny = !(amax >= 0x1p-100f);
    const float inv = tiny ? 0.0f : 448.0f / amax;
    const float sq = tiny ? 0.0f : amax / 448.0f;
    for (int d = 0; d < p->head_dim_qk; ++d) {
      const float x = (float)qr[d] * inv;
      qr[d] = oracle_e4m3_to_double(oracle_e4m3_encode(x)) * (double)sq;
    }
  }
}

static int check_problem(const oracle_problem *p, const oracle_inputs *in) {
  if (!p || !in || !in->q || !in->k || !in->v || !in->seq_lens) return ORACLE_BAD_ARG;
  if (p->batch < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->q_len < 0 ||
      p->sparse_batch < 0 || p->sparse_heads < 0)
    return ORACLE_BAD_ARG;
  if (p->num_q_heads % p->num_kv_heads) return ORACLE_BAD_ARG;
  if (p->is_mla) {
    if (p->num_kv_heads != 1 || !in->q_pe || p->kv_fp8) return ORACLE_BAD_ARG;
    if (p->head_dim_qk != p->ckv_dim + p->kpe_dim || p->head_dim_v != p->ckv_dim)
      return ORACLE_BAD_ARG;
  }
  if (p->paged && (!in->block_table || p->page_size <= 0 || p->max_pages_per_seq < 0))
    return ORACLE_BAD_ARG;
  if (p->kv_fp8 == 1 && (!in->k_scale || !in->v_scale)) return ORACLE_BAD_ARG;
  if (p->kv_fp8 == 2 && (!in->k_scale_shift || !in->v_scale_shift || p->is_mla)) return ORACLE_BAD_ARG;
  if (p->kv_fp8 < 0 || p->kv_fp8 > 3) return ORACLE_BAD_ARG;
  if (p->kv_fp8 == 3) {
    const int ng = p->kv_groups;
    if (p->is_mla || !(ng == 1 || ng == 2 || ng == 4 || ng == 8)) return ORACLE_BAD_ARG;
    if (p->head_dim_qk % (8 * ng) || p->head_dim_v % (8 * ng)) return ORACLE_BAD_ARG;
  }
  if (p->sparse_block_size > 0 && (!in->kv_num_blks || !in->kv_idx)) return ORACLE_BAD_ARG;
  if ((in->kv_full_num_blks != NULL) != (in->kv_full_idx != NULL)) return ORACLE_BAD_ARG;
  if (in->kv_full_num_blks && p->sparse_block_size <= 0) return ORACLE_BAD_ARG;
  if (in->mask_sink && !in->mask_window) return ORACLE_BAD_ARG;
  /* a soft cap and ALiBi together would need an order of the two score_mods */
  if (in->alibi_slopes && in->softcap > 0.0) return ORACLE_BAD_ARG;
  if (p->fp8_mma && (p->kv_fp8 != 1 || p->is_mla)) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* one (b, hq) row, optionally cut into chunks of the position list    */
/* ------------------------------------------------------------------ */

typedef struct {
  const oracle_problem *p;
  const oracle_inputs *in;
  int num_chunks;              /* 0: unsplit */
  const int64_t *chunk_bounds; /* [num_chunks + 1] list-index boundaries */
  double *out;                 /* unsplit: [B][HQ][Dv]; split: [B][HQ][C][Dv] */
  double *lse;                 /* unsplit: [B][HQ];     split: [B][HQ][C] */
  int64_t next_row;
  int64_t rows;
  pthread_mutex_t lock;
  int status;
} job_t;

static int run_row(job_t *job, int64_t row, int64_t *pos, double *s, double *vrows, double *qr,
                   double *kr) {
  const oracle_problem *p = job->p;
  const oracle_inputs *in = job->in;
  const int Q = q_tokens(p);
  int b = (int)(row / ((int64_t)p->num_q_heads * Q));
  int hq = (int)((row / Q) % p->num_q_heads);
  int t = (int)(row % Q);
  int G = p->num_q_heads / p->num_kv_heads;
  int h = hq / G;
  int dq = p->head_dim_qk, dv = p->head_dim_v;

  int64_t n_masked = 0;
  int64_t n = positions(p, in, b, h, pos, &n_masked);
  if (n < 0) return (int)n;
  /* the query token's position: the row's new tokens are its last Q positions */
  const int64_t q_pos = (int64_t)in->seq_lens[b] - Q + t;
  if (in->mask_window) {
    /* the sink/window mask_mod, per query head, on the positions it applies to */
    const int64_t sink = in->mask_sink ? in->mask_sink[hq] : 0, win = in->mask_window[hq];
    int64_t kept = 0, kept_masked = 0;
    for (int64_t j = 0; j < n; ++j) {
      const int keep = j >= n_masked || pos[j] < sink || win < 0 || pos[j] > q_pos - win;
      if (keep) {
        pos[kept++] = pos[j];
        if (j < n_masked) ++kept_masked;
      }
    }
    n = kept;
    n_masked = kept_masked;
  }
  if (Q > 1) {
    /* Several new query tokens (speculative decoding): they are the row's last
     * Q positions. Token t sees every older position and, among the new ones,
     * those up to its own, n <= N_b - Q + t (the causal mask of the split-K
     * decode kernel, splitk_kernels.py `_fwd_kernel_splitK`, IS_CAUSAL), or
     * those its tree-mask row selects (XQA mha.cu, SPEC_DEC). */
    const int64_t first_new = (int64_t)in->seq_lens[b] - Q;
    const int64_t words = (Q + 31) / 32;
    const uint32_t *mrow = in->spec_mask ? in->spec_mask + ((int64_t)b * Q + t) * words : NULL;
    int64_t kept = 0;
    for (int64_t j = 0; j < n; ++j) {
      const int64_t d = pos[j] - first_new; /* index among the new positions, < 0: an old one */
      int keep;
      if (d < 0)
        keep = 1;
      else if (mrow) /* the tree mask (XQA SPEC_DEC): bit d of the token's mask row */
        keep = (int)((mrow[d / 32] >> (d % 32)) & 1u);
      else
        keep = d <= t; /* causal */
      if (keep) pos[kept++] = pos[j];
    }
    n = kept;
  }
  fetch_q(p, in, b, hq, t, qr);
  for (int64_t j = 0; j < n; ++j) {
    int st = fetch_kv(p, in, b, h, pos[j], kr, vrows + j * (int64_t)dv);
    if (st) return st;
    double dot = 0.0;
    for (int d = 0; d < dq; ++d) dot += qr[d] * kr[d];
    s[j] = in->scale * dot;
    /* tanh soft-capping of the scaled score (the FlashAttention-3 page:
     * tanh(scores * softmax_scale / softcap_val) * softcap_val) */
    if (in->softcap > 0.0) s[j] = in->softcap * tanh(s[j] / in->softcap);
    /* the ALiBi score_mod: a per-head slope times the distance to the query */
    if (in->alibi_slopes) s[j] += (double)in->alibi_slopes[hq] * (double)(pos[j] - q_pos);
  }
  if (job->num_chunks == 0) {
    if (p->fp8_mma)
      oracle_softmax_attend_p8(n, s, vrows, dv, job->out + row * dv, job->lse + row,
                               in->p8_bound ? in->p8_bound + row * dv : NULL);
    else
      oracle_softmax_attend(n, s, vrows, dv, job->out + row * dv, job->lse + row);
    return ORACLE_OK;
  }
  if (p->fp8_mma) return ORACLE_BAD_ARG; /* split decode is defined on exact weights */
  for (int c = 0; c < job->num_chunks; ++c) {
    int64_t lo = job->chunk_bounds[c], hi = job->chunk_bounds[c + 1];
    if (lo > n) lo = n;
    if (hi > n) hi = n;
    if (hi < lo) hi = lo;
    oracle_softmax_attend(hi - lo, s + lo, vrows + lo * (int64_t)dv, dv,
                          job->out + (row * job->num_chunks + c) * dv,
                          job->lse + row * job->num_chunks + c);
  }
  return ORACLE_OK;
}

static void *worker(void *arg) {
  job_t *job = (job_t *)arg;
  const oracle_problem *p = job->p;
  int64_t cap = max_positions(p);
  int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
  double *s = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
  double *vrows = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1) * p->head_dim_v);
  double *qr = (double *)malloc(sizeof(double) * p->head_dim_qk);
  double *kr = (double *)malloc(sizeof(double) * p->head_dim_qk);
  int status = (pos && s && vrows && qr && kr) ? ORACLE_OK : ORACLE_NO_MEM;
  while (status == ORACLE_OK) {
    pthread_mutex_lock(&job->lock);
    int64_t row = job->next_row++;
    int failed = job->status;
    pthread_mutex_unlock(&job->lock);
    if (row >= job->rows || failed) break;
    status = run_row(job, row, pos, s, vrows, qr, kr);
  }
  if (status) {
    pthread_mutex_lock(&job->lock);
    if (!job->status) job->status = status;
    pthread_mutex_unlock(&job->lock);
  }
  free(pos);
  free(s);
  free(vrows);
  free(qr);
  free(kr);
  return NULL;
}

static int run_job(job_t *job, int num_threads) {
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  pthread_t tid[256];
  pthread_mutex_init(&job->lock, NULL);
  job->next_row = 0;
  job->status = ORACLE_OK;
  int started = 0;
  for (int t = 1; t < num_threads; ++t) {
    if (pthread_create(&tid[started], NULL, worker, job) == 0) ++started;
  }
  worker(job);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&job->lock);
  return job->status;
}

/*
 * Full decode attention: out [B][HQ][Q][Dv] and lse [B][HQ][Q] (natural log;
 * Q = q_len, the [Q] axis absent for one query token).
 * Returns 0, or a negative code (bad argument, or an index outside the cache:
 * a page id outside [0, num_pages), a sparse block outside the cache, a
 * sequence length over the cache capacity).
 */
int oracle_decode(const oracle_problem *p, const oracle_inputs *in, double *out, double *lse,
                  int num_threads) {
  int st = check_problem(p, in);
  if (st) return st;
  job_t job;
  memset(&job, 0, sizeof job);
  job.p = p;
  job.in = in;
  job.num_chunks = 0;
  job.out = out;
  job.lse = lse;
  job.rows = (int64_t)p->batch * p->num_q_heads * q_tokens(p);
  return run_job(&job, num_threads);
}

/*
 * Split decode: the position list of every row is cut at the list indices
 * chunk_bounds[0..num_chunks] (clipped to the row's length; chunks may be
 * empty), and each chunk is attended on its own, giving per-chunk o
 * [B][HQ][C][Dv] and lse [B][HQ][C] -- the per-split results the split-K
 * kernel stores before its reduce.
 */
int oracle_split(const oracle_problem *p, const oracle_inputs *in, int num_chunks,
                 const int64_t *chunk_bounds, double *o, double *lse, int num_threads) {
  int st = check_problem(p, in);
  if (st) return st;
  if (num_chunks <= 0 || !chunk_bounds) return ORACLE_BAD_ARG;
  for (int c = 0; c < num_chunks; ++c)
    if (chunk_bounds[c] < 0 || chunk_bounds[c + 1] < chunk_bounds[c]) return ORACLE_BAD_ARG;
  job_t job;
  memset(&job, 0, sizeof job);
  job.p = p;
  job.in = in;
  job.num_chunks = num_chunks;
  job.chunk_bounds = chunk_bounds;
  job.out = o;
  job.lse = lse;
  job.rows = (int64_t)p->batch * p->num_q_heads * q_tokens(p);
  return run_job(&job, num_threads);
}

/* Merge for many rows at once: o [rows][S][dv], lse_s [rows][S]. */
void oracle_merge_rows(int64_t rows, int num_splits, int dv, const double *o,
                       const double *lse_s, double *out, double *lse) {
  for (int64_t r = 0; r < rows; ++r)
    oracle_merge(num_splits, dv, o + r * num_splits * (int64_t)dv, lse_s + r * num_splits,
                 out + r * dv, lse + r);
}

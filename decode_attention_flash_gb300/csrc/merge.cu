// merge.cu -- LSE-weighted merge of per-split decode results.
//
// For every output row: M = max_s lse_s, w_s = exp(lse_s - M),
// out = sum_s w_s * O_s / sum_s w_s, lse = M + ln(sum_s w_s); a row whose
// splits are all empty (M = -inf) gets out = 0 and lse = -inf. This is the
// reduce of the split-K Triton decode page (mslk splitk_kernels.py,
// `_splitK_reduce`), also the merge step of FlashInfer mla.cuh
// (`DevicePersistentMergeStates`). Splits marked empty (lse = -inf) are
// skipped without reading their O.
//
// One warp per row; each lane owns float4 columns of the head dimension, so a
// split's O row is read with one coalesced 16-byte load per lane.
#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) lse_merge_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarpsPerBlock + warp;
  if (row >= p.rows) return;
  const int R = p.rows_per_unit, S = p.num_splits;
  const int64_t u = row / R, g = row % R;
  const float *lse_s = p.lse_part + u * S * R + g;  // element s at s*R
  const float ninf = -__int_as_float(0x7f800000);

  float M = ninf;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse_s[(int64_t)s * R]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  const int nvec = p.dv >> 2;
  __nv_bfloat16 *out_row = p.out + (int64_t)row * p.dv;
  if (M == ninf) {
    for (int c = lane; c < nvec; c += 32) {
      __nv_bfloat162 z = __floats2bfloat162_rn(0.f, 0.f);
      reinterpret_cast<__nv_bfloat162 *>(out_row)[2 * c] = z;
      reinterpret_cast<__nv_bfloat162 *>(out_row)[2 * c + 1] = z;
    }
    if (lane == 0 && p.lse) p.lse[row] = ninf;
    return;
  }

  float wsum = 0.f;
  for (int s = lane; s < S; s += 32) wsum += ex2((lse_s[(int64_t)s * R] - M) * kLog2e);
#pragma unroll
  for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float inv = 1.f / wsum;

  // up to 8 float4 columns per lane (dv <= 1024)
  float4 acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float *o_base = p.o_part + (u * S * R + g) * (int64_t)p.dv;  // split s at s*R*dv
  for (int s = 0; s < S; ++s) {
    const float l = lse_s[(int64_t)s * R];
    if (l == ninf) continue;
    const float w = ex2((l - M) * kLog2e);
    const float4 *src = reinterpret_cast<const float4 *>(o_base + (int64_t)s * R * p.dv);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = lane + 32 * k;
      if (c < nvec) {
        const float4 v = src[c];
        acc[k].x += w * v.x;
        acc[k].y += w * v.y;
        acc[k].z += w * v.z;
        acc[k].w += w * v.w;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = lane + 32 * k;
    if (c < nvec) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
      reinterpret_cast<__nv_bfloat162 *>(out_row)[2 * c] = lo;
      reinterpret_cast<__nv_bfloat162 *>(out_row)[2 * c + 1] = hi;
    }
  }
  if (lane == 0 && p.lse) p.lse[row] = M + __log2f(wsum) * kLn2;
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const int blocks = (p.rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  lse_merge_kernel<<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace da

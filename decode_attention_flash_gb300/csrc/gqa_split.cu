// gqa_split.cu -- host side of the persistent GQA decode kernel: shared-memory
// sizes, one-time attributes and the launch, dispatched to the translation
// unit of the cache's element kind (gqa_kind_*.cu, compiled in parallel).
// The kernel itself is in gqa_split.cuh.
#include "gqa_split.cuh"

namespace da {

int gqa_smem_bytes(bool fp8, int group, bool token_scale, bool int4) {
  if (int4) return group <= 8 ? Cfg<true, 1, false, true>::kTotal : Cfg<true, 2, false, true>::kTotal;
  if (fp8 && token_scale) return group <= 8 ? Cfg<true, 1, true>::kTotal : Cfg<true, 2, true>::kTotal;
  if (fp8) return group <= 8 ? Cfg<true, 1>::kTotal : Cfg<true, 2>::kTotal;
  return group <= 8 ? Cfg<false, 1>::kTotal : Cfg<false, 2>::kTotal;
}
int gqa_threads() { return kMaxThreads; }

int gqa_box_tokens(const da_problem &p) {
  if (p.kv_layout == DA_KV_PAGED && p.page_size < kTile) return p.page_size;
  return kTile;
}

cudaError_t gqa_prepare(int /*device*/) {
  cudaError_t e;
  if ((e = gqa_prepare_kind_bf16()) != cudaSuccess) return e;
  if ((e = gqa_prepare_kind_e4m3()) != cudaSuccess) return e;
  if ((e = gqa_prepare_kind_e4m3_token()) != cudaSuccess) return e;
  if ((e = gqa_prepare_kind_e4m3_mma()) != cudaSuccess) return e;
  return gqa_prepare_kind_int4();
}

cudaError_t launch_gqa(bool fp8, int group, const CUtensorMap &kmap, const CUtensorMap &vmap,
                       const CUtensorMap &qmap, const CUtensorMap &kssmap,
                       const CUtensorMap &vssmap, const GqaParams &p, int ctas,
                       cudaStream_t stream) {
  // score and mask modifications (several query tokens, a draft-tree mask, a
  // soft cap, the sink/window mask_mod, ALiBi) take their own instantiation:
  // the plain decode keeps the shorter softmax
  const int mod = (p.mask_window != nullptr || p.alibi_slopes != nullptr)
                      ? 2
                      : (p.q_len > 1 || p.spec_mask != nullptr || p.softcap_l2 > 0.f) ? 1 : 0;
  const bool two = group > 8;
  if (!fp8) return gqa_launch_kind_bf16(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
  if (p.kv_groups > 0)
    return gqa_launch_kind_int4(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
  if (p.token_scale)
    return gqa_launch_kind_e4m3_token(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
  if (p.fp8_mma)
    return gqa_launch_kind_e4m3_mma(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
  return gqa_launch_kind_e4m3(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
}

}  // namespace da

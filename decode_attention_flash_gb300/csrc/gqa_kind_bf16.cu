// gqa_kind_bf16.cu -- the GQA decode kernel's instantiations for bf16 K/V.
#include "gqa_split.cuh"

namespace da {

cudaError_t gqa_prepare_kind_bf16() { return prepare_kind<false, false, false>(); }

cudaError_t gqa_launch_kind_bf16(bool two, int mod, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, const CUtensorMap &qmap,
                                 const CUtensorMap &kssmap, const CUtensorMap &vssmap,
                                 const GqaParams &p, int ctas, cudaStream_t stream) {
  return launch_kind<false, false, false>(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
}

}  // namespace da

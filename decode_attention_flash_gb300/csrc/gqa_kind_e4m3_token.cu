// gqa_kind_e4m3_token.cu -- the GQA decode kernel's instantiations for e4m3 K/V with a scale and shift
// per token.
#include "gqa_split.cuh"

namespace da {

cudaError_t gqa_prepare_kind_e4m3_token() { return prepare_kind<true, true, false>(); }

cudaError_t gqa_launch_kind_e4m3_token(bool two, int mod, const CUtensorMap &kmap,
                                       const CUtensorMap &vmap, const CUtensorMap &qmap,
                                       const CUtensorMap &kssmap, const CUtensorMap &vssmap,
                                       const GqaParams &p, int ctas, cudaStream_t stream) {
  return launch_kind<true, true, false>(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
}

}  // namespace da

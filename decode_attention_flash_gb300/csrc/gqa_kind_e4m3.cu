// gqa_kind_e4m3.cu -- the GQA decode kernel's instantiations for e4m3 K/V with a scale per kv
// head.
#include "gqa_split.cuh"

namespace da {

cudaError_t gqa_prepare_kind_e4m3() { return prepare_kind<true, false, false>(); }

cudaError_t gqa_launch_kind_e4m3(bool two, int mod, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, const CUtensorMap &qmap,
                                 const CUtensorMap &kssmap, const CUtensorMap &vssmap,
                                 const GqaParams &p, int ctas, cudaStream_t stream) {
  return launch_kind<true, false, false>(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
}

}  // namespace da

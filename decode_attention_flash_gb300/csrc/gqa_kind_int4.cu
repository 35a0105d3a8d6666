// gqa_kind_int4.cu -- the GQA decode kernel's instantiations for int4 group-wise K/V rows.
#include "gqa_split.cuh"

namespace da {

cudaError_t gqa_prepare_kind_int4() { return prepare_kind<true, false, true>(); }

cudaError_t gqa_launch_kind_int4(bool two, int mod, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, const CUtensorMap &qmap,
                                 const CUtensorMap &kssmap, const CUtensorMap &vssmap,
                                 const GqaParams &p, int ctas, cudaStream_t stream) {
  return launch_kind<true, false, true>(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas, stream);
}

}  // namespace da

// gqa_kind_e4m3_mma.cu -- the GQA decode kernel's instantiations for e4m3 K/V
// with per-kv-head scales on e4m3 tensor cores (e4m3 queries and weights).
#include "gqa_split.cuh"

namespace da {

cudaError_t gqa_prepare_kind_e4m3_mma() { return prepare_kind<true, false, false, true>(); }

cudaError_t gqa_launch_kind_e4m3_mma(bool two, int mod, const CUtensorMap &kmap,
                                     const CUtensorMap &vmap, const CUtensorMap &qmap,
                                     const CUtensorMap &kssmap, const CUtensorMap &vssmap,
                                     const GqaParams &p, int ctas, cudaStream_t stream) {
  return launch_kind<true, false, false, true>(two, mod, kmap, vmap, qmap, kssmap, vssmap, p, ctas,
                                               stream);
}

}  // namespace da

// Instances of the column pass (pass 2) for every head_dim and input type.
#include "imp_pass.cuh"

namespace tsel {

cudaError_t launch_imp_pass2(int head_dim, bool fp8, const CUtensorMap* maps,
                             const ImpPassParams& p, int grid, cudaStream_t stream) {
#define TSEL_PASS2_CASE(DD)                                                                   \
  case DD:                                                                                    \
    return fp8 ? launch_pass_t<2, DD, true, false>(maps, p, grid, stream)                     \
               : launch_pass_t<2, DD, false, false>(maps, p, grid, stream);
  switch (head_dim) {
    TSEL_PASS2_CASE(64)
    TSEL_PASS2_CASE(80)
    TSEL_PASS2_CASE(96)
    TSEL_PASS2_CASE(112)
    TSEL_PASS2_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef TSEL_PASS2_CASE
}

}  // namespace tsel

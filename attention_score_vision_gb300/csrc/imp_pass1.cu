// Instances of the row-LSE pass (pass 1) for every head_dim and input type,
// with and without key chunks.
#include "imp_pass.cuh"

namespace tsel {

cudaError_t launch_imp_pass1(int head_dim, bool fp8, bool ksplit, const CUtensorMap* maps,
                             const ImpPassParams& p, int grid, cudaStream_t stream) {
#define TSEL_PASS1_CASE(DD)                                                                   \
  case DD:                                                                                    \
    if (fp8)                                                                                  \
      return ksplit ? launch_pass_t<1, DD, true, true>(maps, p, grid, stream)                 \
                    : launch_pass_t<1, DD, true, false>(maps, p, grid, stream);               \
    return ksplit ? launch_pass_t<1, DD, false, true>(maps, p, grid, stream)                  \
                  : launch_pass_t<1, DD, false, false>(maps, p, grid, stream);
  switch (head_dim) {
    TSEL_PASS1_CASE(64)
    TSEL_PASS1_CASE(80)
    TSEL_PASS1_CASE(96)
    TSEL_PASS1_CASE(112)
    TSEL_PASS1_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef TSEL_PASS1_CASE
}

}  // namespace tsel

// Backward kernel instantiations for head dimension 256.
#include "fa_bwd256.cuh"

namespace fa {

int launch_bwd_d256(bool causal, bool bf16, const CUtensorMap* maps, const BwdParams& prm, int grid,
                    cudaStream_t stream) {
  if (bf16)
    return causal ? launch_bwd256<true, true>(maps, prm, grid, stream)
                  : launch_bwd256<false, true>(maps, prm, grid, stream);
  return causal ? launch_bwd256<true, false>(maps, prm, grid, stream)
                : launch_bwd256<false, false>(maps, prm, grid, stream);
}

}  // namespace fa

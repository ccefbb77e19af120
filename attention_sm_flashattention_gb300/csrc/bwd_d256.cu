// Backward kernel instantiations for head dimension 256.
#include "fa_bwd.cuh"

namespace fa {

int launch_bwd_d256(bool causal, const CUtensorMap* maps, const BwdParams& prm, int grid, cudaStream_t stream) {
  return causal ? launch_bwd<256, true>(maps, prm, grid, stream) : launch_bwd<256, false>(maps, prm, grid, stream);
}

}  // namespace fa

// Backward kernel instantiations for head dimension 64.
#include "fa_bwd.cuh"

namespace fa {

int launch_bwd_d64(bool causal, const CUtensorMap* maps, const BwdParams& prm, int grid, cudaStream_t stream) {
  return causal ? launch_bwd<64, true>(maps, prm, grid, stream) : launch_bwd<64, false>(maps, prm, grid, stream);
}

}  // namespace fa

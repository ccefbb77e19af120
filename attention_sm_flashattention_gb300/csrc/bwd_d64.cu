// Backward kernel instantiations for head dimension 64: Delta preprocess,
// then the dK/dV kernel and the dQ kernel.
#include "fa_bwd.cuh"
#include "fa_bwd2.cuh"

namespace fa {

int launch_bwd_d64(bool causal, const CUtensorMap* maps, const BwdParams& prm, int grid, cudaStream_t stream) {
  return causal ? launch_bwd2<64, true>(maps, prm, grid, stream) : launch_bwd2<64, false>(maps, prm, grid, stream);
}

}  // namespace fa

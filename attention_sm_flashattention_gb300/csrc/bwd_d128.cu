// Backward kernel instantiations for head dimension 128.
#include "fa_bwd.cuh"

namespace fa {

int launch_bwd_d128(bool causal, const CUtensorMap* maps, const BwdParams& prm, int grid, cudaStream_t stream) {
  return causal ? launch_bwd<128, true>(maps, prm, grid, stream) : launch_bwd<128, false>(maps, prm, grid, stream);
}

}  // namespace fa

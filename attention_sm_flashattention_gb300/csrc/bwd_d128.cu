// Backward kernel instantiations for head dimension 128: the dQ kernel (which
// also forms Delta and lse2), then the dK/dV kernel.
#include "fa_bwd2.cuh"

namespace fa {

int launch_bwd_d128(bool causal, bool bf16, const CUtensorMap* maps, const BwdParams& prm, int grid,
                    cudaStream_t stream) {
  if (bf16)
    return causal ? launch_bwd2<128, true, true>(maps, prm, grid, stream)
                  : launch_bwd2<128, false, true>(maps, prm, grid, stream);
  return causal ? launch_bwd2<128, true, false>(maps, prm, grid, stream)
                : launch_bwd2<128, false, false>(maps, prm, grid, stream);
}

}  // namespace fa

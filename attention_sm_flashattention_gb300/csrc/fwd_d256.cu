// Forward kernel instantiations for head dimension 256.
#include "fa_fwd.cuh"

namespace fa {

int launch_fwd_d256(bool causal, const CUtensorMap* maps, const FwdParams& prm, int num_sms, cudaStream_t stream) {
  return causal ? launch_fwd<256, true>(maps, prm, num_sms, stream) : launch_fwd<256, false>(maps, prm, num_sms, stream);
}

}  // namespace fa

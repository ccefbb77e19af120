// Forward kernel instantiations for head dimension 256 over dense K/V (the
// paged, selected-block and split modes use fa_fwd.cuh's kernel).
#include "fa_fwd256.cuh"

namespace fa {

int launch_fwd_d256(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                    cudaStream_t stream) {
  if (bf16)
    return causal ? launch_fwd256<true, true>(maps, prm, num_sms, stream)
                  : launch_fwd256<false, true>(maps, prm, num_sms, stream);
  return causal ? launch_fwd256<true, false>(maps, prm, num_sms, stream)
                : launch_fwd256<false, false>(maps, prm, num_sms, stream);
}

}  // namespace fa

// Forward kernel instantiations over a paged K/V cache, head dimension 64.
#include "fa_fwd.cuh"

namespace fa {

int launch_fwd_paged_d64(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                         cudaStream_t stream) {
  if (bf16)
    return causal ? launch_fwd<64, true, true, kPaged>(maps, prm, num_sms, stream)
                  : launch_fwd<64, false, true, kPaged>(maps, prm, num_sms, stream);
  return causal ? launch_fwd<64, true, false, kPaged>(maps, prm, num_sms, stream)
                : launch_fwd<64, false, false, kPaged>(maps, prm, num_sms, stream);
}

}  // namespace fa

// Forward kernel instantiations over a paged K/V cache with split key
// ranges, head dimension 256, followed by the merge of the slices.
#include "fa_fwd.cuh"

namespace fa {

int launch_fwd_paged_split_d256(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                               cudaStream_t stream) {
  int rc;
  if (bf16)
    rc = causal ? launch_fwd<256, true, true, kPagedSplit>(maps, prm, num_sms, stream)
                : launch_fwd<256, false, true, kPagedSplit>(maps, prm, num_sms, stream);
  else
    rc = causal ? launch_fwd<256, true, false, kPagedSplit>(maps, prm, num_sms, stream)
                : launch_fwd<256, false, false, kPagedSplit>(maps, prm, num_sms, stream);
  if (rc != 0) return rc;
  return launch_split_combine(prm.part_o, prm.part_lse, prm.o, prm.lse, static_cast<long long>(prm.heads) * prm.Nq,
                              256, prm.splits, bf16, num_sms, stream);
}

}  // namespace fa

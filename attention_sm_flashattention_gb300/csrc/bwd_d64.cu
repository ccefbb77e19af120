// Backward kernel instantiations for head dimension 64.
#include "fa_kernels.h"

namespace fa {

int launch_bwd_d64(bool, const CUtensorMap*, const BwdParams&, int, cudaStream_t) { return -2; }

}  // namespace fa

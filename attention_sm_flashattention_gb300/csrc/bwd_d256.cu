// Backward kernel instantiations for head dimension 256.
#include "fa_kernels.h"

namespace fa {

int launch_bwd_d256(bool, const CUtensorMap*, const BwdParams&, int, cudaStream_t) { return -2; }

}  // namespace fa

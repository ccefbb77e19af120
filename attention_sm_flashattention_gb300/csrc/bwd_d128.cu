// Backward kernel instantiations for head dimension 128.
#include "fa_kernels.h"

namespace fa {

int launch_bwd_d128(bool, const CUtensorMap*, const BwdParams&, int, cudaStream_t) { return -2; }

}  // namespace fa

// Kernel parameter blocks and the per-instantiation launchers shared between
// the C-ABI translation unit and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fa {

struct FwdParams {
  __half* o;         // [heads, N, D] (written through the O tensor map)
  float* lse;        // [heads, N]
  int heads;         // Z * H
  int N;             // sequence length (multiple of 128)
  float scale_log2;  // scale * log2(e)
  int* status;       // device status word
};

struct BwdParams {
  const __half* o;     // [heads, N, D] forward output
  const __half* dout;  // [heads, N, D]
  const float* lse;    // [heads, N] natural-log lse from the forward
  __half* dq;          // [heads, N, D]
  __half* dk;
  __half* dv;
  float* delta;        // workspace [heads, N]: rowsum(O * dO)
  float* lse2;         // workspace [heads, N]: lse * log2(e)
  float* dq_acc;       // workspace [grid, N, D]: per-CTA fp32 dQ accumulator (D = 256 only)
  int heads;
  int N;
  float scale;         // softmax scale
  float scale_log2;    // scale * log2(e)
  int* status;
};

// One launcher per head dimension; `causal` and `bf16` (bf16 instead of
// fp16 inputs and outputs) select the instantiation.  Return 0 on success.
// For the backward, `grid` caps the persistent grid: for D = 256 it is the
// number of per-CTA dQ accumulators in the workspace, for D <= 128 (no
// accumulators) the SM count.  The tensor maps carry the element type.
#define FA_DECLARE_LAUNCHERS(D)                                                                      \
  int launch_fwd_d##D(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm,       \
                      int num_sms, cudaStream_t stream);                                              \
  /* bwd maps: q, k, v, dout, dq, dk, dv */                                                         \
  int launch_bwd_d##D(bool causal, bool bf16, const CUtensorMap* maps, const BwdParams& prm,       \
                      int grid, cudaStream_t stream);

FA_DECLARE_LAUNCHERS(64)
FA_DECLARE_LAUNCHERS(128)
FA_DECLARE_LAUNCHERS(256)
#undef FA_DECLARE_LAUNCHERS

// Tile sizes the host needs to build tensor maps and size grids.
inline int fwd_block_n(int D) { return D == 256 ? 64 : 128; }

}  // namespace fa

// FlashAttention backward preprocess for sm_103a.
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
// §二 -- Delta = rowsum(O * dO), the row term of dS = scale * P * (dP -
// Delta); P is recomputed from the saved log-sum-exp.  §七 -- for D = 256
// the row sum over both D halves is the same sum.
//
// fa_bwd_prep_kernel: Delta in fp32 and lse2 = lse * log2(e) for every query
// row (HBM-bound, one pass over O and dO), into the padded [heads, Nq_pad]
// workspace vectors that the dK/dV and dQ kernels read per query tile (D =
// 64 in fa_bwd2.cuh, D = 256 in fa_bwd256.cuh).  For D = 128 the dQ kernel
// (fa_bwd2.cuh) forms the same two vectors itself, from the dO tile it holds
// anyway.
#pragma once

#include "fa_kernels.h"
#include "ptx.cuh"

namespace fa {

// -------------------------------------------------------------- preprocess

// Rows are those of the padded [heads, Nq_pad] workspace vectors: a query
// row past Nq (the rest of a ragged last tile) gets Delta = 0 and lse2 =
// +inf, so its recomputed P is exactly 0 and it adds nothing to dK or dV.
template <int D, bool BF>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __half* __restrict__ o,
                                                          const __half* __restrict__ dout,
                                                          const float* __restrict__ lse, float* __restrict__ delta,
                                                          float* __restrict__ lse2, int heads, int Nq, int Nq_pad) {
  constexpr int TPR = D / 8;  // threads per row, 8 fp16 (16 bytes) each
  constexpr int RPB = 256 / TPR;
  const int r = blockIdx.x * RPB + threadIdx.x / TPR;  // padded row
  const int part = threadIdx.x % TPR;
  const int rows = heads * Nq_pad;
  const int head = r / Nq_pad, i = r - head * Nq_pad;
  const bool live = r < rows && i < Nq;
  const size_t src = static_cast<size_t>(head) * Nq + i;  // row of O, dO and lse
  float acc = 0.f;
  if (live) {
    const uint4 a = reinterpret_cast<const uint4*>(o + src * D)[part];
    const uint4 b = reinterpret_cast<const uint4*>(dout + src * D)[part];
    const uint32_t* ha = reinterpret_cast<const uint32_t*>(&a);
    const uint32_t* hb = reinterpret_cast<const uint32_t*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa2 = unpack2<BF>(ha[e]);
      const float2 fb2 = unpack2<BF>(hb[e]);
      acc = fmaf(fa2.x, fb2.x, acc);
      acc = fmaf(fa2.y, fb2.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (r < rows && part == 0) {
    delta[r] = acc;
    lse2[r] = live ? lse[src] * 1.4426950408889634f : INFINITY;
  }
}

template <int D, bool BF>
int launch_prep(const BwdParams& prm, cudaStream_t stream) {
  const long long rows = static_cast<long long>(prm.heads) * prm.Nq_pad;
  constexpr int RPB = 256 / (D / 8);
  fa_bwd_prep_kernel<D, BF><<<static_cast<unsigned>((rows + RPB - 1) / RPB), 256, 0, stream>>>(
      prm.o, prm.dout, prm.lse, prm.delta, prm.lse2, prm.heads, prm.Nq, prm.Nq_pad);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

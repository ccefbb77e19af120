// Merge of a split-key-range forward (the paged forward with every work
// item's key tiles cut into slices).
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战», §一
// -- the online softmax keeps, per row, a running max and a running sum so
// that blocks of keys can be processed one at a time and merged; the same
// merge applies to whole slices of keys.  A slice s that reports the
// log-sum-exp lse_s of its scores and O_s = (its exp-weighted V rows) / (its
// row sum) combines as
//     lse = log sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) * O_s,
// since exp(lse_s - lse) is slice s's share of the full row sum.  A slice
// with no visible key has lse_s = -inf and weight 0 (its O_s is not read).
//
// HBM-bound and small (splits x rows x D fp32 in, rows x D 16-bit out): one
// warp per row, each lane a 16-byte column group.
#include <cstdint>
#include <cuda_runtime.h>

#include "fa_kernels.h"
#include "ptx.cuh"

namespace fa {

template <int D, bool BF>
__global__ void __launch_bounds__(256) fa_split_combine_kernel(const float* __restrict__ part_o,
                                                               const float* __restrict__ part_lse,
                                                               uint16_t* __restrict__ o, float* __restrict__ lse,
                                                               long long rows, int splits) {
  constexpr int G = D / 4;                 // float4 column groups per row
  constexpr int PER = (G + 31) / 32;       // groups per lane
  const int lane = threadIdx.x % 32;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += warps) {
    float mx = -INFINITY;
    for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, __ldg(part_lse + s * rows + row));
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    float sum = 0.f;
    if (mx != -INFINITY)
      for (int s = lane; s < splits; s += 32) sum += expf(__ldg(part_lse + s * rows + row) - mx);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, k);
    const float total = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    float4 acc[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) acc[p] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (total != -INFINITY) {
      for (int s = 0; s < splits; ++s) {
        const float ls = __ldg(part_lse + s * rows + row);
        if (ls == -INFINITY) continue;  // nothing visible in the slice
        const float w = expf(ls - total);
        const float4* src = reinterpret_cast<const float4*>(part_o + (s * rows + row) * D);
#pragma unroll
        for (int p = 0; p < PER; ++p) {
          const int g = lane + 32 * p;
          if (g < G) {
            const float4 v = __ldg(src + g);
            acc[p].x = fmaf(w, v.x, acc[p].x);
            acc[p].y = fmaf(w, v.y, acc[p].y);
            acc[p].z = fmaf(w, v.z, acc[p].z);
            acc[p].w = fmaf(w, v.w, acc[p].w);
          }
        }
      }
    }
    uint2* dst = reinterpret_cast<uint2*>(o + row * D);
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int g = lane + 32 * p;
      if (g < G) dst[g] = make_uint2(pack2<BF>(acc[p].x, acc[p].y), pack2<BF>(acc[p].z, acc[p].w));
    }
    if (lane == 0) lse[row] = total;
  }
}

template <int D, bool BF>
static int combine(const float* part_o, const float* part_lse, void* o, float* lse, long long rows, int splits,
                   int num_sms, cudaStream_t stream) {
  long long blocks = (rows + 7) / 8;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fa_split_combine_kernel<D, BF><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      part_o, part_lse, static_cast<uint16_t*>(o), lse, rows, splits);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_split_combine(const float* part_o, const float* part_lse, void* o, float* lse, long long rows, int D,
                         int splits, bool bf16, int num_sms, cudaStream_t stream) {
  switch (D) {
    case 64:
      return bf16 ? combine<64, true>(part_o, part_lse, o, lse, rows, splits, num_sms, stream)
                  : combine<64, false>(part_o, part_lse, o, lse, rows, splits, num_sms, stream);
    case 128:
      return bf16 ? combine<128, true>(part_o, part_lse, o, lse, rows, splits, num_sms, stream)
                  : combine<128, false>(part_o, part_lse, o, lse, rows, splits, num_sms, stream);
    case 256:
      return bf16 ? combine<256, true>(part_o, part_lse, o, lse, rows, splits, num_sms, stream)
                  : combine<256, false>(part_o, part_lse, o, lse, rows, splits, num_sms, stream);
    default:
      return -1;
  }
}

}  // namespace fa

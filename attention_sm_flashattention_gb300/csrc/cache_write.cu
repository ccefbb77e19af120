// Paged K/V cache write (ReshapeAndCache).
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战», the
// contest section's ReshapeAndCache part: new tokens' K and V, laid out one
// token after another, go to the physical block slot // block_size at
// offset slot % block_size given by slot_mapping; a negative slot means the
// token is skipped.
//
// With the cache laid out [num_pages, page_size, Hkv, D], block b offset o is
// flat row b * page_size + o = slot of a [num_pages * page_size, Hkv * D]
// matrix, so the write is a row scatter: token t's Hkv * D 16-bit values go
// to row slot_mapping[t].  HBM-bound: one warp per token row, 16 bytes per
// lane per step (rows are 16-byte aligned: Hkv * D * 2 is a multiple of 128).
#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

__global__ void __launch_bounds__(256) fa_cache_write_kernel(const uint4* __restrict__ k_new,
                                                             const uint4* __restrict__ v_new,
                                                             const long long* __restrict__ slots, uint4* k_cache,
                                                             uint4* v_cache, int tokens, int row_vec,
                                                             long long cache_rows) {
  const int warps = blockDim.x / 32;
  const int lane = threadIdx.x % 32;
  for (long long t = static_cast<long long>(blockIdx.x) * warps + threadIdx.x / 32; t < tokens;
       t += static_cast<long long>(gridDim.x) * warps) {
    const long long slot = __ldg(slots + t);
    if (slot < 0 || slot >= cache_rows) continue;  // skipped token (or a slot outside the cache)
    const uint4* ks = k_new + t * row_vec;
    const uint4* vs = v_new + t * row_vec;
    uint4* kd = k_cache + slot * row_vec;
    uint4* vd = v_cache + slot * row_vec;
    for (int e = lane; e < row_vec; e += 32) {
      kd[e] = __ldg(ks + e);
      vd[e] = __ldg(vs + e);
    }
  }
}

int launch_cache_write(const void* k_new, const void* v_new, const long long* slots, void* k_cache, void* v_cache,
                       int tokens, int Hkv, int D, long long cache_rows, int num_sms, cudaStream_t stream) {
  const int row_vec = Hkv * D * 2 / 16;  // 16-byte vectors per token row
  const int warps_per_block = 8;
  long long blocks = (static_cast<long long>(tokens) + warps_per_block - 1) / warps_per_block;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fa_cache_write_kernel<<<static_cast<unsigned>(blocks), 32 * warps_per_block, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), tokens, row_vec, cache_rows);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

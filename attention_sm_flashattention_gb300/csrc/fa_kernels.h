// Kernel parameter blocks and the per-instantiation launchers shared between
// the C-ABI translation unit and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_once.h"

namespace fa {

// Shapes: queries (and O, dO, dQ) are [heads, Nq, D]; keys and values (and
// dK, dV) are [heads / group, Nk, D]; query head h reads K/V head h / group.
// Causal: query i sees key j iff j <= i + causal_off, causal_off = Nk - Nq
// (the queries are the last Nq positions of the sequence; Nq <= Nk).
struct FwdParams {
  __half* o;         // [heads, Nq, D] (written through the O tensor map)
  float* lse;        // [heads, Nq]
  int heads;         // query heads, Z * H
  int group;         // query heads per K/V head
  int Nq, Nk;        // query and key lengths (any >= 1)
  int causal_off;    // Nk - Nq
  float scale_log2;  // scale * log2(e)
  int* status;       // device status word
  // Paged K/V cache (paged launchers only).  K and V are [num_pages,
  // page_size, Hkv, D]; query head h of sequence b = head / H reads K/V head
  // (head % H) / group of its cache pages; sequence b's key p lives in page
  // block_table[b * max_pages + p / page_size] at row p % page_size, and its
  // key count is context_lens[b], clamped to [causal ? Nq : 1, max_pages *
  // page_size].
  const int* block_table;
  const int* context_lens;
  int H;             // query heads per sequence
  int num_pages, page_size, max_pages;
  // Selected blocks (sparse launchers): for sequence b and K/V head kvh, list
  // entries e < sel_count[b * Hkv + kvh] (at most max_pages) name physical
  // page sel_pages[(b * Hkv + kvh) * max_pages + e] holding logical block
  // sel_blocks[...]; row r of it is the token at logical position block *
  // page_size + r, visible iff below context_lens[b] (and, causal, at most
  // the query's own position, the queries being the context's last Nq).
  const int* sel_pages;
  const int* sel_blocks;
  const int* sel_count;
  int Hkv;
  // Packed grouped heads (0 = off): the G query heads that share a K/V head
  // run as one head of G * q_period rows (they are consecutive in memory);
  // row r is query position r % q_period, and `heads`, `group`, `Nq` and `H`
  // describe the packed problem (group 1).
  int q_period;
  // Split key range (paged split launchers): each work item's key tiles are
  // cut into `splits` contiguous slices, one work unit each.  A unit writes
  // its rows' partial result to part_o ([splits, heads * Nq, D] fp32, O
  // normalised by the slice's own row sum) and part_lse ([splits, heads *
  // Nq] fp32, natural log; -inf for a slice with no visible key), and the
  // combine kernel merges the slices into o and lse.
  int splits;
  float* part_o;
  float* part_lse;
};

struct BwdParams {
  const __half* v;     // [heads / group, Nk, D] (read directly by the D = 256 dK/dV kernel)
  const __half* o;     // [heads, Nq, D] forward output
  const __half* dout;  // [heads, Nq, D]
  const float* lse;    // [heads, Nq] natural-log lse from the forward
  __half* dq;          // [heads, Nq, D]
  __half* dk;          // [heads / group, Nk, D]
  __half* dv;
  float* delta;        // workspace [heads, Nq_pad]: rowsum(O * dO), 0 in the padding
  float* lse2;         // workspace [heads, Nq_pad]: lse * log2(e), +inf in the padding
  int heads;           // query heads
  int group;           // query heads per K/V head
  int Nq, Nk;
  int Nq_pad;          // Nq rounded up to the 128-row query tile
  int causal_off;      // Nk - Nq
  float scale;         // softmax scale
  float scale_log2;    // scale * log2(e)
  int* status;
};

// One launcher per head dimension; `causal` and `bf16` (bf16 instead of
// fp16 inputs and outputs) select the instantiation.  Return 0 on success.
// For the backward, `grid` caps each persistent grid (the SM count).  The
// tensor maps carry the element type.
// Dense forward maps: q, k, v, o (D = 256: v with 64-row boxes; o unused).
#define FA_DECLARE_LAUNCHERS(D)                                                                      \
  int launch_fwd_d##D(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm,       \
                      int num_sms, cudaStream_t stream);                                              \
  /* bwd maps: q, k, v, dout, dq, dk, dv, q and k with the D = 256 dQ kernel's boxes, o */                     \
  int launch_bwd_d##D(bool causal, bool bf16, const CUtensorMap* maps, const BwdParams& prm,       \
                      int grid, cudaStream_t stream);

FA_DECLARE_LAUNCHERS(64)
FA_DECLARE_LAUNCHERS(128)
FA_DECLARE_LAUNCHERS(256)
#undef FA_DECLARE_LAUNCHERS

// Paged cache write: token t's K and V rows ([Hkv, D] 16-bit values each) to
// cache row slots[t] of [cache_rows, Hkv, D] caches; negative slots and slots
// >= cache_rows are skipped.
int launch_cache_write(const void* k_new, const void* v_new, const long long* slots, void* k_cache, void* v_cache,
                       int tokens, int Hkv, int D, long long cache_rows, int num_sms, cudaStream_t stream);

// Forward over a paged K/V cache; maps: q, k cache, v cache (4-D, one page
// row block per box), o.
int launch_fwd_paged_d64(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                         cudaStream_t stream);
int launch_fwd_paged_d128(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                          cudaStream_t stream);
int launch_fwd_paged_d256(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                          cudaStream_t stream);
// Forward over selected blocks of a paged cache; maps as for the paged launchers.
int launch_fwd_sparse_d64(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                          cudaStream_t stream);
int launch_fwd_sparse_d128(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                           cudaStream_t stream);
int launch_fwd_sparse_d256(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                           cudaStream_t stream);

// Forward over a paged K/V cache with the key range of every work item split
// into prm.splits slices (partial results into prm.part_o / part_lse), then
// the combine kernel (o, lse); maps as for the paged launchers.
int launch_fwd_paged_split_d64(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                               cudaStream_t stream);
int launch_fwd_paged_split_d128(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                                cudaStream_t stream);
int launch_fwd_paged_split_d256(bool causal, bool bf16, const CUtensorMap* maps, const FwdParams& prm, int num_sms,
                                cudaStream_t stream);
// Merge `splits` partial results per row: rows = heads * Nq, O and lse as
// described for FwdParams::part_o / part_lse.
int launch_split_combine(const float* part_o, const float* part_lse, void* o, float* lse, long long rows, int D,
                         int splits, bool bf16, int num_sms, cudaStream_t stream);

// Index of the current device, or -1 if the runtime cannot tell.
inline int current_device_index() {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

// Tile sizes the host needs to build tensor maps and size grids: keys per
// tile of the paged, selected-block and split forward, and of the dense one
// (which at D = 256 moves each 128-key tile as two halves: K by halves of
// the contraction, 128-row boxes; V by halves of the keys, 64-row boxes).
inline int fwd_block_n(int D) { return D == 256 ? 64 : 128; }
inline int fwd_dense_block_n(int) { return 128; }

}  // namespace fa

/*
 * fa.h -- C ABI of libfa.so: exact FlashAttention forward and backward for
 * one NVIDIA GB300 (sm_103a): fp16 inputs and outputs (fa_fwd, fa_bwd; bf16
 * through fa_fwd_bf16, fa_bwd_bf16 and the _ex calls), fp32 accumulation.
 *
 * What is computed (source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV
 * Pipeline 优化实战»):
 *   forward  (§一)  S = Q K^T * scale,  P = softmax(S),  O = P V, computed
 *                   tile by tile with the online softmax (running row max m,
 *                   denominator l, unnormalised fp32 accumulator), exp2 with
 *                   log2(e) folded into the scale; causal mode visits only
 *                   key tiles at or below the diagonal and masks exactly only
 *                   inside diagonal tiles (§一, §八).
 *   backward (§二)  Delta = rowsum(O * dO), P recomputed from the saved
 *                   log-sum-exp, dP = dO V^T, dS = scale * P * (dP - Delta),
 *                   dQ = dS K, dK = dS^T Q, dV = P^T dO, with every gradient
 *                   tile written by exactly one CTA and a workspace that does
 *                   not grow with the number of heads times N^2 (§二's three
 *                   rules).
 *
 * Layout and types (all calls):
 *   q, k, v, o, dout, dq, dk, dv : fp16 (IEEE binary16), contiguous
 *                                  [Z, H, N, D] row-major, 16-byte aligned.
 *   lse                          : fp32 [Z, H, N]; lse[z,h,i] is the natural
 *                                  log of sum_j exp(S_ij) over the visible
 *                                  keys j (j <= i when causal).
 *   Every (z, h) pair is an independent head; queries and keys have the same
 *   length N (any N >= 1; a last partial 128-row tile is masked).  Causal
 *   means key j is visible to query i iff j <= i.  fa_fwd_ex / fa_bwd_ex
 *   below add grouped K/V heads and different query and key lengths.
 *
 * Ownership: every pointer is device memory owned by the caller; the library
 * keeps no pointer after a call returns and allocates no device memory on
 * these paths.  The only library state is one device status word per device.
 *
 * Asynchrony: fa_fwd / fa_bwd validate their arguments on the host, enqueue
 * kernels on `stream` and return.  A return of FA_OK means "enqueued".
 * Results are ready when the stream reaches that point.
 *
 * Errors: argument problems are reported synchronously, before anything is
 * enqueued, with a negative code (below).  A device-side wait that gives up
 * (bounded by about one second; it never hangs the GPU) is reported through
 * fa_device_status().  Not thread-safe with respect to concurrent first calls
 * on the same device from several host threads.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK 0
#define FA_ERR_INVALID_ARG (-1) /* null pointer, a size <= 0, H not a multiple of Hkv, bad causal flag or
                                   dtype, non-finite or <= 0 scale, misaligned pointer */
#define FA_ERR_UNSUPPORTED (-2) /* D not in {64, 128, 256}, causal with Nq > Nk, or sizes past 32-bit indexing */
#define FA_ERR_WORKSPACE (-3)   /* workspace null, misaligned or smaller than its size query
                                   (fa_bwd_workspace_size, fa_fwd_paged_split_workspace_size) */
#define FA_ERR_CUDA (-4)        /* a CUDA runtime call or kernel launch failed */
#define FA_ERR_DEVICE (-5)      /* current device is not a compute capability 10.3 GPU */
#define FA_ERR_TIMEOUT (-6)     /* (fa_device_status) a kernel wait gave up; results invalid */
#define FA_ERR_SCRATCH_LIMIT (-7) /* (fa_bwd_noalloc) problem needs more than the built-in scratch buffer */

/*
 * Forward pass.  Source: «把 FlashAttention 搬上昇腾» §一 (tiled online
 * softmax, exp2, fp32 m/l/acc, fp16 P into the matrix unit, causal loop
 * bound + diagonal-only mask), §七 (D256: the key and value tiles move in
 * halves; the 256-column accumulator fits whole).
 *   q, k, v : inputs [Z,H,N,D] fp16.
 *   o       : output [Z,H,N,D] fp16, O = softmax(Q K^T scale) V, rounded to
 *             nearest from the fp32 accumulator divided by l.
 *   lse     : output [Z,H,N] fp32 (natural-log log-sum-exp of each row of S).
 *   Z, H, N : batch, heads, sequence length (N >= 1).
 *   D       : head dimension, 64, 128 or 256.
 *   causal  : 0 or 1.
 *   scale   : softmax scale applied to Q K^T (usually 1/sqrt(D)); finite, > 0.
 *   stream  : CUDA stream the kernel is enqueued on (0 = legacy default).
 * Returns FA_OK or a negative FA_ERR_* code.
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int H, int N, int D,
           int causal, float scale, cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd (or fa_bwd_bf16) needs: Delta and the
 * log2-scaled lse (2 x Z*H*N' fp32, N' = N rounded up to a multiple of 128,
 * each vector rounded up to 256 bytes).  It grows with Z*H*N, never with N^2
 * over all heads (§二, third rule): every dQ, dK and dV tile is accumulated
 * on chip by the one CTA that writes it.  Returns 0 for unsupported
 * arguments.
 */
FA_API size_t fa_bwd_workspace_size(int Z, int H, int N, int D, int causal);

/*
 * Backward pass.  Source: «把 FlashAttention 搬上昇腾» §二 (equations and
 * the three rules), §五 (persistent programs: here one per SM, each taking
 * (head, tile) work units in turn, and every dQ/dK/dV tile has one writer),
 * §七 (D256: the accumulators split so that they fit; here one gradient at a
 * time).
 *   q, k, v, o, dout : inputs [Z,H,N,D] fp16; o must be fa_fwd's output for
 *                      the same q, k, v, causal and scale.
 *   lse              : input [Z,H,N] fp32 from the same fa_fwd call.
 *   dq, dk, dv       : outputs [Z,H,N,D] fp16, overwritten (not accumulated).
 *   workspace        : device scratch of at least workspace_bytes >=
 *                      fa_bwd_workspace_size(Z,H,N,D,causal) bytes, 256-byte
 *                      aligned; contents on entry are ignored, on exit
 *                      undefined.  Must not be used by another call that runs
 *                      concurrently on the GPU.
 *   other arguments  : as for fa_fwd.
 * Enqueues two persistent kernels on `stream`: first the dQ kernel, which
 * also forms Delta = rowsum(O * dO) and the log2-scaled lse of every query
 * row into the workspace, then the dK/dV kernel, which reads them.
 * Returns FA_OK or a negative FA_ERR_* code.
 */
FA_API int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int Z, int H, int N, int D,
           int causal, float scale, cudaStream_t stream);

/*
 * bf16 forward and backward.  Source: «把 FlashAttention 搬上昇腾» §九 (every
 * candidate version is checked for correctness in FP16 and in BF16).  Identical to fa_fwd / fa_bwd
 * except that every [Z,H,N,D] tensor (q, k, v, o, dout, dq, dk, dv) is
 * bf16, and P and dS are rounded to bf16 before the matrix unit; lse, Delta,
 * the accumulators and the softmax statistics stay fp32.  Same layout,
 * alignment, ownership, workspace (fa_bwd_workspace_size) and error codes.
 */
FA_API int fa_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int H, int N,
                       int D, int causal, float scale, cudaStream_t stream);

FA_API int fa_bwd_bf16(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                       int Z, int H, int N, int D, int causal, float scale, cudaStream_t stream);

/*
 * Grouped K/V heads and different query / key lengths.  Source: «把
 * FlashAttention 搬上昇腾», the GQA Paged Attention part of the contest
 * section: the number of query heads is an integer multiple of the number
 * of K/V heads, several query heads share one K/V head, each sequence has
 * its own context length and the last incomplete block is masked.
 *
 *   q, o, dout, dq : [Z, H, Nq, D]        lse : fp32 [Z, H, Nq]
 *   k, v, dk, dv   : [Z, Hkv, Nk, D]      (H a multiple of Hkv; g = H / Hkv)
 *   Query head h of batch z reads K/V head h / g of batch z (consecutive
 *   query heads share a K/V head).  dk, dv of a shared head are the sums of
 *   the gradients of its g query heads, each written once by one CTA.
 *   Nq, Nk : any lengths >= 1.
 *   causal : the queries are the last Nq positions of an Nk-long sequence:
 *            query i sees key j iff j <= i + (Nk - Nq).  Needs Nq <= Nk
 *            (otherwise some row would see no key): FA_ERR_UNSUPPORTED.
 *   dtype  : FA_DTYPE_F16 or FA_DTYPE_BF16, the element type of every
 *            [.., D] tensor (lse, Delta and accumulation stay fp32).
 * Layout, alignment, ownership, asynchrony and errors as for fa_fwd /
 * fa_bwd; workspace from fa_bwd_ex_workspace_size (0 = unsupported shape).
 * fa_fwd(q, k, v, o, lse, Z, H, N, D, c, s, st) is
 * fa_fwd_ex(q, k, v, o, lse, Z, H, H, N, N, D, c, s, FA_DTYPE_F16, st).
 */
#define FA_DTYPE_F16 0
#define FA_DTYPE_BF16 1
FA_API int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int H, int Hkv, int Nq,
                     int Nk, int D, int causal, float scale, int dtype, cudaStream_t stream);

/*
 * Forward over a paged K/V cache.  Source: «把 FlashAttention 搬上昇腾», the
 * contest section's ReshapeAndCache and GQA Paged Attention parts: the cache
 * is kept in physical blocks ("pages") of page_size tokens (token slot s in
 * page s / page_size, row s % page_size); block_tables maps each sequence's
 * logical blocks to physical ones; context_lens gives each sequence's real
 * length and the invalid tokens of its last block are masked; query heads
 * share K/V heads as in fa_fwd_ex.
 *
 *   q, o         : [B, H, Nq, D] (dtype), contiguous, 16-byte aligned.
 *   lse          : fp32 [B, H, Nq].
 *   k_cache,
 *   v_cache      : [num_pages, page_size, Hkv, D] (dtype), 16-byte aligned.
 *   block_table  : int32 [B, max_pages], device memory: sequence b's key p
 *                  is in page block_table[b * max_pages + p / page_size].
 *                  Entries outside [0, num_pages) read as zero keys/values
 *                  (never out of bounds).
 *   context_lens : int32 [B], device memory: sequence b attends to its first
 *                  context_lens[b] keys, clamped to [causal ? Nq : 1,
 *                  max_pages * page_size].
 *   causal       : the Nq queries are the last Nq of the sequence's
 *                  context_lens[b] tokens (query i sees key p iff p <= i +
 *                  context_lens[b] - Nq).
 *   page_size    : 16, 32, 64 or 128, and at most 64 when D = 256.
 * Returns FA_OK (enqueued), FA_ERR_INVALID_ARG (null / misaligned pointer,
 * a size <= 0, H % Hkv != 0, bad dtype / causal / scale),
 * FA_ERR_UNSUPPORTED (D or page_size not supported, sizes past 32-bit
 * indexing), FA_ERR_DEVICE or FA_ERR_CUDA.
 */
/*
 * Paged cache write (ReshapeAndCache).  Source: «把 FlashAttention 搬上昇腾»,
 * the contest section's ReshapeAndCache part: token t's K and V go to block
 * slot_mapping[t] / page_size at offset slot_mapping[t] % page_size of the
 * caches; a negative slot skips the token.
 *   k_new, v_new : [tokens, Hkv, D] 16-bit (fp16 or bf16; copied bit for
 *                  bit), contiguous, 16-byte aligned.
 *   slot_mapping : int64 [tokens], device memory.  Slots >= num_pages *
 *                  page_size are skipped as well (never written out of
 *                  bounds).
 *   k_cache,
 *   v_cache      : [num_pages, page_size, Hkv, D], same element type,
 *                  written in place.
 * tokens == 0 enqueues nothing.  Two tokens with the same slot: one of them
 * wins (unspecified which).  Returns FA_OK, FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED (D not 64/128/256), FA_ERR_DEVICE or FA_ERR_CUDA.
 */
FA_API int fa_reshape_and_cache(const void* k_new, const void* v_new, const long long* slot_mapping, void* k_cache,
                                void* v_cache, int tokens, int Hkv, int D, int num_pages, int page_size,
                                cudaStream_t stream);

FA_API int fa_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                        const int* context_lens, void* o, float* lse, int B, int H, int Hkv, int Nq, int D,
                        int num_pages, int page_size, int max_pages, int causal, float scale, int dtype,
                        cudaStream_t stream);

/*
 * Paged forward with each sequence's key range split into slices, for calls
 * with too few (sequence, head) work items to fill the GPU (decode with a
 * small batch and long contexts).  Source: «把 FlashAttention 搬上昇腾», §一
 * -- the online softmax merges blocks of keys through a running max and sum;
 * whole slices of keys merge the same way: slice s reports lse_s and its own
 * normalised O_s, and lse = log sum_s exp(lse_s), O = sum_s exp(lse_s - lse)
 * O_s.  The result equals fa_fwd_paged's up to rounding.
 *
 *   all arguments as fa_fwd_paged, plus
 *   num_splits      : slices per work item, 1 .. 256; a work item with T key
 *                     tiles (128 keys, 64 at D = 256) uses min(num_splits, T)
 *                     balanced slices.  1 runs fa_fwd_paged's path.
 *   workspace       : device memory of at least
 *                     fa_fwd_paged_split_workspace_size(B, H, Nq, D,
 *                     num_splits) bytes, 16-byte aligned, caller-owned, only
 *                     used by this call on `stream` (fp32 per-slice lse and O).
 *
 * Launches the paged kernel over (work item, slice) units, then a merge
 * kernel that writes o and lse.  Errors as fa_fwd_paged, plus
 * FA_ERR_INVALID_ARG for num_splits out of range and FA_ERR_WORKSPACE for a
 * missing, misaligned or short workspace.
 */
FA_API int fa_fwd_paged_split(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                              const int* context_lens, void* o, float* lse, void* workspace, size_t workspace_bytes,
                              int B, int H, int Hkv, int Nq, int D, int num_pages, int page_size, int max_pages,
                              int num_splits, int causal, float scale, int dtype, cudaStream_t stream);

/* Bytes of workspace fa_fwd_paged_split needs (0 for invalid arguments). */
FA_API size_t fa_fwd_paged_split_workspace_size(int B, int H, int Nq, int D, int num_splits);

/*
 * A slice count for fa_fwd_paged_split on the current device: the largest
 * that keeps every (work item, slice) unit in one wave of the SM count (1
 * when the work items alone fill the GPU), at most the key tiles of the
 * longest context (max_pages * page_size keys) and 256.  Returns 1 for
 * invalid arguments.
 */
FA_API int fa_fwd_paged_split_count(int B, int H, int Hkv, int Nq, int D, int page_size, int max_pages, int causal);

/*
 * Forward over selected blocks of a paged cache.  Source: «把 FlashAttention
 * 搬上昇腾», the contest section's Quest Sparse Attention part: only the
 * chosen (Top-K) blocks of a sequence get exact attention, read through the
 * paged mapping, with per-sequence context lengths and grouped heads.  The
 * choice itself (block scoring, Top-K) is an input of this call.
 *
 *   q, o, lse, k_cache, v_cache, page_size, causal, dtype : as fa_fwd_paged.
 *   sel_pages    : int32 [B, Hkv, max_sel], device: physical pages of the
 *                  selected blocks of sequence b for K/V head kvh.
 *   sel_blocks   : int32 [B, Hkv, max_sel], device: the logical block each
 *                  of them holds (row r is the token at position block *
 *                  page_size + r).
 *   sel_count    : int32 [B, Hkv], device: entries in use (clamped to
 *                  [0, max_sel]).
 *   context_lens : int32 [B], device: tokens at positions >= context_lens[b]
 *                  never take part (the last block's invalid tokens); with
 *                  causal, the queries are the last Nq tokens of the context
 *                  and see positions up to their own.
 * Selected blocks may come in any order.  A query row that sees no selected
 * token gets O = 0 and lse = -inf.  Errors as for fa_fwd_paged.
 */
FA_API int fa_fwd_sparse(const void* q, const void* k_cache, const void* v_cache, const int* sel_pages,
                         const int* sel_blocks, const int* sel_count, const int* context_lens, void* o, float* lse,
                         int B, int H, int Hkv, int Nq, int D, int num_pages, int page_size, int max_sel, int causal,
                         float scale, int dtype, cudaStream_t stream);

FA_API size_t fa_bwd_ex_workspace_size(int Z, int H, int Hkv, int Nq, int Nk, int D, int causal);

FA_API int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int Z,
                     int H, int Hkv, int Nq, int Nk, int D, int causal, float scale, int dtype, cudaStream_t stream);

/*
 * Backward pass that allocates nothing and takes no workspace.
 *
 * The attention pages have no counterpart to this call; it exists for
 * callers that cannot allocate device memory when they run the backward --
 * for example code that runs inside a fixed memory pool or arena it does not
 * own, or an embedding host whose allocator must not be re-entered.
 *
 * It computes exactly what fa_bwd computes (same kernels, same arguments
 * without workspace/workspace_bytes, same outputs bit for bit), but the
 * scratch that fa_bwd takes from the caller (Delta and the log2-scaled
 * lse) lives in one static device buffer of FA_NOALLOC_SCRATCH_BYTES (64 MiB)
 * compiled into libfa.so.  Every GPU on which the library is used holds that
 * buffer until the process exits.
 *
 *   Limit  : fa_bwd_workspace_size(Z,H,N,D,causal) (about 8*Z*H*N bytes) must
 *            fit in the buffer; otherwise FA_ERR_SCRATCH_LIMIT is returned
 *            before anything is enqueued.
 *   Set-up : the first call on a device (with that device current) looks up
 *            the buffer's device address; make that first call before any
 *            stream capture.
 *   Sharing: all calls share the one buffer and it keeps the last call's
 *            contents.  Nothing in it needs clearing -- each call writes
 *            every scratch element it reads -- but calls whose kernels may
 *            overlap on the GPU (different streams, other host threads)
 *            race on it: serialise them.
 * Returns FA_OK or a negative FA_ERR_* code.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64ull << 20)
FA_API int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, int Z, int H, int N, int D, int causal,
                          float scale, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: FA_OK, FA_ERR_TIMEOUT (a kernel wait gave up; the
 * outputs of the calls since the last check are invalid) or FA_ERR_CUDA.
 */
FA_API int fa_device_status(cudaStream_t stream);

/*
 * Like fa_device_status but also returns the raw status word (timeout site in
 * bits 8 and up) through *raw when raw is not NULL.
 */
FA_API int fa_device_status_raw(cudaStream_t stream, int* raw);

/*
 * Self-test of the failure-detection path: enqueues one tiny kernel on
 * `stream` that waits on a shared-memory barrier nothing ever signals, using
 * the same bounded wait as every kernel of the library.  The wait gives up
 * after about one second, records FA_ERR_TIMEOUT with site code 200 in the
 * device status word and the kernel returns normally, so the context stays
 * usable.  Callers then see FA_ERR_TIMEOUT from fa_device_status().
 * Returns FA_OK once enqueued, FA_ERR_CUDA or FA_ERR_DEVICE otherwise.
 */
FA_API int fa_selftest_wait_timeout(cudaStream_t stream);

/* Static, human-readable description of an FA_* code. */
FA_API const char* fa_error_string(int code);

/*
 * Number of (query tile, key tile) pairs one head's pass visits with the
 * dense forward's tiling (128-row query tiles and 128-key tiles for every D,
 * the last of each possibly partial): the causal loop bound of §八 (T*T tiles
 * non-causal, 1+2+...+T causal for square tiles).  Host-only helper used
 * for the FLOP model; -1 on bad arguments.
 */
FA_API long long fa_fwd_tile_count(int N, int D, int causal);

/*
 * Algorithmic FLOPs of one call over all heads (the work the method must do,
 * not counting what it avoids): forward 4*N*N*D non-causal, 2*N*(N+1)*D
 * causal, per head; backward 2.5x that (five GEMMs incl. the recompute of P).
 */
FA_API double fa_fwd_flops(int Z, int H, int N, int D, int causal);
FA_API double fa_bwd_flops(int Z, int H, int N, int D, int causal);

/*
 * The same for the fa_fwd_ex / fa_bwd_ex shapes: 4*D per visible (query,
 * key) pair per query head, Nq*Nk pairs non-causal, Nq*(Nq+1)/2 +
 * Nq*(Nk-Nq) causal; backward 2.5x.
 */
FA_API double fa_fwd_ex_flops(int Z, int H, int Nq, int Nk, int D, int causal);
FA_API double fa_bwd_ex_flops(int Z, int H, int Nq, int Nk, int D, int causal);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */

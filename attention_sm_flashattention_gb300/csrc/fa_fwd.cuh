// FlashAttention forward for sm_103a: persistent, warp-specialised, TMA-fed,
// tcgen05 MMAs accumulating in TMEM.
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
// §一 -- one Q tile stays on chip and streams K/V tiles; the online softmax
// keeps the running row max m, the denominator l and the unnormalised fp32
// accumulator, rescaling l and acc when the max moves; exp2 with log2(e)
// folded into the scale; m, l, acc in fp32 and P rounded to fp16 before the
// matrix unit; causal shortens the key-tile loop and masks only diagonal
// tiles; D = 256 keeps two 128-wide accumulator halves; O is written once.
//
// Roles (512 threads, one CTA per SM):
//   warps 0-7   softmax: two warpgroups split the columns of each tile; thread
//               (g, r) owns query row r and half g of the key columns of S.
//               Both halves of a row read the whole S row to take the same
//               row max (TMEM reads are cheap), then each exponentiates its
//               own half and keeps its own partial l.  They write P (fp16)
//               back to TMEM and rescale O when m moved; at the end of an
//               item they publish l and m and go straight on to the next
//               item.
//   warps 8-11  epilogue: O / l -> fp16 into the item's (now unused) Q
//               buffer, lse; this overlaps the softmax of the next item.
//               Warp 8 then writes the tile out with a TMA store and
//               releases the Q buffer.  (Split key ranges: fp32 O / l and
//               lse of the slice straight to global memory instead.)
//   warp 12     TMA producer: Q tile per work item, K tiles into a ring.
//   warp 13     QK^T issuer (converged warp, one elected lane per MMA) and
//               TMEM owner.  It walks the CTA's tiles as one flat sequence
//               (across work items) and issues S = Q K^T up to two tiles
//               ahead of P V, into one of two S buffers.
//   warp 14     TMA producer: V tiles into their own ring.
//   warp 15     P V issuer: O += P V (P read from TMEM) as soon as a tile's
//               P is ready, over the same flat tile sequence.
// The softmax warpgroups run with more registers than the others
// (setmaxnreg), since they hold a whole S half-row and its P.
#pragma once

#include "fa_kernels.h"
#include "ptx.cuh"

namespace fa {

template <int D, bool CAUSAL>
struct FwdTraits {
  static constexpr int BM = 128;                    // query rows per tile
  static constexpr int BN = (D == 256) ? 64 : 128;  // keys per tile
  // K is released right after Q K^T, V only after P V (a softmax later), so
  // the two tiles travel in separate rings, each with its own producer warp.
  static constexpr int K_STAGES = (D == 64) ? 4 : (D == 128) ? 2 : 3;
  static constexpr int V_STAGES = (D == 64) ? 4 : 2;
  static constexpr int Q_STAGES = (D == 256) ? 1 : 3;
  static constexpr int DSUB = D / 64;               // 64-column sub-tiles per row
  static constexpr int Q_SUB = BM * 128;            // bytes of a [BM x 64] fp16 sub-tile
  static constexpr int KV_SUB = BN * 128;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OH = (D > 128) ? 128 : D;    // width of one O accumulator half
  static constexpr int NOH = D / OH;                // number of O halves
  // TMEM columns (fp32 columns; 512 allocated)
  static constexpr int S_COL = 0;       // S buffer b: [b*BN, b*BN + BN)
  static constexpr int P_COL = 2 * BN;  // P buffer b: [2BN + b*BN/2, +BN/2) packed fp16 pairs
  static constexpr int O_COL = 3 * BN;  // O: [3BN, 3BN + D)
  static constexpr int TMEM_COLS = 512;
  static_assert(O_COL + D <= TMEM_COLS, "TMEM budget");
  // shared memory layout (offsets from a 1024-byte aligned base)
  static constexpr int SM_Q = 0;
  static constexpr int SM_K = SM_Q + Q_STAGES * Q_BYTES;
  static constexpr int SM_V = SM_K + K_STAGES * KV_BYTES;
  // partial row sums l of both column halves and the row max m of the item
  // the epilogue works on next
  static constexpr int SM_LM = SM_V + V_STAGES * KV_BYTES;  // [3][128] fp32
  static constexpr int SM_BAR = SM_LM + 3 * BM * 4;
  static constexpr int SM_BYTES = SM_BAR + 512;
  // never below 120 KB so that a second CTA can never share the SM (each
  // CTA takes all 512 TMEM columns)
  static constexpr int SMEM_ALLOC = (SM_BYTES > 120 * 1024) ? SM_BYTES : 120 * 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static constexpr int THREADS = 512;
  static constexpr int SOFTMAX_THREADS = 256;
  static constexpr int EPI_THREADS = 128;  // warps 8-11
  static constexpr int PRODUCER_WARP = 12;  // Q and K
  static constexpr int MMA_WARP = 13;
  static constexpr int V_PRODUCER_WARP = 14;
  static constexpr int PV_MMA_WARP = 15;
  // registers per thread after the split (launch: 65536 / 512 = 128):
  // 256 x 184 + 256 x 64 = 63488 <= 65536
  static constexpr int SOFTMAX_REGS = 184;
  static constexpr int OTHER_REGS = 64;
};

// Threshold (log2 units) of the lazy online-softmax rescale.
constexpr float kRescaleLog2 = 8.0f;

// Barrier slots inside the SM_BAR area.
struct FwdBars {
  uint64_t q_full[3], q_empty[3];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], s_free[2], p_full[2];
  uint64_t o_free, mma_done[2];
  // P V of a tile that used P buffer b completed (and with it every earlier
  // P V).  Waits name the tile's buffer and phase, never "the latest P V":
  // Q K^T of later tiles is issued ahead of P V, so a completed S does not
  // imply that all earlier P V completed, and one shared barrier could be
  // two phases behind.
  uint64_t pv_done[2];
  uint64_t epi_full[3];  // O tile written into Q buffer b
  uint64_t lm_full, lm_empty;  // l, m of one item, handed to the epilogue warps
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(FwdBars) <= 512, "barrier area");

// Static schedule.  Non-causal: one work unit per (head, query tile), head
// major so that the CTAs running at the same time share K/V through L2.
// Causal: one unit pairs query tiles qt and nqt-1-qt of the same head, so
// every unit costs the same number of key tiles (nqt + 1 for square tiles)
// and a static stride over units balances the SMs.
template <bool CAUSAL>
__device__ __forceinline__ int fwd_num_units(int heads, int nqt) {
  return CAUSAL ? heads * ((nqt + 1) / 2) : heads * nqt;
}

template <bool CAUSAL>
__device__ __forceinline__ void fwd_decode(int u, int nqt, int& head, int& qa, int& qb) {
  if (CAUSAL) {
    const int npair = (nqt + 1) / 2;
    head = u / npair;
    const int p = u - head * npair;
    qa = nqt - 1 - p;
    qb = (p != qa) ? p : -1;
  } else {
    head = u / nqt;
    qa = u - head * nqt;
    qb = -1;
  }
}

// Key tiles query tile qt visits: all of them, or (causal) those up to the
// last key its last row sees, key (qt + 1) * BM - 1 + off.
template <int D, bool CAUSAL>
__device__ __forceinline__ int fwd_num_kv(int qt, int nkv_full, int Nk, int off) {
  using T = FwdTraits<D, CAUSAL>;
  if (!CAUSAL) return nkv_full;
  const int end = min((qt + 1) * T::BM + off, Nk);  // one past the last visible key
  return (end + T::BN - 1) / T::BN;
}

// Last key row `qi` sees (Nk - 1, or qi + off when causal).  A tile whose
// last key is past the smallest such limit over its rows needs the mask.
template <bool CAUSAL>
__device__ __forceinline__ int fwd_key_limit(int qi, int Nk, int off) {
  return CAUSAL ? min(qi + off, Nk - 1) : Nk - 1;
}

// Work modes of the forward kernel: K/V dense [heads / group, Nk, D]; a
// paged cache read in key order through a block table; a paged cache read
// through a per-(sequence, K/V head) list of selected blocks; the paged
// cache with every work item's key tiles split into slices that are
// separate work units writing partial results (FwdParams::splits).
enum FwdMode : int { kDense = 0, kPaged = 1, kSparse = 2, kPagedSplit = 3 };

// Work units of a launch: the schedule's units, times the key-range slices
// in split mode; unit u is then slice u % splits of schedule unit u / splits.
template <bool CAUSAL, int MODE>
__device__ __forceinline__ int fwd_units(const FwdParams& prm, int nqt) {
  return fwd_num_units<CAUSAL>(prm.heads, nqt) * (MODE == kPagedSplit ? prm.splits : 1);
}

template <bool CAUSAL, int MODE>
__device__ __forceinline__ void fwd_unit(const FwdParams& prm, int u, int nqt, int& head, int& qa, int& qb,
                                         int& split) {
  split = 0;
  if (MODE == kPagedSplit) {
    split = u % prm.splits;
    u /= prm.splits;
  }
  fwd_decode<CAUSAL>(u, nqt, head, qa, qb);
}

// Key count, causal offset and key tiles of the work items of query head
// `head`.  Dense: the call's Nk.  Paged: the sequence's context length,
// clamped to [causal ? Nq : 1, max_pages * page_size].  Sparse: key slots of
// the selected blocks (at least one block, so that every item has a tile);
// `ctx` is the context length that the keys' logical positions are masked
// against, `sel` the number of selected blocks.
// Key tiles of query tile qt: all of them when sparse, or when packed
// grouped heads put every query position in every tile (then up to the last
// key the last position sees); otherwise fwd_num_kv.
template <int D, bool CAUSAL, int MODE>
__device__ __forceinline__ int fwd_item_tiles(int qt, int nkv_full, int nk, int off, int qp) {
  if (MODE == kSparse) return nkv_full;
  if (CAUSAL && qp > 0) return (min(qp + off, nk) + FwdTraits<D, CAUSAL>::BN - 1) / FwdTraits<D, CAUSAL>::BN;
  return fwd_num_kv<D, CAUSAL>(qt, nkv_full, nk, off);
}

// The key tiles a work unit visits for query tile qt: [j0, j0 + return).
// Without splitting, all of the item's tiles from 0.  Split: slice `split`
// of min(splits, tiles) balanced slices of them (each slice non-empty), and
// none for a slice index past that.
template <int D, bool CAUSAL, int MODE>
__device__ __forceinline__ int fwd_range(int qt, int nkv_full, int nk, int off, int qp, int split, int nsplit,
                                         int& j0) {
  const int total = fwd_item_tiles<D, CAUSAL, MODE>(qt, nkv_full, nk, off, qp);
  j0 = 0;
  if (MODE != kPagedSplit) return total;
  const int ns = min(nsplit, total);
  if (split >= ns) return 0;
  j0 = split * total / ns;
  return (split + 1) * total / ns - j0;
}

template <int D, bool CAUSAL, int MODE>
struct FwdItemShape {
  int nk, off, nkv_full, ctx, sel, qp, split, nsplit;
  __device__ __forceinline__ FwdItemShape(const FwdParams& prm, int head, int split_ = 0) {
    int n = prm.Nk;
    ctx = 0;
    sel = 0;
    qp = prm.q_period;
    split = split_;
    nsplit = MODE == kPagedSplit ? prm.splits : 1;
    const int nq_pos = qp > 0 ? qp : prm.Nq;  // query positions per head
    if (MODE == kPaged || MODE == kPagedSplit) {
      n = __ldg(prm.context_lens + head / prm.H);
      n = min(max(n, CAUSAL ? nq_pos : 1), prm.max_pages * prm.page_size);
    } else if (MODE == kSparse) {
      const int b = head / prm.H, kvh = (head % prm.H) / prm.group;
      ctx = max(__ldg(prm.context_lens + b), 0);
      sel = min(max(__ldg(prm.sel_count + b * prm.Hkv + kvh), 0), prm.max_pages);
      n = max(sel, 1) * prm.page_size;
    }
    nk = n;
    off = (MODE == kSparse ? ctx : n) - nq_pos;
    nkv_full = (n + FwdTraits<D, CAUSAL>::BN - 1) / FwdTraits<D, CAUSAL>::BN;
  }
  // key tiles of query tile qt (selected blocks carry arbitrary positions,
  // so the causal bound does not shorten a sparse item)
  __device__ __forceinline__ int tiles(int qt) const { return fwd_item_tiles<D, CAUSAL, MODE>(qt, nkv_full, nk, off, qp); }
  // this unit's tiles of query tile qt: [j0, j0 + return)
  __device__ __forceinline__ int range(int qt, int& j0) const {
    return fwd_range<D, CAUSAL, MODE>(qt, nkv_full, nk, off, qp, split, nsplit, j0);
  }
};

// Sparse mode: which of key tile j's BN columns query row qi may see, as a
// bit mask over BN / 32 words (bit c of word w = column 32 w + c).  Column c
// is row c % page_size of list entry j * BN / page_size + c / page_size,
// logical position block * page_size + c % page_size; it is visible iff the
// entry is selected and the position is at most the row's limit (the last
// context position, or the query's own position when causal).  Within an
// entry the visible rows are a prefix, so each entry adds one bit range.
template <int D, bool CAUSAL>
__device__ __forceinline__ void fwd_sparse_mask(const FwdParams& prm, int head, int j, int sel, int limit,
                                                uint32_t* mask) {
  using T = FwdTraits<D, CAUSAL>;
  constexpr int W = T::BN / 32;
  const int ps = prm.page_size, epb = T::BN / ps;
  const int b = head / prm.H, kvh = (head % prm.H) / prm.group;
  const int* blk = prm.sel_blocks + (static_cast<size_t>(b) * prm.Hkv + kvh) * prm.max_pages;
#pragma unroll
  for (int w = 0; w < W; ++w) mask[w] = 0u;
#pragma unroll
  for (int e = 0; e < T::BN / 16; ++e) {
    if (e >= epb) break;
    const int eg = j * epb + e;
    if (eg >= sel) break;
    const int n = min(max(limit - __ldg(blk + eg) * ps + 1, 0), ps);  // visible rows of the entry
    const int lo = e * ps, hi = lo + n;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const int a = max(lo - 32 * w, 0), z = min(hi - 32 * w, 32);
      if (z > a) mask[w] |= (z - a == 32 ? 0xffffffffu : ((1u << (z - a)) - 1u)) << a;
    }
  }
}

// Bounded wait that ignores the abort flag: used only while draining at exit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_test(a, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// The CTA's tiles in the order it processes them: work items (query tiles)
// in schedule order, the key tiles of each item in order.  Global tile index
// `tile` also indexes the K and V rings, which hold one tile per key tile.
template <int D, bool CAUSAL, int MODE>
struct FwdCursor {
  int u, half, head, qt, qb, j, nkv, j0, split;  // j: index within the unit's tiles; key tile j0 + j
  uint32_t item, tile;
  bool valid;
  int units, nqt, nkv_full, Nk, off, ctx, sel, qp;
  const FwdParams* prm;

  __device__ void start(int first_unit, int units_, int nqt_, const FwdParams* prm_) {
    units = units_;
    nqt = nqt_;
    prm = prm_;
    item = 0;
    tile = 0;
    j = 0;
    j0 = 0;
    u = first_unit;
    half = 0;
    load_unit();
  }
  __device__ int range(int q) {
    if (MODE != kPagedSplit) return fwd_item_tiles<D, CAUSAL, MODE>(q, nkv_full, Nk, off, qp);
    return fwd_range<D, CAUSAL, MODE>(q, nkv_full, Nk, off, qp, split, prm->splits, j0);
  }
  __device__ void load_unit() {
    if constexpr (MODE != kPagedSplit) {
      valid = u < units;
      if (!valid) return;
      int qa;
      fwd_decode<CAUSAL>(u, nqt, head, qa, qb);
      const FwdItemShape<D, CAUSAL, MODE> sh(*prm, head);
      Nk = sh.nk;
      off = sh.off;
      nkv_full = sh.nkv_full;
      ctx = sh.ctx;
      sel = sh.sel;
      qp = sh.qp;
      qt = qa;
      half = 0;
      nkv = fwd_item_tiles<D, CAUSAL, MODE>(qt, nkv_full, Nk, off, qp);
    } else {
      load_split_unit();
    }
  }
  // split mode: the next unit (from u on) with at least one tile; only split
  // units can have none, and every role skips them the same way
  __device__ void load_split_unit() {
    for (;;) {
      valid = u < units;
      if (!valid) return;
      int qa;
      fwd_unit<CAUSAL, MODE>(*prm, u, nqt, head, qa, qb, split);
      const FwdItemShape<D, CAUSAL, MODE> sh(*prm, head, split);
      Nk = sh.nk;
      off = sh.off;
      nkv_full = sh.nkv_full;
      ctx = sh.ctx;
      sel = sh.sel;
      qp = sh.qp;
      qt = qa;
      half = 0;
      nkv = range(qt);
      if (nkv > 0) return;
      if (qb >= 0) {
        half = 1;
        qt = qb;
        nkv = range(qt);
        if (nkv > 0) return;
      }
      u += gridDim.x;
    }
  }
  __device__ void advance() {
    ++tile;
    if (++j < nkv) return;
    j = 0;
    ++item;
    if constexpr (MODE != kPagedSplit) {
      if (half == 0 && qb >= 0) {
        half = 1;
        qt = qb;
        nkv = fwd_item_tiles<D, CAUSAL, MODE>(qt, nkv_full, Nk, off, qp);
      } else {
        u += gridDim.x;
        load_unit();
      }
    } else {
      if (half == 0 && qb >= 0) {
        half = 1;
        qt = qb;
        nkv = range(qt);
        if (nkv > 0) return;
      }
      u += gridDim.x;
      load_unit();
    }
  }
};

// One K or V tile (BN keys, tile j of query head `head`) from the paged
// cache: BN / page_size boxes per 64-column sub-tile, box p going to rows
// [p * page_size, (p + 1) * page_size) of the sub-tile (page_size is a
// multiple of 8, so every box starts on a 1024-byte swizzle atom).  Pages
// wholly past the sequence's key count get an out-of-range page coordinate,
// which TMA fills with zeros; so does a block-table entry outside [0,
// num_pages).  Every box counts its full size towards the barrier.
// Sparse mode: the tile's pages are entries j * BN / page_size ... of the
// item's selected-block list; entries past the selection count load zeros.
template <int D, bool CAUSAL, int MODE>
__device__ __forceinline__ void fwd_load_paged_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                                    const FwdParams& prm, int head, int j, int nk, int sel,
                                                    uint64_t pol) {
  using T = FwdTraits<D, CAUSAL>;
  const int ps = prm.page_size;
  const int ppt = T::BN / ps;                  // pages per tile
  const int b = head / prm.H, kvh = (head % prm.H) / prm.group;
  const int lp0 = j * (T::BN / ps);            // first logical page (list entry) of the tile
  const int* row = MODE == kSparse ? prm.sel_pages + (static_cast<size_t>(b) * prm.Hkv + kvh) * prm.max_pages
                                   : prm.block_table + static_cast<size_t>(b) * prm.max_pages;
  for (int pg = 0; pg < ppt; ++pg) {
    const int lp = lp0 + pg;
    const bool live = MODE == kSparse ? lp < sel : lp * ps < nk;
    const int page = live ? __ldg(row + lp) : prm.num_pages;
    for (int s = 0; s < T::DSUB; ++s)
      tma_load_4d_hint(dst + s * T::KV_SUB + pg * ps * 128, map, bar, s * 64, kvh, 0, page, pol);
  }
}

template <int D, bool CAUSAL, bool BF, int MODE>
__global__ void __launch_bounds__(512, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams prm) {
  using T = FwdTraits<D, CAUSAL>;
  constexpr bool PAGED = MODE != kDense;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128-byte-swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) record_timeout(prm.status, 99);
    return;
  }
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + T::SM_BAR);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars->q_full[i], 1);
      // a Q buffer is free once its last Q K^T completed (MMA commit) and the
      // O tile written into it has been stored (store warp)
      mbar_init(&bars->q_empty[i], 2);
      mbar_init(&bars->epi_full[i], T::EPI_THREADS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], T::SOFTMAX_THREADS);
      mbar_init(&bars->p_full[i], T::SOFTMAX_THREADS);
    }
    mbar_init(&bars->lm_full, T::SOFTMAX_THREADS);
    mbar_init(&bars->lm_empty, T::EPI_THREADS);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    mbar_init(&bars->pv_done[0], 1);
    mbar_init(&bars->pv_done[1], 1);
    mbar_init(&bars->o_free, T::EPI_THREADS);
    mbar_init(&bars->mma_done[0], 1);
    mbar_init(&bars->mma_done[1], 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == T::MMA_WARP) {
    tmem_alloc(&bars->tmem_base, T::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == T::PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  const int Nq = prm.Nq;
  const int nqt = (Nq + T::BM - 1) / T::BM;
  const int units = fwd_units<CAUSAL, MODE>(prm, nqt);
  // split mode: a row can see no key of its slice; it then keeps m = -inf
  // and l = 0 (an empty partial softmax), as a sparse row can
  constexpr bool kEmptyRows = MODE == kSparse || MODE == kPagedSplit;

  if (warp < 8) {
    reg_alloc<T::SOFTMAX_REGS>();
      // ----------------------------------------------------- softmax warps
      constexpr int HC = T::BN / 2;  // S columns per thread
      constexpr int HD = D / 2;      // O columns per thread
      const int wg = warp >> 2;      // column half
      const int quad = warp & 3;
      const int r = quad * 32 + lane;  // query row inside the tile, == TMEM lane
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      float* lm = reinterpret_cast<float*>(smem + T::SM_LM);
      const float sl2 = prm.scale_log2;
      uint32_t t = 0, q_item = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int head, qa, qb, sp;
        fwd_unit<CAUSAL, MODE>(prm, u, nqt, head, qa, qb, sp);
        const FwdItemShape<D, CAUSAL, MODE> sh(prm, head, sp);
        const int Nk = sh.nk, off = sh.off;
        for (int half = 0; ok && half < 2; ++half) {
          const int qt = half ? qb : qa;
          if (qt < 0) break;
          int j0 = 0;
          const int nkv = MODE == kPagedSplit ? sh.range(qt, j0) : sh.tiles(qt);
          if (MODE == kPagedSplit && nkv == 0) continue;
          const int jb = MODE == kPagedSplit ? j0 : 0;  // the unit's first key tile
          const int qi = qt * T::BM + r;  // query row within the head
          const int qpos = sh.qp > 0 ? qi % sh.qp : qi;  // its query position
          const int lim = fwd_key_limit<CAUSAL>(qpos, Nk, off);  // this row's last key
          // the tile's smallest limit (packed heads: every tile holds position 0)
          const int lim_lo = fwd_key_limit<CAUSAL>(sh.qp > 0 ? 0 : qt * T::BM, Nk, off);
          // sparse: the row's last visible logical position
          const int slim = CAUSAL ? min(qpos + sh.off, sh.ctx - 1) : sh.ctx - 1;
          float m = -INFINITY, l = 0.f;   // l: this half's partial row sum
          for (int j = jb; j < jb + nkv; ++j) {
            uint32_t vis[T::BN / 32];  // sparse: visible columns of this tile
            if (MODE == kSparse) fwd_sparse_mask<D, CAUSAL>(prm, head, j, sh.sel, slim, vis);
            const int b = t & 1;
            ok = mbar_wait(&bars->s_full[b], (t >> 1) & 1, wc, 5);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // other half of the row: only its max is needed
            uint32_t sr[HC];
            float pm[8];
  #pragma unroll
            for (int c = 0; c < HC; c += 32) tmem_ld32(lane_base + T::S_COL + b * T::BN + (wg ^ 1) * HC + c, sr + c);
            tmem_wait_ld();
            reg_fence<HC>(sr);
            if (MODE == kSparse) {
  #pragma unroll
              for (int c = 0; c < HC; ++c) {
                const uint32_t wv = (wg ^ 1) ? vis[(HC + c) / 32] : vis[c / 32];
                if (!((wv >> (c % 32)) & 1u)) sr[c] = __float_as_uint(-INFINITY);
              }
            } else if ((j + 1) * T::BN - 1 > lim_lo) {
              if constexpr (CAUSAL) {
                // visibility as one bit per column of each 32-column word
                const int nv = lim - (j * T::BN + (wg ^ 1) * HC) + 1;  // visible columns of the half
  #pragma unroll
                for (int w = 0; w < HC / 32; ++w) {
                  const int n = min(max(nv - 32 * w, 0), 32);
                  const uint32_t keep = n == 32 ? 0xffffffffu : ((1u << n) - 1u);
  #pragma unroll
                  for (int c = 0; c < 32; ++c)
                    sr[32 * w + c] = ((keep >> c) & 1u) ? sr[32 * w + c] : __float_as_uint(-INFINITY);
                }
              } else {
                const int k0 = j * T::BN + (wg ^ 1) * HC;
  #pragma unroll
                for (int c = 0; c < HC; ++c)
                  if (k0 + c > lim) sr[c] = __float_as_uint(-INFINITY);
              }
            }
  #pragma unroll
            for (int i = 0; i < 8; ++i) pm[i] = fmaxf(__uint_as_float(sr[i]), __uint_as_float(sr[i + 8]));
  #pragma unroll
            for (int c = 16; c < HC; c += 16)
  #pragma unroll
              for (int i = 0; i < 8; ++i) pm[i] = fmax3(pm[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
            // own half
  #pragma unroll
            for (int c = 0; c < HC; c += 32) tmem_ld32(lane_base + T::S_COL + b * T::BN + wg * HC + c, sr + c);
            tmem_wait_ld();
            reg_fence<HC>(sr);
            tc_fence_before();
            mbar_arrive(&bars->s_free[b]);  // S buffer b may take the S of tile t + 2
            float s[HC];
  #pragma unroll
            for (int c = 0; c < HC; ++c) s[c] = __uint_as_float(sr[c]);
            if (MODE == kSparse) {
  #pragma unroll
              for (int c = 0; c < HC; ++c) {
                const uint32_t wv = wg ? vis[(HC + c) / 32] : vis[c / 32];
                if (!((wv >> (c % 32)) & 1u)) s[c] = -INFINITY;
              }
            } else if ((j + 1) * T::BN - 1 > lim_lo) {
              if constexpr (CAUSAL) {
                const int nv = lim - (j * T::BN + wg * HC) + 1;
  #pragma unroll
                for (int w = 0; w < HC / 32; ++w) {
                  const int n = min(max(nv - 32 * w, 0), 32);
                  const uint32_t keep = n == 32 ? 0xffffffffu : ((1u << n) - 1u);
  #pragma unroll
                  for (int c = 0; c < 32; ++c)
                    s[32 * w + c] = ((keep >> c) & 1u) ? s[32 * w + c] : -INFINITY;
                }
              } else {
                const int k0 = j * T::BN + wg * HC;
  #pragma unroll
                for (int c = 0; c < HC; ++c)
                  if (k0 + c > lim) s[c] = -INFINITY;
              }
            }
  #pragma unroll
            for (int c = 0; c < HC; c += 16)
  #pragma unroll
              for (int i = 0; i < 8; ++i) pm[i] = fmax3(pm[i], s[c + i], s[c + 8 + i]);
            const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
            // The running max m only moves when this tile's max exceeds it by
            // more than kRescaleLog2: below that the stale m keeps every P value
            // under 2^kRescaleLog2 (exact range for fp16 P and fp32 l), so O and
            // l need no rescaling.  O / l and lse use the max actually applied,
            // which gives the same result as always tracking the exact max.
            // Both halves of a row compute the same row max, so they take the
            // same decision.
            const float m_tile = mx * sl2;
            const float m_new = (m_tile > m + kRescaleLog2) ? m_tile : m;
            // sparse: a row that has seen no visible key yet keeps m = -inf;
            // its P must be 0, not exp2(-inf + inf)
            const float neg = (kEmptyRows && m_new == -INFINITY) ? 0.f : -m_new;
            // x = s * c - m and the row sum in packed fp32 pairs (one f32x2
            // instruction per two columns)
            const uint64_t c2 = f2_pack(sl2, sl2), neg2 = f2_pack(neg, neg);
            uint64_t ps2[4];
  #pragma unroll
            for (int i = 0; i < 4; ++i) ps2[i] = 0ull;
            uint32_t pk[HC / 2];
  #pragma unroll
            for (int c = 0; c < HC; c += 2) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), c2, neg2), x0, x1);
              const float p0 = ex2_approx(x0);
              const float p1 = ex2_approx(x1);
              ps2[(c >> 1) & 3] = f2_add(ps2[(c >> 1) & 3], f2_pack(p0, p1));
              pk[c / 2] = pack2<BF>(p0, p1);
            }
            float ps[8];
  #pragma unroll
            for (int i = 0; i < 4; ++i) f2_unpack(ps2[i], ps[2 * i], ps[2 * i + 1]);
            const float rs = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            const float alpha = (kEmptyRows && m_new == -INFINITY)
                                    ? 1.f
                                    : ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)
            l = l * alpha + rs;
            m = m_new;
            // P V of this tile may start while the previous P V still runs
            // (the tensor pipe executes one issuer's MMAs in order); only a
            // rescale has to wait for it.  Every wait names the barrier of
            // the tile's own P buffer and the phase of that use, and the
            // previous use of the same buffer (tile t - 3) is known to be
            // complete (waited at tile t - 1), so no wait can pass on a
            // phase two uses old.
            if (j > jb && __any_sync(0xffffffffu, alpha != 1.f)) {
              // O holds P V of the previous tiles: wait for the last P V, then
              // rescale (this half's columns of) rows whose max moved.
              ok = mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, wc, 6);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
              tc_fence_after();
              if (__any_sync(0xffffffffu, alpha != 1.f)) {
  #pragma unroll 1
                for (int c = 0; c < HD; c += 32) {
                  uint32_t o[32];
                  tmem_ld32(lane_base + T::O_COL + wg * HD + c, o);
                  tmem_wait_ld();
                  reg_fence<32>(o);
  #pragma unroll
                  for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st32(lane_base + T::O_COL + wg * HD + c, o);
                }
              }
            }
            // P buffer b was last read by the P V of tile t - 2
            if (t >= 2) {
              ok = mbar_wait(&bars->pv_done[b], ((t - 2) >> 1) & 1, wc, 15);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
              tc_fence_after();
            }
            const uint32_t pcol = lane_base + T::P_COL + b * (T::BN / 2) + wg * (HC / 2);
            if (HC / 2 == 32) {
              tmem_st32(pcol, pk);
            } else {
              tmem_st16(pcol, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[b]);
            ++t;
          }
          if (!ok) break;
          // ---- hand l (this half's partial row sum) and m to the epilogue
          // warps, once they have read the previous item's
          if (q_item >= 1) {
            ok = mbar_wait(&bars->lm_empty, (q_item - 1) & 1, wc, 14);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          }
          lm[wg * T::BM + r] = l;
          if (wg == 0) lm[2 * T::BM + r] = m;
          mbar_arrive(&bars->lm_full);
          ++q_item;
        }
      }
  } else {
    reg_dealloc<T::OTHER_REGS>();
    if (warp == T::PRODUCER_WARP) {
      // ------------------------------------------------ producer: Q and K tiles
      if (lane == 0) {
        const uint64_t pol_kv = l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_first();
        uint32_t q_it = 0, k_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
          int head, qa, qb, sp;
          fwd_unit<CAUSAL, MODE>(prm, u, nqt, head, qa, qb, sp);
          const FwdItemShape<D, CAUSAL, MODE> sh(prm, head, sp);
          for (int half = 0; ok && half < 2; ++half) {
            const int qt = half ? qb : qa;
            if (qt < 0) break;
            int j0 = 0;
            const int nkv = MODE == kPagedSplit ? sh.range(qt, j0) : sh.tiles(qt);
            if (MODE == kPagedSplit && nkv == 0) continue;
            const int qs = q_it % T::Q_STAGES;
            if (!(ok = mbar_wait(&bars->q_empty[qs], ((q_it / T::Q_STAGES) & 1) ^ 1, wc, 1))) break;
            mbar_arrive_expect_tx(&bars->q_full[qs], T::Q_BYTES);
            uint8_t* sq = smem + T::SM_Q + qs * T::Q_BYTES;
            for (int s = 0; s < T::DSUB; ++s)
              tma_load_3d_hint(sq + s * T::Q_SUB, &tm_q, &bars->q_full[qs], s * 64, qt * T::BM, head, pol_q);
            ++q_it;
            for (int j = j0; j < j0 + nkv; ++j) {
              const int st = k_it % T::K_STAGES;
              if (!(ok = mbar_wait(&bars->k_empty[st], ((k_it / T::K_STAGES) & 1) ^ 1, wc, 2))) break;
              uint8_t* sk = smem + T::SM_K + st * T::KV_BYTES;
              mbar_arrive_expect_tx(&bars->k_full[st], T::KV_BYTES);
              if (PAGED) {
                fwd_load_paged_tile<D, CAUSAL, MODE>(sk, &tm_k, &bars->k_full[st], prm, head, j, sh.nk, sh.sel, pol_kv);
              } else {
                for (int s = 0; s < T::DSUB; ++s)
                  tma_load_3d_hint(sk + s * T::KV_SUB, &tm_k, &bars->k_full[st], s * 64, j * T::BN, head / prm.group,
                                   pol_kv);
              }
              ++k_it;
            }
          }
        }
        // Drain: every load issued must have landed before the CTA may exit.
        for (uint32_t i = (k_it > T::K_STAGES ? k_it - T::K_STAGES : 0); i < k_it; ++i)
          drain_wait(&bars->k_full[i % T::K_STAGES], (i / T::K_STAGES) & 1);
        for (uint32_t i = (q_it > T::Q_STAGES ? q_it - T::Q_STAGES : 0); i < q_it; ++i)
          drain_wait(&bars->q_full[i % T::Q_STAGES], (i / T::Q_STAGES) & 1);
      }
    } else if (warp == T::V_PRODUCER_WARP) {
      // ------------------------------------------------------ producer: V tiles
      if (lane == 0) {
        const uint64_t pol_kv = l2_policy_evict_last();
        uint32_t v_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
          int head, qa, qb, sp;
          fwd_unit<CAUSAL, MODE>(prm, u, nqt, head, qa, qb, sp);
          const FwdItemShape<D, CAUSAL, MODE> sh(prm, head, sp);
          for (int half = 0; ok && half < 2; ++half) {
            const int qt = half ? qb : qa;
            if (qt < 0) break;
            int j0 = 0;
            const int nkv = MODE == kPagedSplit ? sh.range(qt, j0) : sh.tiles(qt);
            if (MODE == kPagedSplit && nkv == 0) continue;
            for (int j = j0; j < j0 + nkv; ++j) {
              const int st = v_it % T::V_STAGES;
              if (!(ok = mbar_wait(&bars->v_empty[st], ((v_it / T::V_STAGES) & 1) ^ 1, wc, 8))) break;
              uint8_t* sv = smem + T::SM_V + st * T::KV_BYTES;
              mbar_arrive_expect_tx(&bars->v_full[st], T::KV_BYTES);
              if (PAGED) {
                fwd_load_paged_tile<D, CAUSAL, MODE>(sv, &tm_v, &bars->v_full[st], prm, head, j, sh.nk, sh.sel, pol_kv);
              } else {
                for (int s = 0; s < T::DSUB; ++s)
                  tma_load_3d_hint(sv + s * T::KV_SUB, &tm_v, &bars->v_full[st], s * 64, j * T::BN, head / prm.group,
                                   pol_kv);
              }
              ++v_it;
            }
          }
        }
        for (uint32_t i = (v_it > T::V_STAGES ? v_it - T::V_STAGES : 0); i < v_it; ++i)
          drain_wait(&bars->v_full[i % T::V_STAGES], (i / T::V_STAGES) & 1);
      }
    } else if (warp == T::MMA_WARP || warp == T::PV_MMA_WARP) {
      // ------------------------------------------------------------ MMA issuers
      // The whole warp runs the loop; one elected lane issues each MMA.
      constexpr uint32_t idesc_qk = idesc_16<BF>(128, T::BN, false, false);
      constexpr uint32_t idesc_pv = idesc_16<BF>(128, T::OH, false, true);
      const uint32_t sbase = smem_u32(smem);
      bool ok = true;

      // S = Q K^T of the cursor's tile into S buffer tile % 2, which the
      // softmax of tile - 2 has read by then.
      auto issue_s = [&](const FwdCursor<D, CAUSAL, MODE>& c) -> bool {
        const int qs = c.item % T::Q_STAGES;
        const int st = c.tile % T::K_STAGES;
        const int b = c.tile & 1;
        if (c.j == 0 && !warp_wait(&bars->q_full[qs], (c.item / T::Q_STAGES) & 1, wc, 3)) return false;
        if (!warp_wait(&bars->k_full[st], (c.tile / T::K_STAGES) & 1, wc, 4)) return false;
        if (c.tile >= 2 && !warp_wait(&bars->s_free[b], ((c.tile - 2) >> 1) & 1, wc, 16)) return false;
        tc_fence_after();
        const uint64_t qdesc = sdesc_sw128(sbase + T::SM_Q + qs * T::Q_BYTES, 16, 1024);
        const uint64_t kdesc = sdesc_sw128(sbase + T::SM_K + st * T::KV_BYTES, 16, 1024);
  #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_f16_ss_warp(tmem + T::S_COL + b * T::BN, sdesc_add(qdesc, (kk / 4) * T::Q_SUB + (kk % 4) * 32),
                          sdesc_add(kdesc, (kk / 4) * T::KV_SUB + (kk % 4) * 32), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit_warp(&bars->s_full[b]);
        mma_commit_warp(&bars->k_empty[st]);
        if (c.j == c.nkv - 1) mma_commit_warp(&bars->q_empty[qs]);
        return true;
      };

      // O += P V of the cursor's tile; the first tile of an item overwrites O,
      // which the previous item's epilogue must have read.
      auto issue_pv = [&](const FwdCursor<D, CAUSAL, MODE>& c) -> bool {
        const int b = c.tile & 1;
        const int st = c.tile % T::V_STAGES;
        const bool first = (c.j == 0);
        if (first && c.item > 0 && !warp_wait(&bars->o_free, (c.item - 1) & 1, wc, 10)) return false;
        if (!warp_wait(&bars->p_full[b], (c.tile >> 1) & 1, wc, 11)) return false;
        if (!warp_wait(&bars->v_full[st], (c.tile / T::V_STAGES) & 1, wc, 12)) return false;
        tc_fence_after();
        if (MODE == kSparse) {
          // Sparse: a selected block that holds the context's end carries
          // stale cache rows past it; zero those V rows (blocks past the
          // selection count were loaded as zeros).
          const int ps = prm.page_size, epb = T::BN / ps;
          const int sb = c.head / prm.H, kvh = (c.head % prm.H) / prm.group;
          const int* blk = prm.sel_blocks + (static_cast<size_t>(sb) * prm.Hkv + kvh) * prm.max_pages;
          const uint32_t sv = smem_u32(smem + T::SM_V + st * T::KV_BYTES);
          bool wrote = false;
          for (int e = 0; e < epb; ++e) {
            const int eg = (c.j0 + c.j) * epb + e;
            if (eg >= c.sel) break;
            const int valid = min(max(c.ctx - __ldg(blk + eg) * ps, 0), ps);
            if (valid == ps) continue;
            for (int idx = lane; idx < (ps - valid) * 8 * T::DSUB; idx += 32) {
              const int row = e * ps + valid + idx / (8 * T::DSUB), rem = idx % (8 * T::DSUB);
              st_shared_v4(sv + (rem / 8) * T::KV_SUB + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
            }
            wrote = true;
          }
          if (wrote) {
            fence_proxy_async_smem();
            __syncwarp();
          }
        } else if (PAGED && (c.j0 + c.j + 1) * T::BN > c.Nk) {
          // Rows of the sequence's last page past its key count hold whatever
          // the cache holds there; P is 0 for them, but 0 * NaN is NaN, so
          // zero those V rows before P V reads them.  (Each row is the same
          // 128 bytes of its sub-tile under the 128-byte swizzle.)
          const int valid = c.Nk - (c.j0 + c.j) * T::BN;
          const uint32_t sv = smem_u32(smem + T::SM_V + st * T::KV_BYTES);
          for (int idx = lane; idx < (T::BN - valid) * 8 * T::DSUB; idx += 32) {
            const int row = valid + idx / (8 * T::DSUB), rem = idx % (8 * T::DSUB);
            st_shared_v4(sv + (rem / 8) * T::KV_SUB + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        const uint64_t vdesc = sdesc_sw128(sbase + T::SM_V + st * T::KV_BYTES, T::KV_SUB, 1024);
  #pragma unroll
        for (int kk = 0; kk < T::BN / 16; ++kk) {
  #pragma unroll
          for (int h = 0; h < T::NOH; ++h) {
            mma_f16_ts_warp(tmem + T::O_COL + h * 128, tmem + T::P_COL + b * (T::BN / 2) + kk * 8,
                            sdesc_add(vdesc, (h * 2) * T::KV_SUB + kk * 16 * 128), idesc_pv,
                            (first && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit_warp(&bars->v_empty[st]);
        mma_commit_warp(&bars->pv_done[b]);
        return true;
      };

      // Two issuing warps: this one issues Q K^T, bounded only by the two S
      // buffers (S(t + 2) as soon as the softmax has read S(t)), so it runs
      // two tiles ahead of the softmax, across work items; warp 15 issues
      // P V as each tile's P becomes ready.  Neither waits behind the
      // other's dependencies.
      FwdCursor<D, CAUSAL, MODE> c;
      c.start(blockIdx.x, units, nqt, &prm);
      const bool s_side = (warp == T::MMA_WARP);
      while (ok && c.valid) {
        ok = s_side ? issue_s(c) : issue_pv(c);
        c.advance();
      }
      // Drain: all MMAs issued by this warp complete before TMEM is freed.
      mma_commit_warp(&bars->mma_done[s_side ? 0 : 1]);
      drain_wait(&bars->mma_done[s_side ? 0 : 1], 0);
    } else {
      // -------------------------------------------- epilogue warps (8-11)
      // (warp 8 also writes each finished O tile out with a TMA store)
      // O / l -> fp16 into the item's Q buffer (swizzled like a Q tile; the
      // store warp writes it out with TMA), lse direct.  Runs while the
      // softmax warps start on the next item.
      const int quad = warp & 3;
      const int r = quad * 32 + lane;  // query row inside the tile, == TMEM lane
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      const float* lm = reinterpret_cast<const float*>(smem + T::SM_LM);
      uint32_t t = 0, q_item = 0;
      bool ok = true;
      const size_t part_rows = static_cast<size_t>(prm.heads) * Nq;  // rows of one slice's partial result
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int head, qa, qb, sp;
        fwd_unit<CAUSAL, MODE>(prm, u, nqt, head, qa, qb, sp);
        const FwdItemShape<D, CAUSAL, MODE> sh(prm, head, sp);
        for (int half = 0; ok && half < 2; ++half) {
          const int qt = half ? qb : qa;
          if (qt < 0) break;
          int j0 = 0;
          const int nkv = MODE == kPagedSplit ? sh.range(qt, j0) : sh.tiles(qt);
          // split mode: this row's slot in the slice's partial result
          const size_t prow = MODE == kPagedSplit ? static_cast<size_t>(sp) * part_rows +
                                                        static_cast<size_t>(head) * Nq + qt * T::BM + r
                                                  : 0;
          if (MODE == kPagedSplit && nkv == 0) {
            // a slice past the item's tiles: nothing visible
            if (qt * T::BM + r < Nq) prm.part_lse[prow] = -INFINITY;
            continue;
          }
          t += nkv;
          ok = mbar_wait(&bars->lm_full, q_item & 1, wc, 17);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          const float l_row = lm[r] + lm[T::BM + r];
          const float m = lm[2 * T::BM + r];
          mbar_arrive(&bars->lm_empty);
          // the item's last P V has completed
          ok = mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, wc, 7);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          // sparse: a row with no visible key at all has an empty softmax
          const float inv_l = (kEmptyRows && !(l_row > 0.f)) ? 0.f : 1.f / l_row;
          if constexpr (MODE == kPagedSplit) {
            // the slice's partial O (normalised by its own row sum) in fp32
            // and its lse, straight to global memory
            const bool live_row = qt * T::BM + r < Nq;
  #pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld32(lane_base + T::O_COL + c, o);
              tmem_wait_ld();
              reg_fence<32>(o);
              if (live_row) {
                float4* dst = reinterpret_cast<float4*>(prm.part_o + prow * D + c);
  #pragma unroll
                for (int i = 0; i < 8; ++i)
                  dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                       __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
              }
            }
            mbar_arrive(&bars->epi_full[q_item % T::Q_STAGES]);
            if (live_row)
              prm.part_lse[prow] = !(l_row > 0.f) ? -INFINITY : (m + log2f(l_row)) * 0.69314718055994530942f;
          } else {
            const uint32_t so = smem_u32(smem + T::SM_Q + (q_item % T::Q_STAGES) * T::Q_BYTES) + r * 128;
  #pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld32(lane_base + T::O_COL + c, o);
              tmem_wait_ld();
              reg_fence<32>(o);
              uint32_t h[16];
  #pragma unroll
              for (int i = 0; i < 16; ++i)
                h[i] = pack2<BF>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
              const uint32_t sub = so + (c / 64) * T::Q_SUB;
  #pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int ch = ((c % 64) / 8 + i) ^ (r & 7);
                st_shared_v4(sub + ch * 16, h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
              }
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->epi_full[q_item % T::Q_STAGES]);
            if (qt * T::BM + r < Nq)
              prm.lse[static_cast<size_t>(head) * Nq + qt * T::BM + r] =
                  (MODE == kSparse && !(l_row > 0.f)) ? -INFINITY : (m + log2f(l_row)) * 0.69314718055994530942f;
          }
          tc_fence_before();
          mbar_arrive(&bars->o_free);
          if (warp == 8) {
            // all 128 rows are staged: store the tile with TMA, then release
            // the Q buffer once TMA has read it
            const int qs = q_item % T::Q_STAGES;
            if (!(ok = warp_wait(&bars->epi_full[qs], (q_item / T::Q_STAGES) & 1, wc, 13))) break;
            if (lane == 0) {
              if (MODE != kPagedSplit) {  // split: the partial result went straight to global memory
                const uint8_t* so_tile = smem + T::SM_Q + qs * T::Q_BYTES;
                for (int sub = 0; sub < T::DSUB; ++sub)
                  tma_store_3d(&tm_o, so_tile + sub * T::Q_SUB, sub * 64, qt * T::BM, head);
                bulk_commit();
                bulk_wait_read<0>();
              }
              mbar_arrive(&bars->q_empty[qs]);
            }
            __syncwarp();
          }
          ++q_item;
        }
      }
      if (warp == 8 && lane == 0) bulk_wait<0>();  // all O stores complete before the CTA exits
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == T::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF, int MODE = kDense>
int launch_fwd(const CUtensorMap* maps, const FwdParams& prm, int num_sms, cudaStream_t stream) {
  using T = FwdTraits<D, CAUSAL>;
  // Function attributes belong to the device current when they are set: set
  // them once per device.
  static DeviceOnceFlags attr_done;
  const int rc = once_per_device(attr_done, current_device_index(), [] {
    if (cudaFuncSetAttribute(fa_fwd_kernel<D, CAUSAL, BF, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T::SMEM_ALLOC) != cudaSuccess)
      return -1;
    // the kernel splits its launch registers between warpgroups
    // (setmaxnreg); refuse to launch if the build gave it fewer than the
    // split needs, rather than let the raising warpgroups wait forever
    cudaFuncAttributes fa_attr;
    if (cudaFuncGetAttributes(&fa_attr, fa_fwd_kernel<D, CAUSAL, BF, MODE>) != cudaSuccess ||
        fa_attr.numRegs * T::THREADS < T::SOFTMAX_THREADS * T::SOFTMAX_REGS + (T::THREADS - T::SOFTMAX_THREADS) * T::OTHER_REGS)
      return -1;
    return 0;
  });
  if (rc != 0) return -1;
  const int nqt = (prm.Nq + T::BM - 1) / T::BM;
  const long long units = (CAUSAL ? static_cast<long long>(prm.heads) * ((nqt + 1) / 2)
                                  : static_cast<long long>(prm.heads) * nqt) *
                          (MODE == kPagedSplit ? prm.splits : 1);
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  fa_fwd_kernel<D, CAUSAL, BF, MODE><<<grid, T::THREADS, T::SMEM_ALLOC, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                                                  prm);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

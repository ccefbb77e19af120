// FlashAttention backward for D = 64 and D = 128 on sm_103a: two persistent
// kernels, each gradient tile written by exactly one CTA, no atomics and no
// accumulator in global memory.
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
// §二 -- the backward equations (Delta = rowsum(O * dO), P recomputed from
// the saved log-sum-exp, dP = dO V^T, dS = scale * P * (dP - Delta),
// dQ = dS K, dK = dS^T Q, dV = P^T dO) and the rules "recompute P, never
// store it", "one writer per gradient tile", "scratch does not grow with N^2
// over all heads"; §七 (D128: dK and dV fused into one sweep over the query
// tiles).
//
//  fa_bwd_dkdv_kernel: one work unit per (head, key tile j).  K_j and V_j stay
//    in shared memory; Q_i (with the tile's lse2) and dO_i (with its Delta)
//    stream through two separate rings.  Per tile, with M = keys:
//      S^T  = K_j Q_i^T                 -> TMEM
//      P^T  = exp2(S^T * c - lse2)      -> fp16, TMEM (over S^T)
//      dP^T = V_j dO_i^T                -> TMEM
//      dS^T = P^T * (dP^T - Delta)      -> fp16, TMEM (over dP^T)
//      dV_j += P^T dO_i                 (A from TMEM)
//      dK_j += dS^T Q_i                 (A from TMEM)
//    and dK_j (times scale), dV_j are written once at the end of the unit.
//  fa_bwd_dq_kernel (runs first): one work unit per (head, query tile i).
//    Q_i and dO_i stay in shared memory; K_j and V_j stream through separate
//    rings.  For D = 128, in its first key tile the compute warps form Delta_i =
//    rowsum(O_i * dO_i) from dO_i in shared memory and O_i read from global
//    memory (prefetched into L2 during the previous unit), and write Delta_i
//    and lse2_i to the workspace that the dK/dV kernel reads.  Per tile,
//    with M = queries: S = Q_i K_j^T, P = exp2(S * c - lse2_i),
//    dP = dO_i V_j^T (double-buffered in TMEM), dS = P * (dP - Delta_i)
//    (fp16 into TMEM over its dP), dQ_i += dS K_j (A from TMEM); dQ_i (times
//    scale) is written once at the end of the unit.  S is released as soon
//    as it is read, so the next S overlaps this tile's dS work, and the two
//    dP/dS buffers let dP of the next tile run before dQ of this one ends.
//
// The second kernel recomputes S and dP (7 GEMMs instead of 5) in exchange
// for having no cross-tile reduction at all.  Scale is applied to dK and dQ
// at write-out (dS is kept as P * (dP - Delta) in fp16).
#pragma once

#include "fa_kernels.h"
#include "ptx.cuh"

namespace fa {

template <int D>
struct Bwd2Traits {
  static_assert(D == 64 || D == 128, "two-kernel backward covers D = 64 and 128");
  static constexpr int BM = 128;  // queries per tile
  static constexpr int BN = 128;  // keys per tile
  static constexpr int DSUB = D / 64;
  static constexpr int SUB = 128 * 128;    // bytes of a [128 x 64] fp16 sub-tile
  static constexpr int TILE = 128 * D * 2; // bytes of a [128 x D] fp16 tile
  static constexpr int QC = 64;            // columns per compute warpgroup
  static constexpr int MIN_SMEM = 120 * 1024;  // keeps one CTA per SM (512 TMEM columns each)

  // ---- dK/dV kernel: Q ring of A_QS stages, dO ring of A_OS stages; each
  // Q stage carries the tile's lse2, each dO stage its Delta
  static constexpr int A_QS = (D == 64) ? 4 : 3;
  static constexpr int A_OS = (D == 64) ? 4 : 2;
  static constexpr int A_DV = 0, A_DK = D, A_R = 2 * D;  // region r of the query tiles at A_R + r * BM
  static constexpr int A_SM_K = 0, A_SM_V = TILE, A_SM_Q = 2 * TILE;
  static constexpr int A_SM_DO = A_SM_Q + A_QS * TILE;
  static constexpr int A_SM_L2 = A_SM_DO + A_OS * TILE;       // lse2[128] per Q stage
  static constexpr int A_SM_DL = A_SM_L2 + A_QS * BM * 4;     // Delta[128] per dO stage
  static constexpr int A_SM_BAR = A_SM_DL + A_OS * BM * 4;
  static constexpr int A_SM_BYTES = A_SM_BAR + 512;
  static constexpr int A_SMEM = A_SM_BYTES > MIN_SMEM ? A_SM_BYTES : MIN_SMEM;
  static_assert(A_SMEM <= 232448, "dK/dV kernel shared memory budget");
  static_assert(A_R + 2 * BM <= 512, "dK/dV kernel TMEM budget");

  // ---- dQ kernel.  TMEM: dQ, then Q_i and dO_i as MMA A operands (16-bit
  // pairs: D / 2 columns each), then two 128-column regions for the key
  // tiles.  Shared memory: staging buffers for the next item's Q and dO (the
  // Q buffer then receives dQ for its store), a K ring and a V ring.
  // O_i, for Delta: staged by TMA beside Q_i and dO_i where shared memory
  // has room (D = 64); at D = 128 the compute warps read it from global
  // memory (a single V stage to make room measured slower).
  static constexpr bool kStageO = (D == 64);
  static constexpr int B_K_STAGES = (D == 64) ? 4 : 3;
  static constexpr int B_V_STAGES = (D == 64) ? 4 : 2;
  static constexpr int B_DQ = 0, B_QT = D, B_OT = D + D / 2, B_R = 2 * D;  // region r at B_R + r * BN
  static constexpr int B_SM_Q = 0, B_SM_DO = TILE, B_SM_O = 2 * TILE, B_SM_K = (kStageO ? 3 : 2) * TILE;
  static constexpr int B_SM_V = B_SM_K + B_K_STAGES * TILE;
  static constexpr int B_SM_BAR = B_SM_V + B_V_STAGES * TILE;
  static constexpr int B_SM_DX = B_SM_BAR + 512;        // Delta halves: [item parity][warpgroup][BM] fp32
  static constexpr int B_SM_BYTES = B_SM_DX + 2 * 2 * BM * 4;
  static constexpr int B_SMEM = B_SM_BYTES > MIN_SMEM ? B_SM_BYTES : MIN_SMEM;
  static_assert(B_SMEM <= 232448, "dQ kernel shared memory budget");
  static_assert(B_R + 2 * BN <= 512, "dQ kernel TMEM budget");
};

// Work units of the two kernels.  Non-causal: one unit per (head, tile),
// head-major.  Causal: tiles t and n-1-t of a head form one unit so that all
// units cost the same number of tile pairs (n + 1).
template <bool CAUSAL>
__device__ __forceinline__ int bwd2_units(int heads, int ntiles) {
  return CAUSAL ? heads * ((ntiles + 1) / 2) : heads * ntiles;
}

template <bool CAUSAL>
__device__ __forceinline__ void bwd2_decode(int u, int ntiles, int& head, int& ta, int& tb) {
  if (CAUSAL) {
    const int npair = (ntiles + 1) / 2;
    head = u / npair;
    const int p = u - head * npair;
    ta = ntiles - 1 - p;
    tb = (p != ta) ? p : -1;
  } else {
    head = u / ntiles;
    ta = u - head * ntiles;
    tb = -1;
  }
}

__device__ __forceinline__ void bwd2_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_test(a, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Write 32 fp16 values (16 packed words) of row `row`, columns col0..col0+31
// (col0 a multiple of 32) into a [128 x D] tile laid out as 128-byte-swizzled
// [128 x 64] sub-tiles -- the layout a TMA store of 64 x 128 boxes reads.
__device__ __forceinline__ void stage_row32(uint32_t tile, int row, int col0, const uint32_t* h) {
  const uint32_t base = tile + (col0 / 64) * (128 * 128) + row * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ch = ((col0 % 64) / 8 + i) ^ (row & 7);
    st_shared_v4(base + ch * 16, h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
  }
}

// Site code reported when the dynamic shared memory base is not 1024-byte
// aligned (the 128-byte-swizzled tiles need it); the kernel then does nothing.
constexpr int kSiteSmemAlign = 99;

// ===================================================================== dK, dV

struct DkdvBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[4], q_empty[4], o_full[4], o_empty[4];
  uint64_t s_full, s_free, dp_full;
  // per TMEM region (phase = the region's use count): P^T written, dS^T
  // written, the tile's dK MMA (and the dV MMA before it) read the region
  uint64_t p_full[2], ds_full[2], dk_done[2];
  uint64_t dkv_full, dkv_free, epi_full, mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DkdvBars) <= 512, "barrier area");

// TMEM use per key tile j: the dV_j and dK_j accumulators and two 128-column
// regions that the query tiles use in turn.  Query tile t works in region
// t % 2 from start to end: S^T, read into registers at once; then dP^T in
// the same columns; then P^T and dS^T in fp16 (the A operands of dV += P^T
// dO and dK += dS^T Q; per warpgroup half of the 128 query columns, P^T
// takes the first 32 TMEM columns and dS^T the next 32).  A region is free
// again once the tile's dK MMA (issued after its dV MMA) completed, so the
// MMAs of tile t+1 run in the other region while the compute warps turn dP^T
// of tile t into P^T and dS^T, and no tile waits on the previous one's MMAs.
//
// Unit boundaries: K_j and V_j are released after the last dP^T of the unit,
// so the next unit's K, V load overlaps the unit's last dV, dK MMAs and its
// write-out.  dK_j and dV_j are staged in the Q and dO ring slots of the
// unit's last query tile (free once its dK and dV MMAs completed) and written
// with TMA stores by warp 11, which then hands those two slots back to the
// producer.
template <int D, bool CAUSAL, bool BF>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const BwdParams prm) {
  using T = Bwd2Traits<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_timeout(prm.status, kSiteSmemAlign);
    return;
  }
  DkdvBars* bars = reinterpret_cast<DkdvBars*>(smem + T::A_SM_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int PRODUCER_WARP = 8, MMA_WARP = 9, GRAD_MMA_WARP = 10, STORE_WARP = 11, NCOMPUTE = 256;
  constexpr int QS = T::A_QS, OS = T::A_OS;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, NCOMPUTE / 32);
    mbar_init(&bars->dp_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->p_full[i], NCOMPUTE / 32);
      mbar_init(&bars->ds_full[i], NCOMPUTE / 32);
      mbar_init(&bars->dk_done[i], 1);
    }
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_free, NCOMPUTE / 32);
    mbar_init(&bars->epi_full, NCOMPUTE / 32);
    mbar_init(&bars->mma_done[0], 1);
    mbar_init(&bars->mma_done[1], 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  } else if (warp == STORE_WARP && lane == 0) {
    tma_prefetch_desc(&tm_dk);
    tma_prefetch_desc(&tm_dv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  // Unit = (K/V head, key tile j).  It sweeps the query tiles of each of the
  // G query heads that read this K/V head (one writer for dK_j and dV_j,
  // which sum over the group), from the first query tile that sees key
  // j * BN (causal) to the last.
  const int G = prm.group, coff = prm.causal_off, Nq_pad = prm.Nq_pad;
  const int nqt = (prm.Nq + T::BM - 1) / T::BM, nkv = (prm.Nk + T::BN - 1) / T::BN;
  const int units = bwd2_units<CAUSAL>(prm.heads / G, nkv);
  auto first_q = [&](int j) { return CAUSAL ? max(0, j * T::BN - coff) / T::BM : 0; };

  if (warp == PRODUCER_WARP) {
    // --------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_last();
      const uint64_t pol_kv = l2_policy_evict_first();
      uint32_t t = 0, kc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int kvh, ja, jb;
        bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
        for (int half = 0; ok && half < 2; ++half) {
          const int j = half ? jb : ja;
          if (j < 0) break;
          if (!(ok = mbar_wait(&bars->kv_empty, (kc & 1) ^ 1, wc, 51))) break;
          mbar_arrive_expect_tx(&bars->kv_full, 2 * T::TILE);
          for (int s = 0; s < T::DSUB; ++s) {
            tma_load_3d_hint(smem + T::A_SM_K + s * T::SUB, &tm_k, &bars->kv_full, s * 64, j * T::BN, kvh, pol_kv);
            tma_load_3d_hint(smem + T::A_SM_V + s * T::SUB, &tm_v, &bars->kv_full, s * 64, j * T::BN, kvh, pol_kv);
          }
          ++kc;
          const int i0 = first_q(j), nqi = nqt - i0;
          for (int x = 0; x < G * nqi; ++x) {
            const int qh = kvh * G + x / nqi, i = i0 + x % nqi;
            const size_t vrow = static_cast<size_t>(qh) * Nq_pad + i * T::BM;  // lse2 / Delta row
            const int qs = t % QS, os = t % OS;
            if (!(ok = mbar_wait(&bars->q_empty[qs], ((t / QS) & 1) ^ 1, wc, 52))) break;
            mbar_arrive_expect_tx(&bars->q_full[qs], T::TILE + 512);
            for (int s = 0; s < T::DSUB; ++s)
              tma_load_3d_hint(smem + T::A_SM_Q + qs * T::TILE + s * T::SUB, &tm_q, &bars->q_full[qs], s * 64,
                               i * T::BM, qh, pol_q);
            bulk_load(smem + T::A_SM_L2 + qs * 512, prm.lse2 + vrow, 512, &bars->q_full[qs]);
            if (!(ok = mbar_wait(&bars->o_empty[os], ((t / OS) & 1) ^ 1, wc, 53))) break;
            mbar_arrive_expect_tx(&bars->o_full[os], T::TILE + 512);
            for (int s = 0; s < T::DSUB; ++s)
              tma_load_3d_hint(smem + T::A_SM_DO + os * T::TILE + s * T::SUB, &tm_do, &bars->o_full[os], s * 64,
                               i * T::BM, qh, pol_q);
            bulk_load(smem + T::A_SM_DL + os * 512, prm.delta + vrow, 512, &bars->o_full[os]);
            // warm L2 with the tiles that will refill these slots, so their
            // loads are short once the slots free up
            ++t;
          }
        }
      }
      if (kc > 0) bwd2_drain(&bars->kv_full, (kc - 1) & 1);
      for (uint32_t i = (t > QS ? t - QS : 0); i < t; ++i) bwd2_drain(&bars->q_full[i % QS], (i / QS) & 1);
      for (uint32_t i = (t > OS ? t - OS : 0); i < t; ++i) bwd2_drain(&bars->o_full[i % OS], (i / OS) & 1);
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------- MMA warp: S^T = K Q^T, dP^T = V dO^T
    constexpr uint32_t id_s = idesc_16<BF>(128, T::BM, false, false);  // S^T, dP^T: M keys, N queries
    const uint32_t sb = smem_u32(smem);
    const uint64_t kdesc = sdesc_sw128(sb + T::A_SM_K, 16, 1024), vdesc = sdesc_sw128(sb + T::A_SM_V, 16, 1024);
    uint32_t t = 0, kc = 0;
    bool ok = true;
    // S^T(tile) = K Q^T into region tile % 2, free once the dK MMA of tile
    // - 2 completed
    auto issue_s = [&](uint32_t tile) -> bool {
      const int qs = tile % QS, r = tile & 1;
      if (!warp_wait(&bars->q_full[qs], (tile / QS) & 1, wc, 62)) return false;
      if (tile >= 2 && !warp_wait(&bars->dk_done[r], ((tile - 2) >> 1) & 1, wc, 63)) return false;
      tc_fence_after();
      const uint64_t qdesc = sdesc_sw128(sb + T::A_SM_Q + qs * T::TILE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * T::SUB + (kk % 4) * 32;
        mma_f16_ss_warp(tmem + T::A_R + r * T::BM, sdesc_add(kdesc, off), sdesc_add(qdesc, off), id_s,
                        kk > 0 ? 1u : 0u);
      }
      mma_commit_warp(&bars->s_full);
      return true;
    };
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        if (!(ok = warp_wait(&bars->kv_full, kc & 1, wc, 61))) break;
        tc_fence_after();
        if (!(ok = issue_s(t))) break;
        const int nx = G * (nqt - first_q(j));
        for (int x = 0; x < nx; ++x) {
          const bool last = (x == nx - 1);
          const int os = t % OS;
          // dP^T = V dO^T over S^T in the tile's region, once the compute
          // warps have read S^T
          if (!(ok = warp_wait(&bars->o_full[os], (t / OS) & 1, wc, 64))) break;
          if (!(ok = warp_wait(&bars->s_free, t & 1, wc, 65))) break;
          tc_fence_after();
          const uint64_t odesc = sdesc_sw128(sb + T::A_SM_DO + os * T::TILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * T::SUB + (kk % 4) * 32;
            mma_f16_ss_warp(tmem + T::A_R + (t & 1) * T::BM, sdesc_add(vdesc, off), sdesc_add(odesc, off), id_s,
                            kk > 0 ? 1u : 0u);
          }
          mma_commit_warp(&bars->dp_full);
          if (last) {
            mma_commit_warp(&bars->kv_empty);  // K_j, V_j are not read again
          } else if (!(ok = issue_s(t + 1))) {
            break;
          }
          ++t;
        }
        ++kc;
      }
    }
    mma_commit_warp(&bars->mma_done[0]);
    bwd2_drain(&bars->mma_done[0], 0);
  } else if (warp == GRAD_MMA_WARP) {
    // ---------------------------- MMA warp: dV += P^T dO, dK += dS^T Q
    constexpr uint32_t id_g = idesc_16<BF>(128, D, false, true);  // dV, dK: N = D, B MN-major
    const uint32_t sb = smem_u32(smem);
    uint32_t t = 0, kc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        const int nx = G * (nqt - first_q(j));
        for (int x = 0; x < nx; ++x) {
          const bool first = (x == 0), last = (x == nx - 1);
          const int qs = t % QS, os = t % OS;
          const uint64_t qdesc_mn = sdesc_sw128(sb + T::A_SM_Q + qs * T::TILE, T::SUB, 1024);
          const uint64_t odesc_mn = sdesc_sw128(sb + T::A_SM_DO + os * T::TILE, T::SUB, 1024);
          // the first tile of a unit overwrites the accumulators, which the
          // previous unit's write-out must have read
          if (first && kc > 0 && !(ok = warp_wait(&bars->dkv_free, (kc - 1) & 1, wc, 67))) break;
          if (!(ok = warp_wait(&bars->o_full[os], (t / OS) & 1, wc, 60))) break;
          if (!(ok = warp_wait(&bars->p_full[t & 1], (t >> 1) & 1, wc, 68))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < T::BM / 16; ++kk) {
            const uint32_t a_t = tmem + T::A_R + (t & 1) * T::BM + (kk / 4) * T::QC + (kk % 4) * 8;
            mma_f16_ts_warp(tmem + T::A_DV, a_t, sdesc_add(odesc_mn, kk * 2048), id_g, (first && kk == 0) ? 0u : 1u);
          }
          // dO_i is free once this dV MMA completed (dP^T of the tile
          // completed before the compute warps could signal p_full); the
          // last tile's slot receives dV_j and is released by the store warp
          if (!last) mma_commit_warp(&bars->o_empty[os]);
          if (!(ok = warp_wait(&bars->q_full[qs], (t / QS) & 1, wc, 59))) break;
          if (!(ok = warp_wait(&bars->ds_full[t & 1], (t >> 1) & 1, wc, 69))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < T::BM / 16; ++kk) {
            const uint32_t a_t = tmem + T::A_R + (t & 1) * T::BM + T::QC / 2 + (kk / 4) * T::QC + (kk % 4) * 8;
            mma_f16_ts_warp(tmem + T::A_DK, a_t, sdesc_add(qdesc_mn, kk * 2048), id_g, (first && kk == 0) ? 0u : 1u);
          }
          // dV and dK of this tile (in issue order) have read P^T and dS^T
          mma_commit_warp(&bars->dk_done[t & 1]);
          if (last) {
            // the Q and dO slots of the last tile receive dK_j and dV_j; the
            // store warp releases them after writing those out
            mma_commit_warp(&bars->dkv_full);
          } else {
            // Q_i is free: S^T of this tile completed before the compute
            // warps could signal p_full
            mma_commit_warp(&bars->q_empty[qs]);
          }
          ++t;
        }
        ++kc;
      }
    }
    mma_commit_warp(&bars->mma_done[1]);
    bwd2_drain(&bars->mma_done[1], 0);
  } else if (warp == STORE_WARP) {
    // -------------- write dK_j, dV_j (staged by the compute warps in the Q
    // and dO slots of the unit's last tile), then release those slots
    uint32_t t = 0, kc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        t += G * (nqt - first_q(j));
        const int qs = (t - 1) % QS, os = (t - 1) % OS;
        if (!(ok = warp_wait(&bars->epi_full, kc & 1, wc, 58))) break;
        if (lane == 0) {
          for (int s = 0; s < T::DSUB; ++s) {
            tma_store_3d(&tm_dk, smem + T::A_SM_Q + qs * T::TILE + s * T::SUB, s * 64, j * T::BN, kvh);
            tma_store_3d(&tm_dv, smem + T::A_SM_DO + os * T::TILE + s * T::SUB, s * 64, j * T::BN, kvh);
          }
          bulk_commit();
          bulk_wait_read<0>();
          mbar_arrive(&bars->q_empty[qs]);
          mbar_arrive(&bars->o_empty[os]);
        }
        __syncwarp();
        ++kc;
      }
    }
    if (lane == 0) bulk_wait<0>();  // all stores complete before the CTA exits
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = key row of the tile
    const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = prm.scale_log2;
    uint32_t t = 0, kc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        const int key = j * T::BN + row;
        const int i0 = first_q(j), nqi = nqt - i0;
        for (int x = 0; x < G * nqi; ++x) {
          const int i = i0 + x % nqi;
          const int qs = t % QS, os = t % OS;
          // key k is hidden from query q iff k > q + coff: only tiles whose
          // last key passes their first query's limit need the mask
          const bool diag = CAUSAL && (j + 1) * T::BN - 1 > i * T::BM + coff;
          const int q0 = i * T::BM + wg * T::QC + coff;  // limit of this warpgroup's first query column
          // ---- P^T = exp2(S^T * c - lse2); the region takes dP^T once S^T
          // has been read
          ok = mbar_wait(&bars->q_full[qs], (t / QS) & 1, wc, 71) && mbar_wait(&bars->s_full, t & 1, wc, 72);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          uint32_t sr[T::QC];
          const uint32_t rb = lb + T::A_R + (t & 1) * T::BM + wg * T::QC;  // this warpgroup's columns
          tmem_ld32(rb, sr);
          tmem_ld32(rb + 32, sr + 32);
          tmem_wait_ld();
          reg_fence<T::QC>(sr);
          tc_fence_before();
          mbar_arrive_warp(&bars->s_free);
          // y = lse2 - S^T * c in packed fp32 pairs, P^T = exp2(-y)
          const float4* l4 = reinterpret_cast<const float4*>(smem + T::A_SM_L2 + qs * 512) + wg * (T::QC / 4);
          const uint64_t nc2 = f2_pack(-sl2, -sl2);
          // diagonal tile: the query columns this key row sees (a suffix,
          // query >= key - coff) as one bit per column of each 32-column word
          uint32_t keep[T::QC / 32];
          if (diag) {
            const int nh = key - q0;  // hidden columns
#pragma unroll
            for (int w = 0; w < T::QC / 32; ++w) {
              const int h = min(max(nh - 32 * w, 0), 32);
              keep[w] = h == 32 ? 0u : (0xffffffffu << h);
            }
          }
          uint64_t p2[T::QC / 2];
#pragma unroll
          for (int c = 0; c < T::QC; c += 4) {
            const float4 L = l4[c / 4];
            float y[4];
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), nc2, f2_pack(L.x, L.y)), y[0],
                      y[1]);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), nc2, f2_pack(L.z, L.w)),
                      y[2], y[3]);
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pv[e] = ex2_approx(-y[e]);
              if (diag) pv[e] = ((keep[(c + e) / 32] >> ((c + e) % 32)) & 1u) ? pv[e] : 0.f;
            }
            p2[c / 2] = f2_pack(pv[0], pv[1]);
            p2[c / 2 + 1] = f2_pack(pv[2], pv[3]);
          }
          // ---- P^T (fp16) over the first half of dP^T once that half is
          // read; dS^T = P^T * (dP^T - Delta) over the second half.  The
          // halves are read one at a time to keep register pressure low.
          uint32_t pk[T::QC / 2];
#pragma unroll
          for (int c = 0; c < T::QC / 2; ++c) pk[c] = f2_to_pack2<BF>(p2[c]);
          ok = mbar_wait(&bars->o_full[os], (t / OS) & 1, wc, 73) && mbar_wait(&bars->dp_full, t & 1, wc, 74);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          tmem_ld32(rb, sr);
          tmem_wait_ld();
          reg_fence<32>(sr);
          tmem_st32(rb, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive_warp(&bars->p_full[t & 1]);
          const float4* d4 = reinterpret_cast<const float4*>(smem + T::A_SM_DL + os * 512) + wg * (T::QC / 4);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 1) {
              tmem_ld32(rb + 32, sr);
              tmem_wait_ld();
              reg_fence<32>(sr);
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const float4 Dl = d4[(32 * h + c) / 4];
              const uint64_t d01 = f2_sub(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), f2_pack(Dl.x, Dl.y));
              const uint64_t d23 =
                  f2_sub(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), f2_pack(Dl.z, Dl.w));
              pk[16 * h + c / 2] = f2_to_pack2<BF>(f2_mul(p2[(32 * h + c) / 2], d01));
              pk[16 * h + c / 2 + 1] = f2_to_pack2<BF>(f2_mul(p2[(32 * h + c) / 2 + 1], d23));
            }
          }
          tmem_st32(rb + T::QC / 2, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive_warp(&bars->ds_full[t & 1]);
          ++t;
        }
        if (!ok) break;
        // ---- dV_j and dK_j (times scale) -> fp16, staged in the dO and Q
        // slots of the unit's last tile; the store warp writes them out
        ok = mbar_wait(&bars->dkv_full, kc & 1, wc, 75);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const int ql = (t - 1) % QS, ol = (t - 1) % OS;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = (which == 0 ? T::A_DV : T::A_DK) + wg * (D / 2);
          const float mul = which == 0 ? 1.f : prm.scale;
          const uint32_t tile = smem_u32(smem + (which == 0 ? T::A_SM_DO + ol * T::TILE : T::A_SM_Q + ql * T::TILE));
#pragma unroll
          for (int c = 0; c < D / 2; c += 32) {
            uint32_t v[32];
            tmem_ld32(lb + col + c, v);
            tmem_wait_ld();
            reg_fence<32>(v);
            uint32_t h[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              h[e] = pack2<BF>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
            stage_row32(tile, row, wg * (D / 2) + c, h);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(&bars->dkv_free);
        mbar_arrive_warp(&bars->epi_full);
        ++kc;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ========================================================================= dQ

// The query-tile items of one CTA in processing order: units blockIdx.x,
// blockIdx.x + gridDim.x, ...; a causal unit is two items (tiles t and
// n-1-t of one head).
template <bool CAUSAL>
struct DqItems {
  int u, units, nt, head, ta, tb, half;
  __device__ DqItems(int units_, int nt_) : u(blockIdx.x), units(units_), nt(nt_), head(0), ta(0), tb(-1), half(0) {
    if (u < units) bwd2_decode<CAUSAL>(u, nt, head, ta, tb);
  }
  __device__ bool valid() const { return u < units; }
  __device__ int tile() const { return half ? tb : ta; }
  __device__ void next() {
    if (half == 0 && tb >= 0) {
      half = 1;
      return;
    }
    half = 0;
    u += gridDim.x;
    if (u < units) bwd2_decode<CAUSAL>(u, nt, head, ta, tb);
  }
};

struct DqBars {
  // Q_n, dO_n landed in the staging buffers; the compute warps have read
  // them (copied into TMEM, Delta formed); Q_n and dO_n are in TMEM
  uint64_t qo_full, qo_empty, qo_tmem;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  // per TMEM region (phase = the region's use count): S landed; dS written;
  // the dQ MMA has read the region
  uint64_t s_full[2], ds_full[2], dq_done[2];
  uint64_t s_free, dp_full;
  uint64_t dq_full, dq_free, mma_done[2];
  uint64_t epi_full[2];  // dQ of item n staged for its store (barrier n % 2)
  uint64_t dx_full[2];   // both Delta halves of an item's rows are in shared memory
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 512, "barrier area");

// TMEM of the dQ kernel: dQ_i, then Q_i and dO_i as MMA A operands (16-bit
// pairs, one query row per lane), then two 128-column regions that the key
// tiles use in turn.  Key tile t works in region t % 2 from start to end: S,
// read into registers at once; then dP over it; then dS (16-bit) over the
// first half of each warpgroup's dP columns, the A operand of dQ += dS K.
// The region is free again once that dQ MMA completed, so S of tile t+1
// runs while the compute warps work on tile t.  S and dP read only K and V
// from shared memory (their A operands are in TMEM), which keeps the MMAs
// below the shared-memory bandwidth that the K/V loads also use.
//
// Item boundaries: Q_n and dO_n arrive in shared-memory staging buffers
// during item n-1.  At the boundary the compute warps copy them into TMEM
// (and form Delta_n from dO_n and O_n), then stage dQ of item n-1 (times
// scale, 16-bit) in the Q staging buffer they just emptied; the producer
// writes it out with a TMA store before loading Q_{n+1} there.  The last
// item's dQ goes to the dO staging buffer.
template <int D, bool CAUSAL, bool BF>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_o,
                     const BwdParams prm) {
  using T = Bwd2Traits<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_timeout(prm.status, kSiteSmemAlign);
    return;
  }
  DqBars* bars = reinterpret_cast<DqBars*>(smem + T::B_SM_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // warp 9 issues S and dP (and owns TMEM); warp 11 issues dQ; warp 8 loads
  // Q, dO and K and stores dQ; warp 10 loads V
  constexpr int PRODUCER_WARP = 8, S_MMA_WARP = 9, V_PRODUCER_WARP = 10, GRAD_MMA_WARP = 11, NCOMPUTE = 256;
  constexpr int KS = T::B_K_STAGES, VS = T::B_V_STAGES;

  if (threadIdx.x == 0) {
    mbar_init(&bars->qo_full, 1);
    mbar_init(&bars->qo_empty, NCOMPUTE / 32);
    mbar_init(&bars->qo_tmem, NCOMPUTE / 32);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->ds_full[i], NCOMPUTE / 32);
      mbar_init(&bars->dq_done[i], 1);
      mbar_init(&bars->epi_full[i], NCOMPUTE / 32);
      mbar_init(&bars->dx_full[i], NCOMPUTE / 32);
      mbar_init(&bars->mma_done[i], 1);
    }
    mbar_init(&bars->s_free, NCOMPUTE / 32);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, NCOMPUTE / 32);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == S_MMA_WARP) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
    tma_prefetch_desc(&tm_o);
  } else if (warp == V_PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  // Item = (query head, query tile i); K/V come from head / G.  Causal: key
  // tiles up to the last key the tile's last query sees.
  const int G = prm.group, Nk = prm.Nk, coff = prm.causal_off, Nq_pad = prm.Nq_pad;
  const int nqt = (prm.Nq + T::BM - 1) / T::BM, nkv = (Nk + T::BN - 1) / T::BN;
  const int units = bwd2_units<CAUSAL>(prm.heads, nqt);
  auto num_kv = [&](int i) { return CAUSAL ? (min((i + 1) * T::BM + coff, Nk) + T::BN - 1) / T::BN : nkv; };

  if (warp == PRODUCER_WARP) {
    // ------------------------------------- producer: Q, dO, K; dQ write-out
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t n = 0, qc = 0, k_it = 0;  // items begun, Q/dO loads issued, K loads issued
      int h1 = 0, i1 = 0, h2 = 0, i2 = 0;  // (head, tile) of items n-1 and n-2
      bool ok = true;
      // write dQ of item m (query head h, tile i), staged in buffer `buf`
      auto store_dq = [&](uint32_t m, int h, int i, int buf) -> bool {
        if (!mbar_wait(&bars->epi_full[m & 1], (m >> 1) & 1, wc, 84)) return false;
        for (int s = 0; s < T::DSUB; ++s) tma_store_3d(&tm_dq, smem + buf + s * T::SUB, s * 64, i * T::BM, h);
        bulk_commit();
        bulk_wait_read<0>();
        return true;
      };
      // Q_n, dO_n (and O_n where staged) into the (empty) staging buffers
      auto load_qo = [&](int head, int i) {
        mbar_arrive_expect_tx(&bars->qo_full, (T::kStageO ? 3 : 2) * T::TILE);
        for (int s = 0; s < T::DSUB; ++s) {
          tma_load_3d_hint(smem + T::B_SM_Q + s * T::SUB, &tm_q, &bars->qo_full, s * 64, i * T::BM, head, pol_q);
          tma_load_3d_hint(smem + T::B_SM_DO + s * T::SUB, &tm_do, &bars->qo_full, s * 64, i * T::BM, head, pol_q);
          if (T::kStageO)
            tma_load_3d_hint(smem + T::B_SM_O + s * T::SUB, &tm_o, &bars->qo_full, s * 64, i * T::BM, head, pol_q);
        }
        ++qc;
      };
      DqItems<CAUSAL> it(units, nqt);
      if (it.valid()) load_qo(it.head, it.tile());
      for (; ok && it.valid(); ++n) {
        const int head = it.head, i = it.tile(), nj = num_kv(i);
        DqItems<CAUSAL> nx = it;
        nx.next();
        for (int j = 0; ok && j < nj; ++j) {
          const int ks = k_it % KS;
          if (!(ok = mbar_wait(&bars->k_empty[ks], ((k_it / KS) & 1) ^ 1, wc, 82))) break;
          mbar_arrive_expect_tx(&bars->k_full[ks], T::TILE);
          for (int s = 0; s < T::DSUB; ++s)
            tma_load_3d_hint(smem + T::B_SM_K + ks * T::TILE + s * T::SUB, &tm_k, &bars->k_full[ks], s * 64,
                             j * T::BN, head / G, pol_kv);
          ++k_it;
          // Once the item's first two K tiles are on their way (they load
          // during the previous item), the next item's Q and dO go into the
          // staging buffers: the compute warps empty them at this item's
          // start, after which dQ of the previous item, staged in the Q
          // buffer, is written out.  They then land a whole item ahead.
          if (j == min(1, nj - 1) && nx.valid()) {
            if (n >= 1 && !(ok = store_dq(n - 1, h1, i1, T::B_SM_Q))) break;
            if (!(ok = mbar_wait(&bars->qo_empty, n & 1, wc, 81))) break;
            load_qo(nx.head, nx.tile());
          }
        }
        h2 = h1;
        i2 = i1;
        h1 = head;
        i1 = i;
        it = nx;
      }
      // the last two items' dQ: item n-2 (staged in the Q buffer at the
      // start of the last item, which loaded no successor) and item n-1, the
      // CTA's last (in the dO buffer)
      if (ok && n >= 2) ok = store_dq(n - 2, h2, i2, T::B_SM_Q);
      if (ok && n >= 1) ok = store_dq(n - 1, h1, i1, T::B_SM_DO);
      bulk_wait<0>();  // all stores complete before the CTA exits
      if (qc > 0) bwd2_drain(&bars->qo_full, (qc - 1) & 1);
      for (uint32_t x = (k_it > KS ? k_it - KS : 0); x < k_it; ++x) bwd2_drain(&bars->k_full[x % KS], (x / KS) & 1);
    }
  } else if (warp == V_PRODUCER_WARP) {
    // --------------------------------------------------------- producer: V
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t v_it = 0;
      bool ok = true;
      for (DqItems<CAUSAL> it(units, nqt); ok && it.valid(); it.next()) {
        for (int j = 0; j < num_kv(it.tile()); ++j) {
          const int vs = v_it % VS;
          if (!(ok = mbar_wait(&bars->v_empty[vs], ((v_it / VS) & 1) ^ 1, wc, 83))) break;
          mbar_arrive_expect_tx(&bars->v_full[vs], T::TILE);
          for (int s = 0; s < T::DSUB; ++s)
            tma_load_3d_hint(smem + T::B_SM_V + vs * T::TILE + s * T::SUB, &tm_v, &bars->v_full[vs], s * 64,
                             j * T::BN, it.head / G, pol_kv);
          ++v_it;
        }
      }
      for (uint32_t x = (v_it > VS ? v_it - VS : 0); x < v_it; ++x) bwd2_drain(&bars->v_full[x % VS], (x / VS) & 1);
    }
  } else if (warp == S_MMA_WARP) {
    // -------------------------------- MMA warp: S = Q K^T and dP = dO V^T
    // The tensor pipe runs its queue in issue order.  This warp issues per
    // key tile dP(t), then S(t+1): the compute warps need dP(t) first, and
    // S(t+1) (into region (t+1) % 2, free once the dQ MMA of tile t-1
    // completed) runs while they turn dP(t) into dS(t).
    constexpr uint32_t id_s = idesc_16<BF>(128, T::BN, false, false);  // S, dP: M queries, N keys
    const uint32_t sb = smem_u32(smem);
    uint32_t ts = 0, tp = 0, n = 0, k_it = 0, v_it = 0;  // tiles whose S / dP is issued
    bool ok = true;
    // S(ts); the first tile of item m also needs the item's Q in TMEM
    auto issue_s = [&](bool first_of_item, uint32_t m) -> bool {
      const int ks = k_it % KS, r = ts & 1;
      if (first_of_item && !warp_wait(&bars->qo_tmem, m & 1, wc, 91)) return false;
      if (!warp_wait(&bars->k_full[ks], (k_it / KS) & 1, wc, 92)) return false;
      if (ts >= 2 && !warp_wait(&bars->dq_done[r], ((ts - 2) >> 1) & 1, wc, 93)) return false;
      tc_fence_after();
      const uint64_t kdesc = sdesc_sw128(sb + T::B_SM_K + ks * T::TILE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_f16_ts_warp(tmem + T::B_R + r * T::BN, tmem + T::B_QT + kk * 8,
                        sdesc_add(kdesc, (kk / 4) * T::SUB + (kk % 4) * 32), id_s, kk > 0 ? 1u : 0u);
      mma_commit_warp(&bars->s_full[r]);
      ++ts;
      ++k_it;
      return true;
    };
    DqItems<CAUSAL> it(units, nqt);
    if (it.valid()) ok = issue_s(true, 0);
    for (; ok && it.valid(); ++n) {
      const int nj = num_kv(it.tile());
      DqItems<CAUSAL> nx = it;
      nx.next();
      for (int j = 0; ok && j < nj; ++j) {
        // dP(tp) over S in the tile's region, once the compute warps have read S
        const int vs = v_it % VS, r = tp & 1;
        if (!(ok = warp_wait(&bars->v_full[vs], (v_it / VS) & 1, wc, 95))) break;
        if (!(ok = warp_wait(&bars->s_free, tp & 1, wc, 96))) break;
        tc_fence_after();
        const uint64_t vdesc = sdesc_sw128(sb + T::B_SM_V + vs * T::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16_ts_warp(tmem + T::B_R + r * T::BN, tmem + T::B_OT + kk * 8,
                          sdesc_add(vdesc, (kk / 4) * T::SUB + (kk % 4) * 32), id_s, kk > 0 ? 1u : 0u);
        mma_commit_warp(&bars->dp_full);
        mma_commit_warp(&bars->v_empty[vs]);
        ++tp;
        ++v_it;
        // then S of the next tile: this item's next one, or the next item's first
        if (j + 1 < nj) {
          ok = issue_s(false, n);
        } else if (nx.valid()) {
          ok = issue_s(true, n + 1);
        }
      }
      it = nx;
    }
    mma_commit_warp(&bars->mma_done[0]);
    bwd2_drain(&bars->mma_done[0], 0);
  } else if (warp == GRAD_MMA_WARP) {
    // ------------------------------------------------ MMA warp: dQ += dS K
    constexpr uint32_t id_q = idesc_16<BF>(128, D, false, true);  // dQ: N = D, B = K MN-major
    const uint32_t sb = smem_u32(smem);
    uint32_t t = 0, n = 0, k_it = 0;
    bool ok = true;
    for (DqItems<CAUSAL> it(units, nqt); ok && it.valid(); it.next(), ++n) {
      const int nj = num_kv(it.tile());
      for (int j = 0; j < nj; ++j) {
        const int ks = k_it % KS, r = t & 1;
        // the item's first tile overwrites dQ, which the previous item's
        // write-out must have read; dS of the tile is in its region
        if (j == 0 && n > 0 && !(ok = warp_wait(&bars->dq_free, (n - 1) & 1, wc, 97))) break;
        if (!(ok = warp_wait(&bars->ds_full[r], (t >> 1) & 1, wc, 98))) break;
        tc_fence_after();
        const uint64_t kdesc_mn = sdesc_sw128(sb + T::B_SM_K + ks * T::TILE, T::SUB, 1024);
#pragma unroll
        for (int kk = 0; kk < T::BN / 16; ++kk) {
          const uint32_t a_t = tmem + T::B_R + r * T::BN + (kk / 4) * T::QC + (kk % 4) * 8;
          mma_f16_ts_warp(tmem + T::B_DQ, a_t, sdesc_add(kdesc_mn, kk * 2048), id_q, (j == 0 && kk == 0) ? 0u : 1u);
        }
        // the region is free and K_t read (S of this tile completed before
        // the compute warps could signal ds_full)
        mma_commit_warp(&bars->dq_done[r]);
        mma_commit_warp(&bars->k_empty[ks]);
        if (j == nj - 1) mma_commit_warp(&bars->dq_full);
        ++t;
        ++k_it;
      }
    }
    mma_commit_warp(&bars->mma_done[1]);
    bwd2_drain(&bars->mma_done[1], 0);
  } else {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = query row of the tile
    const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = prm.scale_log2;
    constexpr int CH = D / 16;  // 16-byte chunks of this warpgroup's half of a row
    uint32_t t = 0, n = 0;
    bool ok = true;
    // Delta and lse2 of this thread's row of the current item, packed for
    // the f32x2 arithmetic (negated)
    uint64_t nd2 = 0ull, nl2 = 0ull;

    // Item `nx` (index m) begins: Q_m and dO_m are copied from the staging
    // buffers into TMEM, and this warpgroup's half of rowsum(O * dO) is
    // formed: with O staged beside them, from the dO words just read; else
    // with O read coalesced from global memory (CH lanes per row, 32 / CH rows
    // per load, the sum gathered by the row's owner) and dO re-read from the
    // staging buffer in the same pattern.  `lse_raw` is the row's
    // natural-log lse, requested an item earlier.
    auto load_item = [&](const DqItems<CAUSAL>& nx, uint32_t m, float lse_raw, float& lse2, float& part) -> bool {
      const bool live = nx.tile() * T::BM + row < prm.Nq;
      lse2 = live ? lse_raw * 1.4426950408889634f : INFINITY;
      constexpr int RPL = 32 / CH;  // rows per coalesced load
      uint4 ov[T::kStageO ? 1 : CH];
      if constexpr (!T::kStageO) {
#pragma unroll
        for (int k = 0; k < CH; ++k) {
          const int qr = nx.tile() * T::BM + quad * 32 + RPL * k + lane / CH;
          ov[k] = qr < prm.Nq ? ldg_nc_v4(prm.o + (static_cast<size_t>(nx.head) * prm.Nq + qr) * D + wg * (D / 2) +
                                          (lane % CH) * 8)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      const bool got = mbar_wait(&bars->qo_full, m & 1, wc, 104);
      if (!__all_sync(0xffffffffu, got)) return false;
      // chunk c of row r's half wg * D / 2 .. of a 128-byte-swizzled tile
      auto chunk = [&](int buf, int r, int c) {
        const int g = wg * CH + c;
        return ld_shared_v4(smem_u32(smem + buf) + (g / 8) * T::SUB + r * 128 + (((g % 8) ^ (r & 7)) << 4));
      };
      uint32_t w[4 * CH];
#pragma unroll
      for (int which = 0; which < 2; ++which) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const uint4 x = chunk(which == 0 ? T::B_SM_Q : T::B_SM_DO, row, c);
          w[4 * c] = x.x;
          w[4 * c + 1] = x.y;
          w[4 * c + 2] = x.z;
          w[4 * c + 3] = x.w;
        }
        const uint32_t col = (which == 0 ? T::B_QT : T::B_OT) + wg * (D / 4);
        if constexpr (D == 128) {
          tmem_st32(lb + col, w);
        } else {
          tmem_st16(lb + col, w);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&bars->qo_tmem);  // Q_m, dO_m are in TMEM: the item's S can start
      if constexpr (T::kStageO) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const uint4 o4 = chunk(T::B_SM_O, row, c);
          const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 x = unpack2<BF>(ow[q]), y = unpack2<BF>(w[4 * c + q]);
            acc0 = fmaf(x.x, y.x, acc0);
            acc1 = fmaf(x.y, y.y, acc1);
          }
        }
        part = acc0 + acc1;
      } else {
#pragma unroll
        for (int k = 0; k < CH; ++k) {
          const uint4 d4 = chunk(T::B_SM_DO, quad * 32 + RPL * k + lane / CH, lane % CH);
          const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
          const uint32_t ow[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
          float acc = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 x = unpack2<BF>(ow[q]), y = unpack2<BF>(dw[q]);
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
          }
#pragma unroll
          for (int o = 1; o < CH; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          // row RPL * k + lane / CH of the warp; its owner is lane RPL * k + that
          const float v = __shfl_sync(0xffffffffu, acc, (lane % RPL) * CH);
          if (lane / RPL == k) part = v;
        }
      }
      mbar_arrive_warp(&bars->qo_empty);  // the staging buffers are no longer read
      return true;
    };
    // Delta of item m's rows: both warpgroups' halves through shared memory;
    // written to the workspace (with lse2) for the dK/dV kernel
    auto finish_delta = [&](const DqItems<CAUSAL>& nx, uint32_t m, float lse2, float part) -> bool {
      float* dx = reinterpret_cast<float*>(smem + T::B_SM_DX) + (m & 1) * 2 * T::BM;
      dx[wg * T::BM + row] = part;
      mbar_arrive_warp(&bars->dx_full[m & 1]);
      const bool got = mbar_wait(&bars->dx_full[m & 1], (m >> 1) & 1, wc, 105);
      if (!__all_sync(0xffffffffu, got)) return false;
      const float delta = dx[row] + dx[T::BM + row];  // the same sum in both warpgroups
      if (wg == 0) {
        const size_t grow = static_cast<size_t>(nx.head) * Nq_pad + nx.tile() * T::BM + row;
        prm.delta[grow] = delta;
        prm.lse2[grow] = lse2;
      }
      nd2 = f2_pack(-delta, -delta);
      return true;
    };

    // The current item's lse2 and this warpgroup's half of its Delta, until
    // the halves are combined in its first key tile (after S is read, so that
    // dP of that tile is already queued)
    float lse2 = 0.f, part = 0.f;
    // an item ahead: this row's lse (and, at D = 128, its O half for the
    // coalesced reads) into L2.  No load into a register here: a warp's
    // tcgen05.wait::ld also waits for its global loads in flight, so a load
    // issued an item ahead would stall the item's first TMEM read.
    auto prefetch_item = [&](const DqItems<CAUSAL>& x) {
      const int q = x.tile() * T::BM + row;
      if (!x.valid() || q >= prm.Nq) return;
      const size_t src = static_cast<size_t>(x.head) * prm.Nq + q;
      if (!T::kStageO) prefetch_l2(prm.o + src * D + wg * (D / 2));
      prefetch_l2(prm.lse + src);
    };
    auto lse_of = [&](const DqItems<CAUSAL>& x) {
      const int q = x.tile() * T::BM + row;
      return x.valid() && q < prm.Nq ? __ldg(prm.lse + static_cast<size_t>(x.head) * prm.Nq + q) : 0.f;
    };
    DqItems<CAUSAL> it(units, nqt);
    if (it.valid()) {
      ok = load_item(it, 0, lse_of(it), lse2, part);
      ok = __all_sync(0xffffffffu, ok);
      nl2 = f2_pack(-lse2, -lse2);
    }
    for (; ok && it.valid(); ++n) {
      const int head = it.head, i = it.tile();
      const int query = i * T::BM + row;
      DqItems<CAUSAL> nx = it;
      nx.next();
      prefetch_item(nx);
      // last key this row sees; key tiles past the tile's smallest limit
      // (the causal diagonal, or the ragged end of the keys) are masked
      const int lim = CAUSAL ? min(query + coff, Nk - 1) : Nk - 1;
      const int lim_lo = CAUSAL ? min(i * T::BM + coff, Nk - 1) : Nk - 1;
      const uint64_t c2 = f2_pack(sl2, sl2);
      for (int j = 0; j < num_kv(i); ++j) {
        const int r = t & 1;
        const int k0 = j * T::BN + wg * T::QC;  // first key column of this warpgroup
        const uint32_t rb = lb + T::B_R + r * T::BN + wg * T::QC;  // this warpgroup's columns of the region
        // ---- P = exp2(S * c - lse2)
        ok = mbar_wait(&bars->s_full[r], (t >> 1) & 1, wc, 101);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[T::QC];
        tmem_ld32(rb, sr);
        tmem_ld32(rb + 32, sr + 32);
        tmem_wait_ld();
        reg_fence<T::QC>(sr);
        tc_fence_before();
        mbar_arrive_warp(&bars->s_free);  // the region takes dP
        if (j == 0) {
          ok = finish_delta(it, n, lse2, part);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        uint64_t p2[T::QC / 2];
        const bool masked = (j + 1) * T::BN - 1 > lim_lo;
        // causal: the row's visible columns of this warpgroup's half as one
        // bit per column of each 32-column word
        uint32_t keep[T::QC / 32];
        if constexpr (CAUSAL) {
          const int nv = lim - k0 + 1;
#pragma unroll
          for (int w = 0; w < T::QC / 32; ++w) {
            const int nvis = min(max(nv - 32 * w, 0), 32);
            keep[w] = nvis == 32 ? 0xffffffffu : ((1u << nvis) - 1u);
          }
        }
#pragma unroll
        for (int c = 0; c < T::QC; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, nl2), x0, x1);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if constexpr (CAUSAL) {
            if (masked) {
              p0 = ((keep[c / 32] >> (c % 32)) & 1u) ? p0 : 0.f;
              p1 = ((keep[c / 32] >> ((c + 1) % 32)) & 1u) ? p1 : 0.f;
            }
          } else if (masked) {
            if (k0 + c > lim) p0 = 0.f;
            if (k0 + c + 1 > lim) p1 = 0.f;
          }
          p2[c / 2] = f2_pack(p0, p1);
        }
        // ---- dS = P * (dP - Delta), 16-bit over the first half of this
        // warpgroup's dP columns
        ok = mbar_wait(&bars->dp_full, t & 1, wc, 102);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        tmem_ld32(rb, sr);
        tmem_ld32(rb + 32, sr + 32);
        tmem_wait_ld();
        reg_fence<T::QC>(sr);
        uint32_t pk[T::QC / 2];
#pragma unroll
        for (int c = 0; c < T::QC; c += 2)
          pk[c / 2] = f2_to_pack2<BF>(
              f2_mul(p2[c / 2], f2_add(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), nd2)));
        tmem_st32(rb, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&bars->ds_full[r]);
        ++t;
      }
      if (!ok) break;
      // ---- item boundary: the next item's Q, dO into TMEM first (its S can
      // start) and its Delta halves, then this item's dQ out
      const bool has_next = nx.valid();
      if (has_next) {
        ok = load_item(nx, n + 1, lse_of(nx), lse2, part);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        nl2 = f2_pack(-lse2, -lse2);
      }
      // dQ_i (times scale) -> 16-bit, staged in the Q staging buffer (just
      // emptied by this thread's own reads of the same row and columns), or
      // in the dO buffer after the CTA's last item; the producer stores it
      ok = mbar_wait(&bars->dq_full, n & 1, wc, 103);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tile = smem_u32(smem + (has_next ? T::B_SM_Q : T::B_SM_DO));
#pragma unroll
      for (int c = 0; c < D / 2; c += 32) {
        uint32_t v[32];
        tmem_ld32(lb + T::B_DQ + wg * (D / 2) + c, v);
        tmem_wait_ld();
        reg_fence<32>(v);
        const float sc = prm.scale;
        uint32_t h[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) h[e] = pack2<BF>(__uint_as_float(v[2 * e]) * sc, __uint_as_float(v[2 * e + 1]) * sc);
        stage_row32(tile, row, wg * (D / 2) + c, h);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(&bars->dq_free);
      mbar_arrive_warp(&bars->epi_full[n & 1]);
      it = nx;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == S_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The dQ kernel (which also writes Delta and lse2 of every query row), then
// the dK/dV kernel, on the same stream.  `max_ctas` caps each persistent
// grid (normally the SM count).  maps: [0] q, [1] k, [2] v, [3] dout, [4] dq,
// [5] dk, [6] dv, [9] o.
template <int D, bool CAUSAL, bool BF>
int launch_bwd2(const CUtensorMap* maps, const BwdParams& prm, int max_ctas, cudaStream_t stream) {
  using T = Bwd2Traits<D>;
  static DeviceOnceFlags attr_done;  // the attributes are per device
  if (once_per_device(attr_done, current_device_index(), [] {
        return cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D, CAUSAL, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    T::A_SMEM) == cudaSuccess &&
                       cudaFuncSetAttribute(fa_bwd_dq_kernel<D, CAUSAL, BF>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, T::B_SMEM) == cudaSuccess
                   ? 0
                   : -1;
      }) != 0)
    return -1;
  auto grid_for = [&](int heads, int tiles) {
    const long long units = CAUSAL ? static_cast<long long>(heads) * ((tiles + 1) / 2) : static_cast<long long>(heads) * tiles;
    return static_cast<int>(units < max_ctas ? units : max_ctas);
  };
  const int nqt = (prm.Nq + T::BM - 1) / T::BM, nkv = (prm.Nk + T::BN - 1) / T::BN;
  fa_bwd_dq_kernel<D, CAUSAL, BF><<<grid_for(prm.heads, nqt), 384, T::B_SMEM, stream>>>(maps[0], maps[1], maps[2],
                                                                                       maps[3], maps[4], maps[9], prm);
  if (cudaGetLastError() != cudaSuccess) return -1;
  fa_bwd_dkdv_kernel<D, CAUSAL, BF><<<grid_for(prm.heads / prm.group, nkv), 384, T::A_SMEM, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[5], maps[6], prm);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

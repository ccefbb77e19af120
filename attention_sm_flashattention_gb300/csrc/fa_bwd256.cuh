// FlashAttention backward for D = 256 on sm_103a: two persistent kernels,
// each gradient tile written by exactly one CTA, no atomics and no
// accumulator in global memory.
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
// §二 -- the backward equations (Delta = rowsum(O * dO), P recomputed from
// the saved log-sum-exp, dP = dO V^T, dS = scale * P * (dP - Delta),
// dQ = dS K, dK = dS^T Q, dV = P^T dO) and the rules "recompute P", "one
// writer per gradient tile", "scratch does not grow with N^2 over all
// heads"; §七 -- D256 handled as two D128 halves.
//
// At D = 256 a 128-row tile of K, V, Q or dO is 64 KB, and TMEM (512
// columns) cannot hold 256-wide dK and dV accumulators next to S and dP.
// The two kernels make room by keeping one stationary operand in TMEM as
// the A operand of a tcgen05 MMA (packed 16-bit pairs, one row per lane)
// instead of in shared memory:
//
//  fa_bwd256_dkdv_kernel: one work unit per (K/V head, key tile j of 128
//    keys); the unit sweeps the 64-row query tiles of the G query heads that
//    read its K/V head twice, once per gradient:
//      dV pass:  S^T  = K_j Q_i^T               (K in shared memory)
//                P^T  = exp2(S^T * c - lse2)    -> 16-bit, TMEM (over S^T)
//                dV_j += P^T dO_i               (N = 256: all of D)
//      dK pass:  S^T as above, P^T in registers
//                dP^T = V_j dO_i^T              (V_j in TMEM, loaded once per unit)
//                dS^T = P^T * (dP^T - Delta)    -> 16-bit, TMEM (over dP^T)
//                dK_j += dS^T Q_i               (N = 256)
//    S^T is computed in both passes (five 128 x 64 x 256 GEMM blocks per
//    query tile instead of four): the 256-wide dV and dK accumulators do not
//    fit in TMEM together (§七 splits D for the same reason), one at a time
//    they do.  TMEM: the pass's accumulator (256 columns), V_j (128), two
//    64-column regions that the query tiles use in turn.  Shared memory:
//    K_j (64 KB), three Q stages and two dO stages of 32 KB.
//  fa_bwd256_dq_kernel: one work unit per (query head, 128-row query tile
//    i); 64-key tiles of K and V stream through rings:
//      S = Q_i K_j^T, P = exp2(S * c - lse2), dP = dO_i V_j^T (dO_i in TMEM),
//      dS = P * (dP - Delta) -> fp16 into TMEM over dP, dQ_i += dS K_j.
//    TMEM: dO_i (128 columns), dQ_i (256), two 64-column regions that the
//    key tiles use in turn (S, then dP over it, then dS).  Shared memory:
//    Q_i (64 KB), three K stages and two V stages of 32 KB.
// The compute warps write the TMEM-resident operand from global memory at the
// start of a unit, and at its end stage dK, dV and dQ (times the scale where
// §二 puts it) as 16-bit tiles in ring slots that the last tile no longer
// needs, which a TMA store writes out.
#pragma once

#include "fa_bwd2.cuh"

namespace fa {

struct B256 {
  static constexpr int D = 256;
  static constexpr int NCOMPUTE = 256;  // warps 0-7
  // ---- dK/dV kernel
  static constexpr int A_BN = 128, A_BM = 64;   // keys per unit (MMA M), queries per tile (MMA N)
  static constexpr int A_QC = 32;               // query columns per compute warpgroup
  static constexpr int A_QSUB = 64 * 128;       // [64 x 64] 16-bit sub-tile, 8 KB
  static constexpr int A_KSUB = 128 * 128;      // [128 x 64], 16 KB
  static constexpr int A_QTILE = 4 * A_QSUB;    // 32 KB
  static constexpr int A_KTILE = 4 * A_KSUB;    // 64 KB
  static constexpr int A_QS = 3, A_OS = 2;
  // TMEM columns: the pass's gradient accumulator (dV, then dK; N = 256),
  // V_j as an MMA A operand, region r at A_R + 64 r
  static constexpr int A_ACC = 0, A_V = 256, A_R = 384;
  static constexpr int A_SM_K = 0, A_SM_Q = A_KTILE, A_SM_DO = A_SM_Q + A_QS * A_QTILE;
  static constexpr int A_SM_L2 = A_SM_DO + A_OS * A_QTILE;  // lse2[64] per Q stage
  static constexpr int A_SM_DL = A_SM_L2 + A_QS * 256;      // Delta[64] per dO stage
  static constexpr int A_SM_BAR = A_SM_DL + A_OS * 256;
  static constexpr int A_SMEM = A_SM_BAR + 256;
  static constexpr int A_THREADS = 384;  // 8 compute warps, producer, three MMA warps
  static_assert(A_SMEM <= 232448, "dK/dV kernel shared memory budget");
  static_assert(A_R + 2 * A_BM <= 512, "dK/dV kernel TMEM budget");
  // ---- dQ kernel
  static constexpr int B_BM = 128, B_BN = 64;   // queries per unit (MMA M), keys per tile
  static constexpr int B_KC = 32;               // key columns per compute warpgroup
  static constexpr int B_QSUB = 128 * 128;      // [128 x 64], 16 KB
  static constexpr int B_KSUB = 64 * 128;       // [64 x 64], 8 KB
  static constexpr int B_QTILE = 4 * B_QSUB;    // 64 KB
  static constexpr int B_KTILE = 4 * B_KSUB;    // 32 KB
  static constexpr int B_KS = 3, B_VS = 2;
  static constexpr int B_DO = 0, B_DQ = 128, B_R = 384;  // TMEM columns; region r (S, then dP, then dS) at B_R + 64 r
  static constexpr int B_SM_Q = 0, B_SM_K = B_QTILE, B_SM_V = B_SM_K + B_KS * B_KTILE;
  static constexpr int B_SM_BAR = B_SM_V + B_VS * B_KTILE;
  static constexpr int B_SM_DX = B_SM_BAR + 256;   // Delta halves: [item parity][warpgroup][B_BM] fp32
  static constexpr int B_SMEM = B_SM_DX + 2 * 2 * B_BM * 4;
  static constexpr int B_THREADS = 416;  // 8 compute warps, two producers, three MMA warps
  static_assert(B_SMEM <= 232448, "dQ kernel shared memory budget");
  static_assert(B_R + 2 * B_BN <= 512, "dQ kernel TMEM budget");
};

// 128 16-bit values (256 bytes) of one row from global memory, as 64 packed
// words in column order; zeros past the end of the matrix.  32-byte loads
// (one whole sector each) when the row is 32-byte aligned -- rows are 512
// bytes apart, so that is a property of the tensor's base address and the
// same for every thread -- else 16-byte loads.
__device__ __forceinline__ void load_row128(const __half* src, bool live, uint32_t* w) {
  if (!live) {
#pragma unroll
    for (int k = 0; k < 64; ++k) w[k] = 0u;
  } else if ((reinterpret_cast<uintptr_t>(src) & 31u) == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                   : "=r"(w[8 * e]), "=r"(w[8 * e + 1]), "=r"(w[8 * e + 2]), "=r"(w[8 * e + 3]), "=r"(w[8 * e + 4]),
                     "=r"(w[8 * e + 5]), "=r"(w[8 * e + 6]), "=r"(w[8 * e + 7])
                   : "l"(src + 16 * e));
  } else {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint4 x = __ldg(s4 + e);
      w[4 * e] = x.x;
      w[4 * e + 1] = x.y;
      w[4 * e + 2] = x.z;
      w[4 * e + 3] = x.w;
    }
  }
}

// Ask L2 to fetch the 256 bytes at `p` (two 128-byte lines) ahead of a
// load_row128 of them.
__device__ __forceinline__ void prefetch_row128(const __half* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p + 64));
}

// 32 fp32 TMEM columns of this thread's row, times `mul`, as 16-bit values
// into row `row`, columns col0..col0+31, of a [128 x 128] staging tile in
// shared memory laid out as two 128-byte-swizzled [128 x 64] boxes (what a
// TMA store of 64 x 128 boxes reads).  A 32-KB ring slot holds one tile.
template <bool BF>
__device__ __forceinline__ void stage_tmem32(uint32_t taddr, float mul, uint32_t tile, int row, int col0) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_wait_ld();
  reg_fence<32>(v);
  uint32_t h[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) h[e] = pack2<BF>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
  stage_row32(tile, row, col0, h);
}

// ===================================================================== dK, dV

struct Bwd256ABars {
  uint64_t k_full, k_empty, v_full, v_free;
  uint64_t q_full[3], q_empty[3], o_full[2], o_empty[2];
  // per TMEM region (phase = the region's use count): S^T landed; the
  // tile's gradient A operand (P^T in the dV pass, dS^T in the dK pass) is
  // written; the tile's gradient MMA has read the region
  uint64_t s_full[2], a_full[2], dk_done[2];
  uint64_t s_free, dp_full;  // dK pass only, one use per dK-pass tile
  uint64_t dkv_full, dkv_free, mma_done[3];
  uint64_t epi_full;  // the pass's gradient staged in the last tile's Q and dO slots
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bwd256ABars) <= 256, "barrier area");

template <bool CAUSAL, bool BF>
__global__ void __launch_bounds__(384, 1)
    fa_bwd256_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dk,
                          const __grid_constant__ CUtensorMap tm_dv, const BwdParams prm) {
  using T = B256;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_timeout(prm.status, kSiteSmemAlign);
    return;
  }
  Bwd256ABars* bars = reinterpret_cast<Bwd256ABars*>(smem + T::A_SM_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int PRODUCER_WARP = 8, MMA_WARP = 9, GRAD_MMA_WARP = 10, DP_MMA_WARP = 11;
  constexpr int QS = T::A_QS, OS = T::A_OS;

  if (threadIdx.x == 0) {
    mbar_init(&bars->k_full, 1);
    mbar_init(&bars->k_empty, 1);
    mbar_init(&bars->v_full, T::NCOMPUTE);
    mbar_init(&bars->v_free, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_empty[i], 1);
      mbar_init(&bars->dk_done[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->a_full[i], T::NCOMPUTE);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&bars->mma_done[i], 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->s_free, T::NCOMPUTE);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->epi_full, T::NCOMPUTE);
    mbar_init(&bars->dkv_free, T::NCOMPUTE);
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
    tma_prefetch_desc(&tm_do);
  } else if (warp == GRAD_MMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_dk);
    tma_prefetch_desc(&tm_dv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  // Unit = (K/V head, key tile j); the query tiles of its G query heads are
  // swept once per D half, from the first tile that sees key j * BN (causal).
  const int G = prm.group, coff = prm.causal_off, Nq_pad = prm.Nq_pad, Nk = prm.Nk;
  const int nqt = (prm.Nq + T::A_BM - 1) / T::A_BM, nkv = (Nk + T::A_BN - 1) / T::A_BN;
  const int units = bwd2_units<CAUSAL>(prm.heads / G, nkv);
  auto first_q = [&](int j) { return CAUSAL ? max(0, j * T::A_BN - coff) / T::A_BM : 0; };

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------- producer
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
          if (!(ok = mbar_wait(&bars->k_empty, (kc & 1) ^ 1, wc, 151))) break;
          mbar_arrive_expect_tx(&bars->k_full, T::A_KTILE);
          for (int s = 0; s < 4; ++s)
            tma_load_3d_hint(smem + T::A_SM_K + s * T::A_KSUB, &tm_k, &bars->k_full, s * 64, j * T::A_BN, kvh, pol_kv);
          ++kc;
          const int i0 = first_q(j), nqi = nqt - i0;
          for (int h = 0; ok && h < 2; ++h) {
            for (int x = 0; x < G * nqi; ++x) {
              const int qh = kvh * G + x / nqi, i = i0 + x % nqi;
              const size_t vrow = static_cast<size_t>(qh) * Nq_pad + i * T::A_BM;  // lse2 / Delta row
              const int qs = t % QS, os = t % OS;
              if (!(ok = mbar_wait(&bars->q_empty[qs], ((t / QS) & 1) ^ 1, wc, 152))) break;
              mbar_arrive_expect_tx(&bars->q_full[qs], T::A_QTILE + 256);
              for (int s = 0; s < 4; ++s)
                tma_load_3d_hint(smem + T::A_SM_Q + qs * T::A_QTILE + s * T::A_QSUB, &tm_q, &bars->q_full[qs],
                                 s * 64, i * T::A_BM, qh, pol_q);
              bulk_load(smem + T::A_SM_L2 + qs * 256, prm.lse2 + vrow, 256, &bars->q_full[qs]);
              if (!(ok = mbar_wait(&bars->o_empty[os], ((t / OS) & 1) ^ 1, wc, 153))) break;
              mbar_arrive_expect_tx(&bars->o_full[os], T::A_QTILE + 256);
              for (int s = 0; s < 4; ++s)
                tma_load_3d_hint(smem + T::A_SM_DO + os * T::A_QTILE + s * T::A_QSUB, &tm_do, &bars->o_full[os],
                                 s * 64, i * T::A_BM, qh, pol_q);
              bulk_load(smem + T::A_SM_DL + os * 256, prm.delta + vrow, 256, &bars->o_full[os]);
              ++t;
            }
          }
        }
      }
      if (kc > 0) bwd2_drain(&bars->k_full, (kc - 1) & 1);
      for (uint32_t i = (t > QS ? t - QS : 0); i < t; ++i) bwd2_drain(&bars->q_full[i % QS], (i / QS) & 1);
      for (uint32_t i = (t > OS ? t - OS : 0); i < t; ++i) bwd2_drain(&bars->o_full[i % OS], (i / OS) & 1);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------ MMA warp: S^T = K Q^T
    // S^T(t) goes into region t % 2 as soon as that region is free (the dK
    // MMA of tile t - 2 completed) and Q_t has landed: it runs ahead of the
    // compute warps, independent of the dP^T issuer.
    constexpr uint32_t id_s = idesc_16<BF>(128, T::A_BM, false, false);  // M keys, N queries
    const uint32_t sb = smem_u32(smem);
    const uint64_t kdesc = sdesc_sw128(sb + T::A_SM_K, 16, 1024);
    uint32_t t = 0, kc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        if (!(ok = warp_wait(&bars->k_full, kc & 1, wc, 161))) break;
        const int nx = G * (nqt - first_q(j));
        for (int h = 0; ok && h < 2; ++h) {
          for (int x = 0; x < nx; ++x) {
            const int qs = t % QS, r = t & 1;
            if (!(ok = warp_wait(&bars->q_full[qs], (t / QS) & 1, wc, 162))) break;
            if (t >= 2 && !(ok = warp_wait(&bars->dk_done[r], ((t - 2) >> 1) & 1, wc, 163))) break;
            tc_fence_after();
            const uint64_t qdesc = sdesc_sw128(sb + T::A_SM_Q + qs * T::A_QTILE, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_f16_ss_warp(tmem + T::A_R + r * T::A_BM, sdesc_add(kdesc, (kk / 4) * T::A_KSUB + (kk % 4) * 32),
                              sdesc_add(qdesc, (kk / 4) * T::A_QSUB + (kk % 4) * 32), id_s, kk > 0 ? 1u : 0u);
            mma_commit_warp(&bars->s_full[r]);
            if (h == 1 && x == nx - 1) mma_commit_warp(&bars->k_empty);  // K_j is not read again
            ++t;
          }
        }
        ++kc;
      }
    }
    mma_commit_warp(&bars->mma_done[0]);
    bwd2_drain(&bars->mma_done[0], 0);
  } else if (warp == DP_MMA_WARP) {
    // ----------------------------------------- MMA warp: dP^T = V dO^T
    // dK pass only: over S^T in the tile's region once the compute warps have
    // read S^T; V_j must be in TMEM (written at the start of the unit)
    constexpr uint32_t id_s = idesc_16<BF>(128, T::A_BM, false, false);
    const uint32_t sb = smem_u32(smem);
    uint32_t t = 0, t1 = 0, kc = 0;  // tiles, dK-pass tiles
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        const int nx = G * (nqt - first_q(j));
        t += nx;  // the dV pass
        for (int x = 0; x < nx; ++x) {
          const int os = t % OS;
          if (!(ok = warp_wait(&bars->o_full[os], (t / OS) & 1, wc, 164))) break;
          if (!(ok = warp_wait(&bars->s_free, t1 & 1, wc, 165))) break;
          if (x == 0 && !(ok = warp_wait(&bars->v_full, kc & 1, wc, 166))) break;
          tc_fence_after();
          const uint64_t odesc = sdesc_sw128(sb + T::A_SM_DO + os * T::A_QTILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_f16_ts_warp(tmem + T::A_R + (t & 1) * T::A_BM, tmem + T::A_V + kk * 8,
                            sdesc_add(odesc, (kk / 4) * T::A_QSUB + (kk % 4) * 32), id_s, kk > 0 ? 1u : 0u);
          mma_commit_warp(&bars->dp_full);
          if (x == nx - 1) mma_commit_warp(&bars->v_free);  // V_j is not read again
          ++t;
          ++t1;
        }
        ++kc;
      }
    }
    mma_commit_warp(&bars->mma_done[2]);
    bwd2_drain(&bars->mma_done[2], 0);
  } else if (warp == GRAD_MMA_WARP) {
    // ------------------- MMA warp: dV += P^T dO (dV pass), dK += dS^T Q (dK pass)
    // N = 256: the whole of D in one accumulator.  It also writes out each
    // pass's gradient, which the compute warps stage in the Q and dO slots of
    // the pass's last tile: before the first MMA of the next pass (which
    // needs the compute warps' next P^T or dS^T anyway) and at the end.
    constexpr uint32_t id_g = idesc_16<BF>(128, 256, false, true);  // N = D, B MN-major
    const uint32_t sb = smem_u32(smem);
    uint32_t t = 0, sc = 0;  // tiles, passes
    int p_kvh = 0, p_j = 0, p_pass = 0;  // the previous pass (kvh, key tile, dV or dK)
    bool ok = true;
    // store the staged tile of pass `sc - 1` (last tile t - 1), then release its slots
    auto store_prev = [&]() -> bool {
      if (!warp_wait(&bars->epi_full, (sc - 1) & 1, wc, 158)) return false;
      if (lane == 0) {
        const int qs = (t - 1) % QS, os = (t - 1) % OS;
        const CUtensorMap* map = p_pass == 0 ? &tm_dv : &tm_dk;
        for (int s2 = 0; s2 < 2; ++s2) {
          tma_store_3d(map, smem + T::A_SM_Q + qs * T::A_QTILE + s2 * 16384, s2 * 64, p_j * T::A_BN, p_kvh);
          tma_store_3d(map, smem + T::A_SM_DO + os * T::A_QTILE + s2 * 16384, 128 + s2 * 64, p_j * T::A_BN, p_kvh);
        }
        bulk_commit();
        bulk_wait_read<0>();
        mbar_arrive(&bars->q_empty[qs]);
        mbar_arrive(&bars->o_empty[os]);
      }
      __syncwarp();
      return true;
    };
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        const int nx = G * (nqt - first_q(j));
        for (int pass = 0; ok && pass < 2; ++pass) {
          for (int x = 0; x < nx; ++x) {
            const bool first = (x == 0), last = (x == nx - 1);
            // the first tile of a pass overwrites the accumulator, which the
            // previous pass's write-out must have read
            if (first && sc > 0) {
              if (!(ok = warp_wait(&bars->dkv_free, (sc - 1) & 1, wc, 167))) break;
              if (!(ok = store_prev())) break;
            }
            const int qs = t % QS, os = t % OS;
            // dV pass: B = dO_i (all 256 columns), A = P^T; dK pass: B = Q_i, A = dS^T
            const uint64_t bdesc = pass == 0 ? sdesc_sw128(sb + T::A_SM_DO + os * T::A_QTILE, T::A_QSUB, 1024)
                                             : sdesc_sw128(sb + T::A_SM_Q + qs * T::A_QTILE, T::A_QSUB, 1024);
            if (!(ok = pass == 0 ? warp_wait(&bars->o_full[os], (t / OS) & 1, wc, 160)
                                 : warp_wait(&bars->q_full[qs], (t / QS) & 1, wc, 159)))
              break;
            if (!(ok = warp_wait(&bars->a_full[t & 1], (t >> 1) & 1, wc, 168))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < T::A_BM / 16; ++kk) {
              const uint32_t a_t = tmem + T::A_R + (t & 1) * T::A_BM + (kk / 2) * T::A_QC + (kk % 2) * 8;
              mma_f16_ts_warp(tmem + T::A_ACC, a_t, sdesc_add(bdesc, kk * 2048), id_g, (first && kk == 0) ? 0u : 1u);
            }
            mma_commit_warp(&bars->dk_done[t & 1]);  // the region is free again
            if (last) {
              mma_commit_warp(&bars->dkv_full);  // the Q and dO slots receive the gradient; released after its store
            } else {
              // S^T (and in the dK pass dP^T) of the tile completed before the
              // compute warps could signal a_full
              mma_commit_warp(&bars->q_empty[qs]);
              mma_commit_warp(&bars->o_empty[os]);
            }
            ++t;
          }
          p_kvh = kvh;
          p_j = j;
          p_pass = pass;
          ++sc;
        }
      }
    }
    if (ok && sc > 0) store_prev();
    if (lane == 0) bulk_wait<0>();  // all stores complete before the CTA exits
    __syncwarp();
    mma_commit_warp(&bars->mma_done[1]);
    bwd2_drain(&bars->mma_done[1], 0);
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = key row of the tile
    const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = prm.scale_log2;
    uint32_t t = 0, t1 = 0, kc = 0, sc = 0;  // tiles, dK-pass tiles, unit halves, passes
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int kvh, ja, jb;
      bwd2_decode<CAUSAL>(u, nkv, kvh, ja, jb);
      for (int half = 0; ok && half < 2; ++half) {
        const int j = half ? jb : ja;
        if (j < 0) break;
        const int key = j * T::A_BN + row;
        const bool key_live = key < Nk;
        const size_t kv_row = static_cast<size_t>(kvh) * Nk + key;
        // ---- V_j (this thread: its key row, D columns [128 wg, 128 wg + 128))
        // into TMEM, once the previous unit's last dP^T has read the old one
        {
          uint32_t w[64];
          load_row128(prm.v + kv_row * T::D + wg * 128, key_live, w);
          ok = mbar_wait(&bars->v_free, (kc & 1) ^ 1, wc, 170);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          tmem_st32(lb + T::A_V + wg * 64, w);
          tmem_st32(lb + T::A_V + wg * 64 + 32, w + 32);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->v_full);
        }
        const int i0 = first_q(j), nqi = nqt - i0;
        {
          // the CTA's next key tile: its V rows into L2 while this one runs
          int nkvh = kvh, nj = -1;
          if (half == 0 && jb >= 0) {
            nj = jb;
          } else if (u + static_cast<int>(gridDim.x) < units) {
            int nb;
            bwd2_decode<CAUSAL>(u + gridDim.x, nkv, nkvh, nj, nb);
          }
          if (nj >= 0 && nj * T::A_BN + row < Nk)
            prefetch_row128(prm.v + (static_cast<size_t>(nkvh) * Nk + nj * T::A_BN + row) * T::D + wg * 128);
        }
        // two passes over the query tiles: dV (S^T, P^T), then dK (S^T,
        // dP^T, dS^T); each ends with its gradient written out
        for (int pass = 0; ok && pass < 2; ++pass) {
          for (int x = 0; x < G * nqi; ++x) {
            const int i = i0 + x % nqi;
            const int qs = t % QS, os = t % OS;
            // key k is hidden from query q iff k > q + coff
            const bool diag = CAUSAL && (j + 1) * T::A_BN - 1 > i * T::A_BM + coff;
            const int q0 = i * T::A_BM + wg * T::A_QC + coff;  // limit of this warpgroup's first query column
            ok = mbar_wait(&bars->q_full[qs], (t / QS) & 1, wc, 171) &&
                 mbar_wait(&bars->s_full[t & 1], (t >> 1) & 1, wc, 172);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[T::A_QC];
            const uint32_t rb = lb + T::A_R + (t & 1) * T::A_BM + wg * T::A_QC;  // this warpgroup's columns
            tmem_ld32(rb, sr);
            tmem_wait_ld();
            reg_fence<T::A_QC>(sr);
            if (pass == 1) {
              tc_fence_before();
              mbar_arrive(&bars->s_free);  // the region takes dP^T
            }
            // P^T = exp2(S^T * c - lse2) in packed fp32 pairs
            const float4* l4 = reinterpret_cast<const float4*>(smem + T::A_SM_L2 + qs * 256) + wg * (T::A_QC / 4);
            const uint64_t nc2 = f2_pack(-sl2, -sl2);
            // diagonal tile: the query columns this key row sees (a suffix)
            // as one bit per column
            uint32_t keep = 0xffffffffu;
            if (diag) {
              const int h = min(max(key - q0, 0), 32);  // hidden columns
              keep = h == 32 ? 0u : (0xffffffffu << h);
            }
            uint64_t p2[T::A_QC / 2];
#pragma unroll
            for (int c = 0; c < T::A_QC; c += 4) {
              const float4 L = l4[c / 4];
              float y[4];
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), nc2, f2_pack(L.x, L.y)),
                        y[0], y[1]);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), nc2, f2_pack(L.z, L.w)),
                        y[2], y[3]);
              float pv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pv[e] = ex2_approx(-y[e]);
                if (diag) pv[e] = ((keep >> (c + e)) & 1u) ? pv[e] : 0.f;
              }
              p2[c / 2] = f2_pack(pv[0], pv[1]);
              p2[c / 2 + 1] = f2_pack(pv[2], pv[3]);
            }
            uint32_t pk[T::A_QC / 2];
            if (pass == 0) {
              // ---- P^T (16-bit) over the first half of this warpgroup's S^T
              // columns (only this warpgroup reads them)
#pragma unroll
              for (int c = 0; c < T::A_QC / 2; ++c) pk[c] = f2_to_pack2<BF>(p2[c]);
              tmem_st16(rb, pk);
              tmem_wait_st();
              tc_fence_before();
              mbar_arrive(&bars->a_full[t & 1]);
            } else {
              // ---- dS^T = P^T * (dP^T - Delta) (16-bit) over the first half
              // of this warpgroup's dP^T columns
              ok = mbar_wait(&bars->o_full[os], (t / OS) & 1, wc, 173) && mbar_wait(&bars->dp_full, t1 & 1, wc, 174);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
              tc_fence_after();
              tmem_ld32(rb, sr);
              tmem_wait_ld();
              reg_fence<T::A_QC>(sr);
              const float4* d4 = reinterpret_cast<const float4*>(smem + T::A_SM_DL + os * 256) + wg * (T::A_QC / 4);
#pragma unroll
              for (int c = 0; c < T::A_QC; c += 4) {
                const float4 Dl = d4[c / 4];
                const uint64_t d01 =
                    f2_sub(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), f2_pack(Dl.x, Dl.y));
                const uint64_t d23 =
                    f2_sub(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), f2_pack(Dl.z, Dl.w));
                pk[c / 2] = f2_to_pack2<BF>(f2_mul(p2[c / 2], d01));
                pk[c / 2 + 1] = f2_to_pack2<BF>(f2_mul(p2[c / 2 + 1], d23));
              }
              tmem_st16(rb, pk);
              tmem_wait_st();
              tc_fence_before();
              mbar_arrive(&bars->a_full[t & 1]);
              ++t1;
            }
            ++t;
          }
          if (!ok) break;
          // ---- the pass's gradient, dV_j or dK_j (times scale), -> 16-bit:
          // columns 0-127 staged in the Q slot and 128-255 in the dO slot of
          // the pass's last tile; the gradient MMA warp writes them out (rows
          // past Nk are dropped by the TMA store)
          ok = mbar_wait(&bars->dkv_full, sc & 1, wc, 175);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = wg == 0 ? smem_u32(smem + T::A_SM_Q + ((t - 1) % QS) * T::A_QTILE)
                                      : smem_u32(smem + T::A_SM_DO + ((t - 1) % OS) * T::A_QTILE);
          const float mul = pass == 0 ? 1.f : prm.scale;
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) stage_tmem32<BF>(lb + T::A_ACC + wg * 128 + c, mul, st, row, c);
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&bars->dkv_free);
          mbar_arrive(&bars->epi_full);
          ++sc;
        }
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

struct Bwd256BBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t do_full, do_free;
  uint64_t s_full[2], s_free, dp_full[2], ds_full[2], dq_done[2];  // [2]: per TMEM region
  uint64_t dq_full, dq_free, mma_done[3];
  uint64_t epi_full;  // dQ_i staged in the last tile's K and V slots
  uint64_t dx_full[2];  // both Delta halves of an item's rows are in shared memory
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bwd256BBars) <= 256, "barrier area");

template <bool CAUSAL, bool BF>
__global__ void __launch_bounds__(416, 1)
    fa_bwd256_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dq,
                        const BwdParams prm) {
  using T = B256;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_timeout(prm.status, kSiteSmemAlign);
    return;
  }
  Bwd256BBars* bars = reinterpret_cast<Bwd256BBars*>(smem + T::B_SM_BAR);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int PRODUCER_WARP = 8, MMA_WARP = 9, V_PRODUCER_WARP = 10, DQ_MMA_WARP = 11, DP_MMA_WARP = 12;
  constexpr int KS = T::B_KS, VS = T::B_VS;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->dp_full[i], 1);
      mbar_init(&bars->ds_full[i], T::NCOMPUTE);
      mbar_init(&bars->dq_done[i], 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&bars->mma_done[i], 1);
    mbar_init(&bars->do_full, T::NCOMPUTE);
    mbar_init(&bars->do_free, 1);
    mbar_init(&bars->dx_full[0], T::NCOMPUTE);
    mbar_init(&bars->dx_full[1], T::NCOMPUTE);
    mbar_init(&bars->s_free, T::NCOMPUTE);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->epi_full, T::NCOMPUTE);
    mbar_init(&bars->dq_free, T::NCOMPUTE);
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
  } else if (warp == DQ_MMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  // Unit = (query head, 128-row query tile i); K/V come from head / G.
  // Causal: 64-key tiles up to the last key the tile's last query sees.
  const int G = prm.group, Nq = prm.Nq, Nk = prm.Nk, coff = prm.causal_off, Nq_pad = prm.Nq_pad;
  const int nqt = (Nq + T::B_BM - 1) / T::B_BM, nkv = (Nk + T::B_BN - 1) / T::B_BN;
  const int units = bwd2_units<CAUSAL>(prm.heads, nqt);
  auto num_kv = [&](int i) {
    return CAUSAL ? (min((i + 1) * T::B_BM + coff, Nk) + T::B_BN - 1) / T::B_BN : nkv;
  };

  if (warp == PRODUCER_WARP) {
    // -------------------------------------------------- producer: Q and K
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t qc = 0, k_it = 0;
      bool ok = true;
      auto load_k = [&](int head, int j) -> bool {
        const int ks = k_it % KS;
        if (!mbar_wait(&bars->k_empty[ks], ((k_it / KS) & 1) ^ 1, wc, 182)) return false;
        mbar_arrive_expect_tx(&bars->k_full[ks], T::B_KTILE);
        for (int s = 0; s < 4; ++s)
          tma_load_3d_hint(smem + T::B_SM_K + ks * T::B_KTILE + s * T::B_KSUB, &tm_k, &bars->k_full[ks], s * 64,
                           j * T::B_BN, head / G, pol_kv);
        ++k_it;
        return true;
      };
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int head, ia, ib;
        bwd2_decode<CAUSAL>(u, nqt, head, ia, ib);
        for (int half = 0; ok && half < 2; ++half) {
          const int i = half ? ib : ia;
          if (i < 0) break;
          // the item's first K tile before its Q tile: its slot frees early,
          // the Q buffer only after the previous item's last S
          if (!(ok = load_k(head, 0))) break;
          if (!(ok = mbar_wait(&bars->q_empty, (qc & 1) ^ 1, wc, 181))) break;
          mbar_arrive_expect_tx(&bars->q_full, T::B_QTILE);
          for (int s = 0; s < 4; ++s)
            tma_load_3d_hint(smem + T::B_SM_Q + s * T::B_QSUB, &tm_q, &bars->q_full, s * 64, i * T::B_BM, head, pol_q);
          ++qc;
          for (int j = 1; ok && j < num_kv(i); ++j) ok = load_k(head, j);
        }
      }
      if (qc > 0) bwd2_drain(&bars->q_full, (qc - 1) & 1);
      for (uint32_t i = (k_it > KS ? k_it - KS : 0); i < k_it; ++i) bwd2_drain(&bars->k_full[i % KS], (i / KS) & 1);
    }
  } else if (warp == V_PRODUCER_WARP) {
    // ----------------------------------------------------------- producer: V
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t v_it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int head, ia, ib;
        bwd2_decode<CAUSAL>(u, nqt, head, ia, ib);
        for (int half = 0; ok && half < 2; ++half) {
          const int i = half ? ib : ia;
          if (i < 0) break;
          for (int j = 0; j < num_kv(i); ++j) {
            const int vs = v_it % VS;
            if (!(ok = mbar_wait(&bars->v_empty[vs], ((v_it / VS) & 1) ^ 1, wc, 183))) break;
            mbar_arrive_expect_tx(&bars->v_full[vs], T::B_KTILE);
            for (int s = 0; s < 4; ++s)
              tma_load_3d_hint(smem + T::B_SM_V + vs * T::B_KTILE + s * T::B_KSUB, &tm_v, &bars->v_full[vs], s * 64,
                               j * T::B_BN, head / G, pol_kv);
            ++v_it;
          }
        }
      }
      for (uint32_t i = (v_it > VS ? v_it - VS : 0); i < v_it; ++i) bwd2_drain(&bars->v_full[i % VS], (i / VS) & 1);
    }
  } else if (warp == MMA_WARP) {
    // --------------------------------------------- MMA warp: S = Q K^T
    // S(t) goes into region t % 2 once that region is free (the dQ MMA of
    // tile t - 2 read its dS) and K_t has landed.
    constexpr uint32_t id_s = idesc_16<BF>(128, T::B_BN, false, false);  // M queries, N keys
    const uint32_t sb = smem_u32(smem);
    const uint64_t qdesc = sdesc_sw128(sb + T::B_SM_Q, 16, 1024);
    uint32_t t = 0, k_it = 0, qc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int head, ia, ib;
      bwd2_decode<CAUSAL>(u, nqt, head, ia, ib);
      for (int half = 0; ok && half < 2; ++half) {
        const int i = half ? ib : ia;
        if (i < 0) break;
        const int nj = num_kv(i);
        if (!(ok = warp_wait(&bars->q_full, qc & 1, wc, 193))) break;
        for (int j = 0; j < nj; ++j) {
          const int ks = k_it % KS, r = t & 1;
          if (!(ok = warp_wait(&bars->k_full[ks], (k_it / KS) & 1, wc, 191))) break;
          if (t >= 2 && !(ok = warp_wait(&bars->dq_done[r], ((t - 2) >> 1) & 1, wc, 192))) break;
          tc_fence_after();
          const uint64_t kdesc = sdesc_sw128(sb + T::B_SM_K + ks * T::B_KTILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_f16_ss_warp(tmem + T::B_R + r * T::B_BN, sdesc_add(qdesc, (kk / 4) * T::B_QSUB + (kk % 4) * 32),
                            sdesc_add(kdesc, (kk / 4) * T::B_KSUB + (kk % 4) * 32), id_s, kk > 0 ? 1u : 0u);
          mma_commit_warp(&bars->s_full[r]);
          if (j == nj - 1) mma_commit_warp(&bars->q_empty);  // Q_i is not read again
          ++t;
          ++k_it;
        }
        ++qc;
      }
    }
    mma_commit_warp(&bars->mma_done[0]);
    bwd2_drain(&bars->mma_done[0], 0);
  } else if (warp == DP_MMA_WARP) {
    // -------------------------------------------- MMA warp: dP = dO V^T
    // over S in the tile's region once the compute warps have read S; dO_i
    // must be in TMEM (first tile of the item)
    constexpr uint32_t id_s = idesc_16<BF>(128, T::B_BN, false, false);
    const uint32_t sb = smem_u32(smem);
    uint32_t t = 0, v_it = 0, qc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int head, ia, ib;
      bwd2_decode<CAUSAL>(u, nqt, head, ia, ib);
      for (int half = 0; ok && half < 2; ++half) {
        const int i = half ? ib : ia;
        if (i < 0) break;
        const int nj = num_kv(i);
        for (int j = 0; j < nj; ++j) {
          const int vs = v_it % VS;
          if (!(ok = warp_wait(&bars->v_full[vs], (v_it / VS) & 1, wc, 194))) break;
          if (!(ok = warp_wait(&bars->s_free, t & 1, wc, 195))) break;
          if (j == 0 && !(ok = warp_wait(&bars->do_full, qc & 1, wc, 196))) break;
          tc_fence_after();
          const uint64_t vdesc = sdesc_sw128(sb + T::B_SM_V + vs * T::B_KTILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_f16_ts_warp(tmem + T::B_R + (t & 1) * T::B_BN, tmem + T::B_DO + kk * 8,
                            sdesc_add(vdesc, (kk / 4) * T::B_KSUB + (kk % 4) * 32), id_s, kk > 0 ? 1u : 0u);
          mma_commit_warp(&bars->dp_full[t & 1]);
          if (j == nj - 1) {
            mma_commit_warp(&bars->do_free);  // dO_i is not read again
          } else {
            mma_commit_warp(&bars->v_empty[vs]);  // the item's last V slot receives half of dQ_i
          }
          ++t;
          ++v_it;
        }
        ++qc;
      }
    }
    mma_commit_warp(&bars->mma_done[2]);
    bwd2_drain(&bars->mma_done[2], 0);
  } else if (warp == DQ_MMA_WARP) {
    // ------------------------------------------------- MMA warp: dQ += dS K
    constexpr uint32_t id_q = idesc_16<BF>(128, T::D, false, true);  // N = 256, B = K MN-major
    const uint32_t sb = smem_u32(smem);
    uint32_t t = 0, k_it = 0, qc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int head, ia, ib;
      bwd2_decode<CAUSAL>(u, nqt, head, ia, ib);
      for (int half = 0; ok && half < 2; ++half) {
        const int i = half ? ib : ia;
        if (i < 0) break;
        const int nj = num_kv(i);
        for (int j = 0; j < nj; ++j) {
          const bool first = (j == 0), last = (j == nj - 1);
          const int ks = k_it % KS;
          // the first tile overwrites dQ, which the previous item's write-out
          // must have read
          if (first && qc > 0 && !(ok = warp_wait(&bars->dq_free, (qc - 1) & 1, wc, 197))) break;
          if (!(ok = warp_wait(&bars->ds_full[t & 1], (t >> 1) & 1, wc, 198))) break;
          tc_fence_after();
          const uint64_t kdesc_mn = sdesc_sw128(sb + T::B_SM_K + ks * T::B_KTILE, T::B_KSUB, 1024);
#pragma unroll
          for (int kk = 0; kk < T::B_BN / 16; ++kk) {
            const uint32_t a_t = tmem + T::B_R + (t & 1) * T::B_BN + (kk / 2) * T::B_KC + (kk % 2) * 8;
            mma_f16_ts_warp(tmem + T::B_DQ, a_t, sdesc_add(kdesc_mn, kk * 2048), id_q, (first && kk == 0) ? 0u : 1u);
          }
          mma_commit_warp(&bars->dq_done[t & 1]);
          if (last) {
            mma_commit_warp(&bars->dq_full);  // the K slot receives half of dQ_i
          } else {
            mma_commit_warp(&bars->k_empty[ks]);  // S of the tile completed before ds_full
          }
          ++t;
          ++k_it;
        }
        if (!ok) break;
        // the compute warps stage dQ_i in the K and V slots of the item's
        // last tile (columns 0-127 and 128-255); store it with TMA, then
        // release both slots
        if (!(ok = warp_wait(&bars->epi_full, qc & 1, wc, 199))) break;
        if (lane == 0) {
          const int kl = (t - 1) % KS, vl = (t - 1) % VS;  // one K and one V stage per tile
          for (int s = 0; s < 2; ++s) {
            tma_store_3d(&tm_dq, smem + T::B_SM_K + kl * T::B_KTILE + s * 16384, s * 64, i * T::B_BM, head);
            tma_store_3d(&tm_dq, smem + T::B_SM_V + vl * T::B_KTILE + s * 16384, 128 + s * 64, i * T::B_BM, head);
          }
          bulk_commit();
          bulk_wait_read<0>();
          mbar_arrive(&bars->k_empty[kl]);
          mbar_arrive(&bars->v_empty[vl]);
        }
        __syncwarp();
        ++qc;
      }
    }
    if (lane == 0) bulk_wait<0>();  // all stores complete before the CTA exits
    __syncwarp();
    mma_commit_warp(&bars->mma_done[1]);
    bwd2_drain(&bars->mma_done[1], 0);
  } else {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = query row of the tile
    const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = prm.scale_log2;
    uint32_t t = 0, qc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int head, ia, ib;
      bwd2_decode<CAUSAL>(u, nqt, head, ia, ib);
      for (int half = 0; ok && half < 2; ++half) {
        const int i = half ? ib : ia;
        if (i < 0) break;
        const int query = i * T::B_BM + row;
        const bool q_live = query < Nq;
        const size_t q_row = static_cast<size_t>(head) * Nq + query;
        const size_t grow = static_cast<size_t>(head) * Nq_pad + query;  // padded: lse2 = +inf past Nq
        const float lse2 = q_live ? __ldg(prm.lse + q_row) * 1.4426950408889634f : INFINITY;
        // last key this row sees; key tiles past the tile's smallest limit are masked
        const int lim = CAUSAL ? min(query + coff, Nk - 1) : Nk - 1;
        const int lim_lo = CAUSAL ? min(i * T::B_BM + coff, Nk - 1) : Nk - 1;
        // ---- dO_i (this thread: its query row, D columns [128 wg, 128 wg +
        // 128)) into TMEM, once the previous item's last dP has read the old one
        {
          uint32_t w[64];
          load_row128(prm.dout + q_row * T::D + wg * 128, q_live, w);
          ok = mbar_wait(&bars->do_free, (qc & 1) ^ 1, wc, 204);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          tmem_st32(lb + T::B_DO + wg * 64, w);
          tmem_st32(lb + T::B_DO + wg * 64 + 32, w + 32);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->do_full);
          // Delta_i = rowsum(O_i * dO_i): this warpgroup's 128 columns, O read
          // in 16-word chunks (the next chunk requested before this one is
          // used), dO from the words just written to TMEM
          const uint4* orow = reinterpret_cast<const uint4*>(prm.o + q_row * T::D + wg * 128);
          uint4 oc[2][4];
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) oc[0][e] = q_live ? ldg_nc_v4(orow + e) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c + 1 < 4) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                oc[(c + 1) & 1][e] = q_live ? ldg_nc_v4(orow + 4 * (c + 1) + e) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t ow[4] = {oc[c & 1][e].x, oc[c & 1][e].y, oc[c & 1][e].z, oc[c & 1][e].w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 x = unpack2<BF>(ow[q]), y = unpack2<BF>(w[16 * c + 4 * e + q]);
                acc0 = fmaf(x.x, y.x, acc0);
                acc1 = fmaf(x.y, y.y, acc1);
              }
            }
          }
          float* dx = reinterpret_cast<float*>(smem + T::B_SM_DX) + (qc & 1) * 2 * T::B_BM;
          dx[wg * T::B_BM + row] = acc0 + acc1;
          mbar_arrive(&bars->dx_full[qc & 1]);
        }
        float delta;
        {
          ok = mbar_wait(&bars->dx_full[qc & 1], (qc >> 1) & 1, wc, 205);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          const float* dx = reinterpret_cast<const float*>(smem + T::B_SM_DX) + (qc & 1) * 2 * T::B_BM;
          delta = dx[row] + dx[T::B_BM + row];  // the same sum in both warpgroups
          if (wg == 0) {  // for the dK/dV kernel, launched after this one
            prm.delta[grow] = delta;
            prm.lse2[grow] = lse2;
          }
        }
        const uint64_t c2 = f2_pack(sl2, sl2), nl2 = f2_pack(-lse2, -lse2), nd2 = f2_pack(-delta, -delta);
        {
          // the CTA's next item: its dO rows into L2 while this one runs
          int nhead = head, ni = -1;
          if (half == 0 && ib >= 0) {
            ni = ib;
          } else if (u + static_cast<int>(gridDim.x) < units) {
            int nb;
            bwd2_decode<CAUSAL>(u + gridDim.x, nqt, nhead, ni, nb);
          }
          if (ni >= 0 && ni * T::B_BM + row < Nq) {
            const size_t nrow = static_cast<size_t>(nhead) * Nq + ni * T::B_BM + row;
            prefetch_row128(prm.dout + nrow * T::D + wg * 128);
            prefetch_row128(prm.o + nrow * T::D + wg * 128);
            if (wg == 0 && lane == 0)  // one line of lse covers this warp's 32 rows
              asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(prm.lse + nrow));
          }
        }
        for (int j = 0; j < num_kv(i); ++j) {
          const int k0 = j * T::B_BN + wg * T::B_KC;  // first key column of this warpgroup
          const uint32_t rb = lb + T::B_R + (t & 1) * T::B_BN + wg * T::B_KC;  // this warpgroup's columns
          ok = mbar_wait(&bars->s_full[t & 1], (t >> 1) & 1, wc, 201);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          uint32_t sr[T::B_KC];
          tmem_ld32(rb, sr);
          tmem_wait_ld();
          reg_fence<T::B_KC>(sr);
          tc_fence_before();
          mbar_arrive(&bars->s_free);
          // P = exp2(S * c - lse2) in packed fp32 pairs
          uint64_t p2[T::B_KC / 2];
          const bool masked = (j + 1) * T::B_BN - 1 > lim_lo;
          // causal: the row's visible prefix of columns as one bit per column
          uint32_t keep = 0xffffffffu;
          if constexpr (CAUSAL) {
            const int n = min(max(lim - k0 + 1, 0), 32);
            keep = n == 32 ? 0xffffffffu : ((1u << n) - 1u);
          }
#pragma unroll
          for (int c = 0; c < T::B_KC; c += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, nl2), x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if constexpr (CAUSAL) {
              if (masked) {
                p0 = ((keep >> c) & 1u) ? p0 : 0.f;
                p1 = ((keep >> (c + 1)) & 1u) ? p1 : 0.f;
              }
            } else if (masked) {
              if (k0 + c > lim) p0 = 0.f;
              if (k0 + c + 1 > lim) p1 = 0.f;
            }
            p2[c / 2] = f2_pack(p0, p1);
          }
          // ---- dS = P * (dP - Delta), 16-bit into TMEM over dP
          ok = mbar_wait(&bars->dp_full[t & 1], (t >> 1) & 1, wc, 202);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          tmem_ld32(rb, sr);
          tmem_wait_ld();
          reg_fence<T::B_KC>(sr);
          uint32_t pk[T::B_KC / 2];
#pragma unroll
          for (int c = 0; c < T::B_KC; c += 2)
            pk[c / 2] = f2_to_pack2<BF>(f2_mul(p2[c / 2], f2_add(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), nd2)));
          tmem_st16(rb, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->ds_full[t & 1]);
          ++t;
        }
        if (!ok) break;
        // ---- dQ_i (times scale) -> 16-bit, staged in the K slot (columns
        // 0-127, warpgroup 0) and the V slot (128-255, warpgroup 1) of the
        // item's last tile; the dQ MMA warp writes it out (rows past Nq are
        // dropped by the TMA store)
        ok = mbar_wait(&bars->dq_full, qc & 1, wc, 203);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t st_q = smem_u32(smem + (wg == 0 ? T::B_SM_K + ((t - 1) % KS) * T::B_KTILE
                                                       : T::B_SM_V + ((t - 1) % VS) * T::B_KTILE));
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) stage_tmem32<BF>(lb + T::B_DQ + wg * 128 + c, prm.scale, st_q, row, c);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->dq_free);
        mbar_arrive(&bars->epi_full);
        ++qc;
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

// The dQ kernel (which also writes Delta and lse2 of every query row), then
// the dK/dV kernel, on the same stream.  maps: [0] q (64-row boxes), [1] k
// (128-row boxes), [3] dout (64-row boxes) for the dK/dV kernel; [7] q
// (128-row boxes), [8] k (64-row boxes), [2] v (64-row boxes) for the dQ
// kernel.
template <bool CAUSAL, bool BF>
int launch_bwd256(const CUtensorMap* maps, const BwdParams& prm, int max_ctas, cudaStream_t stream) {
  using T = B256;
  static DeviceOnceFlags attr_done;  // the attributes are per device
  if (once_per_device(attr_done, current_device_index(), [] {
        return cudaFuncSetAttribute(fa_bwd256_dkdv_kernel<CAUSAL, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    T::A_SMEM) == cudaSuccess &&
                       cudaFuncSetAttribute(fa_bwd256_dq_kernel<CAUSAL, BF>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, T::B_SMEM) == cudaSuccess
                   ? 0
                   : -1;
      }) != 0)
    return -1;
  auto grid_for = [&](int heads, int tiles) {
    const long long units = CAUSAL ? static_cast<long long>(heads) * ((tiles + 1) / 2) : static_cast<long long>(heads) * tiles;
    return static_cast<int>(units < max_ctas ? units : max_ctas);
  };
  const int nkv = (prm.Nk + T::A_BN - 1) / T::A_BN, nqt = (prm.Nq + T::B_BM - 1) / T::B_BM;
  fa_bwd256_dq_kernel<CAUSAL, BF><<<grid_for(prm.heads, nqt), T::B_THREADS, T::B_SMEM, stream>>>(
      maps[7], maps[8], maps[2], maps[4], prm);
  if (cudaGetLastError() != cudaSuccess) return -1;
  fa_bwd256_dkdv_kernel<CAUSAL, BF><<<grid_for(prm.heads / prm.group, nkv), T::A_THREADS, T::A_SMEM, stream>>>(
      maps[0], maps[1], maps[3], maps[5], maps[6], prm);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

// FlashAttention backward for sm_103a.
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
// §二 -- Delta = rowsum(O * dO); P recomputed from Q K^T * scale and the saved
// log-sum-exp; dP = dO V^T; dS = scale * P * (dP - Delta); dQ += dS K;
// dK += dS^T Q; dV += P^T dO; the three design rules (recompute P, one writer
// per gradient tile, scratch per physical core that does not grow with N^2
// over all heads); §五 -- persistent programs that each own whole heads, so a
// program produces a head's complete dQ/dK/dV and nothing is reduced across
// programs; §七 -- D256 handled as two D128 halves.
//
// Two kernels:
//  1. fa_bwd_prep_kernel: Delta = rowsum(O * dO) in fp32 and lse2 = lse *
//     log2(e) for every row (HBM-bound, one pass over O and dO).
//  2. fa_bwd_kernel: persistent CTAs, CTA b owns heads b, b + grid, ...  For
//     each key tile j (128 keys; K_j, V_j resident in shared memory) it
//     streams the query tiles i and, with M = keys on the tensor cores:
//        S^T  = K_j Q_i^T              (TMEM)
//        P^T  = exp2(S^T * c - lse2)   (compute warps; fp16 back into TMEM)
//        dP^T = V_j dO_i^T             (TMEM)
//        dS^T = P^T * (dP^T - Delta)   (compute warps; fp16 into smem)
//        dV_j += P^T dO_i              (A operand read from TMEM)
//        dK_j += dS^T Q_i
//        dQ_i  = dS K_j                (or its transpose for D = 256)
//     dK_j and dV_j accumulate in TMEM and are written once per key tile.
//     dQ_i is added into the CTA's own fp32 accumulator in global memory
//     (N x D per CTA, independent of the number of heads); the CTA converts
//     it to fp16 after its head's last key tile.  The scale of dS is applied
//     once, to dK and dQ at write-out.
//   For D = 256 (query tiles of 64 rows) the key tile is swept twice, once per
//   128-wide half of D: S^T and dP^T are recomputed (full-D contractions) and
//   each sweep accumulates one half of dK_j and dV_j, which keeps every
//   accumulator 128 columns wide.
//
// Roles (320 threads): warps 0-7 compute (warpgroup w handles half the
// columns; warp%4 selects the TMEM lane quarter), warp 8 TMA producer,
// warp 9 MMA issuer (converged warp, one elected lane per MMA) and TMEM
// owner.
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

// -------------------------------------------------------------- main kernel

template <int D, bool CAUSAL>
struct BwdTraits {
  static constexpr int BN = 128;                    // keys per tile (MMA M)
  static constexpr int BM = (D == 256) ? 64 : 128;  // queries per tile
  static constexpr int NPASS = (D == 256) ? 2 : 1;  // sweeps over D halves
  static constexpr int DH = D / NPASS;              // accumulator width
  static constexpr int Q_STAGES = (D == 256) ? 1 : 2;
  static constexpr bool DQ_T = (D == 256);          // dQ computed transposed
  static constexpr int DSUB = D / 64;
  static constexpr int Q_SUB = BM * 128;   // bytes of a [BM x 64] fp16 sub-tile
  static constexpr int KV_SUB = BN * 128;  // bytes of a [BN x 64] fp16 sub-tile
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int DS_SUB = BN * 128;  // dS^T buffer: [BN keys x 64 queries] sub-tiles
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int QC = BM / 2;        // query columns per compute warpgroup
  // TMEM columns
  static constexpr int DV_COL = 0;
  static constexpr int DK_COL = DH;
  static constexpr int S_COL = 2 * DH;
  static constexpr int DP_COL = 2 * DH + BM;
  static constexpr int DQ_COL = DQ_T ? 2 * DH + 2 * BM : DP_COL;
  static constexpr int DQ_W = DQ_T ? BM : D;  // TMEM columns of the dQ tile
  static constexpr int TMEM_COLS = 512;
  static_assert(DQ_COL + DQ_W <= TMEM_COLS && DP_COL + BM <= TMEM_COLS, "TMEM budget");
  // shared memory
  static constexpr int SM_K = 0;
  static constexpr int SM_V = KV_BYTES;
  static constexpr int SM_Q = 2 * KV_BYTES;
  static constexpr int SM_DO = SM_Q + Q_STAGES * Q_BYTES;
  static constexpr int SM_DS = SM_DO + Q_STAGES * Q_BYTES;
  static constexpr int SM_BAR = SM_DS + DS_BYTES;
  static constexpr int SM_BYTES = SM_BAR + 256;
  static constexpr int SMEM_ALLOC = (SM_BYTES + 1024 > 120 * 1024) ? SM_BYTES + 1024 : 120 * 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static constexpr int THREADS = 320;
  static constexpr int COMPUTE_THREADS = 256;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
};

struct BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, dv_done, dq_full, dq_free, ds_free;
  uint64_t dkv_full, dkv_free, mma_done;
  uint64_t cw_sync;  // compute-warp barrier with a bounded wait
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 256, "barrier area");

__device__ __forceinline__ void bwd_drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_test(a, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void red_add_f32(float* p, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}

template <int D, bool CAUSAL>
__device__ __forceinline__ int bwd_first_qtile(int j) {
  using T = BwdTraits<D, CAUSAL>;
  return CAUSAL ? (j * T::BN) / T::BM : 0;
}

template <int D, bool CAUSAL, bool BF>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams prm) {
  using T = BwdTraits<D, CAUSAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + T::SM_BAR);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, T::COMPUTE_THREADS);
    mbar_init(&bars->ds_full, T::COMPUTE_THREADS);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, T::COMPUTE_THREADS);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_free, T::COMPUTE_THREADS);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->cw_sync, T::COMPUTE_THREADS);
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
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  const int N = prm.N;
  const int nqt = N / T::BM;
  const int nkv = N / T::BN;

  if (warp == T::PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      uint32_t t = 0, kc = 0;
      bool ok = true;
      for (int head = blockIdx.x; ok && head < prm.heads; head += gridDim.x) {
        for (int j = 0; ok && j < nkv; ++j) {
          if (!(ok = mbar_wait(&bars->kv_empty, (kc & 1) ^ 1, wc, 21))) break;
          mbar_arrive_expect_tx(&bars->kv_full, 2 * T::KV_BYTES);
          for (int s = 0; s < T::DSUB; ++s) {
            tma_load_3d_hint(smem + T::SM_K + s * T::KV_SUB, &tm_k, &bars->kv_full, s * 64, j * T::BN, head, pol);
            tma_load_3d_hint(smem + T::SM_V + s * T::KV_SUB, &tm_v, &bars->kv_full, s * 64, j * T::BN, head, pol);
          }
          ++kc;
          for (int h = 0; ok && h < T::NPASS; ++h) {
            for (int i = bwd_first_qtile<D, CAUSAL>(j); i < nqt; ++i) {
              const int st = t % T::Q_STAGES;
              if (!(ok = mbar_wait(&bars->q_empty[st], ((t / T::Q_STAGES) & 1) ^ 1, wc, 22))) break;
              mbar_arrive_expect_tx(&bars->q_full[st], 2 * T::Q_BYTES);
              for (int s = 0; s < T::DSUB; ++s) {
                tma_load_3d_hint(smem + T::SM_Q + st * T::Q_BYTES + s * T::Q_SUB, &tm_q, &bars->q_full[st], s * 64,
                                 i * T::BM, head, pol);
                tma_load_3d_hint(smem + T::SM_DO + st * T::Q_BYTES + s * T::Q_SUB, &tm_do, &bars->q_full[st],
                                 s * 64, i * T::BM, head, pol);
              }
              ++t;
            }
          }
        }
      }
      if (kc > 0) bwd_drain_wait(&bars->kv_full, (kc - 1) & 1);
      for (uint32_t i = (t > T::Q_STAGES ? t - T::Q_STAGES : 0); i < t; ++i)
        bwd_drain_wait(&bars->q_full[i % T::Q_STAGES], (i / T::Q_STAGES) & 1);
    }
  } else if (warp == T::MMA_WARP) {
    // ------------------------------------------------------------- MMA issuer
    {  // the whole warp runs the loop; one elected lane issues each MMA
      constexpr uint32_t id_s = idesc_16<BF>(128, T::BM, false, false);   // S^T, dP^T: M keys, N queries
      constexpr uint32_t id_kv = idesc_16<BF>(128, T::DH, false, true);   // dV, dK: N = DH, B MN-major
      constexpr uint32_t id_dq = T::DQ_T ? idesc_16<BF>(128, T::BM, true, true)  // dQ^T: M = d, N = queries
                                         : idesc_16<BF>(128, D, true, true);     // dQ: M = queries, N = D
      const uint32_t sb = smem_u32(smem);
      const uint32_t sK = sb + T::SM_K, sV = sb + T::SM_V, sDS = sb + T::SM_DS;
      uint32_t t = 0, kc = 0, pc = 0;
      bool ok = true;
      for (int head = blockIdx.x; ok && head < prm.heads; head += gridDim.x) {
        for (int j = 0; ok && j < nkv; ++j) {
          if (!(ok = warp_wait(&bars->kv_full, kc & 1, wc, 31))) break;
          tc_fence_after();
          for (int h = 0; ok && h < T::NPASS; ++h) {
            const int i0 = bwd_first_qtile<D, CAUSAL>(j);
            for (int i = i0; i < nqt; ++i) {
              const bool first = (i == i0);
              const int st = t % T::Q_STAGES;
              if (!(ok = warp_wait(&bars->q_full[st], (t / T::Q_STAGES) & 1, wc, 32))) break;
              tc_fence_after();
              const uint32_t sQ = sb + T::SM_Q + st * T::Q_BYTES;
              const uint32_t sO = sb + T::SM_DO + st * T::Q_BYTES;
              // S^T = K Q^T (the S region still holds P^T of the previous tile
              // until that tile's dV MMA has completed)
              if (t > 0 && !(ok = warp_wait(&bars->dv_done, (t - 1) & 1, wc, 33))) break;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = sdesc_sw128(sK + (kk / 4) * T::KV_SUB + (kk % 4) * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(sQ + (kk / 4) * T::Q_SUB + (kk % 4) * 32, 16, 1024);
                mma_f16_ss_warp(tmem + T::S_COL, a, b, id_s, kk > 0 ? 1u : 0u);
              }
              mma_commit_warp(&bars->s_full);
              // dP^T = V dO^T (the dP region holds the previous dQ until drained)
              if (t > 0 && !(ok = warp_wait(&bars->dq_free, (t - 1) & 1, wc, 34))) break;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = sdesc_sw128(sV + (kk / 4) * T::KV_SUB + (kk % 4) * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(sO + (kk / 4) * T::Q_SUB + (kk % 4) * 32, 16, 1024);
                mma_f16_ss_warp(tmem + T::DP_COL, a, b, id_s, kk > 0 ? 1u : 0u);
              }
              mma_commit_warp(&bars->dp_full);
              // dV += P^T dO (P^T from TMEM); the first tile of a sweep
              // overwrites the accumulators, so the previous sweep's
              // write-out must have read them.
              if (first && pc > 0 && !(ok = warp_wait(&bars->dkv_free, (pc - 1) & 1, wc, 35))) break;
              if (!(ok = warp_wait(&bars->p_full, t & 1, wc, 36))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < T::BM / 16; ++kk) {
                const int q = kk * 16, wg = q / T::QC;
                const uint32_t a_t = tmem + T::S_COL + wg * T::QC + (q - wg * T::QC) / 2;
                const uint64_t b = sdesc_sw128(sO + h * (T::DH / 64) * T::Q_SUB + kk * 2048, T::Q_SUB, 1024);
                mma_f16_ts_warp(tmem + T::DV_COL, a_t, b, id_kv, (first && kk == 0) ? 0u : 1u);
              }
              mma_commit_warp(&bars->dv_done);
              // dK += dS^T Q and dQ (dS^T from shared memory)
              if (!(ok = warp_wait(&bars->ds_full, t & 1, wc, 37))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < T::BM / 16; ++kk) {
                const uint64_t a = sdesc_sw128(sDS + ((kk * 16) / 64) * T::DS_SUB + (kk % 4) * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(sQ + h * (T::DH / 64) * T::Q_SUB + kk * 2048, T::Q_SUB, 1024);
                mma_f16_ss_warp(tmem + T::DK_COL, a, b, id_kv, (first && kk == 0) ? 0u : 1u);
              }
#pragma unroll
              for (int kk = 0; kk < T::BN / 16; ++kk) {
                if (T::DQ_T) {
                  // dQ^T[h half] = K[:, h half]^T dS^T : A = K (MN-major), B = dS^T (MN-major)
                  const uint64_t a = sdesc_sw128(sK + h * 2 * T::KV_SUB + kk * 2048, T::KV_SUB, 1024);
                  const uint64_t b = sdesc_sw128(sDS + kk * 2048, T::DS_SUB, 1024);
                  mma_f16_ss_warp(tmem + T::DQ_COL, a, b, id_dq, kk > 0 ? 1u : 0u);
                } else {
                  // dQ = dS K : A = dS (dS^T buffer read MN-major), B = K (MN-major)
                  const uint64_t a = sdesc_sw128(sDS + kk * 2048, T::DS_SUB, 1024);
                  const uint64_t b = sdesc_sw128(sK + kk * 2048, T::KV_SUB, 1024);
                  mma_f16_ss_warp(tmem + T::DQ_COL, a, b, id_dq, kk > 0 ? 1u : 0u);
                }
              }
              mma_commit_warp(&bars->q_empty[st]);
              mma_commit_warp(&bars->ds_free);
              mma_commit_warp(&bars->dq_full);
              ++t;
            }
            if (!ok) break;
            mma_commit_warp(&bars->dkv_full);
            ++pc;
          }
          if (!ok) break;
          mma_commit_warp(&bars->kv_empty);
          ++kc;
        }
      }
      mma_commit_warp(&bars->mma_done);
      bwd_drain_wait(&bars->mma_done, 0);
    }
  } else {
    // --------------------------------------------------------- compute warps
    const int wg = warp >> 2;             // column half
    const int quad = warp & 3;            // TMEM lane quarter
    const int row = quad * 32 + lane;     // TMEM lane
    const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = prm.scale_log2;
    const float scale = prm.scale;
    float* acc = prm.dq_acc + static_cast<size_t>(blockIdx.x) * N * D;
    const uint32_t sDS = smem_u32(smem + T::SM_DS);
    uint32_t t = 0, pc = 0, sync_phase = 0;
    bool ok = true;
    // Barrier among the 256 compute threads; bounded, so a peer that gave up
    // cannot leave the others blocked.
    auto cw_barrier = [&](int site) -> bool {
      mbar_arrive(&bars->cw_sync);
      const bool r = mbar_wait(&bars->cw_sync, sync_phase & 1, wc, site);
      ++sync_phase;
      return __all_sync(0xffffffffu, r);
    };
    for (int head = blockIdx.x; ok && head < prm.heads; head += gridDim.x) {
      const float* lse2_h = prm.lse2 + static_cast<size_t>(head) * N;
      const float* delta_h = prm.delta + static_cast<size_t>(head) * N;
      for (int j = 0; ok && j < nkv; ++j) {
        const int key = j * T::BN + row;  // this thread's key (S^T, dP^T, dK, dV rows)
        for (int h = 0; ok && h < T::NPASS; ++h) {
          const int i0 = bwd_first_qtile<D, CAUSAL>(j);
          for (int i = i0; i < nqt; ++i) {
            const int q0 = i * T::BM + wg * T::QC;  // first query column of this warpgroup
            // ---- P^T = exp2(S^T * c - lse2), masked above the diagonal
            ok = mbar_wait(&bars->s_full, t & 1, wc, 41);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[T::QC];
#pragma unroll
            for (int c = 0; c < T::QC; c += 32) tmem_ld32(lb + T::S_COL + wg * T::QC + c, sr + c);
            tmem_wait_ld();
            reg_fence<T::QC>(sr);
            float p[T::QC];
            const float4* l4 = reinterpret_cast<const float4*>(lse2_h + q0);
#pragma unroll
            for (int c = 0; c < T::QC; c += 4) {
              const float4 L = __ldg(l4 + c / 4);
              p[c + 0] = ex2_approx(fmaf(__uint_as_float(sr[c + 0]), sl2, -L.x));
              p[c + 1] = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, -L.y));
              p[c + 2] = ex2_approx(fmaf(__uint_as_float(sr[c + 2]), sl2, -L.z));
              p[c + 3] = ex2_approx(fmaf(__uint_as_float(sr[c + 3]), sl2, -L.w));
            }
            if (CAUSAL && (j + 1) * T::BN - 1 > i * T::BM) {
#pragma unroll
              for (int c = 0; c < T::QC; ++c)
                if (key > q0 + c) p[c] = 0.f;
            }
            uint32_t pk[T::QC / 2];
#pragma unroll
            for (int c = 0; c < T::QC / 2; ++c) pk[c] = pack2<BF>(p[2 * c], p[2 * c + 1]);
            if (T::QC / 2 == 32) {
              tmem_st32(lb + T::S_COL + wg * T::QC, pk);
            } else {
              tmem_st16(lb + T::S_COL + wg * T::QC, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full);
            // ---- dS^T = P^T * (dP^T - Delta) -> fp16 -> shared memory
            ok = mbar_wait(&bars->dp_full, t & 1, wc, 42);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < T::QC; c += 32) tmem_ld32(lb + T::DP_COL + wg * T::QC + c, sr + c);
            tmem_wait_ld();
            reg_fence<T::QC>(sr);
            const float4* d4 = reinterpret_cast<const float4*>(delta_h + q0);
#pragma unroll
            for (int c = 0; c < T::QC; c += 4) {
              const float4 Dl = __ldg(d4 + c / 4);
              pk[c / 2] = pack2<BF>(p[c] * (__uint_as_float(sr[c]) - Dl.x), p[c + 1] * (__uint_as_float(sr[c + 1]) - Dl.y));
              pk[c / 2 + 1] =
                  pack2<BF>(p[c + 2] * (__uint_as_float(sr[c + 2]) - Dl.z), p[c + 3] * (__uint_as_float(sr[c + 3]) - Dl.w));
            }
            if (t > 0) {
              ok = mbar_wait(&bars->ds_free, (t - 1) & 1, wc, 43);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            }
#pragma unroll
            for (int c = 0; c < T::QC; c += 8) {
              const int qq = wg * T::QC + c;  // query column inside the tile
              const uint32_t addr = sDS + (qq / 64) * T::DS_SUB + row * 128 + ((((qq % 64) / 8) ^ (row & 7)) * 16);
              st_shared_v4(addr, pk[c / 2], pk[c / 2 + 1], pk[c / 2 + 2], pk[c / 2 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->ds_full);
            // ---- dQ partial -> this CTA's fp32 accumulator
            ok = mbar_wait(&bars->dq_full, t & 1, wc, 44);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            if (!T::DQ_T) {
              // TMEM lane = query row, columns = d; this warpgroup takes D/2 columns
              float* dst = acc + static_cast<size_t>(i * T::BM + row) * D + wg * (D / 2);
#pragma unroll
              for (int c = 0; c < D / 2; c += 32) {
                uint32_t v[32];
                tmem_ld32(lb + T::DQ_COL + wg * (D / 2) + c, v);
                tmem_wait_ld();
                reg_fence<32>(v);
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                  float* pd = dst + c + e;
                  const float a0 = __uint_as_float(v[e]), a1 = __uint_as_float(v[e + 1]);
                  const float a2 = __uint_as_float(v[e + 2]), a3 = __uint_as_float(v[e + 3]);
                  if (j == 0) {
                    *reinterpret_cast<float4*>(pd) = make_float4(a0, a1, a2, a3);
                  } else {
                    red_add_v4(pd, a0, a1, a2, a3);
                  }
                }
              }
            } else {
              // TMEM lane = d inside the half, columns = queries
              const int d = h * T::DH + row;
              uint32_t v[32];
              tmem_ld32(lb + T::DQ_COL + wg * T::QC, v);
              tmem_wait_ld();
              reg_fence<32>(v);
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                float* pd = acc + static_cast<size_t>(q0 + c) * D + d;
                if (j == 0) {
                  *pd = __uint_as_float(v[c]);
                } else {
                  red_add_f32(pd, __uint_as_float(v[c]));
                }
              }
            }
            tc_fence_before();
            mbar_arrive(&bars->dq_free);
            ++t;
          }
          if (!ok) break;
          // ---- write dV_j, dK_j (this sweep's half of D), scale folded into dK
          ok = mbar_wait(&bars->dkv_full, pc & 1, wc, 45);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          const size_t orow = (static_cast<size_t>(head) * N + key) * D + h * T::DH + wg * (T::DH / 2);
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t col = (which == 0 ? T::DV_COL : T::DK_COL) + wg * (T::DH / 2);
            const float mul = which == 0 ? 1.f : scale;
            __half* out = (which == 0 ? prm.dv : prm.dk) + orow;
#pragma unroll
            for (int c = 0; c < T::DH / 2; c += 32) {
              uint32_t v[32];
              tmem_ld32(lb + col + c, v);
              tmem_wait_ld();
              reg_fence<32>(v);
              uint32_t hv[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                hv[e] = pack2<BF>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
              uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
              for (int e = 0; e < 4; ++e) dst[e] = make_uint4(hv[4 * e], hv[4 * e + 1], hv[4 * e + 2], hv[4 * e + 3]);
            }
          }
          tc_fence_before();
          mbar_arrive(&bars->dkv_free);
          ++pc;
        }
      }
      if (!ok) break;
      // ---- dQ = scale * accumulator -> fp16 (all of this head's key tiles are in)
      __threadfence();
      if (!(ok = cw_barrier(46))) break;
      const float4* src = reinterpret_cast<const float4*>(acc);
      uint2* dq = reinterpret_cast<uint2*>(prm.dq + static_cast<size_t>(head) * N * D);
      for (int e = threadIdx.x; e < N * D / 4; e += T::COMPUTE_THREADS) {
        const float4 v = __ldcg(src + e);
        dq[e] = make_uint2(pack2<BF>(v.x * scale, v.y * scale), pack2<BF>(v.z * scale, v.w * scale));
      }
      // the next head's first key tile overwrites the accumulator
      if (!(ok = cw_barrier(47))) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == T::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF>
int launch_bwd(const CUtensorMap* maps, const BwdParams& prm, int grid, cudaStream_t stream) {
  using T = BwdTraits<D, CAUSAL>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(fa_bwd_kernel<D, CAUSAL, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T::SMEM_ALLOC) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  if (launch_prep<D, BF>(prm, stream) != 0) return -1;
  fa_bwd_kernel<D, CAUSAL, BF><<<grid, T::THREADS, T::SMEM_ALLOC, stream>>>(maps[0], maps[1], maps[2], maps[3], prm);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

// FlashAttention forward for D = 256 over dense K/V on sm_103a.
//
// Source: «把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战»,
// §一 (the online softmax over key tiles, exp2 with log2(e) folded into the
// scale, fp32 m, l and accumulator, P rounded to 16 bits before the matrix
// unit, O written once) and §七 (D256: the accumulator split so that it fits;
// here it is one 256-column TMEM accumulator fed by N = 256 MMAs).
//
// Tiles of 128 queries x 128 keys.  A 128-key tile of K or V at D = 256 is
// 64 KB, so K and V travel through rings of 32 KB half tiles: K by halves of
// the contraction (dims 0-127, 128-255), V by halves of the keys (keys 0-63,
// 64-127), each half consumed by its own run of MMAs.  Shared memory: Q (64
// KB, one per work item), three K halves, two V halves.
//
// TMEM: two 128-column regions that the key tiles use in turn -- S(t) fp32,
// then P(t) 16-bit over its first 64 columns once both softmax warpgroups
// have read S(t) -- and O in columns 256-511.  S(t+2) goes into the region
// of tile t once P V(t) has read P(t).
//
// Roles (512 threads, one CTA per SM):
//   warps 0-7   softmax: two warpgroups split each tile's key columns; thread
//               (g, r) owns query row r.  Both read the whole S row (row
//               max), exponentiate their half, keep a partial l, write P.
//   warps 8-11  epilogue: O / l -> 16-bit straight to global memory (each
//               thread its row), lse; overlaps the next item's softmax.
//   warp 12     TMA producer: Q per work item, K halves into their ring.
//   warp 13     Q K^T issuer and TMEM owner.
//   warp 14     TMA producer: V halves into their ring.
//   warp 15     P V issuer (N = 256, P from TMEM).
#pragma once

#include "fa_fwd.cuh"

namespace fa {

struct Fwd256 {
  static constexpr int D = 256, BM = 128, BN = 128;
  static constexpr int KS = 3, VS = 2;        // half-tile ring slots
  static constexpr int SUB = 128 * 128;       // [128 rows x 64] 16-bit sub-tile, 16 KB
  static constexpr int VSUB = 64 * 128;       // [64 keys x 64] sub-tile of a V half, 8 KB
  static constexpr int Q_BYTES = 4 * SUB;     // 64 KB
  static constexpr int HALF = 32 * 1024;      // K half (2 sub-tiles) or V half (4 sub-tiles)
  static constexpr int SM_Q = 0, SM_K = Q_BYTES, SM_V = SM_K + KS * HALF;
  static constexpr int SM_LM = SM_V + VS * HALF;  // [3][BM] fp32: l of both halves, m
  static constexpr int SM_BAR = SM_LM + 3 * BM * 4;
  static constexpr int SMEM = SM_BAR + 512;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr int O_COL = 256;           // TMEM: regions at 0 and 128, O at 256
  static constexpr int THREADS = 512, SOFTMAX_THREADS = 256, EPI_THREADS = 128;
  static constexpr int PRODUCER_WARP = 12, MMA_WARP = 13, V_PRODUCER_WARP = 14, PV_MMA_WARP = 15;
  static constexpr int SOFTMAX_REGS = 184, OTHER_REGS = 64;  // 256 x 184 + 256 x 64 <= 65536
};

struct Fwd256Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[Fwd256::KS], k_empty[Fwd256::KS], v_full[Fwd256::VS], v_empty[Fwd256::VS];
  uint64_t s_full[2], p_full[2], pv_done[2];  // per TMEM region
  uint64_t s_read;                            // both warpgroups have read S(t): P may overwrite it
  uint64_t o_free, lm_full, lm_empty, mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Fwd256Bars) <= 512, "barrier area");

// The work items of one CTA in processing order (units blockIdx.x,
// blockIdx.x + gridDim.x, ...; a causal unit is query tiles qt and nqt-1-qt
// of one head) and the key tiles of each: all of them, or (causal) up to the
// last key the tile's last query sees.  Packed grouped heads (q_period > 0)
// put every query position in every tile.
template <bool CAUSAL>
struct Fwd256Items {
  int u, units, nqt, head, qa, qb, half;
  __device__ Fwd256Items(int units_, int nqt_) : u(blockIdx.x), units(units_), nqt(nqt_), head(0), qa(0), qb(-1), half(0) {
    if (u < units) fwd_decode<CAUSAL>(u, nqt, head, qa, qb);
  }
  __device__ bool valid() const { return u < units; }
  __device__ int qt() const { return half ? qb : qa; }
  __device__ void next() {
    if (half == 0 && qb >= 0) {
      half = 1;
      return;
    }
    half = 0;
    u += gridDim.x;
    if (u < units) fwd_decode<CAUSAL>(u, nqt, head, qa, qb);
  }
  __device__ int tiles(const FwdParams& prm) const {
    const int nkv = (prm.Nk + Fwd256::BN - 1) / Fwd256::BN;
    if (!CAUSAL) return nkv;
    const int end = prm.q_period > 0 ? min(prm.q_period + prm.causal_off, prm.Nk)
                                     : min((qt() + 1) * Fwd256::BM + prm.causal_off, prm.Nk);
    return (end + Fwd256::BN - 1) / Fwd256::BN;
  }
};

template <bool CAUSAL, bool BF>
__global__ void __launch_bounds__(512, 1)
    fa_fwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams prm) {
  using T = Fwd256;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128-byte-swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) record_timeout(prm.status, 99);
    return;
  }
  Fwd256Bars* bars = reinterpret_cast<Fwd256Bars*>(smem + T::SM_BAR);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < T::KS; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < T::VS; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], T::SOFTMAX_THREADS);
      mbar_init(&bars->pv_done[i], 1);
      mbar_init(&bars->mma_done[i], 1);
    }
    mbar_init(&bars->s_read, T::SOFTMAX_THREADS);
    mbar_init(&bars->o_free, T::EPI_THREADS);
    mbar_init(&bars->lm_full, T::SOFTMAX_THREADS);
    mbar_init(&bars->lm_empty, T::EPI_THREADS);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == T::MMA_WARP) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == T::PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  } else if (warp == T::V_PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const WaitCtx wc{prm.status, &bars->abort_flag};
  const uint32_t tmem = bars->tmem_base;
  const int Nq = prm.Nq, Nk = prm.Nk, off = prm.causal_off, qp = prm.q_period;
  const int nqt = (Nq + T::BM - 1) / T::BM;
  const int units = fwd_num_units<CAUSAL>(prm.heads, nqt);

  if (warp < 8) {
    reg_alloc<T::SOFTMAX_REGS>();
    // ------------------------------------------------------- softmax warps
    constexpr int HC = T::BN / 2;  // S columns per thread
    const int wg = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;  // query row inside the tile, == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* lm = reinterpret_cast<float*>(smem + T::SM_LM);
    const float sl2 = prm.scale_log2;
    uint32_t t = 0, n = 0;
    bool ok = true;
    for (Fwd256Items<CAUSAL> it(units, nqt); ok && it.valid(); it.next(), ++n) {
      const int qt = it.qt(), nkv = it.tiles(prm);
      const int qi = qt * T::BM + r;                  // query row within the head
      const int qpos = qp > 0 ? qi % qp : qi;         // its query position
      const int lim = fwd_key_limit<CAUSAL>(qpos, Nk, off);  // this row's last key
      const int lim_lo = fwd_key_limit<CAUSAL>(qp > 0 ? 0 : qt * T::BM, Nk, off);  // the tile's smallest limit
      float m = -INFINITY, l = 0.f;                   // l: this half's partial row sum
      for (int j = 0; j < nkv; ++j) {
        const int b = t & 1;
        const uint32_t sreg = lane_base + b * T::BN;
        ok = mbar_wait(&bars->s_full[b], (t >> 1) & 1, wc, 205);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        // the other half of the row: only its max is needed
        uint32_t sr[HC];
        float pm[8];
#pragma unroll
        for (int c = 0; c < HC; c += 32) tmem_ld32(sreg + (wg ^ 1) * HC + c, sr + c);
        tmem_wait_ld();
        reg_fence<HC>(sr);
        const bool masked = (j + 1) * T::BN - 1 > lim_lo;
        auto mask_half = [&](uint32_t* v, int g) {
          if constexpr (CAUSAL) {
            const int nv = lim - (j * T::BN + g * HC) + 1;  // visible columns of half g
#pragma unroll
            for (int w = 0; w < HC / 32; ++w) {
              const int nvis = min(max(nv - 32 * w, 0), 32);
              const uint32_t keep = nvis == 32 ? 0xffffffffu : ((1u << nvis) - 1u);
#pragma unroll
              for (int c = 0; c < 32; ++c) v[32 * w + c] = ((keep >> c) & 1u) ? v[32 * w + c] : __float_as_uint(-INFINITY);
            }
          } else {
            const int k0 = j * T::BN + g * HC;
#pragma unroll
            for (int c = 0; c < HC; ++c)
              if (k0 + c > lim) v[c] = __float_as_uint(-INFINITY);
          }
        };
        if (masked) mask_half(sr, wg ^ 1);
#pragma unroll
        for (int i = 0; i < 8; ++i) pm[i] = fmaxf(__uint_as_float(sr[i]), __uint_as_float(sr[i + 8]));
#pragma unroll
        for (int c = 16; c < HC; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) pm[i] = fmax3(pm[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
        // own half
#pragma unroll
        for (int c = 0; c < HC; c += 32) tmem_ld32(sreg + wg * HC + c, sr + c);
        tmem_wait_ld();
        reg_fence<HC>(sr);
        tc_fence_before();
        mbar_arrive(&bars->s_read);
        if (masked) mask_half(sr, wg);
#pragma unroll
        for (int c = 0; c < HC; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) pm[i] = fmax3(pm[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
        const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        // lazy rescale: m moves only when the tile's max exceeds it by more
        // than kRescaleLog2 (P then stays below 2^kRescaleLog2); O / l and lse
        // use the max actually applied.  Both halves of a row take the same
        // decision from the same row max.
        const float m_tile = mx * sl2;
        const float m_new = (m_tile > m + kRescaleLog2) ? m_tile : m;
        const uint64_t c2 = f2_pack(sl2, sl2), neg2 = f2_pack(-m_new, -m_new);
        uint64_t ps2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ps2[i] = 0ull;
        uint32_t pk[HC / 2];
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, neg2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          ps2[(c >> 1) & 3] = f2_add(ps2[(c >> 1) & 3], f2_pack(p0, p1));
          pk[c / 2] = pack2<BF>(p0, p1);
        }
        float ps[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(ps2[i], ps[2 * i], ps[2 * i + 1]);
        const float rs = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        const float alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)
        l = l * alpha + rs;
        m = m_new;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds P V of the earlier tiles: once the last of them completed,
          // rescale this half's columns of the rows whose max moved
          ok = mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, wc, 206);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t o[32];
            tmem_ld32(lane_base + T::O_COL + wg * 128 + c, o);
            tmem_wait_ld();
            reg_fence<32>(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + T::O_COL + wg * 128 + c, o);
          }
        }
        // P over the region's first 64 columns (this half: 32 of them) once
        // both warpgroups have read all of S
        ok = mbar_wait(&bars->s_read, t & 1, wc, 207);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tmem_st32(sreg + wg * (HC / 2), pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);
        ++t;
      }
      if (!ok) break;
      // ---- hand l (this half's partial row sum) and m to the epilogue warps
      if (n >= 1) {
        ok = mbar_wait(&bars->lm_empty, (n - 1) & 1, wc, 208);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      lm[wg * T::BM + r] = l;
      if (wg == 0) lm[2 * T::BM + r] = m;
      mbar_arrive(&bars->lm_full);
    }
  } else {
    reg_dealloc<T::OTHER_REGS>();
    if (warp == T::PRODUCER_WARP) {
      // ------------------------------------------- producer: Q and K halves
      if (lane == 0) {
        const uint64_t pol_kv = l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_first();
        uint32_t qc = 0, k_it = 0;  // Q and K-half loads issued
        bool ok = true;
        for (Fwd256Items<CAUSAL> it(units, nqt); ok && it.valid(); it.next()) {
          const int qt = it.qt(), nkv = it.tiles(prm), kvh = it.head / prm.group;
          if (!(ok = mbar_wait(&bars->q_empty, (qc & 1) ^ 1, wc, 201))) break;
          mbar_arrive_expect_tx(&bars->q_full, T::Q_BYTES);
          for (int s = 0; s < 4; ++s)
            tma_load_3d_hint(smem + T::SM_Q + s * T::SUB, &tm_q, &bars->q_full, s * 64, qt * T::BM, it.head, pol_q);
          ++qc;
          for (int j = 0; ok && j < nkv; ++j) {
            for (int h = 0; h < 2; ++h) {
              const int st = k_it % T::KS;
              if (!(ok = mbar_wait(&bars->k_empty[st], ((k_it / T::KS) & 1) ^ 1, wc, 202))) break;
              mbar_arrive_expect_tx(&bars->k_full[st], T::HALF);
              for (int s = 0; s < 2; ++s)
                tma_load_3d_hint(smem + T::SM_K + st * T::HALF + s * T::SUB, &tm_k, &bars->k_full[st],
                                 h * 128 + s * 64, j * T::BN, kvh, pol_kv);
              ++k_it;
            }
          }
        }
        // every load issued must have landed before the CTA may exit
        for (uint32_t i = (k_it > T::KS ? k_it - T::KS : 0); i < k_it; ++i)
          drain_wait(&bars->k_full[i % T::KS], (i / T::KS) & 1);
        if (qc > 0) drain_wait(&bars->q_full, (qc - 1) & 1);
      }
    } else if (warp == T::V_PRODUCER_WARP) {
      // ------------------------------------------------- producer: V halves
      if (lane == 0) {
        const uint64_t pol_kv = l2_policy_evict_last();
        uint32_t v_it = 0;
        bool ok = true;
        for (Fwd256Items<CAUSAL> it(units, nqt); ok && it.valid(); it.next()) {
          const int nkv = it.tiles(prm), kvh = it.head / prm.group;
          for (int j = 0; ok && j < nkv; ++j) {
            for (int h = 0; h < 2; ++h) {
              const int st = v_it % T::VS;
              if (!(ok = mbar_wait(&bars->v_empty[st], ((v_it / T::VS) & 1) ^ 1, wc, 203))) break;
              mbar_arrive_expect_tx(&bars->v_full[st], T::HALF);
              for (int s = 0; s < 4; ++s)
                tma_load_3d_hint(smem + T::SM_V + st * T::HALF + s * T::VSUB, &tm_v, &bars->v_full[st], s * 64,
                                 j * T::BN + h * 64, kvh, pol_kv);
              ++v_it;
            }
          }
        }
        for (uint32_t i = (v_it > T::VS ? v_it - T::VS : 0); i < v_it; ++i)
          drain_wait(&bars->v_full[i % T::VS], (i / T::VS) & 1);
      }
    } else if (warp == T::MMA_WARP) {
      // ------------------------------------------------- Q K^T issuer
      // S(t) into region t % 2 once P V(t-2) has read P(t-2) there; the
      // contraction's two halves come from two K half slots.
      constexpr uint32_t idesc_qk = idesc_16<BF>(128, T::BN, false, false);
      const uint32_t sbase = smem_u32(smem);
      const uint64_t qdesc = sdesc_sw128(sbase + T::SM_Q, 16, 1024);
      uint32_t t = 0, n = 0, k_it = 0;
      bool ok = true;
      for (Fwd256Items<CAUSAL> it(units, nqt); ok && it.valid(); it.next(), ++n) {
        const int nkv = it.tiles(prm);
        if (!(ok = warp_wait(&bars->q_full, n & 1, wc, 209))) break;
        for (int j = 0; ok && j < nkv; ++j) {
          const int b = t & 1;
          if (t >= 2 && !(ok = warp_wait(&bars->pv_done[b], ((t - 2) >> 1) & 1, wc, 210))) break;
          for (int h = 0; h < 2; ++h) {
            const int st = k_it % T::KS;
            if (!(ok = warp_wait(&bars->k_full[st], (k_it / T::KS) & 1, wc, 211))) break;
            tc_fence_after();
            const uint64_t kdesc = sdesc_sw128(sbase + T::SM_K + st * T::HALF, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const int g = h * 8 + kk;  // 16-wide slice of the contraction
              mma_f16_ss_warp(tmem + b * T::BN, sdesc_add(qdesc, (g / 4) * T::SUB + (g % 4) * 32),
                              sdesc_add(kdesc, (kk / 4) * T::SUB + (kk % 4) * 32), idesc_qk, g > 0 ? 1u : 0u);
            }
            mma_commit_warp(&bars->k_empty[st]);
            ++k_it;
          }
          if (!ok) break;
          mma_commit_warp(&bars->s_full[b]);
          if (j == nkv - 1) mma_commit_warp(&bars->q_empty);  // Q is not read again
          ++t;
        }
      }
      mma_commit_warp(&bars->mma_done[0]);
      drain_wait(&bars->mma_done[0], 0);
    } else if (warp == T::PV_MMA_WARP) {
      // ---------------------------------------------------- P V issuer
      // O += P V(t), N = 256, P from TMEM region t % 2, 16 keys per MMA from
      // the V half that holds them; the item's first tile overwrites O,
      // which the previous item's epilogue must have read.
      constexpr uint32_t idesc_pv = idesc_16<BF>(128, 256, false, true);
      const uint32_t sbase = smem_u32(smem);
      uint32_t t = 0, n = 0, v_it = 0;
      bool ok = true;
      for (Fwd256Items<CAUSAL> it(units, nqt); ok && it.valid(); it.next(), ++n) {
        const int nkv = it.tiles(prm);
        for (int j = 0; ok && j < nkv; ++j) {
          const int b = t & 1;
          if (j == 0 && n > 0 && !(ok = warp_wait(&bars->o_free, (n - 1) & 1, wc, 212))) break;
          if (!(ok = warp_wait(&bars->p_full[b], (t >> 1) & 1, wc, 213))) break;
          for (int h = 0; h < 2; ++h) {
            const int st = v_it % T::VS;
            if (!(ok = warp_wait(&bars->v_full[st], (v_it / T::VS) & 1, wc, 214))) break;
            tc_fence_after();
            const uint64_t vdesc = sdesc_sw128(sbase + T::SM_V + st * T::HALF, T::VSUB, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts_warp(tmem + T::O_COL, tmem + b * T::BN + (h * 4 + kk) * 8, sdesc_add(vdesc, kk * 2048),
                              idesc_pv, (j == 0 && h == 0 && kk == 0) ? 0u : 1u);
            mma_commit_warp(&bars->v_empty[st]);
            ++v_it;
          }
          if (!ok) break;
          mma_commit_warp(&bars->pv_done[b]);
          ++t;
        }
      }
      mma_commit_warp(&bars->mma_done[1]);
      drain_wait(&bars->mma_done[1], 0);
    } else {
      // ----------------------------------------------- epilogue warps (8-11)
      // O / l -> 16-bit, each thread its row straight to global memory; lse.
      const int quad = warp & 3;
      const int r = quad * 32 + lane;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      const float* lm = reinterpret_cast<const float*>(smem + T::SM_LM);
      uint32_t t = 0, n = 0;
      bool ok = true;
      for (Fwd256Items<CAUSAL> it(units, nqt); ok && it.valid(); it.next(), ++n) {
        const int qt = it.qt();
        t += it.tiles(prm);
        ok = mbar_wait(&bars->lm_full, n & 1, wc, 215);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const float l_row = lm[r] + lm[T::BM + r];
        const float m = lm[2 * T::BM + r];
        mbar_arrive(&bars->lm_empty);
        // the item's last P V has completed
        ok = mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, wc, 216);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float inv_l = 1.f / l_row;
        const int qi = qt * T::BM + r;
        const bool live = qi < Nq;
        uint4* dst = reinterpret_cast<uint4*>(prm.o + (static_cast<size_t>(it.head) * Nq + qi) * T::D);
#pragma unroll 1
        for (int c = 0; c < T::D; c += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + T::O_COL + c, o);
          tmem_wait_ld();
          reg_fence<32>(o);
          uint32_t h[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            h[i] = pack2<BF>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[c / 8 + i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->o_free);
        if (live) prm.lse[static_cast<size_t>(it.head) * Nq + qi] = (m + log2f(l_row)) * 0.69314718055994530942f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == T::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// maps: q (128-row boxes), k (128-row boxes), v (64-row boxes).
template <bool CAUSAL, bool BF>
int launch_fwd256(const CUtensorMap* maps, const FwdParams& prm, int num_sms, cudaStream_t stream) {
  using T = Fwd256;
  static DeviceOnceFlags attr_done;  // the attributes are per device
  const int rc = once_per_device(attr_done, current_device_index(), [] {
    if (cudaFuncSetAttribute(fa_fwd256_kernel<CAUSAL, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
        cudaSuccess)
      return -1;
    // refuse to launch if the build gave the kernel fewer registers than its
    // warpgroup split needs (the raising warpgroups would wait forever)
    cudaFuncAttributes fa_attr;
    if (cudaFuncGetAttributes(&fa_attr, fa_fwd256_kernel<CAUSAL, BF>) != cudaSuccess ||
        fa_attr.numRegs * T::THREADS < T::SOFTMAX_THREADS * T::SOFTMAX_REGS + (T::THREADS - T::SOFTMAX_THREADS) * T::OTHER_REGS)
      return -1;
    return 0;
  });
  if (rc != 0) return -1;
  const int nqt = (prm.Nq + T::BM - 1) / T::BM;
  const long long units = CAUSAL ? static_cast<long long>(prm.heads) * ((nqt + 1) / 2)
                                 : static_cast<long long>(prm.heads) * nqt;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  fa_fwd256_kernel<CAUSAL, BF><<<grid, T::THREADS, T::SMEM, stream>>>(maps[0], maps[1], maps[2], prm);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace fa

// FlashAttention-2 forward pass, bf16 in / fp32 accumulate, for sm_103a.
//
// Algorithm (the FA2 forward of "FlashAttention-2 from PyTorch to Triton",
// section "What We Are Building", with the masking and block skipping of
// "Writing a FlashAttention kernel in Metal", "Blockwise attention and causal
// masking"): for each 128-row query tile Q_i, loop over key/value tiles
// K_j, V_j; S = Q_i K_j^T; fold S into the running row max m, the rescaled row
// sum l and the unnormalised output O (rescale factor exp(m_old - m_new));
// divide by l once at the end and store L = m + log l.
//
// Mapping onto one GB300 SM (one persistent CTA per SM):
//   * a TMA producer warp streams Q tiles and a ring of NS K/V tiles into
//     128-byte-swizzled shared memory, each slot guarded by full/empty mbarriers;
//   * one MMA warp issues tcgen05.mma: S = Q K^T into tensor memory (TMEM),
//     then O += P V with P read from TMEM and V from shared memory;
//   * softmax warpgroups (one thread per query row = one TMEM lane) read S with
//     tcgen05.ld, apply mask and scale, update m and l, write P as bf16 back
//     into the S columns with tcgen05.st, and rescale O in TMEM when the row
//     max moved by more than a factor 2^8 (the guarded correction of the
//     metal-flash-attention case study, with a threshold);
//   * for d <= 128 a work unit is two query tiles (256 rows) sharing every
//     K/V tile, and the MMA warp alternates between them so that one tile's
//     softmax overlaps the other tile's matrix products (ping-pong);
//     for d = 256 a work unit is one query tile and S is double-buffered;
//   * work units (batch*head, query block) are ordered heaviest first for the
//     causal mask and strided over the persistent CTAs; key tiles wholly in the
//     future of a query tile are never loaded or multiplied.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fa {

struct TcParams {
  int N;                 // sequence length
  int BH;                // batch * heads
  int n_kv;              // number of key tiles: ceil(N / BK)
  int n_qb;              // query blocks per head: ceil(N / (BQ * NQT))
  int total_units;       // BH * n_qb
  float scale_log2;      // softmax scale * log2(e)
  __nv_bfloat16* o;      // [BH][N][D]
  float* lse;            // [BH][N]
  int* status;           // device status word
  unsigned long long limit_ns;  // time limit of each device-side wait
};

template <int D>
struct TcCfg {
  static constexpr int BQ = 128;                       // query rows per tile (= TMEM lanes)
  static constexpr int NQT = (D <= 128) ? 2 : 1;       // query tiles per work unit
  static constexpr int BK = (D <= 128) ? 128 : 64;     // keys per K/V tile
  static constexpr int LA = (NQT == 1) ? 2 : 1;        // K tiles ahead of V in the ring order
  static constexpr int SWB = (D * 2 >= 128) ? 128 : D * 2;  // swizzle span in bytes
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : 4u;   // descriptor swizzle code
  static constexpr int RC = SWB / 2;                   // bf16 columns per swizzle region
  static constexpr int NR = D / RC;                    // regions per tile row
  static constexpr int Q_REGION = BQ * SWB;
  static constexpr int KV_REGION = BK * SWB;
  static constexpr int Q_TILE = BQ * D * 2;
  static constexpr int KV_TILE = BK * D * 2;
  static constexpr int SMEM_LIMIT = 227 * 1024;
  static constexpr int NS_FIT = (SMEM_LIMIT - 2048 - NQT * Q_TILE) / KV_TILE;
  static constexpr int NS = NS_FIT > 8 ? 8 : NS_FIT;   // K/V ring slots
  static constexpr int NO = NQT;                       // O accumulators in TMEM
  // TMEM columns.  Every S/P buffer starts on a multiple of 128 columns and
  // every O accumulator on a multiple of its own width: S/P buffer b at
  // TM_S + b*128, O accumulator t at TM_O + t*D.
  static constexpr int TM_S = (D == 256) ? 256 : 0;
  static constexpr int TM_O = (D == 256) ? 0 : 256;
  static constexpr int TM_SB = 128;                    // column stride of the S/P buffers
  static constexpr int TM_COLS = 512;
  static constexpr int SOFTMAX_WARPS = 4 * NQT;
  static constexpr int MMA_WARP = SOFTMAX_WARPS;
  static constexpr int LOAD_WARP = SOFTMAX_WARPS + 1;
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 2);
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = NQT * Q_TILE;
  static constexpr int OFF_BAR = OFF_KV + NS * KV_TILE;
  // barriers: q_full, q_empty, kv_full[NS], kv_empty[NS], s_full[2], p_full[2],
  // o_done[NO], o_free[NO], drain
  static constexpr int NBAR = 2 + 2 * NS + 4 + 2 * NO + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // TMEM base address, abort flag
  static constexpr int SMEM_USED = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
  // At least ~120 KB so that a second CTA never shares the SM (and its TMEM).
  static constexpr int SMEM_ALLOC = SMEM_USED < 120 * 1024 ? 120 * 1024 : SMEM_USED;
  static_assert(D == 32 || D == 64 || D == 128 || D == 256, "head dim");
  static_assert(NS >= 2, "K/V ring");
  static_assert((D == 256) ? (TM_S + 2 * TM_SB <= TM_COLS && NO * D <= TM_S)
                           : (TM_O + NO * D <= TM_COLS && 2 * TM_SB <= TM_O), "TMEM budget");
  static_assert(SMEM_USED <= SMEM_LIMIT, "shared memory budget");
};

struct TcUnit {
  int bh;    // batch * H + head
  int row0;  // first query row of the unit
  int n[2];  // key tiles visited by each query tile (0 = tile beyond N)
  int nmax;
};

template <int D, bool CAUSAL>
__device__ __forceinline__ TcUnit tc_decode(int u, const TcParams& p) {
  using C = TcCfg<D>;
  TcUnit w;
  const int qb = p.n_qb - 1 - u / p.BH;  // heaviest query blocks first
  w.bh = u % p.BH;
  w.row0 = qb * (C::BQ * C::NQT);
  w.nmax = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int r0 = w.row0 + s * C::BQ;
    int n = 0;
    if (s < C::NQT && r0 < p.N) {
      n = p.n_kv;
      if (CAUSAL) {
        const int last = (r0 + C::BQ - 1) / C::BK + 1;  // tiles holding keys <= last row
        n = last < n ? last : n;
      }
    }
    w.n[s] = n;
    w.nmax = n > w.nmax ? n : w.nmax;
  }
  return w;
}

// Wait without looking at the abort flag (used to drain in-flight copies and
// MMAs before the CTA exits); still time-limited.
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, const WaitGuard& g) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > g.limit_ns) {
      atomicOr(g.status, kStatusTimeoutDrain);
      return false;
    }
  }
  return true;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(TcCfg<D>::THREADS, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = base + C::OFF_BAR;
  const uint32_t q_full = bar0;
  const uint32_t q_empty = bar0 + 8;
  auto kv_full = [&](int i) { return bar0 + 16 + 8u * i; };
  auto kv_empty = [&](int i) { return bar0 + 16 + 8u * (C::NS + i); };
  auto s_full = [&](int b) { return bar0 + 16 + 8u * (2 * C::NS + b); };
  auto p_full = [&](int b) { return bar0 + 16 + 8u * (2 * C::NS + 2 + b); };
  auto o_done = [&](int t) { return bar0 + 16 + 8u * (2 * C::NS + 4 + t); };
  auto o_free = [&](int t) { return bar0 + 16 + 8u * (2 * C::NS + 4 + C::NO + t); };
  const uint32_t drain = bar0 + 16 + 8u * (2 * C::NS + 4 + 2 * C::NO);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(kv_full(i), 1);
      mbar_init(kv_empty(i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), 128);
    }
    for (int t = 0; t < C::NO; ++t) {
      mbar_init(o_done(t), 1);
      mbar_init(o_free(t), 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::LOAD_WARP && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitGuard g{abort_flag, p.status, p.limit_ns};

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t pos = 0;             // K/V loads issued so far (ring position)
      uint32_t issued = 0;          // bit i: slot i has been loaded at least once
      uint32_t last_par = 0;        // bit i: parity of slot i's latest load
      int ui = 0;                   // units started by this CTA
      int last_q = -1;              // unit index of the latest Q load
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x, ++ui) {
        const TcUnit w = tc_decode<D, CAUSAL>(u, p);
        if (!wait_bar(q_empty, (ui & 1) ^ 1, g, kStatusTimeoutLoad)) { ok = false; break; }
        mbar_arrive_expect_tx(q_full, C::NQT * C::Q_TILE);
        for (int s = 0; s < C::NQT; ++s)
          for (int r = 0; r < C::NR; ++r)
            tma_load_3d(base + C::OFF_Q + s * C::Q_TILE + r * C::Q_REGION, &tm_q, q_full, r * C::RC,
                        w.row0 + s * C::BQ, w.bh, pol_q);
        last_q = ui;
        auto load_kv = [&](const CUtensorMap* tm, int j) -> bool {
          const int slot = pos % C::NS;
          const uint32_t par = (pos / C::NS) & 1;
          if (!wait_bar(kv_empty(slot), par ^ 1, g, kStatusTimeoutLoad)) return false;
          mbar_arrive_expect_tx(kv_full(slot), C::KV_TILE);
          for (int r = 0; r < C::NR; ++r)
            tma_load_3d(base + C::OFF_KV + slot * C::KV_TILE + r * C::KV_REGION, tm, kv_full(slot), r * C::RC,
                        j * C::BK, w.bh, pol_kv);
          issued |= 1u << slot;
          last_par = (last_par & ~(1u << slot)) | (par << slot);
          ++pos;
          return true;
        };
        for (int j = 0; ok && j < C::LA && j < w.nmax; ++j) ok = load_kv(&tm_k, j);
        for (int j = 0; ok && j < w.nmax; ++j) {
          ok = load_kv(&tm_v, j);
          if (ok && j + C::LA < w.nmax) ok = load_kv(&tm_k, j + C::LA);
        }
      }
      // Every issued copy must land before the CTA may exit.
      for (int i = 0; i < C::NS; ++i)
        if (issued & (1u << i)) wait_bar_drain(kv_full(i), (last_par >> i) & 1, g);
      if (last_q >= 0) wait_bar_drain(q_full, last_q & 1, g);
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc_bf16(128, C::BK, 0);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, D, 1);
      uint32_t pos = 0;
      uint32_t p_cnt[2] = {0, 0};   // P buffers consumed, per S buffer
      uint32_t o_units[2] = {0, 0}; // units started, per O accumulator
      uint32_t qk_total = 0;        // QK products issued (single-tile mode buffer alternation)
      bool ok = true;
      int ui = 0;

      auto kv_acquire = [&](uint32_t& slot) -> bool {
        slot = pos % C::NS;
        const bool r = wait_bar(kv_full(slot), (pos / C::NS) & 1, g, kStatusTimeoutMma);
        ++pos;
        return r;
      };
      auto issue_qk = [&](int qt, int buf, uint32_t kslot) {
        const uint32_t d_t = tmem + C::TM_S + buf * C::TM_SB;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int k0 = kk * 16;
          const uint32_t off = (k0 % C::RC) * 2;  // byte offset inside the 128-byte swizzle row
          const uint64_t a = make_sdesc(base + C::OFF_Q + qt * C::Q_TILE + (k0 / C::RC) * C::Q_REGION + off, 16,
                                        8 * C::SWB, C::SWZ);
          const uint64_t b = make_sdesc(base + C::OFF_KV + kslot * C::KV_TILE + (k0 / C::RC) * C::KV_REGION + off,
                                        16, 8 * C::SWB, C::SWZ);
          mma_ss(d_t, a, b, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full(buf));
      };
      auto issue_pv = [&](int ot, int buf, uint32_t vslot, bool acc) {
        const uint32_t d_t = tmem + C::TM_O + ot * D;
        const uint32_t a_t = tmem + C::TM_S + buf * C::TM_SB;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint64_t b = make_sdesc(base + C::OFF_KV + vslot * C::KV_TILE + kk * 16 * C::SWB, C::KV_REGION,
                                        8 * C::SWB, C::SWZ);
          mma_ts(d_t, a_t + kk * 8, b, idesc_pv, (acc || kk > 0) ? 1u : 0u);
        }
        mma_commit(o_done(ot));
      };
      // Wait for P in buffer `buf` and, on a unit's first P V into accumulator
      // `ot`, for the epilogue of the previous unit to have read it out.
      auto wait_p = [&](int buf, int ot, bool first) -> bool {
        if (!wait_bar(p_full(buf), p_cnt[buf] & 1, g, kStatusTimeoutMma)) return false;
        ++p_cnt[buf];
        if (first) {
          if (o_units[ot] > 0 && !wait_bar(o_free(ot), (o_units[ot] - 1) & 1, g, kStatusTimeoutMma)) return false;
          ++o_units[ot];
        }
        tc_fence_after();
        return true;
      };

      for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x, ++ui) {
        const TcUnit w = tc_decode<D, CAUSAL>(u, p);
        if (!wait_bar(q_full, ui & 1, g, kStatusTimeoutMma)) { ok = false; break; }
        tc_fence_after();
        if constexpr (C::NQT == 2) {
          uint32_t kslot, vslot;
          if (!(ok = kv_acquire(kslot))) break;
          tc_fence_after();
          for (int s = 0; s < 2; ++s)
            if (w.n[s] > 0) issue_qk(s, s, kslot);
          mma_commit(kv_empty(kslot));
          if (w.nmax == 1) mma_commit(q_empty);
          for (int j = 0; ok && j < w.nmax; ++j) {
            if (!(ok = kv_acquire(vslot))) break;
            bool have_k = false;
            for (int s = 0; ok && s < 2; ++s) {
              if (j < w.n[s]) {
                if (!(ok = wait_p(s, s, j == 0))) break;
                issue_pv(s, s, vslot, j > 0);
              }
              if (j + 1 < w.n[s]) {
                if (!have_k) {
                  if (!(ok = kv_acquire(kslot))) break;
                  tc_fence_after();
                  have_k = true;
                }
                issue_qk(s, s, kslot);
              }
            }
            if (!ok) break;
            mma_commit(kv_empty(vslot));
            if (have_k) {
              mma_commit(kv_empty(kslot));
              if (j + 1 == w.nmax - 1) mma_commit(q_empty);
            }
          }
        } else {
          const int n = w.n[0];
          const uint32_t qk_base = qk_total;
          uint32_t kslot, vslot;
          for (int t = 0; ok && t < C::LA && t < n; ++t) {
            if (!(ok = kv_acquire(kslot))) break;
            tc_fence_after();
            issue_qk(0, qk_total & 1, kslot);
            ++qk_total;
            mma_commit(kv_empty(kslot));
            if (t == n - 1) mma_commit(q_empty);
          }
          for (int j = 0; ok && j < n; ++j) {
            if (!(ok = kv_acquire(vslot))) break;
            const int buf = (qk_base + j) & 1;
            if (!(ok = wait_p(buf, 0, j == 0))) break;
            issue_pv(0, buf, vslot, j > 0);
            mma_commit(kv_empty(vslot));
            if (j + C::LA < n) {
              if (!(ok = kv_acquire(kslot))) break;
              tc_fence_after();
              issue_qk(0, qk_total & 1, kslot);
              ++qk_total;
              mma_commit(kv_empty(kslot));
              if (j + C::LA == n - 1) mma_commit(q_empty);
            }
          }
        }
      }
      // All issued MMAs must complete before TMEM is released.
      mma_commit(drain);
      wait_bar_drain(drain, 0, g);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;          // query tile of the unit this warpgroup owns
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane; // row within the query tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only if the max grew > 2^8
    uint32_t s_waits = 0;   // S buffers consumed by this warpgroup
    uint32_t pv_done = 0;   // P V products into this warpgroup's O completed in earlier units
    bool ok = true;
    const int ot = (C::NQT == 2) ? wg : 0;

    for (int u = blockIdx.x; ok && u < p.total_units; u += gridDim.x) {
      const TcUnit w = tc_decode<D, CAUSAL>(u, p);
      const int n = w.n[wg];
      if (n == 0) continue;
      const int row0 = w.row0 + wg * C::BQ;
      const int row = row0 + r;
      float m = -INFINITY;  // running max of scaled logits, log2 units
      float l = 0.f;        // running sum of exp2(x - m)
      float lw = 0.f;       // the same sum over the bf16-rounded weights
      for (int j = 0; j < n; ++j) {
        const int buf = (C::NQT == 2) ? wg : static_cast<int>(s_waits & 1);
        const uint32_t par = (C::NQT == 2) ? (s_waits & 1) : ((s_waits >> 1) & 1);
        ok = wait_bar(s_full(buf), par, g, kStatusTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++s_waits;
        tc_fence_after();
        const uint32_t ts = tmem + lane_off + C::TM_S + buf * C::TM_SB;

        float s[C::BK];
        {
          uint32_t raw_s[C::BK / 32][32];
#pragma unroll
          for (int c = 0; c < C::BK / 32; ++c) tmem_ld32(ts + c * 32, raw_s[c]);
#pragma unroll
          for (int c = 0; c < C::BK / 32; ++c) tmem_wait_ld(raw_s[c]);
#pragma unroll
          for (int c = 0; c < C::BK / 32; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw_s[c][i]);
        }
        const int key0 = j * C::BK;
        const bool need_mask = (CAUSAL && key0 + C::BK - 1 > row0) || (key0 + C::BK > p.N);
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < C::BK; ++c) {
            const int key = key0 + c;
            if (key >= p.N || (CAUSAL && key > row)) s[c] = -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
        for (int c = 8; c < C::BK; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
        const float rmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_cand = fmaxf(m, rmax * sl2);
        const bool grow = m_cand > m + kRescaleThreshold;  // always true on the first tile
        const float m_new = grow ? m_cand : m;
        const float alpha = grow ? ex2(m - m_new) : 1.f;   // ex2(-inf) = 0 on the first tile
        const float nbase = (m_new == -INFINITY) ? 0.f : -m_new;
        // Two row sums: lsum of the fp32 weights (for L, the logsumexp) and
        // wsum of the bf16-rounded weights that P V multiplies (for O / l, so
        // the division normalises exactly the weights that were applied).
        float lsum[4], wsum[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) lsum[i] = wsum[i] = 0.f;
        uint32_t pk[C::BK / 2];
#pragma unroll
        for (int c = 0; c < C::BK; c += 2) {
          const float p0 = ex2(fmaf(s[c], sl2, nbase));
          const float p1 = ex2(fmaf(s[c + 1], sl2, nbase));
          const uint32_t w = pack_bf16x2(p0, p1);
          pk[c >> 1] = w;
          lsum[(c >> 1) & 3] += p0 + p1;
          wsum[(c >> 1) & 3] += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
        }
        l = l * alpha + ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3]));
        lw = lw * alpha + ((wsum[0] + wsum[1]) + (wsum[2] + wsum[3]));
        m = m_new;
#pragma unroll
        for (int c = 0; c < C::BK / 64; ++c) {
          uint32_t chunk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) chunk[i] = pk[c * 32 + i];
          tmem_st32(ts + c * 32, chunk);
        }
        tmem_wait_st();
        if (j > 0) {
          // Observe the completion of P V number j-1 on this accumulator.  Every
          // completion of o_done is waited for in order: a parity wait that ran
          // two phases ahead of the barrier would read an older phase as done.
          // (At most P V j-1 can be outstanding: P V j needs this tile's P.)
          ok = wait_bar(o_done(ot), (pv_done + j - 1) & 1, g, kStatusTimeoutSoftmax);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        // Rescale the O accumulator of this row when its max grew past the threshold.
        const bool need = grow && j > 0;
        if (__any_sync(0xffffffffu, need)) {
          tc_fence_after();
          const uint32_t to = tmem + lane_off + C::TM_O + ot * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(to + c * 32, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(to + c * 32, v);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(p_full(buf));
      }
      if (!ok) break;
      // ---- epilogue: O / l in bf16, L = (m + log2 l) * ln 2
      // P V number n-1 is the only one not yet observed (see above).
      ok = wait_bar(o_done(ot), (pv_done + n - 1) & 1, g, kStatusTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      pv_done += n;
      tc_fence_after();
      const float inv_l = 1.f / lw;
      const uint32_t to = tmem + lane_off + C::TM_O + ot * D;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(w.bh) * p.N + row) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(to + c * 32, v);
        tmem_wait_ld(v);
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
        if (row < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
      if (row < p.N) p.lse[static_cast<size_t>(w.bh) * p.N + row] = (m + log2f(l)) * 0.69314718055994531f;
      tc_fence_before();
      mbar_arrive(o_free(ot));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

}  // namespace fa

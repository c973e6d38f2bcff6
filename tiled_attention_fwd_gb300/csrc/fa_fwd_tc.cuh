// FlashAttention-2 forward pass, bf16 in / fp32 accumulate, for sm_103a.
//
// Algorithm (the FA2 forward of "FlashAttention-2 from PyTorch to Triton",
// section "What We Are Building", with the masking and block skipping of
// "Writing a FlashAttention kernel in Metal", "Blockwise attention and causal
// masking"): for each 128-row query tile Q_i, loop over key/value tiles
// K_j, V_j; S = Q_i K_j^T; fold S into the running row max m, the rescaled row
// sum l and the unnormalised output O (rescale factor exp(m_old - m_new));
// divide by l once at the end and store L = m + log l.  The rescale of O is
// skipped for rows whose max did not grow (the guarded correction of "Case
// Study: metal-flash-attention").
//
// Mapping onto one GB300 SM (one persistent CTA per SM), by warpgroup:
//   * softmax warpgroup(s), one per 128-row query tile (thread = row = TMEM
//     lane): read S from tensor memory (TMEM), mask, row max, publish the
//     rescale factor alpha, P = exp2(S*scale*log2e - m) with paired fp32
//     arithmetic, write P as bf16 over S in TMEM, keep m and l;
//   * a correction warpgroup: rescales the O accumulators in TMEM by alpha
//     while the softmax computes P, and runs the epilogue (O / l in bf16,
//     L = m + log l) so the softmax can start the next work unit at once; each
//     warp stages its 32 rows of O in shared memory, 32 columns at a time, and
//     a TMA store writes them out, so O is free for the next unit as soon as
//     it has been read;
//   * one MMA warp: tcgen05.mma S = Q K^T into TMEM, then O += P V with P read
//     from TMEM and V from shared memory, issued by an elected lane;
//   * one TMA producer warp: Q tiles and a ring of K/V stages in 128-byte
//     swizzled shared memory, each stage guarded by full/empty mbarriers.
// For d <= 128 a work unit is two query tiles (256 rows) that share every K/V
// tile, and the MMA warp alternates between them so one tile's softmax
// overlaps the other tile's matrix products; for d = 256 a work unit is one
// query tile with a double-buffered S.  Work units (batch*head, query block)
// are ordered heaviest first for the causal mask and dealt to the persistent
// CTAs in snake order; key tiles wholly in the future of a query tile are
// never loaded or multiplied.
//
// The tensor core executes MMAs about as fast as the MMA warp can issue them
// while it shares its scheduler with softmax and correction warps, so the
// issuer is kept lean: one readiness barrier per P V product (the softmax's
// P and the correction's O meet there), one barrier per K/V stage,
// descriptors built once and stepped with 32-bit adds.
//
// Every mbarrier phase is waited for in order by its consumer: a parity wait
// issued two phases ahead of a barrier would read an older phase as complete.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fa {

// Kernel variants (template parameter VAR).
enum : int { kVarBf16 = 0, kVarE4m3 = 1, kVarPair = 2 };

struct TcParams {
  int Nq;                // query rows per head
  int Nk;                // key / value rows per head
  int H;                 // heads (unit index bh = b * H + h)
  int BH;                // batch * heads
  int n_kv;              // number of key tiles: ceil(N / BK)
  int n_qb;              // query blocks per head: ceil(N / (BQ * NQT))
  int total_units;       // BH * n_qb
  float scale_log2;      // softmax scale * log2(e) (e4m3 inputs: times the q and k dequantisation factors)
  float o_scale;         // e4m3 inputs: the v dequantisation factor, applied with 1 / l (unused for bf16)
  float* lse;            // [BH][Nq], contiguous
  int* status;           // device status word
  unsigned long long limit_ns;  // time limit of each device-side wait
};

// NQ: query tiles per work unit.  Two tiles (d <= 128) share every K/V tile;
// one tile with double-buffered S serves d = 256 and, at d <= 128, problems
// with too few 256-row units to occupy the SMs.
// VAR: kVarBf16 (bf16 Q, K, V); kVarE4m3: Q, K, V are e4m3 (one byte per
// element; tcgen05.mma kind::f8f6f4 with K = 32 per instruction, P rounded to
// e4m3 and packed four to a TMEM column; O is bf16 either way); kVarPair:
// bf16 at d = 256 on CTA pairs (cta_group::2, M = 256, BK = 128).
template <int D, int NQ = (D <= 128 ? 2 : 1), int VAR = kVarBf16>
struct TcCfg {
  static constexpr int BQ = 128;                       // query rows per tile (= TMEM lanes)
  static constexpr int NQT = NQ;                       // query tiles per work unit
  static constexpr bool FP8 = (VAR == kVarE4m3);
  static constexpr bool PAIR = (VAR == kVarPair);
  static constexpr int EB = FP8 ? 1 : 2;                // bytes per Q / K / V element
  static constexpr int KM = 32 / EB;                   // K elements per MMA (32 bytes of an operand row)
  static constexpr int BK = (D <= 128 || PAIR) ? 128 : 64;  // keys per K/V tile
  // Query tiles of a work unit (256 rows for a CTA pair: one tile per CTA).
  static constexpr int UNIT_TILES = PAIR ? 2 : NQT;
  // A CTA pair holds half of every K tile (BK / 2 keys) and half of every V
  // tile's columns (D / 2) per CTA.
  static constexpr int K_ROWS = PAIR ? BK / 2 : BK;
  static constexpr int V_COLS = PAIR ? D / 2 : D;
  static constexpr int LA = (NQT == 1) ? 2 : 1;        // K tiles needed before the first P V
  static constexpr int SWB = (D * EB >= 128) ? 128 : D * EB;  // swizzle span in bytes
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : 4u;   // descriptor swizzle code
  static constexpr int RC = SWB / EB;                  // elements per swizzle region
  static constexpr int NR = D / RC;                    // regions per tile row
  static constexpr int Q_REGION = BQ * SWB;
  static constexpr int K_REGION = K_ROWS * SWB;        // one swizzle region of a K tile (slice)
  static constexpr int V_REGION = BK * SWB;            // one swizzle region of a V tile (slice)
  static constexpr int Q_TILE = BQ * D * EB;
  static constexpr int KV_TILE = K_ROWS * D * EB;      // shared-memory slot of one K or V tile (slice)
  static constexpr int P_COLS_64 = 64 * EB / 4;        // TMEM columns holding P of 64 keys
  static constexpr int NO = NQT;                       // O accumulators in TMEM
  // Two-tile mode at d = 128 issues each P V product as two runs over the key
  // halves of P (64 keys each), the first as soon as the softmax has written
  // the first half of P, so the tensor core starts while the second half's
  // exponentials are computed (+1.6 % at d = 128 non-causal and at N = 16384
  // causal; at d <= 64 the extra store wait in the softmax cost 2-3 %).  The
  // e4m3 kernel issues each P V product whole: there its two runs of K = 64
  // keys are half as many MMAs as in bf16, and the split measured 1.1-1.3 %
  // slower on all three d = 128 e4m3 workloads.
  static constexpr bool PV_SPLIT = (NQT == 2 && D == 128 && !FP8);
  // Lazy row max (two-tile kernels): the reference max m moves only when a
  // key tile's row max exceeds it by more than MAX_SLACK (log2 units), so
  // P <= 2^MAX_SLACK (below e4m3's 448) and most steps need no rescale of O.
  // The largest P of a step is then not exactly 1 and its rounding to P's
  // type would no longer be matched by l (the fp32 sum), so O's normaliser
  // adds, per step, that P's rounding residual (round(p) - p, p computed from
  // the row max exactly as the exponential loop computes it); L keeps the
  // fp32 sum.
  static constexpr bool LAZY_MAX = (NQT == 2);
  static constexpr float MAX_SLACK = 8.f;
  // Shared memory: [Q tiles][K/V stages][misc]; misc = barriers, alpha, m/l, TMEM address, abort flag.
  static constexpr int MISC = 7168;
  static constexpr int SMEM_LIMIT = 227 * 1024;
  // A K/V stage holds two tiles: V_j and K_{j+LA} (the first stage of a unit: K_0 .. K_{LA-1}).
  static constexpr int STAGE = 2 * KV_TILE;
  // Epilogue staging: per correction warp OSTB buffers of 32 rows x 32 bf16
  // columns (64-byte swizzled), the source boxes of the TMA stores of O.  Every
  // head dimension stages (at d = 64 the staged TMA stores measured 1-2 %
  // faster than direct 16-byte stores from registers).
  static constexpr int OSTB = 3;
  static constexpr int OST_BUF = 32 * 64;
  static constexpr int OST = 4 * OSTB * OST_BUF;
  static constexpr int NST_FIT = (SMEM_LIMIT - 1024 - MISC - OST - NQT * Q_TILE) / STAGE;
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;  // K/V stages
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = NQT * Q_TILE;
  static constexpr int OFF_MISC = OFF_KV + NST * STAGE;
  static constexpr int OFF_BAR = OFF_MISC;                    // 64 barriers at most
  static constexpr int OFF_ALPHA = OFF_MISC + 512;            // float [NO][2][128] (by step parity)
  // m and l of a finished unit, double-buffered by the parity of the unit's
  // index within the CTA: the softmax may finish the next unit (one key tile)
  // while the correction warpgroup still reads this one's.
  static constexpr int OFF_STAT_M = OFF_ALPHA + 4 * 128 * 4;  // float [2][NO][128]
  static constexpr int OFF_STAT_L = OFF_STAT_M + 4 * 128 * 4; // float [2][NO][128]
  static constexpr int OFF_TMEM_SLOT = OFF_STAT_L + 4 * 128 * 4;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int OFF_OST = OFF_MISC + MISC;             // 1024-byte aligned
  static constexpr int SMEM_USED = OFF_OST + OST + 1024;      // + slack for 1024-byte alignment
  // At least ~120 KB so that a second CTA never shares the SM (and its TMEM).
  static constexpr int SMEM_ALLOC = SMEM_USED < 120 * 1024 ? 120 * 1024 : SMEM_USED;
  // TMEM columns.  S/P buffer b at TM_S + b*128, O accumulator t at TM_O + t*D.
  static constexpr int TM_S = (D == 256) ? 256 : 0;
  static constexpr int TM_O = (D == 256) ? 0 : 256;
  static constexpr int TM_SB = 128;
  static constexpr int TM_COLS = 512;
  // Warp roles.
  static constexpr int SOFTMAX_WARPS = 4 * NQT;
  static constexpr int CORR_WARP0 = SOFTMAX_WARPS;       // four warps
  static constexpr int MMA_WARP = SOFTMAX_WARPS + 4;
  static constexpr int LOAD_WARP = MMA_WARP + 1;
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 8);  // + correction WG + MMA/TMA WG
  // Register split (d <= 128 and CTA pairs).  Two tiles, 512 threads launched at 128
  // registers each: softmax 184 (its lazy row max keeps one more value
  // across the exponential loop; at 176 it spilled 8 bytes), correction 80,
  // MMA/TMA 64 (2*128*184 + 128*144 = 65536; 72 / 72 measured slower).
  // One tile, 384 threads launched at 168:
  // softmax 208, correction 152, MMA/TMA 144; 128*(208 + 296) = 64512
  // (CTA pairs at d = 256: correction 160 for its 256-column rescale, 136).
  // d = 256 on one CTA (64-column S) fits 168 everywhere and is not split.
  static constexpr bool SPLIT_REGS = (D <= 128 || PAIR);
  static constexpr uint32_t REG_SOFTMAX = (NQT == 2) ? 184 : 208;
  static constexpr uint32_t REG_CORR_OTHER = (NQT == 2) ? 144 : 296;
  static constexpr __host__ __device__ uint32_t reg_corr(bool strided) {
    return NQT == 1 ? (PAIR ? 160 : 152) : 80;
  }
  static constexpr int LAUNCH_REGS = 65536 / THREADS > 255 ? 255 : (65536 / THREADS) & ~7;
  static_assert(!SPLIT_REGS || NQT * 128 * REG_SOFTMAX + 128 * REG_CORR_OTHER <= THREADS * LAUNCH_REGS,
                "register split exceeds the launch budget");
  static_assert(D == 32 || D == 64 || D == 128 || D == 256, "head dim");
  static_assert(!FP8 || D == 64 || D == 128, "e4m3 kernels: d = 64 or 128");
  static_assert(SWB == 128 || SWB == 64, "swizzle span");
  static_assert(!PAIR || (D == 256 && NQ == 1 && K_ROWS * D == BK * V_COLS), "CTA pairs: d = 256, one tile per CTA");
  static_assert(NQ == 1 || (NQ == 2 && D <= 128), "query tiles per unit");
  static_assert(NST >= 2, "K/V stages");
  static_assert(LA <= 2, "a stage holds at most two K tiles");
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

template <int D, bool CAUSAL, int NQ, int VAR>
__device__ __forceinline__ TcUnit tc_decode(int u, const TcParams& p) {
  using C = TcCfg<D, NQ, VAR>;
  TcUnit w;
  // Causal: heaviest query blocks first (all heads' block n_qb - 1, then
  // n_qb - 2, ...), which balances the persistent CTAs.  Without the mask
  // every unit costs the same, so units run head by head instead: the CTAs
  // working at one time then share a few heads' K and V in L2.
  int qb;
  if (CAUSAL) {
    qb = p.n_qb - 1 - u / p.BH;
    w.bh = u % p.BH;
  } else {
    qb = u % p.n_qb;
    w.bh = u / p.n_qb;
  }
  w.row0 = qb * (C::BQ * C::UNIT_TILES);
  w.nmax = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int r0 = w.row0 + s * C::BQ;
    int n = 0;
    if (s < C::UNIT_TILES && r0 < p.Nq) {
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

// k-th work unit of this CTA.  Units are numbered heaviest first; CTAs take
// them in rounds of gridDim.x, alternating direction every round (a snake),
// so the CTA that takes the heaviest unit of one round takes the lightest of
// the next and causal work evens out without any shared counter.
template <bool PAIR = false>
__device__ __forceinline__ int tc_unit(int k) {
  // CTA pairs: the cluster (pair) is the unit of scheduling.
  const int g = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int b = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  return k * g + ((k & 1) ? g - 1 - b : b);
}

// Wait without looking at the abort flag (used to drain in-flight copies and
// MMAs before the CTA exits); still time-limited.
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, const WaitGuard& g) {
  const uint64_t t0 = globaltimer_ns();
  while (!guard_try_wait(bar, parity, g)) {
    if (globaltimer_ns() - t0 > g.limit_ns) {
      atomicOr(g.status, kStatusTimeoutDrain);
      return false;
    }
  }
  return true;
}

// Barrier addresses in shared memory.
template <int D, int NQ, int VAR>
struct TcBars {
  using C = TcCfg<D, NQ, VAR>;
  uint32_t b0;
  // Q tile t loaded / free again (one phase per work unit).
  __device__ __forceinline__ uint32_t q_full(int t) const { return b0 + 8u * t; }
  __device__ __forceinline__ uint32_t q_empty(int t) const { return b0 + 16 + 8u * t; }
  __device__ __forceinline__ uint32_t kv_full(int i) const { return b0 + 32 + 8u * i; }
  __device__ __forceinline__ uint32_t kv_empty(int i) const { return b0 + 32 + 8u * (C::NST + i); }
  __device__ __forceinline__ uint32_t s_full(int b) const { return b0 + 32 + 8u * (2 * C::NST + b); }
  // P V number g into accumulator t may start: P written (4 softmax warps) and
  // O ready (4 correction warps: rescaled, or released by the previous
  // epilogue).  Two-tile mode: barrier (t, 0) for the first key half of P
  // (and O), barrier (t, 1) for the second half (softmax warps only).
  // Single-tile mode: barrier (0, g & 1), each completing once per two P V
  // products, because there S of step j+1 is computed before P V j and the
  // softmax may post P j+1 while P V j still waits for the correction
  // warpgroup.
  __device__ __forceinline__ uint32_t pv_go(int t, int k) const { return b0 + 32 + 8u * (2 * C::NST + 2 + 2 * t + k); }
  // alpha of rescale step k of accumulator t published: barrier (t, k & 1), each
  // completing once per two steps (single-tile mode lets the softmax run two
  // steps ahead of the correction warpgroup).
  __device__ __forceinline__ uint32_t a_full(int t, int k) const { return b0 + 32 + 8u * (2 * C::NST + 6 + 2 * t + k); }
  __device__ __forceinline__ uint32_t o_done(int t) const { return b0 + 32 + 8u * (2 * C::NST + 10 + t); }
  __device__ __forceinline__ uint32_t l_full(int t) const { return b0 + 32 + 8u * (2 * C::NST + 12 + t); }
  __device__ __forceinline__ uint32_t drain() const { return b0 + 32 + 8u * (2 * C::NST + 14); }
  static constexpr int COUNT = 4 + 2 * C::NST + 15;
  static_assert(COUNT * 8 <= 512, "barrier area");
};

// ------------------------------------------------------------------ TMA producer
// Run by one thread (lane 0 of the producer warp).
//
// Two-tile mode: the CTA's units form one continuous stream, so that the
// next unit's first S products can be issued while the current unit's last
// P V products run.  Stages: {K_0} of the first unit, then {V_j, K_{j+1}} for
// j < nmax of each unit, where the K slot of a unit's last stage holds K_0 of
// the next unit.  Q tile t of the next unit is loaded after that last stage,
// as soon as the current unit's last S_t product has completed (q_empty(t)).
//
// Single-tile mode: per unit, Q, then {K_0, K_1}, then {V_j, K_{j+2}}.  In a
// CTA pair each CTA loads its own 128 Q rows, its half of the keys of every K
// tile (BK / 2 rows) and its half of the columns of every V tile (D / 2),
// all onto its own barriers.
template <int D, bool CAUSAL, bool STRIDED, int NQ, int VAR>
__device__ __forceinline__ void tc_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                            const TcParams& p, const TcBars<D, NQ, VAR>& bar, uint32_t base,
                                            const WaitGuard& g) {
  using C = TcCfg<D, NQ, VAR>;
  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();
  uint32_t pos = 0;       // stages issued so far
  uint32_t issued = 0;    // bit i: stage i has been loaded at least once
  uint32_t last_par = 0;  // bit i: parity of stage i's latest load
  int last_q[2] = {-1, -1};  // per Q tile: index (within this CTA) of the latest unit whose tile was loaded
  bool ok = true;
  const int rank = C::PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  // K tile j (rows j*BK ..; a pair CTA: its K_ROWS of them) and V tile j (a
  // pair CTA: its V_COLS columns) of unit bh.  Strided tensors are 4-D maps
  // {d, N, H, B} (coordinates h, b), contiguous ones 3-D maps {d, N, B*H}
  // (coordinate bh).
  auto load_slab = [&](const CUtensorMap* tm, uint32_t dst, uint32_t full, int x0, int row, int regions,
                       int region_bytes, int bh) {
    for (int r = 0; r < regions; ++r) {
      if constexpr (STRIDED)
        tma_load_4d(dst + r * region_bytes, tm, full, x0 + r * C::RC, row, bh % p.H, bh / p.H, pol_kv);
      else
        tma_load_3d(dst + r * region_bytes, tm, full, x0 + r * C::RC, row, bh, pol_kv);
    }
  };
  auto load_k = [&](uint32_t dst, uint32_t full, int j, int bh) {
    load_slab(tm_k, dst, full, 0, j * C::BK + rank * C::K_ROWS, C::NR, C::K_REGION, bh);
  };
  auto load_v = [&](uint32_t dst, uint32_t full, int j, int bh) {
    load_slab(tm_v, dst, full, rank * C::V_COLS, j * C::BK, C::V_COLS / C::RC, C::V_REGION, bh);
  };
  // Q tiles of unit x, the qi-th unit of this CTA.
  auto load_q = [&](const TcUnit& x, int qi) -> bool {
    for (int t = 0; t < C::NQT; ++t) {
      if (!wait_bar(bar.q_empty(t), (qi & 1) ^ 1, g, kStatusTimeoutLoad)) return false;
      mbar_arrive_expect_tx(bar.q_full(t), C::Q_TILE);
      for (int r = 0; r < C::NR; ++r)
        if constexpr (STRIDED)
          tma_load_4d(base + C::OFF_Q + t * C::Q_TILE + r * C::Q_REGION, tm_q, bar.q_full(t), r * C::RC,
                      x.row0 + t * C::BQ, x.bh % p.H, x.bh / p.H, pol_q);
        else
          tma_load_3d(base + C::OFF_Q + t * C::Q_TILE + r * C::Q_REGION, tm_q, bar.q_full(t), r * C::RC,
                      x.row0 + (t + rank) * C::BQ, x.bh, pol_q);
      last_q[t] = qi;
    }
    return true;
  };
  // Next free stage: waits for its previous contents to be released; returns
  // its shared address in s0 and arms kv_full for `tiles` tiles.
  auto stage_begin = [&](int tiles, uint32_t& s0, uint32_t& full) -> bool {
    const int st = pos % C::NST;
    const uint32_t par = (pos / C::NST) & 1;
    if (!wait_bar(bar.kv_empty(st), par ^ 1, g, kStatusTimeoutLoad)) return false;
    s0 = base + C::OFF_KV + st * C::STAGE;
    full = bar.kv_full(st);
    mbar_arrive_expect_tx(full, tiles * C::KV_TILE);
    issued |= 1u << st;
    last_par = (last_par & ~(1u << st)) | (par << st);
    ++pos;
    return true;
  };

  if constexpr (C::NQT == 2) {
    int uk = 0;
    int u = tc_unit<C::PAIR>(0);
    if (u < p.total_units) {
      TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
      uint32_t s0, full;
      ok = load_q(w, 0) && stage_begin(1, s0, full);
      if (ok) load_k(s0, full, 0, w.bh);
      while (ok) {
        const int un = tc_unit<C::PAIR>(uk + 1);
        const bool has_next = un < p.total_units;
        const TcUnit wn = tc_decode<D, CAUSAL, NQ, VAR>(has_next ? un : u, p);
        for (int j = 0; ok && j < w.nmax; ++j) {
          const bool k_here = j + 1 < w.nmax;
          const bool k_next = !k_here && has_next;
          if (!(ok = stage_begin((k_here || k_next) ? 2 : 1, s0, full))) break;
          load_v(s0, full, j, w.bh);
          if (k_here) load_k(s0 + C::KV_TILE, full, j + 1, w.bh);
          if (k_next) load_k(s0 + C::KV_TILE, full, 0, wn.bh);
        }
        if (!ok || !has_next) break;
        ++uk;
        ok = load_q(wn, uk);
        u = un;
        w = wn;
      }
    }
  } else {
    for (int uk = 0, u; ok && (u = tc_unit<C::PAIR>(uk)) < p.total_units; ++uk) {
      const TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
      if (!(ok = load_q(w, uk))) break;
      uint32_t s0, full;
      for (int t = -1; t < w.nmax; ++t) {
        if (t < 0) {  // K_0 .. K_{LA-1}
          const int nk = C::LA < w.nmax ? C::LA : w.nmax;
          if (!(ok = stage_begin(nk, s0, full))) break;
          for (int k = 0; k < nk; ++k) load_k(s0 + k * C::KV_TILE, full, k, w.bh);
        } else {  // V_t, K_{t+LA}
          const bool has_k = t + C::LA < w.nmax;
          if (!(ok = stage_begin(has_k ? 2 : 1, s0, full))) break;
          load_v(s0, full, t, w.bh);
          if (has_k) load_k(s0 + C::KV_TILE, full, t + C::LA, w.bh);
        }
      }
    }
  }
  // Every issued copy must land before the CTA may exit.
  for (int i = 0; i < C::NST; ++i)
    if (issued & (1u << i)) wait_bar_drain(bar.kv_full(i), (last_par >> i) & 1, g);
  for (int t = 0; t < C::NQT; ++t)
    if (last_q[t] >= 0) wait_bar_drain(bar.q_full(t), last_q[t] & 1, g);
  // A pair CTA also waits for the leader's last releases of its stages and Q
  // tile: those commits arrive on this CTA's barriers, which must still exist.
  if constexpr (C::PAIR) {
    for (int i = 0; i < C::NST; ++i)
      if (issued & (1u << i)) wait_bar_drain(bar.kv_empty(i), (last_par >> i) & 1, g);
    if (last_q[0] >= 0) wait_bar_drain(bar.q_empty(0), last_q[0] & 1, g);
  }
}

// ------------------------------------------------------------------ MMA issuer
// One warp issues every tcgen05.mma and tcgen05.commit of the CTA: all its
// lanes run the loop (so descriptors and addresses are warp-uniform values)
// and elect.sync picks the lane that issues each operation.  Under load from
// the softmax and correction warps sharing its scheduler this sustains the
// tensor core's rate better than a lone lane-0 thread.  The order lets one
// tile's softmax overlap the other tile's products:
// P V_0 j, S_0 j+1, P V_1 j, S_1 j+1.  Products issued by one warp complete
// in issue order: P V j finishes before S of key tile j + 1 overwrites the
// S/P buffer, and S of key tile j being ready implies P V j - 1 finished.
// (Two issuers, one per tile, would interleave the tiles' products on the
// tensor core and lengthen each tile's softmax-to-softmax cycle.)
//
// Descriptors are kept as (low, high) words and built once: a tile position
// or K step only adds a constant to the low word's address field (bits 0..13
// hold address / 16, and no shared address reaches 2^18, so it never carries).
template <int D, int NQ, int VAR>
struct TcMma {
  using C = TcCfg<D, NQ, VAR>;
  // M = 256 for a CTA pair (each CTA holds 128 of the rows).
  static constexpr int MM = C::PAIR ? 256 : 128;
  static constexpr uint32_t IDESC_QK = C::FP8 ? make_idesc_e4m3(MM, C::BK, 0) : make_idesc_bf16(MM, C::BK, 0);
  static constexpr uint32_t IDESC_PV = C::FP8 ? make_idesc_e4m3(MM, D, 1) : make_idesc_bf16(MM, D, 1);
  static constexpr int N_QK = D * C::EB / 32;      // MMAs per S = Q K^T (K = d)
  static constexpr int N_PV = C::BK / C::KM;       // MMAs per P V (K = BK keys)
  // K-major (Q, K) and MN-major (V) operands share the stride byte offset
  // (8 rows of the swizzle span) and the swizzle mode.
  static constexpr uint32_t DESC_HI = sdesc_hi(8 * C::SWB, C::SWZ);
  // Address-field increments (16-byte units).
  static constexpr __host__ __device__ uint32_t q_step(int kk) {
    return ((kk * C::KM / C::RC) * C::Q_REGION + (kk * C::KM % C::RC) * C::EB) >> 4;
  }
  static constexpr __host__ __device__ uint32_t k_step(int kk) {
    return ((kk * C::KM / C::RC) * C::K_REGION + (kk * C::KM % C::RC) * C::EB) >> 4;
  }
  static constexpr __host__ __device__ uint32_t v_step(int kk) { return (kk * C::KM * C::SWB) >> 4; }
  static constexpr uint32_t TILE_STEP = C::KV_TILE >> 4;
  static constexpr uint32_t QTILE_STEP = C::Q_TILE >> 4;

  uint32_t tmem;
  uint32_t q_lo;  // Q tile 0, K-major
  uint32_t k_lo;  // K/V tile position 0, K-major (K as the B operand of S = Q K^T)
  uint32_t v_lo;  // K/V tile position 0, MN-major (V as the B operand of O = P V)

  __device__ __forceinline__ TcMma(uint32_t tmem_, uint32_t base) : tmem(tmem_) {
    q_lo = sdesc_lo(base + C::OFF_Q, 16);
    k_lo = sdesc_lo(base + C::OFF_KV, 16);
    v_lo = sdesc_lo(base + C::OFF_KV, C::V_REGION);
  }
  // Descriptor increments from K step k-1 to k.
  struct QkSteps {
    static constexpr __host__ __device__ uint32_t da(int k) { return q_step(k) - q_step(k - 1); }
    static constexpr __host__ __device__ uint32_t db(int k) { return k_step(k) - k_step(k - 1); }
  };
  struct PvSteps {
    static constexpr __host__ __device__ uint32_t ta(int) { return 8; }  // KM elements of P = 8 TMEM columns
    static constexpr __host__ __device__ uint32_t db(int) { return C::KM * C::SWB / 16; }  // KM rows of V
  };
  // S[buf] = Q[qt] K^T with K at tile position kpos; completion on s_full_bar.
  __device__ __forceinline__ void qk(int qt, int buf, uint32_t kpos, uint32_t s_full_bar) const {
    const uint32_t d_t = tmem + C::TM_S + buf * C::TM_SB;
    const uint32_t a = q_lo + qt * QTILE_STEP;
    const uint32_t b = k_lo + kpos * TILE_STEP;
    // d <= 128: one block per product (measured faster at d = 32 and 64, equal
    // at d = 128); d = 256: one MMA per block (measured faster there).
    if constexpr (D <= 128) {
      mma_ss_run<N_QK, QkSteps, C::FP8>(d_t, a, DESC_HI, b, DESC_HI, IDESC_QK, 0u);
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        if constexpr (C::PAIR)
          mma_ss_pair(d_t, a + q_step(kk), DESC_HI, b + k_step(kk), DESC_HI, IDESC_QK, kk > 0 ? 1u : 0u);
        else
          mma_ss_elect(d_t, a + q_step(kk), DESC_HI, b + k_step(kk), DESC_HI, IDESC_QK, kk > 0 ? 1u : 0u);
      }
    }
    commit(s_full_bar);
  }
  // O[ot] (+)= P[buf] V with V at tile position vpos.
  __device__ __forceinline__ void pv(int ot, int buf, uint32_t vpos, bool acc) const {
    const uint32_t d_t = tmem + C::TM_O + ot * D;
    const uint32_t a_t = tmem + C::TM_S + buf * C::TM_SB;
    const uint32_t b = v_lo + vpos * TILE_STEP;
    if constexpr (D <= 128) {
      mma_ts_run<N_PV, PvSteps, C::FP8>(d_t, a_t, b, DESC_HI, IDESC_PV, acc ? 1u : 0u);
    } else {
#pragma unroll
      for (int kk = 0; kk < C::BK / 16; ++kk) {
        if constexpr (C::PAIR)
          mma_ts_pair(d_t, a_t + kk * 8, b + v_step(kk), DESC_HI, IDESC_PV, (acc || kk > 0) ? 1u : 0u);
        else
          mma_ts_elect(d_t, a_t + kk * 8, b + v_step(kk), DESC_HI, IDESC_PV, (acc || kk > 0) ? 1u : 0u);
      }
    }
  }
  // O[ot] (+)= P[buf][:, 64h .. 64h+63] V[64h .. 64h+63, :]: one key half of
  // P V (BK = 128); P's half h starts P_COLS_64 TMEM columns in, V's 64 rows in.
  __device__ __forceinline__ void pv_half(int ot, int buf, uint32_t vpos, int h, bool acc) const {
    const uint32_t d_t = tmem + C::TM_O + ot * D;
    const uint32_t a_t = tmem + C::TM_S + buf * C::TM_SB + h * C::P_COLS_64;
    const uint32_t b = v_lo + vpos * TILE_STEP + h * (64 * C::SWB / 16);
    mma_ts_run<N_PV / 2, PvSteps, C::FP8>(d_t, a_t, b, DESC_HI, IDESC_PV, acc ? 1u : 0u);
  }
  // A CTA pair's commits arrive on the barrier at the same offset in both CTAs.
  __device__ __forceinline__ void commit(uint32_t bar) const {
    if constexpr (C::PAIR)
      mma_commit_pair_mc(bar, 3);
    else
      mma_commit_elect(bar);
  }
};

template <int D, bool CAUSAL, int NQ, int VAR>
__device__ __forceinline__ void tc_mma(const TcParams& p, const TcBars<D, NQ, VAR>& bar, uint32_t base, uint32_t tmem,
                                       const WaitGuard& g) {
  using C = TcCfg<D, NQ, VAR>;
  const TcMma<D, NQ, VAR> M(tmem, base);
  // Every lane waits (a non-blocking test first, then the bounded wait); the
  // outcome is made warp-uniform.
  auto wait = [&](uint32_t b, uint32_t par) -> bool {
    const bool r = (C::PAIR ? mbar_test_wait_cl(b, par) : mbar_test_wait(b, par)) ||
                   wait_bar(b, par, g, kStatusTimeoutMma);
    return __all_sync(0xffffffffu, r);
  };
  uint32_t pos = 0;               // K/V stages consumed
  uint32_t go0 = 0, go1 = 0;      // pv_go phases consumed, per O accumulator
  bool ok = true;

  // Acquire the next K/V stage; its tiles sit at positions 2*st and 2*st + 1.
  auto stage_acquire = [&](uint32_t& st) -> bool {
    st = pos % C::NST;
    const bool r = wait(bar.kv_full(st), (pos / C::NST) & 1);
    ++pos;
    if (r) tc_fence_after();
    return r;
  };
  auto pv_wait = [&](int t, uint32_t& go) -> bool {
    const bool r = (C::NQT == 2) ? wait(bar.pv_go(t, 0), go & 1) : wait(bar.pv_go(0, go & 1), (go >> 1) & 1);
    if (!r) return false;
    ++go;
    tc_fence_after();
    return true;
  };

  if constexpr (C::NQT == 2) {
    // One continuous stream over the CTA's units (see the producer).  Per
    // step j of unit w, tile t: P V_t j, then S_t for key tile j + 1, or, in
    // the unit's last step, S_t for key tile 0 of the next unit, whose Q_t
    // has been loaded meanwhile.  Q_t of a unit is released after its last
    // S_t product.  The next unit's first products still wait for O_t to be
    // read out by the epilogue (there is no room in TMEM for a second O).
    int uk = 0;
    int u = tc_unit<C::PAIR>(0);
    // S_t for key tile 0 of unit x (the qi-th unit), K_0 at position kpos.
    auto first_qk = [&](const TcUnit& x, int qi, int t, uint32_t kpos) -> bool {
      if (!wait(bar.q_full(t), qi & 1)) return false;
      tc_fence_after();
      if (x.n[t] > 0) M.qk(t, t, kpos, bar.s_full(t));
      if (x.n[t] <= 1) M.commit(bar.q_empty(t));
      return true;
    };
    // Step j of unit w for tile t, with the stage at st: P V_t j ...
    auto tile_pv = [&](const TcUnit& w, int j, int t, uint32_t st, uint32_t& go) -> bool {
      if (j < w.n[t]) {
        if constexpr (C::PV_SPLIT) {
          // Both halves' barriers complete once per P V: the same phase count.
          if (!wait(bar.pv_go(t, 0), go & 1)) return false;
          tc_fence_after();
          M.pv_half(t, t, 2 * st, 0, j > 0);
          if (!wait(bar.pv_go(t, 1), go & 1)) return false;
          tc_fence_after();
          M.pv_half(t, t, 2 * st, 1, true);
          ++go;
        } else {
          if (!pv_wait(t, go)) return false;
          M.pv(t, t, 2 * st, j > 0);
        }
        if (j == w.n[t] - 1) M.commit(bar.o_done(t));
      }
      return true;
    };
    // ... then S_t for key tile j + 1, or key tile 0 of the next unit.
    auto tile_qk = [&](const TcUnit& w, int j, int t, uint32_t st, bool has_next, const TcUnit& wn, int qn) -> bool {
      if (j + 1 < w.n[t]) {
        M.qk(t, t, 2 * st + 1, bar.s_full(t));
        if (j + 1 == w.n[t] - 1) M.commit(bar.q_empty(t));
      } else if (j == w.nmax - 1 && has_next) {
        return first_qk(wn, qn, t, 2 * st + 1);
      }
      return true;
    };
    if (u < p.total_units) {
      TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
      uint32_t st;
      ok = stage_acquire(st) && first_qk(w, 0, 0, 2 * st) && first_qk(w, 0, 1, 2 * st);
      if (ok) M.commit(bar.kv_empty(st));
      while (ok) {
        const int un = tc_unit<C::PAIR>(uk + 1);
        const bool has_next = un < p.total_units;
        const TcUnit wn = tc_decode<D, CAUSAL, NQ, VAR>(has_next ? un : u, p);
        for (int j = 0; ok && j < w.nmax; ++j) {
          if (!(ok = stage_acquire(st))) break;
          // In a unit's last step both P V products go first: the next unit's
          // S products may have to wait for its Q tiles.
          if (j == w.nmax - 1)
            ok = tile_pv(w, j, 0, st, go0) && tile_pv(w, j, 1, st, go1) &&
                 tile_qk(w, j, 0, st, has_next, wn, uk + 1) && tile_qk(w, j, 1, st, has_next, wn, uk + 1);
          else
            ok = tile_pv(w, j, 0, st, go0) && tile_qk(w, j, 0, st, has_next, wn, uk + 1) &&
                 tile_pv(w, j, 1, st, go1) && tile_qk(w, j, 1, st, has_next, wn, uk + 1);
          if (ok) M.commit(bar.kv_empty(st));
        }
        if (!ok || !has_next) break;
        ++uk;
        u = un;
        w = wn;
      }
    }
  } else {
    uint32_t qk_total = 0;  // S products issued so far
    for (int uk = 0, u; ok && (u = tc_unit<C::PAIR>(uk)) < p.total_units; ++uk) {
      const TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
      if (!(ok = wait(bar.q_full(0), uk & 1))) break;
      uint32_t st;
      if (!(ok = stage_acquire(st))) break;
      const int n = C::PAIR ? w.nmax : w.n[0];  // a pair visits every key tile either CTA's rows need
      const uint32_t qk_base = qk_total;  // S product of key tile j sits in buffer (qk_base + j) & 1
      // First stage: K_0, K_1.
      for (int t = 0; t < C::LA && t < n; ++t) {
        M.qk(0, qk_total & 1, 2 * st + t, bar.s_full(qk_total & 1));
        ++qk_total;
      }
      M.commit(bar.kv_empty(st));
      if (n <= C::LA) M.commit(bar.q_empty(0));
      for (int j = 0; j < n; ++j) {
        // Stage j: V_j at 2*st, K_{j+2} at 2*st + 1.
        if (!(ok = stage_acquire(st))) break;
        if (!(ok = pv_wait(0, go0))) break;
        M.pv(0, (qk_base + j) & 1, 2 * st, j > 0);
        M.commit(bar.o_done(0));
        if (j + C::LA < n) {
          M.qk(0, qk_total & 1, 2 * st + 1, bar.s_full(qk_total & 1));
          ++qk_total;
          if (j + C::LA == n - 1) M.commit(bar.q_empty(0));
        }
        M.commit(bar.kv_empty(st));
      }
    }
  }
  (void)go1;
  // All issued MMAs must complete before TMEM is released (a pair: this CTA's
  // barrier only).
  if constexpr (C::PAIR)
    mma_commit_pair_mc(bar.drain(), 1);
  else
    M.commit(bar.drain());
  wait_bar_drain(bar.drain(), 0, g);
  __syncwarp();
}

// ------------------------------------------------------------------ pair forwarder
// Run by the MMA warp of a CTA pair's second CTA (rank 1), which issues no
// MMAs: in the producer's order, wait for each phase of this CTA's Q and K/V
// barriers (its own copies have landed) and arrive on the leader's barrier at
// the same offset, so that the leader's MMA warp sees both halves loaded.
template <int D, bool CAUSAL, int NQ, int VAR>
__device__ __forceinline__ void tc_forward(const TcParams& p, const TcBars<D, NQ, VAR>& bar, const WaitGuard& g) {
  using C = TcCfg<D, NQ, VAR>;
  const int lane = threadIdx.x & 31;
  uint32_t pos = 0;  // stages forwarded
  auto forward = [&](uint32_t b, uint32_t par) -> bool {
    if (!warp_wait_bar(b, par, g, kStatusTimeoutLoad)) return false;
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(mapa_shared(b, 0));
    return true;
  };
  bool ok = true;
  for (int uk = 0, u; ok && (u = tc_unit<C::PAIR>(uk)) < p.total_units; ++uk) {
    const TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
    ok = forward(bar.q_full(0), uk & 1);
    for (int t = -1; ok && t < w.nmax; ++t) {  // the first stage (K_0, K_1), then one per key tile
      ok = forward(bar.kv_full(pos % C::NST), (pos / C::NST) & 1);
      ++pos;
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ softmax
// Warp arrival on barrier `bar` of the CTA that issues the MMAs: this CTA's
// own, or for a CTA pair the leader's barrier at the same offset.
template <bool PAIR>
__device__ __forceinline__ void arrive_issuer(uint32_t bar) {
  if constexpr (PAIR) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(mapa_shared(bar, 0));
  } else {
    warp_arrive(bar);
  }
}

template <int D, bool CAUSAL, int NQ, int VAR>
__device__ __forceinline__ void tc_softmax(const TcParams& p, const TcBars<D, NQ, VAR>& bar, uint8_t* gbase, uint32_t tmem,
                                           int wg, int quarter, int lane, const WaitGuard& g) {
  using C = TcCfg<D, NQ, VAR>;
  const int r = quarter * 32 + lane;  // row within the query tile = TMEM lane
  const int rank = C::PAIR ? static_cast<int>(cluster_ctarank()) : 0;  // a pair CTA's tile within the unit
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const int ot = (C::NQT == 2) ? wg : 0;
  // alpha of rescale step number k (counted over this accumulator) goes to slot k & 1: in
  // single-tile mode S(j) is computed before P V j-1, so step j's alpha can be written while
  // the correction warpgroup still reads step j-1's.
  float* alpha_s = reinterpret_cast<float*>(gbase + C::OFF_ALPHA) + ot * 256;
  uint32_t a_pub = 0;
  float* stat_m = reinterpret_cast<float*>(gbase + C::OFF_STAT_M) + ot * 128;
  float* stat_l = reinterpret_cast<float*>(gbase + C::OFF_STAT_L) + ot * 128;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  uint32_t s_waits = 0;  // S buffers consumed by this warpgroup
  bool ok = true;

  for (int uk = 0, u; ok && (u = tc_unit<C::PAIR>(uk)) < p.total_units; ++uk) {
    const TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
    // A pair CTA takes part in every key tile of the unit (its rows may see
    // none of a tile's keys: then P = 0 and alpha = 1 for them).
    const int n = C::PAIR ? w.nmax : w.n[wg];
    if (n == 0) continue;
    const int row0 = w.row0 + (wg + rank) * C::BQ;
    const int row = row0 + r;
    float m = -INFINITY;  // running max of scaled logits, log2 units
    float l = 0.f;        // running sum of exp2(x - m)
    float lres = 0.f;     // lazy max: running sum of the steps' largest-P rounding residuals
    for (int j = 0; j < n; ++j) {
      const int buf = (C::NQT == 2) ? wg : static_cast<int>(s_waits & 1);
      const uint32_t par = (C::NQT == 2) ? (s_waits & 1) : ((s_waits >> 1) & 1);
      ok = warp_wait_bar(bar.s_full(buf), par, g, kStatusTimeoutSoftmax);
      if (!ok) break;
      ++s_waits;
      tc_fence_after();
      const uint32_t ts = tmem + lane_off + C::TM_S + buf * C::TM_SB;

      // S is loaded with the maximum of each 32-column chunk (the TMEM load's
      // own reduction), which is the row max wherever no column is masked.
      float s[C::BK];
      float cmax[C::BK / 32];
      {
        uint32_t raw_s[C::BK / 32][32];
#pragma unroll
        for (int c = 0; c < C::BK / 32; ++c) tmem_ld32_max(ts + c * 32, raw_s[c], cmax[c]);
#pragma unroll
        for (int c = 0; c < C::BK / 32; ++c) tmem_wait_ld(raw_s[c], cmax[c]);
#pragma unroll
        for (int c = 0; c < C::BK / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw_s[c][i]);
      }
      const int key0 = j * C::BK;
      const bool need_mask = (CAUSAL && key0 + C::BK - 1 > row0) || (key0 + C::BK > p.Nk);
      float rmax;
      if (need_mask) {
        // Column c of this row is visible iff c <= lim; 32-column blocks that
        // every lane of the warp sees whole are skipped (warp-uniform test).
        const int lim = (CAUSAL ? min(row, p.Nk - 1) : p.Nk - 1) - key0;
        const int lo = __reduce_min_sync(0xffffffffu, lim);
#pragma unroll
        for (int cb = 0; cb < C::BK / 32; ++cb) {
          if (32 * cb + 31 > lo) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * cb + i > lim) s[32 * cb + i] = -INFINITY;
          }
        }
        // Row max of the masked row: 8 chains of three-input maxima over interleaved columns.
        constexpr int KC = C::BK / 8;
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v = fmax3(s[i], s[i + 8], s[i + 16]);
#pragma unroll
          for (int k = 3; k + 1 < KC; k += 2) v = fmax3(v, s[i + 8 * k], s[i + 8 * (k + 1)]);
          if ((KC - 3) % 2 == 1) v = fmaxf(v, s[i + 8 * (KC - 1)]);
          mx[i] = v;
        }
        rmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
      } else {
        rmax = cmax[0];
#pragma unroll
        for (int c = 1; c < C::BK / 32; ++c) rmax = fmaxf(rmax, cmax[c]);
      }
      float m_new, alpha;
      if constexpr (C::LAZY_MAX) {
        const float rm = rmax * sl2;
        m_new = (rm > m + C::MAX_SLACK) ? rm : m;
        // alpha = exp2(m_old - m_new): 0 on the first tile, exactly 1 while m stays.
        alpha = (m_new == m) ? 1.f : ex2(m - m_new);
      } else {
        m_new = fmaxf(m, rmax * sl2);
        // alpha = exp2(m_old - m_new): 0 on the first tile, exactly 1 when the max did not grow.
        alpha = (m_new == -INFINITY) ? 1.f : ex2(m - m_new);
      }
      float nb = (m_new == -INFINITY) ? 0.f : -m_new;
      if (j > 0) {
        alpha_s[(a_pub & 1) * 128 + r] = alpha;
        // The exponentials below are made to depend on the arrival's state
        // word (masked to zero), so the arrival is issued before them and the
        // correction warpgroup rescales O while they run; otherwise the
        // compiler may schedule the arrival after the exponentials, since
        // nothing in this warp depends on it.  (A read-back of alpha from
        // shared memory would order them too, but waits behind the tensor
        // core's operand reads.)
        nb = fmaf(0.f, __uint_as_float(warp_arrive_token(bar.a_full(ot, a_pub & 1))), nb);
        ++a_pub;
      }
      const uint64_t nb2 = f2_pack(nb, nb);
      if constexpr (C::LAZY_MAX) {
        const float pmax = ex2(fmaf(rmax, sl2, nb));  // the step's largest P, as the loop below computes it
        const float pr = C::FP8 ? round_e4m3(pmax) : __uint_as_float(pack_bf16x2(pmax, 0.f) << 16);
        lres = lres * alpha + (pr - pmax);
      }
      uint64_t acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = 0ull;  // (0.f, 0.f)
      // P in chunks of 64 columns (32 bf16x2 words, or 16 words of four e4m3),
      // each stored to TMEM as soon as it is packed.
#pragma unroll
      for (int h = 0; h < C::BK / 64; ++h) {
        if constexpr (C::FP8) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 64 * h; c < 64 * h + 64; c += 4) {
            const float2 x = f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, nb2));
            const float2 y = f2_unpack(f2_fma(f2_pack(s[c + 2], s[c + 3]), sl2x2, nb2));
            const float p0 = ex2(x.x), p1 = ex2(x.y), p2 = ex2(y.x), p3 = ex2(y.y);
            pk[(c >> 2) & 15] = pack_e4m3x4(p0, p1, p2, p3);
            acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(p0, p1));
            acc[((c >> 1) + 1) & 3] = f2_add(acc[((c >> 1) + 1) & 3], f2_pack(p2, p3));
          }
          tmem_st16(ts + h * C::P_COLS_64, pk);
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int c = 64 * h; c < 64 * h + 64; c += 2) {
            const float2 x = f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, nb2));
            const float p0 = ex2(x.x);
            const float p1 = ex2(x.y);
            pk[(c >> 1) & 31] = pack_bf16x2(p0, p1);
            acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(p0, p1));
          }
          tmem_st32(ts + h * C::P_COLS_64, pk);
        }
        if constexpr (C::PV_SPLIT) {
          if (h == 0) {  // first key half of P is in TMEM: its P V may start
            tmem_wait_st();
            tc_fence_before();
            warp_arrive_elect(bar.pv_go(ot, 0));
          }
        }
      }
      const float2 a01 = f2_unpack(f2_add(acc[0], acc[1]));
      const float2 a23 = f2_unpack(f2_add(acc[2], acc[3]));
      l = l * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
      m = m_new;
      tmem_wait_st();
      tc_fence_before();
      // P number s_waits - 1 (counted over this warpgroup) feeds P V number s_waits - 1.
      arrive_issuer<C::PAIR>(C::NQT == 2 ? bar.pv_go(ot, C::PV_SPLIT ? 1 : 0) : bar.pv_go(0, (s_waits - 1) & 1));
    }
    if (!ok) break;
    // Lazy max: the row's log2-sum-exp2 (from the fp32 sum) and O's
    // normaliser; otherwise m and l.
    stat_m[(uk & 1) * 256 + r] = C::LAZY_MAX ? m + log2f(l) : m;
    stat_l[(uk & 1) * 256 + r] = C::LAZY_MAX ? l + lres : l;
    warp_arrive(bar.l_full(ot));
  }
}

// ------------------------------------------------------------------ correction + epilogue
template <int D, bool CAUSAL, bool STRIDED, int NQ, int VAR>
__device__ __forceinline__ void tc_correction(const TcParams& p, const CUtensorMap* tm_o, const TcBars<D, NQ, VAR>& bar,
                                              uint8_t* gbase, uint32_t tmem, int quarter, int lane,
                                              const WaitGuard& g) {
  using C = TcCfg<D, NQ, VAR>;
  const int r = quarter * 32 + lane;
  const int rank = C::PAIR ? static_cast<int>(cluster_ctarank()) : 0;  // a pair CTA's tile within the unit
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const float* alpha_base = reinterpret_cast<const float*>(gbase + C::OFF_ALPHA);
  const float* stat_m = reinterpret_cast<const float*>(gbase + C::OFF_STAT_M);
  const float* stat_l = reinterpret_cast<const float*>(gbase + C::OFF_STAT_L);
  // o_done completes after every P V in single-tile mode (the rescale of step j
  // must wait for P V j-1) and after the last P V of a unit in two-tile mode
  // (S of step j being ready already implies P V j-1 finished).
  constexpr bool PER_PV_DONE = (C::NQT == 1);
  uint32_t a_cnt0 = 0, a_cnt1 = 0, od0 = 0, od1 = 0, lf0 = 0, lf1 = 0;
  uint32_t go_arr = 0;  // single-tile mode: arrivals made on pv_go (= number of the P V they release)
  bool ok = true;
  auto release_o = [&](int t) {
    if (C::NQT == 2) {
      warp_arrive(bar.pv_go(t, 0));
    } else {
      arrive_issuer<C::PAIR>(bar.pv_go(0, go_arr & 1));
      ++go_arr;
    }
  };

  // Rescale step j > 0 of accumulator t.
  auto rescale = [&](int t, uint32_t& a_cnt, uint32_t& od) -> bool {
    bool k = warp_wait_bar(bar.a_full(t, a_cnt & 1), (a_cnt >> 1) & 1, g, kStatusTimeoutSoftmax);
    if (!k) return false;
    const float alpha = alpha_base[t * 256 + (a_cnt & 1) * 128 + r];
    ++a_cnt;
    if (PER_PV_DONE) {
      k = warp_wait_bar(bar.o_done(t), od & 1, g, kStatusTimeoutSoftmax);
      if (!k) return false;
      ++od;
    }
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
      tc_fence_after();
      const uint32_t to = tmem + lane_off + C::TM_O + t * D;
      const uint64_t a2 = f2_pack(alpha, alpha);
      // Chunks of 32 columns in flight per TMEM round trip: single-tile mode
      // (d = 256, no register split, 160 registers a thread) rescales its 256
      // columns in two round trips instead of eight; the two-tile kernels have
      // 80 registers in this warpgroup and keep one chunk.
      constexpr int RG = (C::NQT == 1) ? (D / 32 < 4 ? D / 32 : 4) : 1;
#pragma unroll 1
      for (int c = 0; c < D / 32; c += RG) {
        uint32_t v[RG][32];
#pragma unroll
        for (int k = 0; k < RG; ++k) tmem_ld32(to + (c + k) * 32, v[k]);
#pragma unroll
        for (int k = 0; k < RG; ++k) tmem_wait_ld(v[k]);
#pragma unroll
        for (int k = 0; k < RG; ++k) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 y = f2_unpack(f2_mul(f2_pack(__uint_as_float(v[k][i]), __uint_as_float(v[k][i + 1])), a2));
            v[k][i] = __float_as_uint(y.x);
            v[k][i + 1] = __float_as_uint(y.y);
          }
        }
#pragma unroll
        for (int k = 0; k < RG; ++k) tmem_st32(to + (c + k) * 32, v[k]);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    release_o(t);
    return true;
  };
  // Epilogue of accumulator t: O / l in bf16, L = (m + log2 l) * ln 2.  This
  // warp's 32 rows go out 32 columns at a time: TMEM -> registers -> a staging
  // buffer in shared memory (64-byte swizzle: 16-byte unit k of row i at unit
  // k ^ ((i >> 1) & 3), so a warp's stores hit every bank once) -> TMA store
  // issued by lane 0.  O is released to the next unit right after its last
  // TMEM read; a buffer is rewritten only once the store that read it three
  // chunks earlier has finished reading.
  const uint32_t ost = smem_u32(gbase + C::OFF_OST) + static_cast<uint32_t>(quarter * C::OSTB * C::OST_BUF);
  uint32_t ost_n = 0;  // chunks staged by this warp so far
  auto epilogue = [&](const TcUnit& w, int su, int t, uint32_t& od, uint32_t& lf) -> bool {
    bool k = warp_wait_bar(bar.o_done(t), od & 1, g, kStatusTimeoutSoftmax);
    k = k && warp_wait_bar(bar.l_full(t), lf & 1, g, kStatusTimeoutSoftmax);
    if (!k) return false;
    ++od;
    ++lf;
    tc_fence_after();
    const float mrow = stat_m[su * 256 + t * 128 + r];
    const float lrow = stat_l[su * 256 + t * 128 + r];
    const float inv_l = (C::FP8 ? p.o_scale : 1.f) / lrow;
    const uint64_t il2 = f2_pack(inv_l, inv_l);
    const int row = w.row0 + (t + rank) * C::BQ + r;
    const int wrow0 = w.row0 + (t + rank) * C::BQ + quarter * 32;  // first row of this warp's box
    const uint32_t to = tmem + lane_off + C::TM_O + t * D;
    const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(to + c * 32, v);
      tmem_wait_ld(v);
      if (c == D / 32 - 1) {
        tc_fence_before();
        release_o(t);  // O may be overwritten by the next unit's first P V
      }
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 y = f2_unpack(f2_mul(f2_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), il2));
        packed[i] = pack_bf16x2(y.x, y.y);
      }
      {
        const uint32_t buf = ost + (ost_n % C::OSTB) * C::OST_BUF;
        ++ost_n;
        if (lane == 0) bulk_wait_group_read<C::OSTB - 1>();
        __syncwarp();
        const uint32_t rb = buf + static_cast<uint32_t>(lane) * 64;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(rb + ((static_cast<uint32_t>(u) ^ sw) << 4), packed[4 * u], packed[4 * u + 1],
                       packed[4 * u + 2], packed[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && wrow0 < p.Nq) {
          if constexpr (STRIDED)
            tma_store_4d(tm_o, buf, c * 32, wrow0, w.bh % p.H, w.bh / p.H);
          else
            tma_store_3d(tm_o, buf, c * 32, wrow0, w.bh);
          bulk_commit_group();
        }
      }
    }
    if (row < p.Nq)
      p.lse[static_cast<size_t>(w.bh) * p.Nq + row] = (C::LAZY_MAX ? mrow : mrow + log2f(lrow)) * 0.69314718055994531f;
    return true;
  };

  // O starts free: release it for the first unit's first P V.
  release_o(0);
  if (C::NO == 2) release_o(1);
  for (int uk = 0, u; ok && (u = tc_unit<C::PAIR>(uk)) < p.total_units; ++uk) {
    const TcUnit w = tc_decode<D, CAUSAL, NQ, VAR>(u, p);
    // Same order as the MMA warp's P V products: (tile 0, j), (tile 1, j), (tile 0, j+1), ...
    const int n0 = C::PAIR ? w.nmax : w.n[0];  // a pair CTA takes part in every key tile of the unit
    for (int j = 0; ok && j < w.nmax; ++j) {
      if (ok && j >= 1 && j < n0) ok = rescale(0, a_cnt0, od0);
      if (C::NO == 2 && ok && j >= 1 && j < w.n[1]) ok = rescale(1, a_cnt1, od1);
      if (ok && j == n0 - 1) ok = epilogue(w, uk & 1, 0, od0, lf0);
      if (C::NO == 2 && ok && j == w.n[1] - 1) ok = epilogue(w, uk & 1, 1, od1, lf1);
    }
  }
  // The staged O tiles must be written (and their shared memory read) before the CTA exits.
  if (lane == 0) bulk_wait_group_all();
  __syncwarp();
}

// ------------------------------------------------------------------ kernel
template <int D, bool CAUSAL, bool STRIDED, int NQ, int VAR>
__global__ void __launch_bounds__(TcCfg<D, NQ, VAR>::THREADS, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const TcParams p) {
  using C = TcCfg<D, NQ, VAR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const TcBars<D, NQ, VAR> bar{base + C::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_ABORT);
  // CTA pairs: rank 0 (the leader) issues the MMAs; its Q and K/V barriers
  // also take the arrival forwarded by rank 1, and its P V barriers the
  // arrivals of both CTAs' softmax and correction warps.
  const uint32_t rank = C::PAIR ? cluster_ctarank() : 0;
  const uint32_t full_count = (C::PAIR && rank == 0) ? 2 : 1;
  const uint32_t go_count = C::PAIR ? 16 : 8;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar.q_full(t), full_count);
      mbar_init(bar.q_empty(t), 1);
    }
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(bar.kv_full(i), full_count);
      mbar_init(bar.kv_empty(i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      // Signalled by warps (one arrival each) or by tcgen05.commit (one).
      mbar_init(bar.s_full(b), 1);
      mbar_init(bar.pv_go(b, 0), go_count);  // 4 softmax warps + 4 correction warps (per CTA of a pair)
      mbar_init(bar.pv_go(b, 1), C::PV_SPLIT ? 4 : go_count);  // split P V: second key half, 4 softmax warps
      mbar_init(bar.a_full(b, 0), 4);
      mbar_init(bar.a_full(b, 1), 4);
      mbar_init(bar.o_done(b), 1);
      mbar_init(bar.l_full(b), 4);
    }
    mbar_init(bar.drain(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::LOAD_WARP && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
  }
  if (warp == C::MMA_WARP) {
    if constexpr (C::PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::TM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // Both CTAs of a pair have initialised their barriers before either
  // arrives on, or commits to, the other's.
  if constexpr (C::PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitGuard g{abort_flag, p.status, p.limit_ns, C::PAIR};

  if (warp < C::SOFTMAX_WARPS) {
    if constexpr (C::SPLIT_REGS) regs_increase<C::REG_SOFTMAX>();
    tc_softmax<D, CAUSAL, NQ, VAR>(p, bar, gbase, tmem, warp >> 2, warp & 3, lane, g);
  } else if (warp < C::SOFTMAX_WARPS + 4) {
    if constexpr (C::SPLIT_REGS) regs_decrease<C::reg_corr(STRIDED)>();
    tc_correction<D, CAUSAL, STRIDED, NQ, VAR>(p, &tm_o, bar, gbase, tmem, warp & 3, lane, g);
  } else {
    if constexpr (C::SPLIT_REGS) regs_decrease<C::REG_CORR_OTHER - C::reg_corr(STRIDED)>();
    if (warp == C::LOAD_WARP && lane == 0) tc_producer<D, CAUSAL, STRIDED, NQ, VAR>(&tm_q, &tm_k, &tm_v, p, bar, base, g);
    if (warp == C::MMA_WARP) {
      if (rank == 0)
        tc_mma<D, CAUSAL, NQ, VAR>(p, bar, base, tmem, g);
      else
        tc_forward<D, CAUSAL, NQ, VAR>(p, bar, g);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // A pair CTA leaves only once the other is done with its shared memory,
  // barriers and TMEM (the leader's MMAs read and write both CTAs').
  if constexpr (C::PAIR) cluster_sync_all();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    if constexpr (C::PAIR)
      tmem_dealloc_pair(tmem, C::TM_COLS);
    else
      tmem_dealloc(tmem, C::TM_COLS);
  }
}

}  // namespace fa

// FlashAttention-2 backward pass, bf16 in / fp32 accumulate, for sm_103a.
//
// Given Q, K, V, the forward's O and logsumexp L, and the upstream dO, the
// gradients are (softmax scale s):
//   P = exp(s Q K^T - L)   (recomputed tile by tile from L instead of stored:
//                           "FlashAttention-2 from PyTorch to Triton",
//                           "What We Are Building")
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O),
//   dQ = s dS K,  dK = s dS^T Q.
// As in the metal-flash-attention backward ("Case Study:
// metal-flash-attention"), the work is split into a dK/dV kernel and a dQ
// kernel that each own their outputs, so no float atomics are needed; -D and
// -L * log2(e) (negated, as the elementwise step adds them) come from a small
// preprocessing kernel.
//
// Both kernels share one structure (template parameter MODE):
//   MODE 0, dK/dV: a work unit is a 128-key tile of one head; its K and V
//     tiles stay in shared memory while tiles of Q and dO (64 rows at d = 128,
//     96 at d <= 64) stream past.
//     S^T = K Q^T and dP^T = V dO^T go to TMEM (128 lanes = keys), the
//     elementwise warps form P^T and dS^T in bf16 over them, and the MMA warp
//     accumulates dV += P^T dO and dK += dS^T Q in TMEM.
//   MODE 1, dQ: a work unit is a 128-row query tile; its Q and dO tiles stay,
//     96-key tiles of K and V stream past; S = Q K^T, dP = dO V^T, then
//     dQ += dS K.
// Per CTA (one per SM, persistent): two elementwise warpgroups take the
// streamed tiles alternately (S/dP double-buffered in TMEM), one MMA warp
// issues every tcgen05.mma from an elected lane, one producer thread issues
// the TMA loads.  Every wait is bounded (see ptx.cuh).
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fa {

struct BwdParams {
  int Nq;                // query rows per head
  int Nk;                // key / value rows per head
  int H;                 // heads (unit index bh = b * H + h)
  int BH;                // batch * heads
  int n_pad;             // row stride of the l2 / dsum vectors: N rounded up to 192 (a multiple of every BS)
  int n_m;               // 128-row tiles of the fixed operands per head: ceil(N / 128)
  int n_s;               // streamed tiles per head: ceil(N / BS)
  int total_units;       // BH * n_m * HALVES
  float scale;           // softmax scale (dK and dQ carry one factor of it)
  float scale_log2;      // scale * log2(e)
  const float* l2;       // [BH][n_pad]: -L * log2(e); -inf on rows >= N
  const float* dsum;     // [BH][n_pad]: -D = -rowsum(dO * O); 0 on rows >= N
  __nv_bfloat16* out0;   // MODE 0: dK, MODE 1: dQ: contiguous [BH][rows][D], or (strided
  __nv_bfloat16* out1;   // MODE 0: dV               kernels) row i of (b, h) at b*s[0] + h*s[1] + i*s[2]
  long long out0_s[3];   // element strides {batch, head, row} of out0 / out1 (strided kernels)
  long long out1_s[3];
  int* status;           // device status word
  unsigned long long limit_ns;
};

template <int D, int MODE>
struct BwdCfg {
  static constexpr bool KV = (MODE == 0);
  static constexpr int BM = 128;                         // fixed-tile rows = TMEM lanes
  // Streamed-tile rows: 96 where TMEM holds the double-buffered S and dP and
  // the accumulators (4 * 96 + D in MODE 1; 4 * 96 + 2 * D in MODE 0 for
  // d <= 64), else 64 (MODE 0 at d = 128: 4 * 64 + 2 * 128 = 512 columns).
  // Larger tiles mean fewer, larger S and dP products per FLOP for the MMA warp.
  // d = 256: 32 rows (two 128-row fixed tiles of 64 KB each leave room for
  // two or three stages of 32-row tiles), and in MODE 0 each unit accumulates
  // one half of the dK and dV columns (HALVES units per key tile), so that
  // 4 * 32 + 2 * 128 columns of TMEM suffice.
  static constexpr int BS = (D == 256) ? 32 : (KV && D == 128) ? 64 : 96;
  static constexpr int HALVES = (KV && D == 256) ? 2 : 1;
  static constexpr int OUTW = D / HALVES;                // accumulator columns per output
  static constexpr int SWB = (D * 2 >= 128) ? 128 : D * 2;  // swizzle span in bytes
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : 4u;   // descriptor swizzle code
  static constexpr int RC = SWB / 2;                     // bf16 columns per swizzle region
  static constexpr int NR = D / RC;                      // regions per tile row
  static constexpr int FIX_REGION = BM * SWB;
  static constexpr int S_REGION = BS * SWB;
  static constexpr int FIX_TILE = BM * D * 2;
  static constexpr int S_TILE = BS * D * 2;
  static constexpr int VEC_BYTES = BS * 4;               // one fp32 value per streamed row
  // Shared memory: [fixed A1, A2][stages][misc].  A stage holds the two
  // streamed tiles (B1, B2) and, in MODE 0, their rows' L*log2e and D.
  static constexpr int STAGE = 2 * S_TILE + (KV ? 1024 : 0);
  static constexpr int OFF_FIX = 0;
  static constexpr int OFF_ST = 2 * FIX_TILE;
  static constexpr int MISC = 1024;
  static constexpr int SMEM_LIMIT = 227 * 1024;
  static constexpr int NST_FIT = (SMEM_LIMIT - 1024 - MISC - OFF_ST) / STAGE;
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;
  static constexpr int OFF_MISC = OFF_ST + NST * STAGE;
  static constexpr int OFF_TMEM_SLOT = OFF_MISC + 512;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_USED = OFF_MISC + MISC + 1024;  // + slack for 1024-byte alignment
  static constexpr int SMEM_ALLOC = SMEM_USED < 120 * 1024 ? 120 * 1024 : SMEM_USED;
  // TMEM columns: S buffers at 0 and BS, dP buffers at 2 BS and 3 BS,
  // accumulators from 4 BS (MODE 0: dK, then dV; MODE 1: dQ).
  static constexpr int TM_S = 0;
  static constexpr int TM_DP = 2 * BS;
  static constexpr int TM_OUT = 4 * BS;
  static constexpr int NOUT = KV ? 2 : 1;
  static constexpr int TM_COLS = 512;
  // S and dP issued as runs of MMAs from one block (d >= 64; d = 256 as two
  // runs of 8), or one MMA per block (d = 32, measured faster there).
  static constexpr bool RUNS = D >= 64;
  // Warps: 0-3 and 4-7 elementwise warpgroups (buffer 0 / 1), 8 MMA, 9 TMA.
  static constexpr int MMA_WARP = 8;
  static constexpr int LOAD_WARP = 9;
  static constexpr int THREADS = 320;
  static_assert(D == 32 || D == 64 || D == 128 || D == 256, "head dim of the backward pass");
  static_assert(TM_OUT + NOUT * OUTW <= TM_COLS, "TMEM budget");
  static_assert(NST >= 2, "streamed stages");
  static_assert(SMEM_USED <= SMEM_LIMIT, "shared memory budget");
};

// A work unit: fixed rows [m0, m0 + 128) of head bh, streamed tiles
// [s_begin, s_end), output columns [half * OUTW, (half + 1) * OUTW).
struct BwdUnit {
  int bh;
  int m0;
  int s_begin;
  int s_end;
  int half;
};

// Units are numbered heaviest first under the causal mask: in MODE 0 the
// first key tiles see the most query tiles, in MODE 1 the last query tiles
// see the most key tiles.  Streamed tiles that lie wholly on the masked side
// of the diagonal are skipped.  Without the mask every unit costs the same
// and units are numbered head by head, so that the CTAs at work at one time
// share a few heads' streamed tiles in L2.
template <int D, int MODE, bool CAUSAL>
__device__ __forceinline__ BwdUnit bwd_decode(int u, const BwdParams& p) {
  constexpr int HV = BwdCfg<D, MODE>::HALVES;
  BwdUnit w;
  int mt;
  if (CAUSAL) {
    const int per_tile = p.BH * HV;  // units per fixed tile
    mt = (MODE == 0) ? (u / per_tile) : (p.n_m - 1 - u / per_tile);
    w.half = (u % per_tile) / p.BH;
    w.bh = u % p.BH;
  } else {
    const int per_head = p.n_m * HV;  // units per head
    w.bh = u / per_head;
    mt = (u % per_head) / HV;
    w.half = u % HV;
  }
  w.m0 = mt * 128;
  if (MODE == 0) {
    w.s_begin = CAUSAL ? w.m0 / BwdCfg<D, MODE>::BS : 0;  // query tiles holding some query >= the first key
    w.s_end = p.n_s;
  } else {
    w.s_begin = 0;
    const int last = (w.m0 + 127) / BwdCfg<D, MODE>::BS + 1;  // key tiles holding some key <= the last query
    w.s_end = (CAUSAL && last < p.n_s) ? last : p.n_s;
  }
  if (w.s_begin > w.s_end) w.s_begin = w.s_end;  // MODE 0, causal, keys past the last query: no tile
  return w;
}

// k-th unit of this CTA: rounds of gridDim.x, alternating direction (snake).
__device__ __forceinline__ int bwd_unit(int k) {
  const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  return k * g + ((k & 1) ? g - 1 - b : b);
}

template <int D, int MODE>
struct BwdBars {
  using C = BwdCfg<D, MODE>;
  uint32_t b0;
  __device__ __forceinline__ uint32_t fix_full() const { return b0; }
  __device__ __forceinline__ uint32_t fix_empty() const { return b0 + 8; }
  __device__ __forceinline__ uint32_t st_full(int i) const { return b0 + 16 + 8u * i; }
  __device__ __forceinline__ uint32_t st_empty(int i) const { return b0 + 16 + 8u * (C::NST + i); }
  // S and dP of a streamed tile in buffer b are ready (tcgen05.commit).
  __device__ __forceinline__ uint32_t s_full(int b) const { return b0 + 16 + 8u * (2 * C::NST + b); }
  // P / dS of buffer b are in TMEM (the 4 warps of warpgroup b).
  __device__ __forceinline__ uint32_t p_ready(int b) const { return b0 + 16 + 8u * (2 * C::NST + 2 + b); }
  // The unit's accumulators are final (tcgen05.commit) / read out again (8 warps).
  __device__ __forceinline__ uint32_t out_done() const { return b0 + 16 + 8u * (2 * C::NST + 4); }
  __device__ __forceinline__ uint32_t out_free() const { return b0 + 16 + 8u * (2 * C::NST + 5); }
  __device__ __forceinline__ uint32_t drain() const { return b0 + 16 + 8u * (2 * C::NST + 6); }
  static constexpr int COUNT = 2 + 2 * C::NST + 7;
  static_assert(COUNT * 8 <= 512, "barrier area");
};

// Wait without looking at the abort flag (to drain in-flight copies and MMAs
// before the CTA exits); still time-limited.
__device__ __forceinline__ bool bwd_wait_drain(uint32_t bar, uint32_t parity, const WaitGuard& g) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > g.limit_ns) {
      atomicOr(g.status, kStatusTimeoutDrain);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------------ TMA producer
// One thread.  Per unit: the two fixed tiles (A1, A2: 128 rows each), then one
// stage per streamed tile: B1 and B2 (BS rows each) and, in MODE 0, the
// streamed rows' -L * log2(e) and -D.
//   MODE 0: A1 = K, A2 = V, B1 = Q, B2 = dO.   MODE 1: A1 = Q, A2 = dO, B1 = K, B2 = V.
template <int D, int MODE, bool CAUSAL, bool STRIDED>
__device__ __forceinline__ void bwd_producer(const CUtensorMap* tm_a1, const CUtensorMap* tm_a2,
                                             const CUtensorMap* tm_b1, const CUtensorMap* tm_b2, const BwdParams& p,
                                             const BwdBars<D, MODE>& bar, uint32_t base, const WaitGuard& g) {
  using C = BwdCfg<D, MODE>;
  const uint64_t pol_fix = policy_evict_first();  // read by one unit
  const uint64_t pol_str = policy_evict_last();   // read by every unit of the head
  uint32_t pos = 0;       // stages issued so far
  uint32_t issued = 0;    // bit i: stage i has been loaded at least once
  uint32_t last_par = 0;  // bit i: parity of stage i's latest load
  int last_fix = -1;      // index (within this CTA) of the latest unit whose fixed tiles were loaded
  bool ok = true;
  for (int uk = 0, u; ok && (u = bwd_unit(uk)) < p.total_units; ++uk) {
    const BwdUnit w = bwd_decode<D, MODE, CAUSAL>(u, p);
    if (!(ok = wait_bar(bar.fix_empty(), (uk & 1) ^ 1, g, kStatusTimeoutLoad))) break;
    mbar_arrive_expect_tx(bar.fix_full(), 2 * C::FIX_TILE);
    // Strided tensors are 4-D maps {d, rows, H, B}; contiguous ones 3-D {d, rows, B*H}.
    const int th = STRIDED ? w.bh % p.H : w.bh, tb = STRIDED ? w.bh / p.H : 0;
    auto load = [&](uint32_t dst, const CUtensorMap* tm, uint32_t full, int x, int row, uint64_t pol) {
      if constexpr (STRIDED)
        tma_load_4d(dst, tm, full, x, row, th, tb, pol);
      else
        tma_load_3d(dst, tm, full, x, row, th, pol);
    };
    for (int r = 0; r < C::NR; ++r) {
      load(base + C::OFF_FIX + r * C::FIX_REGION, tm_a1, bar.fix_full(), r * C::RC, w.m0, pol_fix);
      load(base + C::OFF_FIX + C::FIX_TILE + r * C::FIX_REGION, tm_a2, bar.fix_full(), r * C::RC, w.m0, pol_fix);
    }
    last_fix = uk;
    for (int s = w.s_begin; s < w.s_end; ++s) {
      const int st = pos % C::NST;
      const uint32_t par = (pos / C::NST) & 1;
      if (!(ok = wait_bar(bar.st_empty(st), par ^ 1, g, kStatusTimeoutLoad))) break;
      const uint32_t s0 = base + C::OFF_ST + st * C::STAGE;
      const uint32_t full = bar.st_full(st);
      mbar_arrive_expect_tx(full, 2 * C::S_TILE + (C::KV ? 2 * C::VEC_BYTES : 0));
      for (int r = 0; r < C::NR; ++r) {
        load(s0 + r * C::S_REGION, tm_b1, full, r * C::RC, s * C::BS, pol_str);
        load(s0 + C::S_TILE + r * C::S_REGION, tm_b2, full, r * C::RC, s * C::BS, pol_str);
      }
      if constexpr (C::KV) {
        // s * BS + BS <= n_pad (a multiple of BS), and BS * 4 is a multiple of 16: aligned, in bounds.
        const size_t off = static_cast<size_t>(w.bh) * p.n_pad + static_cast<size_t>(s) * C::BS;
        bulk_load(s0 + 2 * C::S_TILE, p.l2 + off, C::VEC_BYTES, full);
        bulk_load(s0 + 2 * C::S_TILE + C::VEC_BYTES, p.dsum + off, C::VEC_BYTES, full);
      }
      issued |= 1u << st;
      last_par = (last_par & ~(1u << st)) | (par << st);
      ++pos;
    }
  }
  // Every issued copy must land before the CTA may exit.
  for (int i = 0; i < C::NST; ++i)
    if (issued & (1u << i)) bwd_wait_drain(bar.st_full(i), (last_par >> i) & 1, g);
  if (last_fix >= 0) bwd_wait_drain(bar.fix_full(), last_fix & 1, g);
}

// ------------------------------------------------------------------ MMA issuer
// The whole MMA warp runs the loop; an elected lane issues each operation.
// Descriptors are (low, high) word pairs built once; positions and K steps
// add constants to the low word's address field (no shared address reaches
// 2^18, so it never carries into the leading-byte-offset field).
template <int D, int MODE>
struct BwdMma {
  using C = BwdCfg<D, MODE>;
  static constexpr uint32_t IDESC_S = make_idesc_bf16(128, C::BS, 0);  // S, dP: B K-major
  static constexpr uint32_t IDESC_O = make_idesc_bf16(128, C::OUTW, 1);  // accumulators: B MN-major
  static constexpr uint32_t DESC_HI = sdesc_hi(8 * C::SWB, C::SWZ);
  static constexpr __host__ __device__ uint32_t a_step(int kk) {
    return ((kk * 16 / C::RC) * C::FIX_REGION + (kk * 16 % C::RC) * 2) >> 4;
  }
  static constexpr __host__ __device__ uint32_t b_step(int kk) {
    return ((kk * 16 / C::RC) * C::S_REGION + (kk * 16 % C::RC) * 2) >> 4;
  }
  static constexpr __host__ __device__ uint32_t mn_step(int kk) { return (kk * 16 * C::SWB) >> 4; }
  static constexpr uint32_t STAGE_STEP = C::STAGE >> 4;

  uint32_t tmem;
  uint32_t a1, a2;          // fixed tiles, K-major
  uint32_t b1, b2;          // stage 0's streamed tiles, K-major (B of S and dP)
  uint32_t b1_mn, b2_mn;    // the same tiles, MN-major (B of the accumulations)

  __device__ __forceinline__ BwdMma(uint32_t tmem_, uint32_t base) : tmem(tmem_) {
    a1 = sdesc_lo(base + C::OFF_FIX, 16);
    a2 = sdesc_lo(base + C::OFF_FIX + C::FIX_TILE, 16);
    b1 = sdesc_lo(base + C::OFF_ST, 16);
    b2 = sdesc_lo(base + C::OFF_ST + C::S_TILE, 16);
    b1_mn = sdesc_lo(base + C::OFF_ST, C::S_REGION);
    b2_mn = sdesc_lo(base + C::OFF_ST + C::S_TILE, C::S_REGION);
  }
  // Descriptor increments from K step k-1 to k (16-byte units; TMEM columns for ta).
  template <int OFF>  // runs that start at K step OFF
  struct SdpSteps {
    static constexpr __host__ __device__ uint32_t da(int k) { return a_step(OFF + k) - a_step(OFF + k - 1); }
    static constexpr __host__ __device__ uint32_t db(int k) { return b_step(OFF + k) - b_step(OFF + k - 1); }
  };
  struct AccSteps {
    static constexpr __host__ __device__ uint32_t ta(int) { return 8; }  // 16 bf16 = 8 TMEM columns
    static constexpr __host__ __device__ uint32_t db(int k) { return mn_step(k) - mn_step(k - 1); }
  };
  static constexpr bool RUNS = C::RUNS;
  // Start of output half h within a streamed tile read MN-major: OUTW / 64 regions per half.
  static constexpr uint32_t HALF_STEP = (C::OUTW / C::RC) * C::S_REGION >> 4;
  // S = A1 B1^T and dP = A2 B2^T of the tile in stage st, into buffer b.
  __device__ __forceinline__ void sdp(uint32_t st, int b) const {
    const uint32_t d_s = tmem + C::TM_S + b * C::BS, d_p = tmem + C::TM_DP + b * C::BS;
    if constexpr (RUNS && D <= 128) {
      mma_ss_run<D / 16, SdpSteps<0>>(d_s, a1, DESC_HI, b1 + st * STAGE_STEP, DESC_HI, IDESC_S, 0u);
      mma_ss_run<D / 16, SdpSteps<0>>(d_p, a2, DESC_HI, b2 + st * STAGE_STEP, DESC_HI, IDESC_S, 0u);
    } else if constexpr (RUNS) {
      const uint32_t bs = b1 + st * STAGE_STEP, bp = b2 + st * STAGE_STEP;
      mma_ss_run<8, SdpSteps<0>>(d_s, a1, DESC_HI, bs, DESC_HI, IDESC_S, 0u);
      mma_ss_run<8, SdpSteps<8>>(d_s, a1 + a_step(8), DESC_HI, bs + b_step(8), DESC_HI, IDESC_S, 1u);
      mma_ss_run<8, SdpSteps<0>>(d_p, a2, DESC_HI, bp, DESC_HI, IDESC_S, 0u);
      mma_ss_run<8, SdpSteps<8>>(d_p, a2 + a_step(8), DESC_HI, bp + b_step(8), DESC_HI, IDESC_S, 1u);
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(d_s, a1 + a_step(kk), DESC_HI, b1 + st * STAGE_STEP + b_step(kk), DESC_HI, IDESC_S, kk > 0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(d_p, a2 + a_step(kk), DESC_HI, b2 + st * STAGE_STEP + b_step(kk), DESC_HI, IDESC_S, kk > 0);
    }
  }
  // MODE 0: dK (+)= dS^T B1 and dV (+)= P^T B2.  MODE 1: dQ (+)= dS B1.
  // dS (bf16) sits over the dP buffer, P (bf16) over the S buffer.  Output
  // half h takes B's columns [h * OUTW, (h + 1) * OUTW).
  __device__ __forceinline__ void accumulate(uint32_t st, int b, bool acc, int half) const {
    const uint32_t a_ds = tmem + C::TM_DP + b * C::BS, a_p = tmem + C::TM_S + b * C::BS;
    const uint32_t hs = static_cast<uint32_t>(half) * HALF_STEP;
    if constexpr (RUNS) {
      mma_ts_run<C::BS / 16, AccSteps>(tmem + C::TM_OUT, a_ds, b1_mn + st * STAGE_STEP + hs, DESC_HI, IDESC_O,
                                       acc ? 1u : 0u);
      if constexpr (C::KV)
        mma_ts_run<C::BS / 16, AccSteps>(tmem + C::TM_OUT + C::OUTW, a_p, b2_mn + st * STAGE_STEP + hs, DESC_HI,
                                         IDESC_O, acc ? 1u : 0u);
    } else {
#pragma unroll
      for (int kk = 0; kk < C::BS / 16; ++kk)
        mma_ts_elect(tmem + C::TM_OUT, a_ds + kk * 8, b1_mn + st * STAGE_STEP + hs + mn_step(kk), DESC_HI,
                     IDESC_O, (acc || kk > 0) ? 1u : 0u);
      if constexpr (C::KV) {
#pragma unroll
        for (int kk = 0; kk < C::BS / 16; ++kk)
          mma_ts_elect(tmem + C::TM_OUT + C::OUTW, a_p + kk * 8, b2_mn + st * STAGE_STEP + hs + mn_step(kk),
                       DESC_HI, IDESC_O, (acc || kk > 0) ? 1u : 0u);
      }
    }
  }
};

// Order per unit of n streamed tiles: S/dP of tiles 0 and 1 (buffers 0, 1);
// then for each tile t: wait for its P / dS, accumulate, release its stage,
// and issue S/dP of tile t + 2 into the freed buffer.  Products from one warp
// complete in issue order, so S/dP of tile t + 2 overwrite buffer t & 1 only
// after the accumulation of tile t has read it.
template <int D, int MODE, bool CAUSAL>
__device__ __forceinline__ void bwd_mma(const BwdParams& p, const BwdBars<D, MODE>& bar, uint32_t base, uint32_t tmem,
                                        const WaitGuard& g) {
  using C = BwdCfg<D, MODE>;
  const BwdMma<D, MODE> M(tmem, base);
  auto wait = [&](uint32_t b, uint32_t par) -> bool {
    const bool r = mbar_test_wait(b, par) || wait_bar(b, par, g, kStatusTimeoutMma);
    return __all_sync(0xffffffffu, r);
  };
  uint32_t pos = 0;            // streamed stages consumed before the current unit
  uint32_t pr0 = 0, pr1 = 0;   // p_ready phases consumed, per buffer
  bool ok = true;
  for (int uk = 0, u; ok && (u = bwd_unit(uk)) < p.total_units; ++uk) {
    const BwdUnit w = bwd_decode<D, MODE, CAUSAL>(u, p);
    const int n = w.s_end - w.s_begin;
    if (!(ok = wait(bar.fix_full(), uk & 1))) break;
    tc_fence_after();
    if (n <= 0) {
      // No streamed tile reaches these fixed rows (MODE 0, causal, with more
      // keys than queries): nothing to multiply; the epilogue writes zeros.
      // The previous unit's epilogue must still release the accumulators
      // first, so that each out_free phase collects the arrivals of one unit.
      if (uk > 0) {
        if (!(ok = wait(bar.out_free(), (uk - 1) & 1))) break;
        tc_fence_after();
      }
      mma_commit_elect(bar.fix_empty());
      mma_commit_elect(bar.out_done());
      continue;
    }
    auto stage_of = [&](int t) -> uint32_t { return (pos + t) % C::NST; };
    auto acquire = [&](int t) -> bool {
      const uint32_t q = pos + t;
      if (!wait(bar.st_full(q % C::NST), (q / C::NST) & 1)) return false;
      tc_fence_after();
      return true;
    };
    for (int t = 0; ok && t < n && t < 2; ++t) {
      if (!(ok = acquire(t))) break;
      M.sdp(stage_of(t), t & 1);
      mma_commit_elect(bar.s_full(t & 1));
      if (t == n - 1) mma_commit_elect(bar.fix_empty());
    }
    for (int t = 0; ok && t < n; ++t) {
      const int b = t & 1;
      uint32_t& pr = b ? pr1 : pr0;
      if (!(ok = wait(bar.p_ready(b), pr & 1))) break;
      ++pr;
      tc_fence_after();
      if (t == 0 && uk > 0) {
        if (!(ok = wait(bar.out_free(), (uk - 1) & 1))) break;
        tc_fence_after();
      }
      M.accumulate(stage_of(t), b, t > 0, w.half);
      mma_commit_elect(bar.st_empty(stage_of(t)));
      if (t + 2 < n) {
        if (!(ok = acquire(t + 2))) break;
        M.sdp(stage_of(t + 2), b);
        mma_commit_elect(bar.s_full(b));
        if (t + 2 == n - 1) mma_commit_elect(bar.fix_empty());
      }
    }
    if (!ok) break;
    pos += n;
    mma_commit_elect(bar.out_done());
  }
  // All issued MMAs must complete before TMEM is released.
  mma_commit_elect(bar.drain());
  bwd_wait_drain(bar.drain(), 0, g);
  __syncwarp();
}

// ------------------------------------------------------------------ elementwise warpgroups
// Warpgroup b (thread = fixed row = TMEM lane) takes the streamed tiles t of
// each unit with t % 2 == b: P = 2^(S * scale * log2e - L * log2e), masked
// entries 0; dS = P * (dP - D); both to TMEM as bf16 (P only in MODE 0, where
// it is the A operand of dV).  At the end of each unit both warpgroups read the
// accumulators out (MODE 0: warpgroup 0 dK, warpgroup 1 dV; MODE 1: dQ, split
// by 32-column chunks) and release them.
template <int D, int MODE, bool CAUSAL, bool STRIDED>
__device__ __forceinline__ void bwd_elementwise(const BwdParams& p, const BwdBars<D, MODE>& bar, uint8_t* gbase,
                                                uint32_t tmem, int b, int quarter, int lane, const WaitGuard& g) {
  using C = BwdCfg<D, MODE>;
  const int r = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const float sl2 = p.scale_log2;
  uint32_t sf = 0;    // s_full(b) phases consumed
  uint32_t pos = 0;   // streamed stages before the current unit
  bool ok = true;
  for (int uk = 0, u; ok && (u = bwd_unit(uk)) < p.total_units; ++uk) {
    const BwdUnit w = bwd_decode<D, MODE, CAUSAL>(u, p);
    const int n = w.s_end - w.s_begin;
    const int row = w.m0 + r;  // key (MODE 0) or query (MODE 1) index of this thread
    float l2_row = -INFINITY, d_row = 0.f;  // this row's -L * log2(e) and -D (MODE 1)
    if (MODE == 1 && row < p.n_pad) {
      l2_row = p.l2[static_cast<size_t>(w.bh) * p.n_pad + row];
      d_row = p.dsum[static_cast<size_t>(w.bh) * p.n_pad + row];
    }
    for (int t = b; ok && t < n; t += 2) {
      ok = warp_wait_bar(bar.s_full(b), sf & 1, g, kStatusTimeoutSoftmax);
      if (!ok) break;
      ++sf;
      const uint32_t q = pos + t;
      const int st = q % C::NST;
      if constexpr (C::KV) {
        // The stage's vectors were written by TMA; observe that completion here too.
        ok = warp_wait_bar(bar.st_full(st), (q / C::NST) & 1, g, kStatusTimeoutSoftmax);
        if (!ok) break;
      }
      tc_fence_after();
      const int s = w.s_begin + t;  // streamed tile
      const int col0 = s * C::BS;  // index of the first streamed row
      bool need_mask;
      if (MODE == 0)
        need_mask = CAUSAL && col0 < w.m0 + C::BM - 1;
      else
        need_mask = (col0 + C::BS > p.Nk) || (CAUSAL && col0 + C::BS - 1 > w.m0);
      const float4* vl2 = reinterpret_cast<const float4*>(gbase + C::OFF_ST + st * C::STAGE + 2 * C::S_TILE);
      const float4* vd = vl2 + C::BS / 4;
      // Two chunks of 32 streamed rows: load S and dP, form P and dS, store
      // both as 16 bf16x2 columns.
#pragma unroll 1
      for (int h = 0; h < C::BS / 32; ++h) {
        uint32_t rs[32], rd[32];
        tmem_ld32(tmem + lane_off + C::TM_S + b * C::BS + h * 32, rs);
        tmem_ld32(tmem + lane_off + C::TM_DP + b * C::BS + h * 32, rd);
        tmem_wait_ld(rs);
        tmem_wait_ld(rd);
        uint32_t pk[16], dk[16];
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        if constexpr (CAUSAL) {
          // Causal kernels: scalar arithmetic (the paired form below measured
          // 3 % slower here, 2-8 % faster in the non-causal kernels).
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            float nl[4], nd[4];  // -L * log2(e) and -D per column
            if constexpr (C::KV) {
              const float4 a = vl2[h * 8 + c4], d4 = vd[h * 8 + c4];
              nl[0] = a.x; nl[1] = a.y; nl[2] = a.z; nl[3] = a.w;
              nd[0] = d4.x; nd[1] = d4.y; nd[2] = d4.z; nd[3] = d4.w;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                nl[e] = l2_row;
                nd[e] = d_row;
              }
            }
            float pv[4], ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = c4 * 4 + e;
              float pe = ex2(fmaf(__uint_as_float(rs[c]), sl2, nl[e]));
              if (need_mask) {
                const int col = col0 + h * 32 + c;
                const bool masked = (MODE == 0) ? (row > col) : (col >= p.Nk || col > row);
                if (masked) pe = 0.f;
              }
              pv[e] = pe;
              ds[e] = pe * (__uint_as_float(rd[c]) + nd[e]);
            }
            pk[c4 * 2] = pack_bf16x2(pv[0], pv[1]);
            pk[c4 * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
            dk[c4 * 2] = pack_bf16x2(ds[0], ds[1]);
            dk[c4 * 2 + 1] = pack_bf16x2(ds[2], ds[3]);
          }
        } else {
  #pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            // -L * log2(e) and -D of the four streamed rows (MODE 0) or of this row (MODE 1).
            uint64_t nl[2], nd[2];
            if constexpr (C::KV) {
              const float4 a = vl2[h * 8 + c4], d4 = vd[h * 8 + c4];
              nl[0] = f2_pack(a.x, a.y);
              nl[1] = f2_pack(a.z, a.w);
              nd[0] = f2_pack(d4.x, d4.y);
              nd[1] = f2_pack(d4.z, d4.w);
            } else {
              nl[0] = nl[1] = f2_pack(l2_row, l2_row);
              nd[0] = nd[1] = f2_pack(d_row, d_row);
            }
  #pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int c = c4 * 4 + e2 * 2;
              const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])), sl2x2, nl[e2]));
              float p0 = ex2(x.x), p1 = ex2(x.y);
              if (need_mask) {
                const int col = col0 + h * 32 + c;
                const bool m0 = (MODE == 0) ? (CAUSAL && row > col) : (col >= p.Nk || (CAUSAL && col > row));
                const bool m1 = (MODE == 0) ? (CAUSAL && row > col + 1) : (col + 1 >= p.Nk || (CAUSAL && col + 1 > row));
                if (m0) p0 = 0.f;
                if (m1) p1 = 0.f;
              }
              const uint64_t pp = f2_pack(p0, p1);
              const float2 ds = f2_unpack(
                  f2_mul(pp, f2_add(f2_pack(__uint_as_float(rd[c]), __uint_as_float(rd[c + 1])), nd[e2])));
              pk[c4 * 2 + e2] = pack_bf16x2(p0, p1);
              dk[c4 * 2 + e2] = pack_bf16x2(ds.x, ds.y);
            }
          }
        }
        // Chunk h's bf16 pairs land in columns [16 h, 16 h + 16) of the
        // buffer, after chunk h's fp32 values have been read (and before the
        // next chunk's fp32 columns [32 (h + 1), ...) are read).
        if constexpr (C::KV) tmem_st16(tmem + lane_off + C::TM_S + b * C::BS + h * 16, pk);
        tmem_st16(tmem + lane_off + C::TM_DP + b * C::BS + h * 16, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar.p_ready(b));
    }
    if (!ok) break;
    pos += n;
    // Read the unit's accumulators out.
    ok = warp_wait_bar(bar.out_done(), uk & 1, g, kStatusTimeoutSoftmax);
    if (!ok) break;
    tc_fence_after();
    const bool second = C::KV && b == 1;
    const uint32_t acc = tmem + lane_off + C::TM_OUT + (second ? C::OUTW : 0);
    __nv_bfloat16* out = second ? p.out1 : p.out0;
    const float f = second ? 1.f : p.scale;  // dK and dQ carry the softmax scale
    const uint64_t f2 = f2_pack(f, f);
    const int n_rows = (MODE == 0) ? p.Nk : p.Nq;  // rows of the fixed operand (and of the outputs)
    __nv_bfloat16* orow;
    if constexpr (STRIDED) {
      const long long* os = second ? p.out1_s : p.out0_s;
      orow = out + (w.bh / p.H) * os[0] + (w.bh % p.H) * os[1] + static_cast<long long>(row) * os[2];
    } else {
      orow = out + (static_cast<size_t>(w.bh) * n_rows + row) * D;
    }
    const bool empty = n <= 0;  // no streamed tile reached these rows: the gradients are zero
#pragma unroll 1
    for (int c = 0; c < C::OUTW / 32; ++c) {
      if (!C::KV && (c & 1) != b) continue;
      uint32_t v[32];
      tmem_ld32(acc + c * 32, v);
      tmem_wait_ld(v);
      if (empty) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 y = f2_unpack(f2_mul(f2_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), f2));
        packed[i] = pack_bf16x2(y.x, y.y);
      }
      if (row < n_rows) {
        uint4* dst = reinterpret_cast<uint4*>(orow + w.half * C::OUTW + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
      }
    }
    tc_fence_before();
    warp_arrive(bar.out_free());
  }
}

// ------------------------------------------------------------------ kernel
template <int D, int MODE, bool CAUSAL, bool STRIDED>
__global__ void __launch_bounds__(BwdCfg<D, MODE>::THREADS, 1)
    fa_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
                     const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                     const BwdParams p) {
  using C = BwdCfg<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const BwdBars<D, MODE> bar{base + C::OFF_MISC};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_ABORT);

  if (threadIdx.x == 0) {
    mbar_init(bar.fix_full(), 1);
    mbar_init(bar.fix_empty(), 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(bar.st_full(i), 1);
      mbar_init(bar.st_empty(i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.s_full(b), 1);
      mbar_init(bar.p_ready(b), 4);
    }
    mbar_init(bar.out_done(), 1);
    mbar_init(bar.out_free(), 8);
    mbar_init(bar.drain(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::LOAD_WARP && lane == 0) {
    prefetch_tmap(&tm_a1);
    prefetch_tmap(&tm_a2);
    prefetch_tmap(&tm_b1);
    prefetch_tmap(&tm_b2);
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

  if (warp < 8) {
    bwd_elementwise<D, MODE, CAUSAL, STRIDED>(p, bar, gbase, tmem, warp >> 2, warp & 3, lane, g);
  } else if (warp == C::MMA_WARP) {
    bwd_mma<D, MODE, CAUSAL>(p, bar, base, tmem, g);
  } else if (warp == C::LOAD_WARP && lane == 0) {
    bwd_producer<D, MODE, CAUSAL, STRIDED>(&tm_a1, &tm_a2, &tm_b1, &tm_b2, p, bar, base, g);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ------------------------------------------------------------------ preprocessing
// Writes -D[row] = -sum_c dO[row, c] * O[row, c] (fp32) and -L[row] * log2(e)
// (negated so that the elementwise step adds them with paired fp32 FMAs),
// for query rows [0, n_pad) of every head (N = the query rows; O and dO are
// read through their strides, L is contiguous [BH][N]); rows >= N get 0 and
// -inf, so their P is exactly 0.  Each row is read by D / 8 lanes,
// 16 bytes per lane.
struct PrepStrides {
  long long o[3];   // element strides {batch, head, row} of O
  long long d[3];   // ... of dO
};

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                          const __nv_bfloat16* __restrict__ dout,
                                                          const float* __restrict__ lse, float* __restrict__ l2,
                                                          float* __restrict__ dsum, int BH, int H, int N, int n_pad,
                                                          const PrepStrides st) {
  constexpr int CPR = D / 8;            // 16-byte chunks per row
  constexpr int RPW = 32 / CPR;         // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / CPR, chunk = lane % CPR;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long total = static_cast<long long>(BH) * n_pad;
  for (long long r0 = (static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5)) * RPW; r0 < total;
       r0 += warps * RPW) {
    const long long rr = r0 + sub;
    const int bh = static_cast<int>(rr / n_pad);
    const int i = static_cast<int>(rr % n_pad);
    const bool valid = rr < total && i < N;
    float acc = 0.f;
    if (valid) {
      const long long hb = bh / H, hh = bh % H;
      const long long oo = hb * st.o[0] + hh * st.o[1] + i * st.o[2] + chunk * 8;
      const long long od = hb * st.d[0] + hh * st.d[1] + i * st.d[2] + chunk * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(o + oo);
      const uint4 c = *reinterpret_cast<const uint4*>(dout + od);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cv[e]));
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int m = CPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (chunk == 0 && rr < total) {
      dsum[rr] = valid ? -acc : 0.f;
      l2[rr] = valid ? -lse[static_cast<size_t>(bh) * N + i] * 1.4426950408889634f : -INFINITY;
    }
  }
}

}  // namespace fa

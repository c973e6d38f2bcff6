// Host launcher of the tensor-core kernel for one head dimension.  Included by
// the per-head-dimension translation units fa_tc_d<D>.cu.
#pragma once

#include <atomic>
#include <cmath>

#include "fa_fwd_tc.cuh"
#include "fa_internal.h"

namespace fa {

template <int D, bool CAUSAL, bool STRIDED, int NQ = TcCfg<D>::NQT, int VAR = kVarBf16>
int launch_tc_impl(const FwdArgs& a, const LaunchCtx& ctx) {
  using C = TcCfg<D, NQ, VAR>;
  static_assert(VAR == kVarBf16 || !STRIDED, "e4m3 and pair kernels take contiguous tensors");
  auto kernel = fa_fwd_tc_kernel<D, CAUSAL, STRIDED, NQ, VAR>;
  if constexpr (C::SPLIT_REGS) {
    // The warpgroups re-split the registers the block was launched with
    // (setmaxnreg); the split is sized for exactly LAUNCH_REGS per thread.  A
    // build with any other count would make setmaxnreg.inc wait forever, so it
    // is refused here.
    // Queried once per instantiation; concurrent first calls may both query
    // (the same value), and the atomic keeps that free of a data race.
    static std::atomic<int> checked_regs{-1};
    int regs = checked_regs.load(std::memory_order_relaxed);
    if (regs < 0) {
      cudaFuncAttributes attr;
      cudaError_t ea = cudaFuncGetAttributes(&attr, kernel);
      if (ea != cudaSuccess) return static_cast<int>(ea);
      regs = attr.numRegs;
      checked_regs.store(regs, std::memory_order_relaxed);
    }
    if (regs != C::LAUNCH_REGS) return -2;
  }
  // The attribute is per function and device; setting it again is cheap and idempotent.
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return static_cast<int>(e);
  CUtensorMap mq, mk, mv, mo;
  // O is stored in boxes of 32 rows x 32 columns (one correction warp, one chunk), 64-byte swizzle.
  if constexpr (STRIDED) {
    if (encode_bf16_map4(&mq, a.q, a.B, a.H, a.Nq, D, a.qs, C::RC, C::BQ, C::SWB) != 0) return -1;
    if (encode_bf16_map4(&mk, a.k, a.B, a.H, a.Nk, D, a.ks, C::RC, C::BK, C::SWB) != 0) return -1;
    if (encode_bf16_map4(&mv, a.v, a.B, a.H, a.Nk, D, a.vs, C::RC, C::BK, C::SWB) != 0) return -1;
    if (encode_bf16_map4(&mo, a.o, a.B, a.H, a.Nq, D, a.os, 32, 32, 64) != 0) return -1;
  } else if constexpr (VAR == kVarE4m3) {
    // e4m3 Q, K, V as bytes; O is bf16 as in every other kernel.
    if (encode_e4m3_map(&mq, a.q, a.B * a.H, a.Nq, D, C::RC, C::BQ, C::SWB) != 0) return -1;
    if (encode_e4m3_map(&mk, a.k, a.B * a.H, a.Nk, D, C::RC, C::BK, C::SWB) != 0) return -1;
    if (encode_e4m3_map(&mv, a.v, a.B * a.H, a.Nk, D, C::RC, C::BK, C::SWB) != 0) return -1;
    if (encode_bf16_map(&mo, a.o, a.B * a.H, a.Nq, D, 32, 32, 64) != 0) return -1;
  } else {
    // K boxes cover a pair CTA's K_ROWS keys; V boxes all BK keys (of one 64-column region).
    if (encode_bf16_map(&mq, a.q, a.B * a.H, a.Nq, D, C::RC, C::BQ, C::SWB) != 0) return -1;
    if (encode_bf16_map(&mk, a.k, a.B * a.H, a.Nk, D, C::RC, C::K_ROWS, C::SWB) != 0) return -1;
    if (encode_bf16_map(&mv, a.v, a.B * a.H, a.Nk, D, C::RC, C::BK, C::SWB) != 0) return -1;
    if (encode_bf16_map(&mo, a.o, a.B * a.H, a.Nq, D, 32, 32, 64) != 0) return -1;
  }
  TcParams p;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.H = a.H;
  p.BH = a.B * a.H;
  p.n_kv = (a.Nk + C::BK - 1) / C::BK;
  p.n_qb = (a.Nq + C::BQ * C::UNIT_TILES - 1) / (C::BQ * C::UNIT_TILES);
  p.total_units = p.BH * p.n_qb;
  if constexpr (VAR == kVarE4m3) {
    // Logits of the dequantised inputs: (qf Q8)(kf K8)^T * scale.
    p.scale_log2 = a.scale * a.q_descale * a.k_descale * 1.4426950408889634f;
    p.o_scale = a.v_descale;
  } else {
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.o_scale = 1.f;
  }
  p.lse = a.lse;
  p.status = ctx.status;
  p.limit_ns = ctx.limit_ns;
  if constexpr (C::PAIR) {
    // Clusters of two CTAs, one work unit (256 rows) per cluster at a time:
    // as many clusters as can be resident together (clusters are placed
    // within a GPC, so that may be fewer than SMs / 2), found once.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> max_clusters{-1};
    int mc = max_clusters.load(std::memory_order_relaxed);
    if (mc < 0) {
      cfg.gridDim = dim3(2 * (ctx.num_sms / 2), 1, 1);
      cudaError_t eo = cudaOccupancyMaxActiveClusters(&mc, kernel, &cfg);
      if (eo != cudaSuccess) return static_cast<int>(eo);
      if (mc < 1) return -3;
      max_clusters.store(mc, std::memory_order_relaxed);
    }
    const int clusters = p.total_units < mc ? p.total_units : mc;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    return static_cast<int>(cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mo, p));
  } else {
    const int grid = p.total_units < ctx.num_sms ? p.total_units : ctx.num_sms;
    kernel<<<grid, C::THREADS, C::SMEM_ALLOC, ctx.stream>>>(mq, mk, mv, mo, p);
    return static_cast<int>(cudaGetLastError());
  }
}

}  // namespace fa

namespace fa {

// At d <= 128 the single-tile kernel (128-row work units, S double-buffered)
// runs when even 128-row units would not outnumber the SMs: there the
// two-tile kernel leaves most SMs idle and the one-tile chain per key tile is
// shorter.
template <int D, bool CAUSAL, bool STRIDED, int VAR = kVarBf16>
int launch_tc_sized(const FwdArgs& a, const LaunchCtx& ctx) {
  if constexpr (D <= 128) {
    const long long units = static_cast<long long>(a.B) * a.H * ((a.Nq + 255) / 256);
    if (2 * units <= ctx.num_sms) return launch_tc_impl<D, CAUSAL, STRIDED, 1, VAR>(a, ctx);
  }
  return launch_tc_impl<D, CAUSAL, STRIDED, TcCfg<D>::NQT, VAR>(a, ctx);
}

}  // namespace fa

// Contiguous [B][H][N][d] tensors (3-D maps, the fast path), in fa_tc_d<D>.cu.
#define FA_DEFINE_TC_LAUNCHER(DIM)                                                                     \
  namespace fa {                                                                                       \
  int launch_tc_d##DIM(const FwdArgs& a, const LaunchCtx& ctx) {                                       \
    return a.causal ? launch_tc_sized<DIM, true, false>(a, ctx) : launch_tc_sized<DIM, false, false>(a, ctx); \
  }                                                                                                    \
  }

// Contiguous tensors at d = 256 on CTA pairs (cta_group::2), in fa_tc_d256.cu.
#define FA_DEFINE_TC_PAIR_LAUNCHER(DIM)                                                                \
  namespace fa {                                                                                       \
  int launch_tc_d##DIM(const FwdArgs& a, const LaunchCtx& ctx) {                                       \
    return a.causal ? launch_tc_impl<DIM, true, false, 1, kVarPair>(a, ctx)                            \
                    : launch_tc_impl<DIM, false, false, 1, kVarPair>(a, ctx);                          \
  }                                                                                                    \
  }

// Any strides with a contiguous d dimension (4-D maps), in fa_tc_d<D>_strided.cu.
#define FA_DEFINE_TC_STRIDED_LAUNCHER(DIM)                                                           \
  namespace fa {                                                                                     \
  int launch_tc_strided_d##DIM(const FwdArgs& a, const LaunchCtx& ctx) {                             \
    return a.causal ? launch_tc_sized<DIM, true, true>(a, ctx) : launch_tc_sized<DIM, false, true>(a, ctx); \
  }                                                                                                  \
  }

// e4m3 Q, K, V (contiguous), bf16 O, in fa_tc_fp8_d<D>.cu.
#define FA_DEFINE_TC_FP8_LAUNCHER(DIM)                                                                     \
  namespace fa {                                                                                           \
  int launch_tc_fp8_d##DIM(const FwdArgs& a, const LaunchCtx& ctx) {                                       \
    return a.causal ? launch_tc_sized<DIM, true, false, kVarE4m3>(a, ctx) : launch_tc_sized<DIM, false, false, kVarE4m3>(a, ctx); \
  }                                                                                                        \
  }

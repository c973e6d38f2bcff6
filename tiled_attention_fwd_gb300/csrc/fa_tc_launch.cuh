// Host launcher of the tensor-core kernel for one head dimension.  Included by
// the per-head-dimension translation units fa_tc_d<D>.cu.
#pragma once

#include <cmath>

#include "fa_fwd_tc.cuh"
#include "fa_internal.h"

namespace fa {

template <int D, bool CAUSAL>
int launch_tc_impl(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N, float scale,
                   const LaunchCtx& ctx) {
  using C = TcCfg<D>;
  auto kernel = fa_fwd_tc_kernel<D, CAUSAL>;
  if constexpr (C::SPLIT_REGS) {
    // The warpgroups re-split the registers the block was launched with
    // (setmaxnreg); the split is sized for exactly LAUNCH_REGS per thread.  A
    // build with any other count would make setmaxnreg.inc wait forever, so it
    // is refused here.
    static int checked_regs = -1;
    if (checked_regs < 0) {
      cudaFuncAttributes attr;
      cudaError_t ea = cudaFuncGetAttributes(&attr, kernel);
      if (ea != cudaSuccess) return static_cast<int>(ea);
      checked_regs = attr.numRegs;
    }
    if (checked_regs != C::LAUNCH_REGS) return -2;
  }
  // The attribute is per function and device; setting it again is cheap and idempotent.
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return static_cast<int>(e);
  CUtensorMap mq, mk, mv;
  if (encode_bf16_map(&mq, q, BH, N, D, C::RC, C::BQ, C::SWB) != 0) return -1;
  if (encode_bf16_map(&mk, k, BH, N, D, C::RC, C::BK, C::SWB) != 0) return -1;
  if (encode_bf16_map(&mv, v, BH, N, D, C::RC, C::BK, C::SWB) != 0) return -1;
  TcParams p;
  p.N = N;
  p.BH = BH;
  p.n_kv = (N + C::BK - 1) / C::BK;
  p.n_qb = (N + C::BQ * C::NQT - 1) / (C::BQ * C::NQT);
  p.total_units = BH * p.n_qb;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = ctx.status;
  p.limit_ns = ctx.limit_ns;
  const int grid = p.total_units < ctx.num_sms ? p.total_units : ctx.num_sms;
  kernel<<<grid, C::THREADS, C::SMEM_ALLOC, ctx.stream>>>(mq, mk, mv, p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace fa

#define FA_DEFINE_TC_LAUNCHER(DIM)                                                                         \
  namespace fa {                                                                                           \
  int launch_tc_d##DIM(bool causal, const void* q, const void* k, const void* v, void* o, float* lse, int BH, \
                       int N, float scale, const LaunchCtx& ctx) {                                         \
    return causal ? launch_tc_impl<DIM, true>(q, k, v, o, lse, BH, N, scale, ctx)                          \
                  : launch_tc_impl<DIM, false>(q, k, v, o, lse, BH, N, scale, ctx);                        \
  }                                                                                                        \
  }

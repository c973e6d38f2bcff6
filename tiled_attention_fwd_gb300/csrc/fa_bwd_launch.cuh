// Host launcher of the backward pass for one head dimension.  Included by the
// per-head-dimension translation units fa_bwd_d<D>.cu.
#pragma once

#include "fa_bwd_tc.cuh"
#include "fa_internal.h"

namespace fa {

template <int D, int MODE, bool CAUSAL>
int launch_bwd_main(const BwdArgs& a, const LaunchCtx& ctx) {
  using C = BwdCfg<D, MODE>;
  auto kernel = fa_bwd_tc_kernel<D, MODE, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return static_cast<int>(e);
  // MODE 0: fixed K, V; streamed Q, dO.  MODE 1: fixed Q, dO; streamed K, V.
  const void* a1 = MODE == 0 ? a.k : a.q;
  const void* a2 = MODE == 0 ? a.v : a.dout;
  const void* b1 = MODE == 0 ? a.q : a.k;
  const void* b2 = MODE == 0 ? a.dout : a.v;
  CUtensorMap m1, m2, m3, m4;
  if (encode_bf16_map(&m1, a1, a.BH, a.N, D, C::RC, C::BM, C::SWB) != 0) return -1;
  if (encode_bf16_map(&m2, a2, a.BH, a.N, D, C::RC, C::BM, C::SWB) != 0) return -1;
  if (encode_bf16_map(&m3, b1, a.BH, a.N, D, C::RC, C::BS, C::SWB) != 0) return -1;
  if (encode_bf16_map(&m4, b2, a.BH, a.N, D, C::RC, C::BS, C::SWB) != 0) return -1;
  BwdParams p;
  p.N = a.N;
  p.BH = a.BH;
  p.n_pad = a.n_pad;
  p.n_m = (a.N + C::BM - 1) / C::BM;
  p.n_s = (a.N + C::BS - 1) / C::BS;
  p.total_units = a.BH * p.n_m;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.l2 = a.l2;
  p.dsum = a.dsum;
  p.out0 = static_cast<__nv_bfloat16*>(MODE == 0 ? a.dk : a.dq);
  p.out1 = static_cast<__nv_bfloat16*>(a.dv);
  p.status = ctx.status;
  p.limit_ns = ctx.limit_ns;
  const int grid = p.total_units < ctx.num_sms ? p.total_units : ctx.num_sms;
  kernel<<<grid, C::THREADS, C::SMEM_ALLOC, ctx.stream>>>(m1, m2, m3, m4, p);
  return static_cast<int>(cudaGetLastError());
}

template <int D>
int launch_bwd_impl(const BwdArgs& a, const LaunchCtx& ctx) {
  constexpr int RPW = 32 / (D / 8);  // rows per warp step of the preprocessing kernel
  const long long rows = static_cast<long long>(a.BH) * a.n_pad;
  const long long blocks_needed = (rows + 8 * RPW - 1) / (8 * RPW);
  const long long cap = 8LL * ctx.num_sms;
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  fa_bwd_prep_kernel<D><<<grid, 256, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.l2, a.dsum, a.BH,
      a.N, a.n_pad);
  int e = static_cast<int>(cudaGetLastError());
  if (e != 0) return e;
  e = a.causal ? launch_bwd_main<D, 0, true>(a, ctx) : launch_bwd_main<D, 0, false>(a, ctx);
  if (e != 0) return e;
  return a.causal ? launch_bwd_main<D, 1, true>(a, ctx) : launch_bwd_main<D, 1, false>(a, ctx);
}

}  // namespace fa

#define FA_DEFINE_BWD_LAUNCHER(DIM)                                                     \
  namespace fa {                                                                        \
  int launch_bwd_d##DIM(const BwdArgs& a, const LaunchCtx& ctx) { return launch_bwd_impl<DIM>(a, ctx); } \
  }

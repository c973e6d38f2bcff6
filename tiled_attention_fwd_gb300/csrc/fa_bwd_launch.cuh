// Host launcher of the backward pass for one head dimension.  Included by the
// per-head-dimension translation units fa_bwd_d<D>.cu (contiguous tensors) and
// fa_bwd_d<D>_strided.cu (any strides with a contiguous head dimension).
#pragma once

#include "fa_bwd_tc.cuh"
#include "fa_internal.h"

namespace fa {

// Tensor-map descriptor of tensor t (0 q, 1 k, 2 v, 4 dO) with `rows` rows per head and a box of box_rows rows.
template <int D, int MODE, bool STRIDED>
int bwd_map(CUtensorMap* m, const BwdArgs& a, const void* ptr, int t, int rows, int box_rows) {
  using C = BwdCfg<D, MODE>;
  if constexpr (STRIDED) return encode_bf16_map4(m, ptr, a.B, a.H, rows, D, a.st[t], C::RC, box_rows, C::SWB);
  return encode_bf16_map(m, ptr, a.B * a.H, rows, D, C::RC, box_rows, C::SWB);
}

template <int D, int MODE, bool CAUSAL, bool STRIDED>
int launch_bwd_main(const BwdArgs& a, const LaunchCtx& ctx) {
  using C = BwdCfg<D, MODE>;
  auto kernel = fa_bwd_tc_kernel<D, MODE, CAUSAL, STRIDED>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return static_cast<int>(e);
  // MODE 0: fixed K, V (Nk rows); streamed Q, dO (Nq rows).
  // MODE 1: fixed Q, dO (Nq rows); streamed K, V (Nk rows).
  const int n_fix = MODE == 0 ? a.Nk : a.Nq, n_str = MODE == 0 ? a.Nq : a.Nk;
  CUtensorMap m1, m2, m3, m4;
  if (bwd_map<D, MODE, STRIDED>(&m1, a, MODE == 0 ? a.k : a.q, MODE == 0 ? 1 : 0, n_fix, C::BM) != 0) return -1;
  if (bwd_map<D, MODE, STRIDED>(&m2, a, MODE == 0 ? a.v : a.dout, MODE == 0 ? 2 : 4, n_fix, C::BM) != 0) return -1;
  if (bwd_map<D, MODE, STRIDED>(&m3, a, MODE == 0 ? a.q : a.k, MODE == 0 ? 0 : 1, n_str, C::BS) != 0) return -1;
  if (bwd_map<D, MODE, STRIDED>(&m4, a, MODE == 0 ? a.dout : a.v, MODE == 0 ? 4 : 2, n_str, C::BS) != 0) return -1;
  BwdParams p;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.H = a.H;
  p.BH = a.B * a.H;
  p.n_pad = a.n_pad;
  p.n_m = (n_fix + C::BM - 1) / C::BM;
  p.n_s = (n_str + C::BS - 1) / C::BS;
  p.total_units = p.BH * p.n_m * C::HALVES;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.l2 = a.l2;
  p.dsum = a.dsum;
  p.out0 = static_cast<__nv_bfloat16*>(MODE == 0 ? a.dk : a.dq);
  p.out1 = static_cast<__nv_bfloat16*>(a.dv);
  for (int i = 0; i < 3; ++i) {
    p.out0_s[i] = a.st[MODE == 0 ? 6 : 5][i];
    p.out1_s[i] = a.st[7][i];
  }
  p.status = ctx.status;
  p.limit_ns = ctx.limit_ns;
  const int grid = p.total_units < ctx.num_sms ? p.total_units : ctx.num_sms;
  kernel<<<grid, C::THREADS, C::SMEM_ALLOC, ctx.stream>>>(m1, m2, m3, m4, p);
  return static_cast<int>(cudaGetLastError());
}

template <int D, bool STRIDED>
int launch_bwd_impl(const BwdArgs& a, const LaunchCtx& ctx) {
  constexpr int RPW = 32 / (D / 8);  // rows per warp step of the preprocessing kernel
  const long long rows = static_cast<long long>(a.B) * a.H * a.n_pad;
  const long long blocks_needed = (rows + 8 * RPW - 1) / (8 * RPW);
  const long long cap = 8LL * ctx.num_sms;
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  PrepStrides ps;
  for (int i = 0; i < 3; ++i) {
    ps.o[i] = a.st[3][i];
    ps.d[i] = a.st[4][i];
  }
  fa_bwd_prep_kernel<D><<<grid, 256, 0, ctx.stream>>>(static_cast<const __nv_bfloat16*>(a.o),
                                                      static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.l2, a.dsum,
                                                      a.B * a.H, a.H, a.Nq, a.n_pad, ps);
  int e = static_cast<int>(cudaGetLastError());
  if (e != 0) return e;
  // The dK/dV and dQ kernels are independent once the preprocessing is done:
  // the dQ kernel runs on a second stream forked after the preprocessing, so
  // that its CTAs take the SMs the dK/dV kernel frees at its tail; the
  // caller's stream then waits for it (ordered on `stream` like one kernel).
  LaunchCtx q_ctx = ctx;
  if (ctx.side != nullptr) {
    if (cudaEventRecord(ctx.ev_fork, ctx.stream) != cudaSuccess ||
        cudaStreamWaitEvent(ctx.side, ctx.ev_fork, 0) != cudaSuccess)
      return -1;
    q_ctx.stream = ctx.side;
  }
  e = a.causal ? launch_bwd_main<D, 0, true, STRIDED>(a, ctx) : launch_bwd_main<D, 0, false, STRIDED>(a, ctx);
  if (e != 0) return e;
  e = a.causal ? launch_bwd_main<D, 1, true, STRIDED>(a, q_ctx) : launch_bwd_main<D, 1, false, STRIDED>(a, q_ctx);
  if (e != 0) return e;
  if (ctx.side != nullptr) {
    if (cudaEventRecord(ctx.ev_join, ctx.side) != cudaSuccess ||
        cudaStreamWaitEvent(ctx.stream, ctx.ev_join, 0) != cudaSuccess)
      return -1;
  }
  return 0;
}

}  // namespace fa

#define FA_DEFINE_BWD_LAUNCHER(DIM)                                                              \
  namespace fa {                                                                                 \
  int launch_bwd_d##DIM(const BwdArgs& a, const LaunchCtx& ctx) { return launch_bwd_impl<DIM, false>(a, ctx); } \
  }

#define FA_DEFINE_BWD_STRIDED_LAUNCHER(DIM)                                                      \
  namespace fa {                                                                                 \
  int launch_bwd_strided_d##DIM(const BwdArgs& a, const LaunchCtx& ctx) {                        \
    return launch_bwd_impl<DIM, true>(a, ctx);                                                   \
  }                                                                                              \
  }

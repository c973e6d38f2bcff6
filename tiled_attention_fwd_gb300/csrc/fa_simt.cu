// fp32 forward pass on the CUDA cores (no tensor cores), for small fp32
// problems and any head dimension 1 <= d <= 256.
//
// The tiled kernel of "Writing a FlashAttention kernel in Metal" (section
// "Shared-memory tiling") stages one K/V tile in shared memory per block and
// lets every thread run the online-softmax recurrence for its own query.
// Here a block of 4 warps owns 16 query rows (4 per warp) and stages 32 keys
// per tile; within a warp, lane j scores key j of the tile against the row
// (so the row max and sum are warp shuffles), the probabilities go through
// shared memory, and lane c accumulates output columns c, c+32, ... of the
// warp's rows (each V element read once for all of them).  State (m, l, O) is fp32, as in the
// FlashAttention-2 forward of "FlashAttention-2 from PyTorch to Triton".
#include <cmath>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kSimtWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kSimtRows = kSimtWarps * kRowsPerWarp;  // query rows per block
constexpr int kSimtKeys = 32;                          // keys per K/V tile

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// DPL: output columns per lane (ceil(d / 32) rounded up to a power of two).
template <int DPL, bool CAUSAL>
__global__ void __launch_bounds__(kSimtWarps * 32)
    fa_fwd_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                       float* __restrict__ o, float* __restrict__ lse, int N, int d, float scale) {
  extern __shared__ float sm[];
  const int ks = d | 1;  // odd row stride of the K tile: lane-strided reads hit distinct banks
  float* qs = sm;                            // [kSimtRows][d]
  float* kt = qs + kSimtRows * d;            // [kSimtKeys][ks]
  float* vt = kt + kSimtKeys * ks;           // [kSimtKeys][d]
  float* pw = vt + kSimtKeys * d;            // [kSimtRows][kSimtKeys]: probabilities of the current tile
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const size_t head = static_cast<size_t>(blockIdx.y) * N;
  const int row_base = blockIdx.x * kSimtRows;

  for (int i = tid; i < kSimtRows * d; i += blockDim.x) {
    const int r = row_base + i / d;
    qs[i] = r < N ? q[(head + r) * d + i % d] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[i][t] = 0.f;
  }

  // Key tiles wholly in the future of every row of the block are skipped.
  int kend = N;
  if (CAUSAL) kend = min(N, row_base + kSimtRows);
  for (int t0 = 0; t0 < kend; t0 += kSimtKeys) {
    __syncthreads();  // the previous tile has been read by every warp
    for (int i = tid; i < kSimtKeys * d; i += blockDim.x) {
      const int j = i / d, c = i % d;
      const int key = t0 + j;
      const bool in = key < N;
      kt[j * ks + c] = in ? k[(head + key) * d + c] : 0.f;
      vt[i] = in ? v[(head + key) * d + c] : 0.f;
    }
    __syncthreads();
    // Scores and softmax statistics of the warp's rows (lane = key of the
    // tile); each row's probabilities go to the warp's slice of pw.
    const int key = t0 + lane;
    float alpha[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int rl = warp * kRowsPerWarp + i;
      const int row = row_base + rl;
      const float* qr = qs + rl * d;
      const float* kr = kt + lane * ks;
      float s0 = 0.f, s1 = 0.f;  // two partial sums for a shorter dependency chain
      int c = 0;
      for (; c + 1 < d; c += 2) {
        s0 = fmaf(qr[c], kr[c], s0);
        s1 = fmaf(qr[c + 1], kr[c + 1], s1);
      }
      if (c < d) s0 = fmaf(qr[c], kr[c], s0);
      float sc = (s0 + s1) * scale;
      const bool valid = key < N && (!CAUSAL || key <= row);
      sc = valid ? sc : -INFINITY;
      const float m_new = fmaxf(m[i], warp_max(sc));
      const float base = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[i] = expf(m[i] - base);  // 0 on the first tile (m = -inf)
      const float pj = expf(sc - base);  // 0 for masked keys
      l[i] = l[i] * alpha[i] + warp_sum(pj);
      pw[(warp * kRowsPerWarp + i) * kSimtKeys + lane] = pj;
      m[i] = m_new;
    }
    __syncwarp();
    // O += P V: each V element is read once for the warp's rows; the
    // probabilities are shared-memory broadcasts.
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
      for (int t = 0; t < DPL; ++t) acc[i][t] *= alpha[i];
    const float* pr = pw + warp * kRowsPerWarp * kSimtKeys;
#pragma unroll 4
    for (int j = 0; j < kSimtKeys; ++j) {
      const float* vr = vt + j * d;
#pragma unroll
      for (int t = 0; t < DPL; ++t) {
        const int c = lane + 32 * t;
        const float vv = c < d ? vr[c] : 0.f;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) acc[i][t] = fmaf(pr[i * kSimtKeys + j], vv, acc[i][t]);
      }
    }
    __syncwarp();  // pw is rewritten by the next tile
  }

#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int row = row_base + warp * kRowsPerWarp + i;
    if (row >= N) continue;
    const float inv_l = 1.f / l[i];
#pragma unroll
    for (int t = 0; t < DPL; ++t) {
      const int c = lane + 32 * t;
      if (c < d) o[(head + row) * d + c] = acc[i][t] * inv_l;
    }
    if (lane == 0) lse[head + row] = m[i] + logf(l[i]);
  }
}

// Whole-head variant for small problems (the fp32 workload has N = 128,
// d = 16).  K and V of the block's head are staged in shared memory once,
// each warp owns one query row, and the row's scores against all keys are
// formed before any exponential (lane j takes keys j, j + 32, ...), so the
// softmax is the plain two-pass one: row max, then exponentials and their
// sum; O is accumulated from the probabilities of all keys at once.  The
// tiled kernel above reloads K/V per tile and serialises one global-memory
// round trip, two block barriers and the online rescale per 32 keys, which at
// this size costs more than the arithmetic.
constexpr int kSmallWarps = 4;  // rows per block

size_t small_smem_bytes(int N, int d) {
  return sizeof(float) * (static_cast<size_t>(N) * (d | 1) + static_cast<size_t>(N) * d +
                          static_cast<size_t>(kSmallWarps) * N + static_cast<size_t>(kSmallWarps) * d);
}

template <int DPL, bool CAUSAL>
__global__ void __launch_bounds__(kSmallWarps * 32)
    fa_fwd_simt_small_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                             float* __restrict__ o, float* __restrict__ lse, int N, int d, float scale) {
  extern __shared__ float sm[];
  const int ks = d | 1;  // odd row stride: lane-strided reads of K hit distinct banks
  float* kt = sm;                                  // [N][ks]
  float* vt = kt + static_cast<size_t>(N) * ks;    // [N][d]
  float* pw = vt + static_cast<size_t>(N) * d;     // [kSmallWarps][N]: the row's scores, then probabilities
  float* qw = pw + kSmallWarps * N;                // [kSmallWarps][d]: the row of Q
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const size_t head = static_cast<size_t>(blockIdx.y) * N;
  const int row = blockIdx.x * kSmallWarps + warp;

  const float* kh = k + head * d;
  const float* vh = v + head * d;
  for (int i = tid; i < N * d; i += blockDim.x) {
    const int j = i / d, c = i - j * d;
    kt[j * ks + c] = kh[i];
    vt[i] = vh[i];
  }
  float* qr = qw + warp * d;
  if (row < N)
    for (int c = lane; c < d; c += 32) qr[c] = q[(head + row) * d + c];
  __syncthreads();
  if (row >= N) return;

  const int kend = CAUSAL ? row + 1 : N;  // keys this row sees
  float* pr = pw + warp * N;
  // Scores, and the row max.
  float mx = -INFINITY;
  for (int key = lane; key < kend; key += 32) {
    const float* kr = kt + key * ks;
    float s0 = 0.f, s1 = 0.f;
    int c = 0;
    for (; c + 1 < d; c += 2) {
      s0 = fmaf(qr[c], kr[c], s0);
      s1 = fmaf(qr[c + 1], kr[c + 1], s1);
    }
    if (c < d) s0 = fmaf(qr[c], kr[c], s0);
    const float sc = (s0 + s1) * scale;
    pr[key] = sc;
    mx = fmaxf(mx, sc);
  }
  mx = warp_max(mx);
  // Probabilities and their sum (every row sees key 0, so mx is finite).
  float sum = 0.f;
  for (int key = lane; key < kend; key += 32) {
    const float p = expf(pr[key] - mx);
    pr[key] = p;
    sum += p;
  }
  sum = warp_sum(sum);
  __syncwarp();
  // O = P V / l: lane c accumulates columns c, c + 32, ...
  float acc[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) acc[t] = 0.f;
  for (int key = 0; key < kend; ++key) {
    const float p = pr[key];
    const float* vr = vt + key * d;
#pragma unroll
    for (int t = 0; t < DPL; ++t) {
      const int c = lane + 32 * t;
      if (c < d) acc[t] = fmaf(p, vr[c], acc[t]);
    }
  }
  const float inv_l = 1.f / sum;
#pragma unroll
  for (int t = 0; t < DPL; ++t) {
    const int c = lane + 32 * t;
    if (c < d) o[(head + row) * d + c] = acc[t] * inv_l;
  }
  if (lane == 0) lse[head + row] = mx + logf(sum);
}

template <int DPL, bool CAUSAL>
int launch_simt_small(const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N, int d,
                      float scale, const LaunchCtx& ctx) {
  const size_t smem = small_smem_bytes(N, d);
  auto kernel = fa_fwd_simt_small_kernel<DPL, CAUSAL>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  const dim3 grid((N + kSmallWarps - 1) / kSmallWarps, BH);
  kernel<<<grid, kSmallWarps * 32, smem, ctx.stream>>>(q, k, v, o, lse, N, d, scale);
  return static_cast<int>(cudaGetLastError());
}

template <int DPL, bool CAUSAL>
int launch_simt_impl(const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N, int d,
                     float scale, const LaunchCtx& ctx) {
  const size_t smem = sizeof(float) * (static_cast<size_t>(kSimtRows) * d + static_cast<size_t>(kSimtKeys) * (d | 1) +
                                       static_cast<size_t>(kSimtKeys) * d +
                                       static_cast<size_t>(kSimtRows) * kSimtKeys);
  auto kernel = fa_fwd_simt_kernel<DPL, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return static_cast<int>(e);
  const dim3 grid((N + kSimtRows - 1) / kSimtRows, BH);
  kernel<<<grid, kSimtWarps * 32, smem, ctx.stream>>>(q, k, v, o, lse, N, d, scale);
  return static_cast<int>(cudaGetLastError());
}

// Problems whose K and V fit in 64 KB of shared memory take the whole-head kernel.
constexpr size_t kSmallSmemLimit = 64 * 1024;

template <bool CAUSAL>
int launch_simt_dpl(const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N, int d,
                    float scale, const LaunchCtx& ctx) {
  if (small_smem_bytes(N, d) <= kSmallSmemLimit) {
    if (d <= 32) return launch_simt_small<1, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
    if (d <= 64) return launch_simt_small<2, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
    if (d <= 128) return launch_simt_small<4, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
    return launch_simt_small<8, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
  }
  if (d <= 32) return launch_simt_impl<1, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
  if (d <= 64) return launch_simt_impl<2, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
  if (d <= 128) return launch_simt_impl<4, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
  return launch_simt_impl<8, CAUSAL>(q, k, v, o, lse, BH, N, d, scale, ctx);
}

}  // namespace

int launch_simt(bool causal, const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N,
                int d, float scale, const LaunchCtx& ctx) {
  return causal ? launch_simt_dpl<true>(q, k, v, o, lse, BH, N, d, scale, ctx)
                : launch_simt_dpl<false>(q, k, v, o, lse, BH, N, d, scale, ctx);
}

}  // namespace fa

// Internal interfaces between the C-ABI translation unit and the kernel
// translation units (one per head dimension, plus the fp32 SIMT kernel).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Everything a launcher needs besides the data pointers.
struct LaunchCtx {
  int* status;                    // device status word of the current device
  unsigned long long limit_ns;    // time limit of each device-side wait
  int num_sms;                    // SMs of the current device
  cudaStream_t stream;
};

// Encode a 3-D TMA descriptor over a contiguous bf16 [BH][N][D] tensor:
// dimensions {D, N, BH}, box {box_cols, box_rows, 1}, swizzle span
// `swizzle_bytes` (64 or 128).  Returns 0 on success.
int encode_bf16_map(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_cols, int box_rows,
                    int swizzle_bytes);

// Resolve the driver's tensor-map encoder (no device state, no allocation).  Returns 0 on success.
int load_tensor_map_encoder();

// Current time limit of the device-side waits (fa_set_wait_limit_ms), in nanoseconds.
unsigned long long wait_limit_ns();

// bf16 tensor-core forward for one head dimension; returns a cudaError_t-like
// code (0 = launched).  Defined in fa_tc_d<D>.cu.
int launch_tc_d32(bool causal, const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                  float scale, const LaunchCtx& ctx);
int launch_tc_d64(bool causal, const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                  float scale, const LaunchCtx& ctx);
int launch_tc_d128(bool causal, const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                   float scale, const LaunchCtx& ctx);
int launch_tc_d256(bool causal, const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                   float scale, const LaunchCtx& ctx);

// Arguments of the backward pass (device pointers; bf16 tensors [BH][N][d],
// lse fp32 [BH][N]; l2 and dsum are workspace vectors [BH][n_pad]).
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int BH;
  int N;
  int n_pad;       // N rounded up to a multiple of 64
  float scale;
  bool causal;
  float* l2;
  float* dsum;
};

// bf16 tensor-core backward (preprocessing, dK/dV kernel, dQ kernel) for one
// head dimension; returns a cudaError_t-like code.  Defined in fa_bwd_d<D>.cu.
int launch_bwd_d32(const BwdArgs& a, const LaunchCtx& ctx);
int launch_bwd_d64(const BwdArgs& a, const LaunchCtx& ctx);
int launch_bwd_d128(const BwdArgs& a, const LaunchCtx& ctx);

// fp32 SIMT forward, 1 <= d <= 256.  Defined in fa_simt.cu.
int launch_simt(bool causal, const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N,
                int d, float scale, const LaunchCtx& ctx);

}  // namespace fa

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
  // Backward pass: a second stream for the dQ kernel and the events that fork
  // it from and join it to `stream` (null: everything on `stream`).
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_join = nullptr;
};

// Arguments of the bf16 forward pass.  Each of q, k, v, o is addressed as
// ptr + b * stride[0] + h * stride[1] + row * stride[2] + c (elements; the d
// dimension is contiguous); q and o have Nq rows per head, k and v Nk.  lse
// is contiguous [B][H][Nq].
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B;
  int H;
  int Nq;
  int Nk;
  long long qs[3];
  long long ks[3];
  long long vs[3];
  long long os[3];
  float scale;
  bool causal;
  // e4m3 inputs only (fa_fwd_fp8): dequantisation factors, real x = factor * x8.
  float q_descale = 1.f;
  float k_descale = 1.f;
  float v_descale = 1.f;
};

// Contiguous [B][H][N][d] strides.
inline void contiguous_strides(long long* st, int H, int N, int d) {
  st[2] = d;
  st[1] = static_cast<long long>(N) * d;
  st[0] = static_cast<long long>(H) * N * d;
}

// Encode a 4-D TMA descriptor over a bf16 tensor addressed as above:
// dimensions {D, N, H, B}, byte strides from `stride` (elements: batch, head,
// row), box {box_cols, box_rows, 1, 1}, swizzle span `swizzle_bytes` (64 or
// 128).  Returns 0 on success.
int encode_bf16_map4(CUtensorMap* map, const void* ptr, int B, int H, int N, int D, const long long* stride,
                     int box_cols, int box_rows, int swizzle_bytes);

// Encode a 3-D TMA descriptor over a contiguous bf16 [BH][N][D] tensor:
// dimensions {D, N, BH}, box {box_cols, box_rows, 1}, swizzle span
// `swizzle_bytes` (64 or 128).  Returns 0 on success.
int encode_bf16_map(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_cols, int box_rows,
                    int swizzle_bytes);

// The same over a contiguous e4m3 [BH][N][D] tensor (one byte per element,
// encoded as 8-bit unsigned data; TMA moves bytes).
int encode_e4m3_map(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_cols, int box_rows,
                    int swizzle_bytes);

// Resolve the driver's tensor-map encoder (no device state, no allocation).  Returns 0 on success.
int load_tensor_map_encoder();

// Current time limit of the device-side waits (fa_set_wait_limit_ms), in nanoseconds.
unsigned long long wait_limit_ns();

// Diagnostic of the bounded waits (fa_selftest.cu): one block whose waits all
// expire after ctx.limit_ns; returns a cudaError_t-like code (0 = launched).
int launch_selftest_wait(const LaunchCtx& ctx);

// bf16 tensor-core forward for one head dimension; returns a cudaError_t-like
// code (0 = launched).  Defined in fa_tc_d<D>.cu.
int launch_tc_d32(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_d64(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_d128(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_d256(const FwdArgs& a, const LaunchCtx& ctx);
// e4m3 Q, K, V, bf16 O (contiguous tensors).  Defined in fa_tc_fp8_d<D>.cu.
int launch_tc_fp8_d64(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_fp8_d128(const FwdArgs& a, const LaunchCtx& ctx);
// The same for strided tensors (4-D tensor maps).  Defined in fa_tc_d<D>_strided.cu.
int launch_tc_strided_d32(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_strided_d64(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_strided_d128(const FwdArgs& a, const LaunchCtx& ctx);
int launch_tc_strided_d256(const FwdArgs& a, const LaunchCtx& ctx);

// Arguments of the backward pass (device pointers).  The bf16 tensors q, o,
// dout, dq have Nq rows per head, k, v, dk, dv Nk rows; tensor t's row i of
// (b, h) starts at element b * st[t][0] + h * st[t][1] + i * st[t][2] (the
// head dimension contiguous), t = 0 q, 1 k, 2 v, 3 o, 4 dout, 5 dq, 6 dk, 7 dv.
// lse is fp32 contiguous [B][H][Nq]; l2 and dsum are workspace vectors
// [B*H][n_pad].
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
  int B;
  int H;
  int Nq;
  int Nk;
  long long st[8][3];
  int n_pad;       // Nq rounded up to a multiple of 192
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
int launch_bwd_d256(const BwdArgs& a, const LaunchCtx& ctx);
// The same for strided tensors (4-D tensor maps).  Defined in fa_bwd_d<D>_strided.cu.
int launch_bwd_strided_d32(const BwdArgs& a, const LaunchCtx& ctx);
int launch_bwd_strided_d64(const BwdArgs& a, const LaunchCtx& ctx);
int launch_bwd_strided_d128(const BwdArgs& a, const LaunchCtx& ctx);
int launch_bwd_strided_d256(const BwdArgs& a, const LaunchCtx& ctx);

// Argument checks shared by the entry points (fa_api.cu); each returns FA_OK
// or the FA_* code of the first violated rule.  check_common: B, H, N >= 1,
// the index ranges, scale finite and > 0.  check_fwd_bf16: the pointers of
// the contiguous bf16 forward (non-null, 16-byte aligned; lse 4-byte aligned),
// check_common and a supported d.
int check_common(int B, int H, int N, int d, float scale);
int check_fwd_bf16(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H, int N,
                   int d, float scale);

// Read and clear fa_fwd_noalloc's status word on the current device
// (fa_noalloc.cu); FA_OK, FA_ERR_TIMEOUT or FA_ERR_CUDA.
int noalloc_take_status();

// Fill `a` for contiguous [B][H][N][d] tensors (N_q = N_k = N).
void contiguous_fwd_args(FwdArgs* a, const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int N, int d, float scale, int causal);

// The bf16 forward for d in {32, 64, 128, 256}; takes the contiguous kernels
// when every tensor is contiguous [B][H][N][d], else the strided ones; returns
// an FA_* code.  Defined in fa_api.cu.
int launch_tc(const FwdArgs& a, int d, const LaunchCtx& ctx);

// fp32 SIMT forward, 1 <= d <= 256.  Defined in fa_simt.cu.
int launch_simt(bool causal, const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N,
                int d, float scale, const LaunchCtx& ctx);

}  // namespace fa

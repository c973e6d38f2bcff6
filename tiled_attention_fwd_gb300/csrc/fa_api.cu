// C ABI of the library (declared in include/fa_gb300.h): argument checks,
// per-device state, TMA descriptor encoding, dispatch to the kernels.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kMaxDevices = 64;

constexpr int kHostChunks = 8;  // fa_fwd_host pipelines its copies and kernels over this many head chunks

// Streams and events of fa_fwd_host's copy/compute pipeline, created on first use.
struct HostPipeline {
  bool ready = false;
  std::mutex mutex;  // one enqueue sequence at a time (the events are reused)
  cudaStream_t s_in = nullptr;
  cudaStream_t s_out = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
  cudaEvent_t in[kHostChunks] = {};
  cudaEvent_t done[kHostChunks] = {};
};

// The backward pass's second stream: the dQ kernel runs on it beside the
// dK/dV kernel (both forked from and joined to the caller's stream).
struct BwdFork {
  bool ready = false;
  std::mutex mutex;  // one enqueue sequence at a time (the events are reused)
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
};

struct DeviceState {
  bool ready = false;
  int* status = nullptr;  // one device int, zeroed at creation
  int num_sms = 0;
  int cc_major = 0;
  int cc_minor = 0;
  HostPipeline pipe;
  BwdFork bwd;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<int> g_wait_limit_ms{2000};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device state of the current device, created on first use.
int current_device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    if (cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    if (s.cc_major != 10 || s.cc_minor != 3) return FA_ERR_ARCH;
    void* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemset(p, 0, 256) != cudaSuccess) return FA_ERR_CUDA;
    s.status = static_cast<int*>(p);
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.ready = true;
  }
  *out = &s;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


LaunchCtx make_ctx(const DeviceState& s, void* stream) {
  LaunchCtx c;
  c.status = s.status;
  c.limit_ns = static_cast<unsigned long long>(g_wait_limit_ms.load()) * 1000000ull;
  c.num_sms = s.num_sms;
  c.stream = static_cast<cudaStream_t>(stream);
  return c;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Create fa_fwd_host's streams and events for device state `s` (once).
int host_pipeline(DeviceState* s, HostPipeline** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  HostPipeline& hp = s->pipe;
  if (!hp.ready) {
    if (cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.join, cudaEventDisableTiming) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int i = 0; i < kHostChunks; ++i)
      if (cudaEventCreateWithFlags(&hp.in[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.done[i], cudaEventDisableTiming) != cudaSuccess)
        return FA_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return FA_OK;
}

}  // namespace

int check_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_BAD_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return FA_ERR_BAD_SHAPE;
  // Work units (B*H*ceil(N/256)) and launch-grid dimensions are 32-bit ints.
  if (bh * ((static_cast<long long>(N) + 255) / 256) > 0x7fffffffLL) return FA_ERR_BAD_SHAPE;
  if (static_cast<long long>(N) * (d > 0 ? d : 1) * 2 >= (1LL << 40)) return FA_ERR_BAD_SHAPE;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_BAD_SCALE;
  return FA_OK;
}

int check_fwd_bf16(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H, int N,
                   int d, float scale) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_POINTER;
  const int rc = check_common(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED_D;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_MISALIGNED;
  return FA_OK;
}

void contiguous_fwd_args(FwdArgs* a, const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int N, int d, float scale, int causal) {
  a->q = q;
  a->k = k;
  a->v = v;
  a->o = o;
  a->lse = lse;
  a->B = B;
  a->H = H;
  a->Nq = N;
  a->Nk = N;
  contiguous_strides(a->qs, H, N, d);
  contiguous_strides(a->ks, H, N, d);
  contiguous_strides(a->vs, H, N, d);
  contiguous_strides(a->os, H, N, d);
  a->scale = scale;
  a->causal = causal != 0;
}

// Dispatch of the bf16 forward by head dimension; maps launch failures to FA_ERR_CUDA.
int launch_tc(const FwdArgs& a, int d, const LaunchCtx& ctx) {
  long long cq[3], ck[3];
  contiguous_strides(cq, a.H, a.Nq, d);
  contiguous_strides(ck, a.H, a.Nk, d);
  bool contiguous = true;
  for (int i = 0; i < 3; ++i)
    contiguous = contiguous && a.qs[i] == cq[i] && a.os[i] == cq[i] && a.ks[i] == ck[i] && a.vs[i] == ck[i];
  int e = 0;
  if (contiguous) {
    switch (d) {
      case 32: e = launch_tc_d32(a, ctx); break;
      case 64: e = launch_tc_d64(a, ctx); break;
      case 128: e = launch_tc_d128(a, ctx); break;
      default: e = launch_tc_d256(a, ctx); break;
    }
  } else {
    switch (d) {
      case 32: e = launch_tc_strided_d32(a, ctx); break;
      case 64: e = launch_tc_strided_d64(a, ctx); break;
      case 128: e = launch_tc_strided_d128(a, ctx); break;
      default: e = launch_tc_strided_d256(a, ctx); break;
    }
  }
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

int encode_bf16_map(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_cols, int box_rows,
                    int swizzle_bytes) {
  if (g_encode == nullptr) return -1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(N) * D * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int encode_e4m3_map(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_cols, int box_rows,
                    int swizzle_bytes) {
  if (g_encode == nullptr) return -1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N) * D};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int encode_bf16_map4(CUtensorMap* map, const void* ptr, int B, int H, int N, int D, const long long* stride,
                     int box_cols, int box_rows, int swizzle_bytes) {
  if (g_encode == nullptr) return -1;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(stride[2]) * 2, static_cast<cuuint64_t>(stride[1]) * 2,
                                 static_cast<cuuint64_t>(stride[0]) * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle swz = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

// Resolve cuTensorMapEncodeTiled without creating any per-device state
// (used by the entry point that allocates nothing).  Returns 0 on success.
int load_tensor_map_encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode != nullptr) return 0;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return -1;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return 0;
}

// Current time limit of the device-side waits, in nanoseconds.
unsigned long long wait_limit_ns() { return static_cast<unsigned long long>(g_wait_limit_ms.load()) * 1000000ull; }

}  // namespace fa

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, void* stream) {
  int rc = fa::check_fwd_bf16(q, k, v, o, lse, B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  fa::DeviceState* s = nullptr;
  rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  fa::FwdArgs a;
  fa::contiguous_fwd_args(&a, q, k, v, o, lse, B, H, N, d, scale, causal);
  return fa::launch_tc(a, d, fa::make_ctx(*s, stream));
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, float q_descale, float k_descale, float v_descale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_POINTER;
  int rc = fa::check_common(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  const float f[3] = {q_descale, k_descale, v_descale};
  for (float x : f)
    if (!(std::isfinite(x) && x > 0.f)) return FA_ERR_BAD_SCALE;
  if (!std::isfinite(scale * q_descale * k_descale) || !(scale * q_descale * k_descale > 0.f)) return FA_ERR_BAD_SCALE;
  if (!fa::aligned16(q) || !fa::aligned16(k) || !fa::aligned16(v) || !fa::aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_MISALIGNED;
  fa::DeviceState* s = nullptr;
  rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  fa::FwdArgs a;
  fa::contiguous_fwd_args(&a, q, k, v, o, lse, B, H, N, d, scale, causal);
  a.q_descale = q_descale;
  a.k_descale = k_descale;
  a.v_descale = v_descale;
  const fa::LaunchCtx ctx = fa::make_ctx(*s, stream);
  const int e = d == 64 ? fa::launch_tc_fp8_d64(a, ctx) : fa::launch_tc_fp8_d128(a, ctx);
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                   int d, const long long* q_stride, const long long* k_stride, const long long* v_stride,
                   const long long* o_stride, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse || !q_stride || !k_stride || !v_stride || !o_stride) return FA_ERR_NULL_POINTER;
  int rc = fa::check_common(B, H, Nq, d, scale);
  if (rc != FA_OK) return rc;
  rc = fa::check_common(B, H, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED_D;
  const long long* all[4] = {q_stride, k_stride, v_stride, o_stride};
  for (const long long* st : all)
    for (int i = 0; i < 3; ++i)
      if (st[i] < 1 || st[i] >= (1LL << 38)) return FA_ERR_BAD_SHAPE;
  for (const long long* st : all)
    for (int i = 0; i < 3; ++i)
      if (st[i] % 8 != 0) return FA_ERR_MISALIGNED;  // 16-byte rows and tiles (TMA, vector stores)
  if (!fa::aligned16(q) || !fa::aligned16(k) || !fa::aligned16(v) || !fa::aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_MISALIGNED;
  fa::DeviceState* s = nullptr;
  rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  fa::FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  for (int i = 0; i < 3; ++i) {
    a.qs[i] = q_stride[i];
    a.ks[i] = k_stride[i];
    a.vs[i] = v_stride[i];
    a.os[i] = o_stride[i];
  }
  a.scale = scale;
  a.causal = causal != 0;
  return fa::launch_tc(a, d, fa::make_ctx(*s, stream));
}

int fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int H, int N, int d,
               float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_POINTER;
  int rc = fa::check_common(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d < 1 || d > 256) return FA_ERR_UNSUPPORTED_D;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_BAD_SHAPE;  // grid.y of the SIMT launch
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(lse);
  if (mis & 3u) return FA_ERR_MISALIGNED;
  fa::DeviceState* s = nullptr;
  rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  const fa::LaunchCtx ctx = fa::make_ctx(*s, stream);
  const int e = fa::launch_simt(causal != 0, q, k, v, o, lse, B * H, N, d, scale, ctx);
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const size_t elems = static_cast<size_t>(B) * H * N * d;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return 4 * fa::round256(elems * 2) + fa::round256(rows * 4);
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_NULL_POINTER;
  int rc = fa::check_common(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED_D;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_MISALIGNED;
  const size_t need = fa_fwd_host_workspace_bytes(B, H, N, d);
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  fa::DeviceState* s = nullptr;
  rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  fa::HostPipeline* hp = nullptr;
  rc = fa::host_pipeline(s, &hp);
  if (rc != FA_OK) return rc;
  const size_t per_head = static_cast<size_t>(N) * d * 2;  // bytes of one head of Q, K, V or O
  const size_t step = fa::round256(static_cast<size_t>(B) * H * per_head);
  char* w = static_cast<char*>(workspace);
  char *dq = w, *dk = w + step, *dv = w + 2 * step, *dout = w + 3 * step;
  float* dl = reinterpret_cast<float*>(w + 4 * step);
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  char* ho = static_cast<char*>(o);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Pipeline over chunks of heads: the copy-in stream brings chunk c's Q, K, V
  // while `stream` runs the kernel of chunk c - 1 and the copy-out stream
  // returns chunk c - 2's O and L.  Both copy streams fork from `stream` and
  // `stream` joins the copy-out stream at the end, so the call is ordered on
  // `stream` like a single kernel.
  const int BH = B * H;
  const int nch = BH < fa::kHostChunks ? BH : fa::kHostChunks;
  std::lock_guard<std::mutex> lock(hp->mutex);
  if (cudaEventRecord(hp->fork, st) != cudaSuccess || cudaStreamWaitEvent(hp->s_in, hp->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->s_out, hp->fork, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int c = 0; c < nch; ++c) {
    const int h0 = static_cast<int>(static_cast<long long>(BH) * c / nch);
    const int h1 = static_cast<int>(static_cast<long long>(BH) * (c + 1) / nch);
    const size_t off = static_cast<size_t>(h0) * per_head, bytes = static_cast<size_t>(h1 - h0) * per_head;
    if (cudaMemcpyAsync(dq + off, hq + off, bytes, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
        cudaMemcpyAsync(dk + off, hk + off, bytes, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
        cudaMemcpyAsync(dv + off, hv + off, bytes, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
        cudaEventRecord(hp->in[c], hp->s_in) != cudaSuccess || cudaStreamWaitEvent(st, hp->in[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    rc = fa_fwd(dq + off, dk + off, dv + off, dout + off, dl + static_cast<size_t>(h0) * N, 1, h1 - h0, N, d, scale,
                causal, stream);
    if (rc != FA_OK) return rc;
    const size_t lrows = static_cast<size_t>(h1 - h0) * N;
    if (cudaEventRecord(hp->done[c], st) != cudaSuccess || cudaStreamWaitEvent(hp->s_out, hp->done[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(ho + off, dout + off, bytes, cudaMemcpyDeviceToHost, hp->s_out) != cudaSuccess ||
        cudaMemcpyAsync(lse + static_cast<size_t>(h0) * N, dl + static_cast<size_t>(h0) * N, lrows * 4,
                        cudaMemcpyDeviceToHost, hp->s_out) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  if (cudaEventRecord(hp->join, hp->s_out) != cudaSuccess || cudaStreamWaitEvent(st, hp->join, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const size_t n_pad = (static_cast<size_t>(N) + 191) / 192 * 192;  // a multiple of both streamed-tile heights
  return 2 * fa::round256(static_cast<size_t>(B) * H * n_pad * 4);
}

namespace fa {
namespace {

// Checks shared by fa_bwd and fa_bwd_strided, then the launch.  The strides in
// a.st are already validated by the caller; `strided` selects the 4-D maps.
// Create the backward pass's second stream and events for device state `s` (once).
int bwd_fork(DeviceState* s, BwdFork** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  BwdFork& f = s->bwd;
  if (!f.ready) {
    if (cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess)
      return FA_ERR_CUDA;
    f.ready = true;
  }
  *out = &f;
  return FA_OK;
}

int run_bwd(BwdArgs& a, int d, bool strided, void* workspace, size_t workspace_bytes, void* stream) {
  if (!a.q || !a.k || !a.v || !a.o || !a.lse || !a.dout || !a.dq || !a.dk || !a.dv || !workspace)
    return FA_ERR_NULL_POINTER;
  if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.o) || !aligned16(a.dout) ||
      !aligned16(a.dq) || !aligned16(a.dk) || !aligned16(a.dv) || (reinterpret_cast<uintptr_t>(a.lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_MISALIGNED;
  if (workspace_bytes < fa_bwd_workspace_bytes(a.B, a.H, a.Nq, d)) return FA_ERR_WORKSPACE;
  DeviceState* s = nullptr;
  int rc = current_device_state(&s);
  if (rc != FA_OK) return rc;
  LaunchCtx ctx = make_ctx(*s, stream);
  BwdFork* f = nullptr;
  rc = bwd_fork(s, &f);
  if (rc != FA_OK) return rc;
  std::lock_guard<std::mutex> lock(f->mutex);
  ctx.side = f->side;
  ctx.ev_fork = f->fork;
  ctx.ev_join = f->join;
  a.n_pad = (a.Nq + 191) / 192 * 192;
  a.l2 = static_cast<float*>(workspace);
  a.dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                    round256(static_cast<size_t>(a.B) * a.H * a.n_pad * 4));
  int e = 0;
  switch (d) {
    case 32: e = strided ? launch_bwd_strided_d32(a, ctx) : launch_bwd_d32(a, ctx); break;
    case 64: e = strided ? launch_bwd_strided_d64(a, ctx) : launch_bwd_d64(a, ctx); break;
    case 128: e = strided ? launch_bwd_strided_d128(a, ctx) : launch_bwd_d128(a, ctx); break;
    default: e = strided ? launch_bwd_strided_d256(a, ctx) : launch_bwd_d256(a, ctx); break;
  }
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* workspace,
           size_t workspace_bytes, void* stream) {
  int rc = fa::check_common(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED_D;
  fa::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Nq = N;
  a.Nk = N;
  for (auto& st : a.st) fa::contiguous_strides(st, H, N, d);
  a.scale = scale;
  a.causal = causal != 0;
  return fa::run_bwd(a, d, false, workspace, workspace_bytes, stream);
}

int fa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, const long long* strides,
                   float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  if (!strides) return FA_ERR_NULL_POINTER;
  int rc = fa::check_common(B, H, Nq, d, scale);
  if (rc != FA_OK) return rc;
  rc = fa::check_common(B, H, Nk, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED_D;
  for (int i = 0; i < 24; ++i)
    if (strides[i] < 1 || strides[i] >= (1LL << 38)) return FA_ERR_BAD_SHAPE;
  for (int i = 0; i < 24; ++i)
    if (strides[i] % 8 != 0) return FA_ERR_MISALIGNED;  // 16-byte rows and tiles (TMA, vector loads and stores)
  fa::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  for (int t = 0; t < 8; ++t)
    for (int i = 0; i < 3; ++i) a.st[t][i] = strides[3 * t + i];
  a.scale = scale;
  a.causal = causal != 0;
  return fa::run_bwd(a, d, true, workspace, workspace_bytes, stream);
}

int fa_status(void* stream) {
  fa::DeviceState* s = nullptr;
  int rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, s->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0 && cudaMemset(s->status, 0, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  const int na = fa::noalloc_take_status();
  if (na == FA_ERR_CUDA) return FA_ERR_CUDA;
  return (word != 0 || na == FA_ERR_TIMEOUT) ? FA_ERR_TIMEOUT : FA_OK;
}

int fa_selftest_wait(void* stream) {
  fa::DeviceState* s = nullptr;
  int rc = fa::current_device_state(&s);
  if (rc != FA_OK) return rc;
  return fa::launch_selftest_wait(fa::make_ctx(*s, stream)) == 0 ? FA_OK : FA_ERR_CUDA;
}

int fa_set_wait_limit_ms(int ms) {
  if (ms < 1) ms = 1;
  return fa::g_wait_limit_ms.exchange(ms);
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "FA_OK: success";
    case FA_ERR_NULL_POINTER: return "FA_ERR_NULL_POINTER: a required pointer is NULL";
    case FA_ERR_BAD_SHAPE: return "FA_ERR_BAD_SHAPE: B, H or N out of range";
    case FA_ERR_UNSUPPORTED_D: return "FA_ERR_UNSUPPORTED_D: head dimension not supported by this entry point";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: pointer not sufficiently aligned";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA runtime or driver call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded device-side wait expired";
    case FA_ERR_ARCH: return "FA_ERR_ARCH: the current device is not compute capability 10.3";
    case FA_ERR_BAD_SCALE: return "FA_ERR_BAD_SCALE: scale (and every dequantisation factor) must be finite and > 0";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace too small";
    case FA_ERR_SCRATCH: return "FA_ERR_SCRATCH: the kernel needs more scratch than fa_fwd_noalloc's static array holds";
    default: return "unknown fa_gb300 error code";
  }
}

int fa_abi_version(void) { return 1; }

}  // extern "C"

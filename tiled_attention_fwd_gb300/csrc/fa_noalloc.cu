// fa_fwd_noalloc: the bf16 tensor-core forward pass for callers that cannot
// allocate device memory (see include/fa_gb300.h).  The only device memory
// the kernel needs besides its inputs and outputs is a small scratch area
// (the status word of its bounded waits); here it lives in a file-scope
// static __device__ array instead of memory the library allocates.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Scratch of the allocation-free entry point: 64 words (256 bytes) per device,
// part of the module image, so every GPU that loads the library holds it until
// exit.  Word 0 is the status word of the kernel's bounded waits.
constexpr int kNoAllocScratchWords = 64;
__device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchWords];

// Scratch words one launch of the tensor-core kernel uses (the status word).
// It does not depend on B, H, N or d.
constexpr int kTcScratchWords = 1;

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};

std::mutex g_na_mutex;
NoAllocDevice g_na_devices[kMaxDevices];

// Once per device, with that device current: look up the device address of
// the scratch array (the host-side symbol is only a stand-in, not a device
// address), the SM count, and the tensor-map encoder.  Allocates nothing.
int noalloc_device(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& s = g_na_devices[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    if (major != 10 || minor != 3) return FA_ERR_ARCH;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    if (load_tensor_map_encoder() != 0) return FA_ERR_CUDA;
    s.scratch = static_cast<int*>(ptr);
    s.num_sms = sms;
    s.ready = true;
  }
  *out = &s;
  return FA_OK;
}

}  // namespace

// Read and clear the status word of the static scratch on the current device
// (fa_status).  Synchronous copies to and from the symbol; allocates nothing.
// Returns FA_OK (word was zero, or no fa_fwd_noalloc call was set up on this
// device), FA_ERR_TIMEOUT (word was set; now cleared) or FA_ERR_CUDA.
int noalloc_take_status() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_na_mutex);
    if (!g_na_devices[dev].ready) return FA_OK;
  }
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_noalloc_scratch, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (word == 0) return FA_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return FA_ERR_TIMEOUT;
}

}  // namespace fa

extern "C" int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int N, int d, float scale, int causal, void* stream) {
  // The same checks, in the same order, as fa_fwd.
  int rc = fa::check_fwd_bf16(q, k, v, o, lse, B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (fa::kTcScratchWords > fa::kNoAllocScratchWords) return FA_ERR_SCRATCH;
  fa::NoAllocDevice* s = nullptr;
  rc = fa::noalloc_device(&s);
  if (rc != FA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word must start at zero for this call; the array keeps whatever the previous call left.
  if (cudaMemsetAsync(s->scratch, 0, sizeof(int) * fa::kTcScratchWords, st) != cudaSuccess) return FA_ERR_CUDA;
  fa::LaunchCtx ctx;
  ctx.status = s->scratch;
  ctx.limit_ns = fa::wait_limit_ns();
  ctx.num_sms = s->num_sms;
  ctx.stream = st;
  fa::FwdArgs a;
  fa::contiguous_fwd_args(&a, q, k, v, o, lse, B, H, N, d, scale, causal);
  return fa::launch_tc(a, d, ctx);
}

// Inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA, commit, ld/st, fences), and a few scalar
// helpers.  Every device-side wait goes through wait_bar(), which gives up
// after a time limit and raises the CTA's abort flag instead of spinning
// forever.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// Non-blocking test of the phase with parity `parity`.
__device__ __forceinline__ uint32_t mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// Cluster-scope forms (CTA pairs): wait with acquire at cluster scope, so that
// what the other CTA of the cluster released before arriving is visible.
__device__ __forceinline__ uint32_t mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}
__device__ __forceinline__ uint32_t mbar_test_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// Address in the shared::cluster window of the same shared-memory offset in
// the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive (release at cluster scope) on a barrier given by its shared::cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Error bits written to the device status word.
enum : int {
  kStatusTimeoutLoad = 1 << 0,
  kStatusTimeoutMma = 1 << 1,
  kStatusTimeoutSoftmax = 1 << 2,
  kStatusTimeoutDrain = 1 << 3,
};

// Shared state of the bounded waits of one CTA.
struct WaitGuard {
  volatile int* abort;  // shared memory flag, set once any wait of the CTA gives up
  int* status;          // device status word (global memory)
  uint64_t limit_ns;
  bool cluster = false;  // CTA pairs: waits acquire at cluster scope
};

__device__ __forceinline__ uint32_t guard_try_wait(uint32_t bar, uint32_t parity, const WaitGuard& g) {
  return g.cluster ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity);
}

// Wait for the phase of `bar` with parity `parity` to complete.  Returns
// false (without completing) if the CTA's abort flag is raised or the wait
// exceeds the time limit; in the latter case this thread raises the flag and
// ORs `code` into the status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitGuard& g, int code) {
  if (guard_try_wait(bar, parity, g)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (guard_try_wait(bar, parity, g)) return true;
    if (*g.abort) return false;
    if (globaltimer_ns() - t0 > g.limit_ns) {
      *g.abort = 1;
      atomicOr(g.status, code);
      return false;
    }
  }
}

// Warp-level forms.  Every lane waits (a warp whose lanes all wait on the
// barrier is suspended and resumed together), the outcome is made uniform
// across the warp; arrivals are made by lane 0 for the whole warp after
// __syncwarp, which orders the memory operations of the warp's lanes before
// lane 0's release.  A barrier signalled this way counts one arrival per warp.
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const WaitGuard& g, int code) {
  const bool ok = wait_bar(bar, parity, g, code);
  return __all_sync(0xffffffffu, ok);
}

// Lane 0 waits for the warp (a non-blocking test first, then the bounded
// wait); the outcome is broadcast and __syncwarp orders the other lanes after
// lane 0's acquire.  For warps whose lanes do nothing but issue on lane 0.
__device__ __forceinline__ bool leader_wait_bar(uint32_t bar, uint32_t parity, const WaitGuard& g, int code) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = (mbar_test_wait(bar, parity) || wait_bar(bar, parity, g, code)) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// The same arrival made by an elect.sync-chosen lane inside one asm block, so
// the compiler sees no divergent branch (keeps register allocation of long
// unrolled loops unchanged where the arrival sits in the middle of them).
__device__ __forceinline__ void warp_arrive_elect(uint32_t bar) {
  __syncwarp();
  asm volatile(
      "{\n\t.reg .pred PE;\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// warp_arrive_elect that also returns a word which is zero but which the
// compiler sees computed from the arrival (its state operand): code that uses
// it is scheduled after the arrival.
__device__ __forceinline__ uint32_t warp_arrive_token(uint32_t bar) {
  __syncwarp();
  uint64_t state = 0;
  asm volatile(
      "{\n\t.reg .pred PE;\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE mbarrier.arrive.shared::cta.b64 %0, [%1];\n\t}"
      : "+l"(state)
      : "r"(bar)
      : "memory");
  uint32_t z;
  asm("and.b32 %0, %1, 0;" : "=r"(z) : "r"(static_cast<uint32_t>(state)));
  return z;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 3-D tiled bulk tensor load global -> shared, completion counted in bytes on `bar`.
// Coordinates are element indices {x (innermost), y, z}; x * 2 bytes is a multiple of 16.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y,
                                            int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// 4-D tiled bulk tensor load global -> shared: coordinates {x (innermost), y, z, w}.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z, int w,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
      : "memory");
}

// 3-D / 4-D tiled bulk tensor store shared -> global, tracked by the issuing
// thread's bulk async-groups.  Elements of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_store_4d(const void* tmap, uint32_t src, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(tmap),
               "r"(src), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Contiguous bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// CTA pairs: one warp in each CTA of the pair executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B,
// A K-major, B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4)                             // D format: f32
         | (1u << 7)                           // A format: bf16
         | (1u << 10)                          // B format: bf16
         | (0u << 15)                          // A major: K
         | (static_cast<uint32_t>(b_mn_major) << 16)  // B major
         | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with e4m3 A and B (format
// code 0 in the A and B fields) and an fp32 accumulator; the other fields as
// in make_idesc_bf16.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int M, int N, int b_mn_major) {
  return (1u << 4)                             // D format: f32
         | (0u << 7)                           // A format: e4m3
         | (0u << 10)                          // B format: e4m3
         | (0u << 15)                          // A major: K
         | (static_cast<uint32_t>(b_mn_major) << 16)  // B major
         | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

// Shared-memory matrix descriptor (tcgen05 format), as two 32-bit words.
// Low word: start address / 16 in bits 0..13, leading byte offset / 16 in
// bits 16..29.  High word: stride byte offset / 16 in bits 0..13 (bits
// 32..45), the fixed 0b001 at bit 14 (bit 46), swizzle mode in bits 29..31
// (bits 61..63; 2 = 128-byte, 4 = 64-byte).
__host__ __device__ constexpr uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi(uint32_t sbo, uint32_t swizzle) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | ((swizzle & 7u) << 29);
}

// tcgen05.mma kind::f16 with the descriptors passed as (low, high) words, so
// that stepping through a tile is a 32-bit add on the low word.  Warp-wide:
// every lane of the warp executes them and one elected lane issues (the
// operands are warp-uniform).  _ss: A and B in shared memory; _ts: A in
// tensor memory.
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                               uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P1, PE;\n\t.reg .b64 DA, DB;\n\t"
      "setp.ne.b32 P1, %6, 0;\n\t"
      "mov.b64 DA, {%1, %2};\n\t"
      "mov.b64 DB, {%3, %4};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, P1;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P1, PE;\n\t.reg .b64 DB;\n\t"
      "setp.ne.b32 P1, %5, 0;\n\t"
      "mov.b64 DB, {%2, %3};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], DB, %4, P1;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A run of n MMAs (n = 2, 4, 6, 8) over consecutive 16-wide K steps, issued by
// one elected lane from a single block: the descriptors advance by the
// compile-time increments S::da(k) / S::db(k) (16-byte units, step k-1 to k;
// for the TMEM A operand S::ta(k) columns), and only the first MMA takes the
// caller's accumulate flag.  One election and no per-MMA operand set-up.
template <class S>
__device__ __forceinline__ void mma_ss_x2(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DA, DB;\n\t"
      "setp.ne.b32 PA, %6, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b64 DA, {%1, %2};\n\t"
      "mov.b64 DB, {%3, %4};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PA;\n\t"
      "add.s64 DA, DA, %7;\n\t"
      "add.s64 DB, DB, %8;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::da(1)), "n"(S::db(1))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ts_x2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DB;\n\t.reg .b32 TA;\n\t"
      "setp.ne.b32 PA, %5, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b32 TA, %1;\n\t"
      "mov.b64 DB, {%2, %3};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PA;\n\t"
      "add.u32 TA, TA, %6;\n\t"
      "add.s64 DB, DB, %7;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::ta(1)), "n"(S::db(1))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ss_x4(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DA, DB;\n\t"
      "setp.ne.b32 PA, %6, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b64 DA, {%1, %2};\n\t"
      "mov.b64 DB, {%3, %4};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PA;\n\t"
      "add.s64 DA, DA, %7;\n\t"
      "add.s64 DB, DB, %10;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %8;\n\t"
      "add.s64 DB, DB, %11;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %9;\n\t"
      "add.s64 DB, DB, %12;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::da(1)), "n"(S::da(2)), "n"(S::da(3)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ts_x4(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DB;\n\t.reg .b32 TA;\n\t"
      "setp.ne.b32 PA, %5, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b32 TA, %1;\n\t"
      "mov.b64 DB, {%2, %3};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PA;\n\t"
      "add.u32 TA, TA, %6;\n\t"
      "add.s64 DB, DB, %9;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %7;\n\t"
      "add.s64 DB, DB, %10;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %8;\n\t"
      "add.s64 DB, DB, %11;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::ta(1)), "n"(S::ta(2)), "n"(S::ta(3)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ss_x6(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DA, DB;\n\t"
      "setp.ne.b32 PA, %6, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b64 DA, {%1, %2};\n\t"
      "mov.b64 DB, {%3, %4};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PA;\n\t"
      "add.s64 DA, DA, %7;\n\t"
      "add.s64 DB, DB, %12;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %8;\n\t"
      "add.s64 DB, DB, %13;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %9;\n\t"
      "add.s64 DB, DB, %14;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %10;\n\t"
      "add.s64 DB, DB, %15;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %11;\n\t"
      "add.s64 DB, DB, %16;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::da(1)), "n"(S::da(2)), "n"(S::da(3)), "n"(S::da(4)), "n"(S::da(5)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3)), "n"(S::db(4)), "n"(S::db(5))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ts_x6(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DB;\n\t.reg .b32 TA;\n\t"
      "setp.ne.b32 PA, %5, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b32 TA, %1;\n\t"
      "mov.b64 DB, {%2, %3};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PA;\n\t"
      "add.u32 TA, TA, %6;\n\t"
      "add.s64 DB, DB, %11;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %7;\n\t"
      "add.s64 DB, DB, %12;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %8;\n\t"
      "add.s64 DB, DB, %13;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %9;\n\t"
      "add.s64 DB, DB, %14;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %10;\n\t"
      "add.s64 DB, DB, %15;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::ta(1)), "n"(S::ta(2)), "n"(S::ta(3)), "n"(S::ta(4)), "n"(S::ta(5)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3)), "n"(S::db(4)), "n"(S::db(5))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ss_x8(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DA, DB;\n\t"
      "setp.ne.b32 PA, %6, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b64 DA, {%1, %2};\n\t"
      "mov.b64 DB, {%3, %4};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PA;\n\t"
      "add.s64 DA, DA, %7;\n\t"
      "add.s64 DB, DB, %14;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %8;\n\t"
      "add.s64 DB, DB, %15;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %9;\n\t"
      "add.s64 DB, DB, %16;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %10;\n\t"
      "add.s64 DB, DB, %17;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %11;\n\t"
      "add.s64 DB, DB, %18;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %12;\n\t"
      "add.s64 DB, DB, %19;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "add.s64 DA, DA, %13;\n\t"
      "add.s64 DB, DB, %20;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %5, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::da(1)), "n"(S::da(2)), "n"(S::da(3)), "n"(S::da(4)), "n"(S::da(5)), "n"(S::da(6)), "n"(S::da(7)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3)), "n"(S::db(4)), "n"(S::db(5)), "n"(S::db(6)), "n"(S::db(7))
      : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ts_x8(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DB;\n\t.reg .b32 TA;\n\t"
      "setp.ne.b32 PA, %5, 0;\n\t"
      "setp.eq.b32 PT, 0, 0;\n\t"
      "mov.b32 TA, %1;\n\t"
      "mov.b64 DB, {%2, %3};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PA;\n\t"
      "add.u32 TA, TA, %6;\n\t"
      "add.s64 DB, DB, %13;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %7;\n\t"
      "add.s64 DB, DB, %14;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %8;\n\t"
      "add.s64 DB, DB, %15;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %9;\n\t"
      "add.s64 DB, DB, %16;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %10;\n\t"
      "add.s64 DB, DB, %17;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %11;\n\t"
      "add.s64 DB, DB, %18;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "add.u32 TA, TA, %12;\n\t"
      "add.s64 DB, DB, %19;\n\t"
      "@PE tcgen05.mma.cta_group::1.kind::f16 [%0], [TA], DB, %4, PT;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::ta(1)), "n"(S::ta(2)), "n"(S::ta(3)), "n"(S::ta(4)), "n"(S::ta(5)), "n"(S::ta(6)), "n"(S::ta(7)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3)), "n"(S::db(4)), "n"(S::db(5)), "n"(S::db(6)), "n"(S::db(7))
      : "memory");
}

// The same runs for kind::f8f6f4 (e4m3 operands, K = 32 per MMA: the same 32
// bytes of each operand row as one kind::f16 MMA), lengths 2 and 4.
#define FA_F8_SS_HEAD                                                       \
  "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DA, DB;\n\t"                   \
  "setp.ne.b32 PA, %6, 0;\n\tsetp.eq.b32 PT, 0, 0;\n\t"                     \
  "mov.b64 DA, {%1, %2};\n\tmov.b64 DB, {%3, %4};\n\t"                      \
  "elect.sync _|PE, 0xffffffff;\n\t"                                        \
  "@PE tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], DA, DB, %5, PA;\n\t"
#define FA_F8_SS_NEXT(IA, IB)                                               \
  "add.s64 DA, DA, %" #IA ";\n\tadd.s64 DB, DB, %" #IB ";\n\t"              \
  "@PE tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], DA, DB, %5, PT;\n\t"
#define FA_F8_TS_HEAD                                                       \
  "{\n\t.reg .pred PE, PA, PT;\n\t.reg .b64 DB;\n\t.reg .b32 TA;\n\t"      \
  "setp.ne.b32 PA, %5, 0;\n\tsetp.eq.b32 PT, 0, 0;\n\t"                     \
  "mov.b32 TA, %1;\n\tmov.b64 DB, {%2, %3};\n\t"                            \
  "elect.sync _|PE, 0xffffffff;\n\t"                                        \
  "@PE tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [TA], DB, %4, PA;\n\t"
#define FA_F8_TS_NEXT(IA, IB)                                               \
  "add.u32 TA, TA, %" #IA ";\n\tadd.s64 DB, DB, %" #IB ";\n\t"              \
  "@PE tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [TA], DB, %4, PT;\n\t"

template <class S>
__device__ __forceinline__ void mma_ss_x2_f8(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                              uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_F8_SS_HEAD FA_F8_SS_NEXT(7, 8) "}"
               ::"r"(d_tmem), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate),
               "n"(S::da(1)), "n"(S::db(1))
               : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ss_x4_f8(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                              uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_F8_SS_HEAD FA_F8_SS_NEXT(7, 10) FA_F8_SS_NEXT(8, 11) FA_F8_SS_NEXT(9, 12) "}"
               ::"r"(d_tmem), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate),
               "n"(S::da(1)), "n"(S::da(2)), "n"(S::da(3)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3))
               : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ts_x2_f8(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_F8_TS_HEAD FA_F8_TS_NEXT(6, 7) "}"
               ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::ta(1)),
               "n"(S::db(1))
               : "memory");
}
template <class S>
__device__ __forceinline__ void mma_ts_x4_f8(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(FA_F8_TS_HEAD FA_F8_TS_NEXT(6, 9) FA_F8_TS_NEXT(7, 10) FA_F8_TS_NEXT(8, 11) "}"
               ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(S::ta(1)),
               "n"(S::ta(2)), "n"(S::ta(3)), "n"(S::db(1)), "n"(S::db(2)), "n"(S::db(3))
               : "memory");
}

// Runs of N = 2, 4, 6 or 8 MMAs (kind::f16), or N = 2 or 4 (kind::f8f6f4 when F8).
template <int N, class S, bool F8 = false>
__device__ __forceinline__ void mma_ss_run(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  if constexpr (F8) {
    static_assert(N == 2 || N == 4, "run length");
    if constexpr (N == 2) mma_ss_x2_f8<S>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 4) mma_ss_x4_f8<S>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, accumulate);
  } else {
    static_assert(N == 2 || N == 4 || N == 6 || N == 8, "run length");
    if constexpr (N == 2) mma_ss_x2<S>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 4) mma_ss_x4<S>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 6) mma_ss_x6<S>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 8) mma_ss_x8<S>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc, accumulate);
  }
}
template <int N, class S, bool F8 = false>
__device__ __forceinline__ void mma_ts_run(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
  if constexpr (F8) {
    static_assert(N == 2 || N == 4, "run length");
    if constexpr (N == 2) mma_ts_x2_f8<S>(d_tmem, a_tmem, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 4) mma_ts_x4_f8<S>(d_tmem, a_tmem, b_lo, b_hi, idesc, accumulate);
  } else {
    static_assert(N == 2 || N == 4 || N == 6 || N == 8, "run length");
    if constexpr (N == 2) mma_ts_x2<S>(d_tmem, a_tmem, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 4) mma_ts_x4<S>(d_tmem, a_tmem, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 6) mma_ts_x6<S>(d_tmem, a_tmem, b_lo, b_hi, idesc, accumulate);
    if constexpr (N == 8) mma_ts_x8<S>(d_tmem, a_tmem, b_lo, b_hi, idesc, accumulate);
  }
}

// CTA-pair MMAs (cta_group::2, M = 256): A rows 0..127 from this CTA, 128..255
// from the peer at the same address; B's N columns half from each CTA; D rows
// split the same way across the two CTAs' TMEM.  Issued by the pair's leader.
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                            uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P1, PE;\n\t.reg .b64 DA, DB;\n\t"
      "setp.ne.b32 P1, %6, 0;\n\t"
      "mov.b64 DA, {%1, %2};\n\t"
      "mov.b64 DB, {%3, %4};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::2.kind::f16 [%0], DA, DB, %5, P1;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred P1, PE;\n\t.reg .b64 DB;\n\t"
      "setp.ne.b32 P1, %5, 0;\n\t"
      "mov.b64 DB, {%2, %3};\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], DB, %4, P1;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at offset `bar` of every CTA in `mask` when the
// pair MMAs this warp issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred PE;\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
      ::"r"(bar), "h"(mask)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the warp issued so far
// has completed (issued by one elected lane).
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred PE;\n\t"
      "elect.sync _|PE, 0xffffffff;\n\t"
      "@PE tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: this thread's TMEM lane, columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for this thread's outstanding tcgen05.ld; the registers are passed
// through so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// tmem_ld32 that also returns, in `mx`, the maximum of the 32 fp32 values
// this thread loads (tcgen05.ld.red, sm_103a); valid after the wait.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr));
}

// tmem_wait_ld for a tmem_ld32_max: its reduced value is passed through as well.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32], float& mx) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+f"(mx)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ register budget
// Re-split the block's registers between warpgroups (all four warps of a
// warpgroup execute the same instruction).
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ math
// Hardware base-2 exponential (MUFU), flushes denormals; ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (one instruction on two lanes of a 64-bit register pair).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two fp32 values to one bf16x2 word, round to nearest even; `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four fp32 values to four e4m3 bytes (round to nearest even, saturating to
// +-448); `p0` in bits 0..7 (the lowest K index first, as a TMEM A operand of
// kind::f8f6f4 holds four consecutive K elements per 32-bit column).
// x rounded to e4m3 as pack_e4m3x4 rounds it (nearest even, saturating),
// back in fp32 (e4m3 -> f16 -> f32 are exact).
__device__ __forceinline__ float round_e4m3(float x) {
  float r;
  asm("{\n\t.reg .b16 b, lo, hi;\n\t.reg .b32 h2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 b, %1, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 h2, b;\n\t"
      "mov.b32 {lo, hi}, h2;\n\t"
      "cvt.f32.f16 %0, lo;\n\t}"
      : "=f"(r)
      : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float p0, float p1, float p2, float p3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(p0), "f"(p1), "f"(p2), "f"(p3));
  return r;
}

}  // namespace fa

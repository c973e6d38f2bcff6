/*
 * fa_gb300.h - C ABI of the GB300 (sm_103a) FlashAttention-2 forward pass.
 *
 * The operation (every entry point below computes it, for each batch b and
 * head h independently):
 *
 *   S = (Q K^T) * scale                         "Writing a FlashAttention kernel in Metal",
 *                                               section "Standard attention"
 *   causal: S[q][k] = -inf for key k > query q  same page, "Blockwise attention and causal
 *                                               masking" (absolute positions, top-left aligned)
 *   O = softmax_rows(S) V                       same page, "Standard attention"
 *   L[q] = log sum_k exp(S[q][k])  (natural log; the tiled method's m + log l)
 *                                               "FlashAttention-2 from PyTorch to Triton",
 *                                               section "What We Are Building"
 *
 * The N x N matrices S and P are never stored: the kernels run the FA2
 * recurrence of the latter page (running row max m, rescaled row sum l,
 * unnormalised O, one division by l at the end) over key/value tiles.
 *
 * Layout: Q, K, V and O are [B][H][N][d] row-major and contiguous (element
 * (b,h,n,c) at ((b*H + h)*N + n)*d + c); L is [B][H][N] fp32.  N_q = N_k = N.
 *
 * Ownership: the caller allocates and owns every buffer passed in.  The
 * library keeps one small device status word per device (allocated on the
 * first call on that device, never freed before process exit).
 *
 * Asynchrony: every call only enqueues work on `stream` (a cudaStream_t
 * passed as void*, NULL = legacy default stream) and returns without
 * synchronising.  Argument errors are detected on the host before anything is
 * enqueued.  A device-side wait that exceeds its time limit ends the kernel
 * early and records FA_ERR_TIMEOUT in the device status word, which
 * fa_status() reports.
 *
 * Return codes: FA_OK (0) or one of the negative FA_ERR_* values below;
 * fa_strerror() names them.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  FA_OK = 0,
  FA_ERR_NULL_POINTER = -1,   /* a required pointer is NULL                                  */
  FA_ERR_BAD_SHAPE = -2,      /* B, H or N < 1, or B*H*N*d does not fit the index types      */
  FA_ERR_UNSUPPORTED_D = -3,  /* head dimension not supported by this entry point            */
  FA_ERR_MISALIGNED = -4,     /* a device pointer is not 16-byte aligned                     */
  FA_ERR_CUDA = -5,           /* a CUDA runtime or driver call failed (launch, tensor map)   */
  FA_ERR_TIMEOUT = -6,        /* a bounded device-side wait expired (reported by fa_status)  */
  FA_ERR_ARCH = -7,           /* the current device is not a compute capability 10.3 GPU     */
  FA_ERR_BAD_SCALE = -8,      /* scale is not a finite number > 0                            */
  FA_ERR_WORKSPACE = -9,      /* the workspace passed to fa_fwd_host or fa_bwd is too small  */
  FA_ERR_SCRATCH = -10        /* the kernel needs more scratch than fa_fwd_noalloc provides  */
};

/*
 * fa_fwd - bf16 forward pass on the tensor cores (tcgen05, TMA, TMEM).
 *
 *   q, k, v : device pointers to bf16 (__nv_bfloat16) [B][H][N][d], 16-byte aligned.
 *   o       : device pointer to bf16 [B][H][N][d], 16-byte aligned; fully overwritten.
 *   lse     : device pointer to fp32 [B][H][N]; fully overwritten with L (natural log).
 *   B, H, N : batch, heads, sequence length; each >= 1.  Any N (ragged tails are masked).
 *   d       : head dimension, one of 32, 64, 128, 256.
 *   scale   : softmax scale applied to Q K^T (the pages use 1/sqrt(d)); finite and > 0.
 *   causal  : nonzero applies the causal mask (key k visible to query q iff k <= q).
 *   stream  : cudaStream_t (as void*) the work is enqueued on.
 *
 * Arithmetic: bf16 products with fp32 accumulation for Q K^T and P V, fp32
 * softmax state, P rounded to bf16 before P V, O rounded to bf16 once at the end.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_fwd_strided - fa_fwd with separate query and key lengths and any layout
 * whose head dimension is contiguous (e.g. [B][N][H][d] as well as
 * [B][H][N][d]), as the Triton kernel of "FlashAttention-2 from PyTorch to
 * Triton" takes N_QUERIES, N_KEYS and per-tensor strides.
 *
 *   q, o    : bf16, Nq rows per head; element (b, h, i, c) at ptr + b*s[0] + h*s[1] + i*s[2] + c,
 *             s = q_stride / o_stride.
 *   k, v    : bf16, Nk rows per head, addressed with k_stride / v_stride likewise.
 *   *_stride: three element strides {batch, head, row}, each >= 1 and a multiple of 8
 *             (16 bytes; else FA_ERR_MISALIGNED); read only during the call.
 *   lse     : fp32, contiguous [B][H][Nq].
 *   causal  : key k visible to query i iff k <= i (positions from the start of
 *             both sequences, as in the pages' kernel); keys >= Nk never visible.
 *   Other arguments, alignment and behaviour as fa_fwd.  o must not overlap q, k, v or itself.
 */
int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int Nq, int Nk, int d,
                   const long long* q_stride, const long long* k_stride,
                   const long long* v_stride, const long long* o_stride,
                   float scale, int causal, void* stream);

/*
 * fa_fwd_fp8 - the forward pass on e4m3 (fp8) inputs with bf16 output.
 * Same computation as fa_fwd on the dequantised inputs: the pages define the
 * method on real-valued inputs ("FlashAttention-2 from PyTorch to Triton",
 * section "What We Are Building") and name low-precision attention only as a
 * later variant ("Case Study: metal-flash-attention", closing section on MFA
 * 2.0); the quantisation reading here is one fp32 dequantisation factor per
 * tensor, real value = factor * e4m3 value.  S = Q8 K8^T runs on the tensor
 * core in e4m3 with fp32 accumulation and is scaled by
 * scale * q_descale * k_descale; the softmax is fa_fwd's (fp32 m and l); P is
 * rounded to e4m3, V's dtype, before O += P V (the Triton kernel of the page
 * above casts P to V's dtype); O = (P V) * v_descale / l is stored in bf16.
 *
 *   q, k, v   : device pointers to e4m3 (OCP E4M3FN, one byte each) [B][H][N][d],
 *               contiguous, 16-byte aligned.
 *   o         : device pointer to bf16 [B][H][N][d], 16-byte aligned.
 *   lse       : device pointer to fp32 [B][H][N] (natural log of the dequantised logits).
 *   d         : 64 or 128 (else FA_ERR_UNSUPPORTED_D).
 *   scale     : softmax scale of the dequantised logits (the pages use 1/sqrt(d)).
 *   q_descale, k_descale, v_descale : dequantisation factors, finite and > 0,
 *               and scale * q_descale * k_descale finite (else FA_ERR_BAD_SCALE).
 *   Other arguments, asynchrony, ownership and return codes as fa_fwd.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int N, int d, float scale,
               float q_descale, float k_descale, float v_descale, int causal, void* stream);

/*
 * fa_fwd_f32 - fp32 forward pass on the CUDA cores (SIMT), all arithmetic in fp32.
 * Same computation as fa_fwd (the plain attention of "FlashAttention-2 from
 * PyTorch to Triton", section "What We Are Building").  Problems whose K and V
 * of one head fit in 64 KB of shared memory (with a score row per warp) run a
 * whole-head kernel with an exact two-pass softmax; larger ones the tiled
 * kernel with the online-softmax rescaling of "Writing a FlashAttention kernel
 * in Metal" (section "Online softmax").
 *
 *   q, k, v, o : device pointers to fp32 [B][H][N][d] (4-byte aligned suffices).
 *   lse        : device pointer to fp32 [B][H][N].
 *   d          : any head dimension 1 <= d <= 256.
 *   Other arguments and behaviour as fa_fwd.
 */
int fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
               int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_fwd_host_workspace_bytes - size of the device workspace fa_fwd_host needs
 * for one bf16 problem of this shape (room for Q, K, V, O and L on the device,
 * each 256-byte aligned).  Returns 0 for invalid shapes.
 */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_fwd_host - fa_fwd on HOST buffers: the host-to-device copies of q, k, v
 * into `workspace`, the forward pass, and the device-to-host copies of O and
 * L into o and lse, pipelined over up to 8 chunks of heads so that copies in,
 * kernels and copies out overlap.  The copies run on two internal streams of
 * the library that start after the work already enqueued on `stream`, and
 * `stream` waits for them at the end: the call is ordered on `stream` like a
 * single kernel (also under stream capture).  Host buffers should be
 * page-locked for the copies to be asynchronous.  The caller synchronises
 * `stream` before reading o and lse or reusing the inputs.
 *
 *   q, k, v   : host pointers to bf16 [B][H][N][d].
 *   o, lse    : host pointers receiving bf16 O and fp32 L.
 *   workspace : device pointer, 256-byte aligned, at least
 *               fa_fwd_host_workspace_bytes(B, H, N, d) bytes (else FA_ERR_WORKSPACE).
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                void* workspace, size_t workspace_bytes,
                int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_bwd_workspace_bytes - size of the device workspace fa_bwd needs: two fp32
 * vectors of B*H*round_up(N, 192) rows (L * log2(e) and D = rowsum(dO * O)),
 * each 256-byte aligned.  For fa_bwd_strided pass N = Nq.  Returns 0 for
 * invalid shapes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_bwd - bf16 backward pass on the tensor cores: the gradients of
 * O = softmax(Q K^T * scale) V (causal mask optional) with respect to Q, K, V
 * given the upstream gradient dO.  P is recomputed from the forward's L as
 * exp(scale * Q K^T - L) ("FlashAttention-2 from PyTorch to Triton", "What We
 * Are Building"); as in the metal-flash-attention backward ("Case Study:
 * metal-flash-attention") a dK/dV kernel and a dQ kernel each own their
 * outputs, so the results are deterministic (no atomics).  Three kernels:
 * D = rowsum(dO * O) and the dK/dV kernel on `stream`, and the dQ kernel on a
 * second stream of the library that starts after the first kernel and that
 * `stream` waits for at the end, so the dQ kernel takes the SMs the dK/dV
 * kernel frees as it finishes; the call is ordered on `stream` like a single
 * kernel (also under stream capture).
 *
 *   q, k, v, o, dout : device pointers to bf16 [B][H][N][d], 16-byte aligned;
 *                      o and lse are the outputs of fa_fwd for q, k, v, scale, causal.
 *   lse              : device pointer to fp32 [B][H][N].
 *   dq, dk, dv       : device pointers to bf16 [B][H][N][d], 16-byte aligned; fully overwritten.
 *   d                : head dimension, one of 32, 64, 128, 256 (else FA_ERR_UNSUPPORTED_D);
 *                      d = 256 runs 32-row streamed tiles and, for dK and dV, one output half
 *                      per work unit (the TMEM of one SM holds no more).
 *   workspace        : device pointer, 256-byte aligned, at least fa_bwd_workspace_bytes(B, H, N, d)
 *                      bytes (else FA_ERR_WORKSPACE); its contents on entry are ignored.
 *   Other arguments and behaviour as fa_fwd.
 *
 * Arithmetic: bf16 products with fp32 accumulation; P and dS are rounded to
 * bf16 before they enter the dV, dK and dQ products; D in fp32; dQ and dK
 * carry the factor `scale`; outputs rounded to bf16 once at the end.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
           void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_strided - fa_bwd with Nq query rows and Nk key rows per head and
 * tensors in any layout whose head dimension is contiguous (the backward
 * counterpart of fa_fwd_strided).  The causal mask keeps key j for query i
 * when j <= i (top-left alignment, as fa_fwd_strided); with causal and
 * Nk > Nq the key rows j >= Nq see no query, so their dK and dV are zero.
 *
 *   q, o, dout, dq : bf16, Nq rows per head.   k, v, dk, dv : bf16, Nk rows per head.
 *   lse            : fp32 contiguous [B][H][Nq], the forward's L.
 *   strides        : host pointer to 24 element strides, three per tensor in
 *                    the order q, k, v, o, dout, dq, dk, dv; for each tensor
 *                    {batch, head, row}: element (b, h, i, c) sits at
 *                    b*s[0] + h*s[1] + i*s[2] + c.  Each stride >= 1 and
 *                    < 2^38 (else FA_ERR_BAD_SHAPE) and a multiple of 8
 *                    (16 bytes; else FA_ERR_MISALIGNED).  The caller keeps
 *                    the three output tensors free of overlap with each other
 *                    and with the inputs.
 *   workspace      : at least fa_bwd_workspace_bytes(B, H, Nq, d) bytes.
 *   Other arguments, checks and arithmetic as fa_bwd.
 */
int fa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                   const long long* strides, float scale, int causal,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_noalloc - fa_fwd for callers that must not allocate device memory.
 * (No counterpart in the pages: this entry point exists for deployment, not
 * for the method.)
 *
 * Who needs it: code that is handed a stream and must not allocate while it
 * runs - an operator or plug-in inside an inference runtime whose enqueue
 * call may not allocate (an allocation can synchronise the device, and memory
 * obtained while a stream is being captured cannot be relied on when the
 * graph replays), a latency-critical serving path that cannot afford the
 * implicit synchronisation and variable latency of cudaMalloc, or a process
 * that reserves all device memory up front.  fa_fwd allocates a small status
 * word on its first call on each device; this entry point never calls
 * cudaMalloc, cudaFree or any allocating routine.
 *
 * Arguments, layout, supported d, asynchrony and return codes are those of
 * fa_fwd (same kernel, same results).  The kernel's scratch - the status word
 * of its bounded device-side waits, 4 bytes, independent of B, H, N and d -
 * lives in a static device array of 256 bytes that every GPU which loads the
 * library holds until the process exits; a kernel that needed more than that
 * would be rejected with FA_ERR_SCRATCH before anything is enqueued.
 *
 * Each call first clears the status word with cudaMemsetAsync on `stream`,
 * then launches.  All calls on a device share the one array: calls whose
 * kernels overlap on the GPU (on different streams) race on it.  A wait that
 * expires ends the kernel early as with fa_fwd and is recorded in this shared
 * word; fa_status() reads (and clears) it as well, so it reports the expiry
 * of the latest fa_fwd_noalloc call on the device (the next call clears the
 * word first).  fa_status allocates its own status word on its first call on
 * a device, so a caller that may not allocate later makes that first call
 * at set-up.
 *
 * The first call on each device does the set-up (with that device current):
 * it looks up the array's device address with cudaGetSymbolAddress, queries
 * the device attributes and resolves the driver's tensor-map encoder.  Make
 * that first call before any stream capture begins.
 */
int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_status - synchronises `stream`, then reads and clears the device status
 * word of the current device, and the status word of fa_fwd_noalloc's static
 * scratch on that device.  Returns FA_OK, FA_ERR_TIMEOUT if a kernel
 * launched since the last call gave up on a bounded wait, or FA_ERR_CUDA if
 * the synchronisation itself failed.
 */
int fa_status(void* stream);

/*
 * fa_set_wait_limit_ms - time limit of every device-side wait in kernels
 * launched afterwards on any device (default 2000 ms; values < 1 are clamped
 * to 1).  Returns the previous limit.
 */
int fa_set_wait_limit_ms(int ms);

/*
 * fa_selftest_wait - diagnostic of the bounded device-side waits; the pages
 * have no counterpart (the waits and their time limit are this library's
 * failure handling).  Enqueues on `stream` one block whose warps wait, through
 * the attention kernels' own bounded-wait code, on barriers that nothing ever
 * signals.  After the current wait limit (fa_set_wait_limit_ms) the first
 * wait gives up, the block's other waits return at once, FA_ERR_TIMEOUT is
 * recorded in the device status word and the kernel ends; fa_status() then
 * reports it (and clears the word), and the device stays usable.  The kernel
 * holds no tensor memory, issues no copies and writes no caller memory.
 * Returns FA_OK when launched, FA_ERR_CUDA or FA_ERR_ARCH otherwise.
 */
int fa_selftest_wait(void* stream);

/* fa_strerror - static, human-readable name of a return code. */
const char* fa_strerror(int code);

/* fa_abi_version - version of this ABI (incremented on incompatible changes). */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

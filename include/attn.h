/*
 * attn.h — C ABI of the B300 (sm_103a) attention library (libswa_attn.so).
 *
 * The operation is the forward pass of a decoder's multi-head attention as the pages define it
 * (and, in attn_bwd, its gradient):
 *   out = softmax(Q^ K^^T / sqrt(D)) V                ("geometry_of_andrea" page,
 *                                                      "O que a Atenção Calcula",
 *                                                      "Escalonamento por sqrt(d_k)")
 * where Q^ and K^ are q and k after rotary position embedding and a parameter-free RMSNorm
 * over the head dimension (habr "Autoresearch" deep dive, train.py listing: apply_rotary_emb,
 * norm, CausalSelfAttention.forward), under a causal mask ("A Máscara Causal") and an optional
 * sliding window passed the way the listing passes window_size=(W, 0) to FlashAttention: query i
 * sees keys j with i - W <= j <= i. The "SSSL" layer pattern (three layers with W = T/2, then one
 * with W = T; listing, _compute_window_sizes) is a per-call `window` choice made by the caller.
 *
 * Conventions shared by every call:
 *  - Tensors are device pointers, row-major, contiguous, owned by the caller.
 *  - q, k, v, out: bf16, layout [B, T, H, D] (element (b, t, h, d) at ((b*T + t)*H + h)*D + d).
 *  - lse: fp32, layout [B, H, T].
 *  - Positions are 0..T-1 for every batch row. The softmax scale is fixed at 1/sqrt(D).
 *  - Q^ and K^ are rounded to bf16 before the products (as the listing's bf16 autocast does);
 *    the norm and rotation before that rounding are evaluated in fp32 (correctly rounded
 *    operations, cos / sin of the double-precision angle). Where the exact value lies within
 *    that evaluation's error of a bf16 rounding midpoint, either neighbouring bf16 value may
 *    result; everywhere else the rounded value is the exact one's.
 *  - Return value: ATTN_OK (0) or one of the negative ATTN_ERR_* codes below. Argument errors
 *    are detected on the host before anything is launched.
 *  - Calls are asynchronous on the given stream; results are ready when the stream is.
 *  - Results are deterministic: the same inputs give bit-identical outputs (except attn_bwd's dq,
 *    whose per-key-tile contributions are summed in the order they arrive).
 */
#ifndef SWA_ATTN_H
#define SWA_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_OK 0
#define ATTN_ERR_NOT_INITIALIZED (-1) /* attn_init has not succeeded yet (or attn_destroy ran) */
#define ATTN_ERR_INVALID_ARG (-2)     /* null / misaligned pointer, bad size, aliasing, bad float */
#define ATTN_ERR_UNSUPPORTED (-3)     /* valid request this build does not implement (e.g. D) */
#define ATTN_ERR_CUDA (-4)            /* a CUDA runtime / driver call failed */
#define ATTN_ERR_DEVICE_TIMEOUT (-5)  /* a kernel gave up on a bounded wait (see attn_device_status) */
#define ATTN_ERR_NO_DEVICE (-6)       /* no usable sm_103 device */
#define ATTN_ERR_SCRATCH_LIMIT (-7)   /* attn_fwd_noalloc: T * D / 2 exceeds its fixed cos/sin scratch */

/*
 * attn_init — prepare the library for CUDA device `device`.
 * Checks the device (compute capability 10.3), records its SM count, raises the kernels'
 * shared-memory limits, resolves the driver's tensor-map encoder, and allocates the device
 * error word. Idempotent for the same device; a different device returns ATTN_ERR_INVALID_ARG
 * until attn_destroy. Thread-safe. Does not change the calling thread's current device.
 */
int attn_init(int device);

/*
 * attn_fwd — one attention forward call.
 *
 *  q, k, v   [in]  bf16 [B, T, H, D], 16-byte aligned device pointers.
 *  out       [out] bf16 [B, T, H, D], 16-byte aligned; must not overlap q, k, v or lse.
 *  lse       [out] fp32 [B, H, T], natural-log log-sum-exp of the scaled scores of each query
 *                  row (ln sum_j exp(q^_i . k^_j / sqrt(D))); may be NULL (not written).
 *  B, H, T         >= 1; B*T*H*D < 2^31.
 *  D               head dimension: 32, 64 or 128 (other values: ATTN_ERR_UNSUPPORTED).
 *  window          < 0: no window. >= 0: query i sees keys j >= i - window (and, when
 *                  causal == 0, also j <= i + window). window >= T - 1 equals no window.
 *  causal          1: keys j <= i only ("A Máscara Causal"); 0: no causal cap.
 *  rope_base       > 0: rotary embedding with this base (the pages use 10000); 0: RoPE off.
 *                  Angle of pair i at position t: t * rope_base^(-2i/D), pairs (d, d + D/2).
 *  eps             >= 0: parameter-free RMSNorm of q and k rows with this epsilon;
 *                  < 0: no norm. (eps < 0 together with rope_base = 0 gives plain
 *                  softmax(Q K^T / sqrt(D)) V.)
 *  stream          a cudaStream_t (NULL = the legacy default stream) on the initialised device.
 *
 * The first call for a new (D, rope_base) pair, or for a T longer than any seen before with
 * that pair, builds the cos/sin table on the device (a cudaMalloc and a synchronous copy);
 * every later call allocates nothing and does not synchronise the host.
 *
 * The persistent kernel (D = 32, 64, 128) hands out work through a pair of device counters owned
 * by the library, and the kernel resets its pair when it finishes. Calls issued one after another
 * on a stream can therefore be repeated without limit. Outside stream capture each call takes the
 * next of 128 such pairs; a pair last used by a call on another stream is taken only after that
 * call's kernel has finished (the new call's stream waits for an event the library records after
 * every launch), so up to 128 calls run at the same time on different streams and further ones
 * wait. A call made while `stream` is being captured into a CUDA graph takes the next of another
 * 128 pairs and records no event (a captured launch cannot wait for work outside its graph):
 * graph launches that run at the same time on different streams must together hold at most 128
 * captured attention calls. Tensor maps of the buffers are cached by (pointer, shape).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int T, int D,
             int window, int causal, float rope_base, float eps, void* stream);

/* attn_fwd_gqa — attn_fwd with grouped K/V heads (habr "Autoresearch" deep dive, train.py
 * listing: GPTConfig.n_kv_head and CausalSelfAttention, where k and v are projected to
 * n_kv_head <= n_head heads, n_head % n_kv_head == 0, and passed to the attention call as
 * they are). Query head h attends with K/V head h / (H / H_kv), the convention of that call.
 *
 *  k, v      [in]  bf16 [B, T, H_kv, D], 16-byte aligned; out must not overlap them.
 *  H_kv            1 <= H_kv <= H and H % H_kv == 0 (else ATTN_ERR_INVALID_ARG).
 *  everything else as attn_fwd (q, out [B, T, H, D]; lse [B, H, T]). H_kv = H is exactly
 *  attn_fwd. The norm and rotation of each K row are applied once per query tile that reads
 *  it, as for attn_fwd.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int H_kv,
                 int T, int D, int window, int causal, float rope_base, float eps, void* stream);

/* attn_fwd_ve — attn_fwd_gqa on a layer with value embeddings (habr "Autoresearch" deep dive,
 * train.py listing, CausalSelfAttention.forward, value residual: layers with `has_ve` replace v by
 *   v' = v + 2 * sigmoid(ve_gate(x[..., :32])) * ve
 * where ve_gate is a bias-free linear map from the first 32 channels of the attention block's input
 * x to one logit per K/V head). A short pass first writes the gate factor 2 * sigmoid(...) of every
 * (b, t, K/V head) to `workspace`; the attention kernel then applies v + factor * ve to every V tile
 * in shared memory while it is staged, so v' never goes through HBM; v and ve are not modified. As in the listing every step is
 * a bf16 value: the logit (a 32-term dot product accumulated in fp32), the sigmoid, the product with
 * ve and the sum with v are each rounded to bf16 (a step whose exact value lies within the fp32
 * evaluation's error of a bf16 midpoint may round either way).
 *
 *  ve        [in]  bf16 [B, T, H_kv, D], 16-byte aligned: the value embeddings of the layer.
 *  x_gate    [in]  bf16, row (b, t) starts at x_gate + (b*T + t)*x_stride; its first 32 elements
 *                  are the gate's input (e.g. x itself with x_stride = n_embd). 16-byte aligned.
 *  x_stride        elements between consecutive rows: >= 32 and a multiple of 8.
 *  w_gate    [in]  bf16 [H_kv, 32], 16-byte aligned: the gate's weights (ve_gate.weight).
 *  workspace [tmp] device buffer of at least attn_fwd_ve_workspace_bytes(B, H_kv, T) bytes, 16-byte
 *                  aligned, caller-owned, not used by other work until the stream reaches the end of
 *                  this call; its contents on entry do not matter.
 *  everything else as attn_fwd_gqa. out, lse and workspace must not overlap ve or each other.
 * Returns ATTN_ERR_INVALID_ARG for a null ve / x_gate / w_gate or a bad stride, ATTN_ERR_UNSUPPORTED
 * when the persistent kernel is not available for D (see attn_fwd_kernel), else as attn_fwd_gqa.
 */
int attn_fwd_ve(const void* q, const void* k, const void* v, const void* ve, const void* x_gate, int x_stride,
                const void* w_gate, void* out, float* lse, void* workspace, size_t workspace_bytes, int B, int H,
                int H_kv, int T, int D, int window, int causal, float rope_base, float eps, void* stream);

/* attn_fwd_ve_workspace_bytes — size of attn_fwd_ve's workspace (0 for a non-positive size). */
size_t attn_fwd_ve_workspace_bytes(int B, int H_kv, int T);

/* attn_fwd_kernel — which kernel attn_fwd launches for head dimension D on the initialised
 * device: 1 = the warp-specialised persistent kernel (TMA-fed K/V ring, tcgen05 MMAs into TMEM,
 * separate prologue, MMA and softmax warps; D = 32, 64 and 128), 0 = the single-warpgroup kernel
 * (only when the warp-specialised kernel was not compiled to the register count its run-time
 * register split needs). ATTN_ERR_UNSUPPORTED for other D, ATTN_ERR_NOT_INITIALIZED
 * before attn_init. Both kernels compute the same function (see attn_fwd). */
int attn_fwd_kernel(int D);

/* attn_bwd_workspace_bytes — size of the scratch buffer attn_bwd needs for this shape (0 for a
 * non-positive size). */
size_t attn_bwd_workspace_bytes(int B, int H, int H_kv, int T, int D);

/* attn_bwd — gradients of sum(out * dout) with respect to q, k and v for the forward that
 * attn_fwd / attn_fwd_gqa compute with the same arguments. The pages train the model (habr
 * "Autoresearch" deep dive, train.py listing: loss.backward() through CausalSelfAttention.forward,
 * i.e. apply_rotary_emb, norm and the attention call under bf16 autocast), so this is that
 * forward's derivative taken where the listing's backward takes it: at the bf16 Q^, K^ (the cast
 * passes gradients through unchanged), then back through the RMSNorm and the rotation:
 *   P = exp(Q^ K^^T / sqrt(D) - lse) on the visible keys, dV = P^T dO, dP = dO V^T,
 *   delta_i = dO_i . out_i, dS = P (dP - delta), dQ^ = dS K^ / sqrt(D), dK^ = dS^T Q^ / sqrt(D),
 *   d(x r) = r dy - (r^3 / D) (x . dy) x for the norm, and the rotation by -angle for RoPE.
 * With grouped K/V heads, dk and dv sum over the query heads sharing a K/V head.
 *
 *  q          [in]  bf16 [B, T, H, D], 16-byte aligned.
 *  k, v       [in]  bf16 [B, T, H_kv, D], 16-byte aligned.
 *  out        [in]  bf16 [B, T, H, D]: the forward's output for these inputs.
 *  lse        [in]  fp32 [B, H, T]: the forward's log-sum-exp (natural log), 4-byte aligned.
 *  dout       [in]  bf16 [B, T, H, D]: gradient of the loss with respect to out.
 *  dq         [out] fp32 [B, T, H, D];  dk, dv [out] fp32 [B, T, H_kv, D]; 16-byte aligned.
 *  workspace  [tmp] device buffer of at least attn_bwd_workspace_bytes(B, H, H_kv, T, D) bytes,
 *                   256-byte aligned, owned by the caller; its contents on entry do not matter
 *                   and it must not be used by other work until the stream reaches the end of
 *                   this call.
 *  B, H, H_kv, T, D, window, causal, rope_base, eps, stream: as attn_fwd_gqa. D = 32, 64, 128.
 * Outputs must not overlap an input, each other or the workspace (ATTN_ERR_INVALID_ARG).
 * Accuracy: P and dS are rounded to bf16 for their products (fp32 accumulation), delta is taken
 * from the bf16 out; dq, dk, dv are fp32. Launches three kernels on `stream`: a prologue pass
 * (Q^, K^, delta), the tcgen05 kernel (one CTA per batch row, K/V head and 128-key tile) and the
 * dq pass. Returns ATTN_OK, ATTN_ERR_NOT_INITIALIZED, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED
 * or ATTN_ERR_CUDA; a bounded wait that gives up is reported through attn_device_status.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
             float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes, int B, int H, int H_kv, int T,
             int D, int window, int causal, float rope_base, float eps, void* stream);

/* attn_destroy — free the cos/sin tables and the error word; idempotent. The caller must make
 * sure no attn_fwd work is still running. After it, attn_init may be called again. */
void attn_destroy(void);

/* attn_status_string — a static, human-readable name for a status code. Never NULL. */
const char* attn_status_string(int status);

/* attn_device_status — synchronise the device, read and clear the device error word.
 * Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, ATTN_ERR_NOT_INITIALIZED or ATTN_ERR_CUDA. */
int attn_device_status(void);

/* attn_selftest_wait_timeout — exercise the kernels' bounded-wait path without any fault.
 * Launches one small kernel on `stream` that waits on a shared-memory barrier nothing will ever
 * arrive on, using the same bounded wait (about 1.5 s of %globaltimer) as the attention kernels.
 * The wait gives up, the kernel writes the timeout code to the device error word and returns
 * normally; the context stays usable. A following attn_device_status() then returns
 * ATTN_ERR_DEVICE_TIMEOUT. Not part of the computation (the pages have no counterpart); it
 * exists so the failure-reporting path can be tested on real hardware. */
int attn_selftest_wait_timeout(void* stream);

/* attn_fwd_noalloc — the same forward call as attn_fwd, for callers that must not allocate.
 *
 * The pages have no counterpart; this is a deployment convenience. Some callers cannot call
 * cudaMalloc: serving processes whose device memory is carved up in advance by a framework
 * allocator or a fixed-size memory pool (a library allocation outside it can fail or break the
 * budget), and plug-in hosts that forbid a library from allocating device memory behind their
 * back. attn_fwd allocates its cos/sin table on the first call for a (D, rope_base) pair and
 * needs attn_init, which allocates the device error word; this entry point needs neither.
 *
 * Arguments, layouts, semantics and return codes are those of attn_fwd. Differences:
 *  - Everything it needs beyond the caller's tensors lives in one file-scope device array of the
 *    library (4 MiB + 256 bytes), which every GPU that loads the library holds until the process
 *    exits: the error word and a cos/sin table of at most 524288 (cos, sin) pairs. Requests with
 *    rope_base > 0 and T * D / 2 > 524288 (for example T > 16384 at D = 64, T > 8192 at D = 128)
 *    return ATTN_ERR_SCRATCH_LIMIT without launching anything.
 *  - It runs on the calling thread's current device; `stream` must belong to that device.
 *    attn_init is not required.
 *  - The first call on a device does a one-time set-up on the host (checks the device, raises the
 *    kernels' shared-memory limits, looks up the array's device address); make that first call
 *    before any stream capture.
 *  - Each call with rope_base > 0 enqueues, on `stream`, a small kernel that rebuilds the table
 *    for (T, D, rope_base) in the array (cos / sin evaluated in double on the device, stored as
 *    fp32), then the attention kernel. All calls share the one array and it keeps the last call's
 *    contents: calls whose work overlaps on the GPU (other streams, other threads) race on it and
 *    must be serialised by the caller.
 *  - A bounded-wait timeout of this path is recorded in that shared error word, where it stays
 *    until attn_noalloc_status reads and clears it; attn_device_status does not see it. */
int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int T,
                     int D, int window, int causal, float rope_base, float eps, void* stream);

/* attn_noalloc_status — read and clear the error word of attn_fwd_noalloc on the current device.
 * The pages have no counterpart. Waits for `stream` (which must belong to the current device),
 * copies the word out of the library's fixed array and writes zero back, both through copies to
 * and from host variables: nothing is allocated. Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT if an
 * attn_fwd_noalloc kernel gave up on a bounded wait since the last read, or ATTN_ERR_CUDA /
 * ATTN_ERR_NO_DEVICE. Like attn_fwd_noalloc, its first call on a device does the one-time set-up. */
int attn_noalloc_status(void* stream);

/* attn_noalloc_selftest_wait_timeout — the bounded-wait self test of attn_selftest_wait_timeout,
 * writing its timeout code to attn_fwd_noalloc's error word instead of attn_init's, so that
 * attn_noalloc_status can be tested on hardware without any fault. Allocates nothing. */
int attn_noalloc_selftest_wait_timeout(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SWA_ATTN_H */

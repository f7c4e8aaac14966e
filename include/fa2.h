/*
 * fa2.h -- C ABI of the GB300 (sm_103a) exact FlashAttention-2 forward pass.
 *
 * The operation (one call = one forward pass over a batch of heads):
 *
 *     for every batch b < B, head h < H, query row i < Lq:
 *         s_ij   = scale * sum_d Q[b,h,i,d] * K[b,h,j,d]      for visible keys j
 *         O[b,h,i,:] = sum_j softmax_j(s_i.) * V[b,h,j,:]
 *         LSE[b,h,i] = ln sum_j exp(s_ij)                       (natural log)
 *
 * with visible keys j < Lk, and additionally j <= i when causal != 0.
 * This is exact scaled-dot-product attention as defined in Olowookere,
 * "FlashAttention-2 from scratch with a custom Triton kernel" (section "The
 * core idea: making attention IO-aware": S = QK^T, P = softmax(S), O = PV,
 * computed by streaming K/V blocks with an online softmax and never writing
 * the score matrix to memory), with the causal rule and the per-row
 * log-sum-exp output of "Chapter 08: Flash Attention -- blocked attention"
 * (sections 3 "LSE" and 4 "causal mask"), and the host-wrapper contract of
 * page 1's section "Host wrapper and kernel launch" (inputs in, O and the
 * per-row statistic out, grid over query blocks x batch*head).
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense, row-major, contiguous:
 *       q, o : bf16 [B, H, Lq, D]      k, v : bf16 [B, H, Lk, D]
 *       lse  : fp32 [B, H, Lq]
 *     bf16 is passed as raw 16-bit storage (void*).
 *   - D must be 64, 128 or 256.  scale must be finite and > 0 (the pages use
 *     1/sqrt(D)).  Causal with Lq != Lk uses the top-left rule j <= i.
 *   - Device pointers must be 16-byte aligned (TMA requirement); lse 4-byte.
 *   - The caller owns every buffer, except the fixed scratch that
 *     fa2_fwd_noalloc takes from the library.  No entry point allocates
 *     device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are stream-ordered and asynchronous: they return once
 *     the work is enqueued, and never synchronise except where stated.
 *   - Re-entrant and thread-safe; the library keeps no per-call state (but
 *     calls of fa2_fwd_noalloc that overlap on the GPU share its scratch).
 *   - O and LSE rows i >= Lq are never written; inputs are never written.
 *   - Per device, the library looks up the device addresses of its own
 *     globals (the error word, fa2_fwd_noalloc's scratch) once and keeps them
 *     for the life of the process.  Tearing the device's context down between
 *     calls (cudaDeviceReset) is not supported.
 */
#ifndef FA2_GB300_H
#define FA2_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa2_status {
    FA2_OK = 0,
    FA2_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad scale */
    FA2_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (D) */
    FA2_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    FA2_ERR_TIMEOUT = 4       /* a kernel wait exceeded its limit (see below) */
} fa2_status;

/*
 * fa2_fwd -- the forward pass on device buffers.
 *
 *   q, k, v  device pointers to the bf16 inputs (read only).
 *   o        device pointer, bf16 [B, H, Lq, D] output.
 *   lse      device pointer, fp32 [B, H, Lq] output, natural-log LSE.
 *   B, H     batch and head counts (>= 1, B*H <= 2^31 - 1).
 *   Lq, Lk   query / key lengths (Lq >= 0, Lk >= 1).  Lq == 0 is a no-op.
 *   D        head dimension: 64, 128 or 256.
 *   causal   0 = full attention, nonzero = key j visible to query i iff j <= i.
 *   scale    score multiplier, finite and > 0.
 *   stream   cudaStream_t as void*.
 *
 * Returns FA2_OK once the kernel is enqueued; FA2_ERR_INVALID_ARG or
 * FA2_ERR_UNSUPPORTED before touching the GPU when an argument is rejected;
 * FA2_ERR_CUDA if building the TMA descriptors or the launch fails.
 * Kernel-side wait time-outs are reported later by fa2_get_device_error().
 */
fa2_status fa2_fwd(const void *q, const void *k, const void *v, void *o,
                   float *lse, int B, int H, int Lq, int Lk, int D,
                   int causal, float scale, void *stream);

/*
 * fa2_fwd_ex -- the forward pass on strided views ("FlashAttention-2 from
 * scratch with a custom Triton kernel", host wrapper and kernel launch: the
 * kernel is given each tensor's batch, head, row and column strides).  Same
 * computation as fa2_fwd, with an optional sliding window (as fa2_fwd_window)
 * and workspace (as fa2_fwd_ws).
 *
 *   q, k, v, o    bf16 [B, H, L, D] views whose rows of D elements are
 *                 contiguous; element (b, h, i, d) of q is at
 *                 q + b*q_strides[0] + h*q_strides[1] + i*q_strides[2] + d,
 *                 likewise k, v (L = Lk) and o (L = Lq).  A NULL stride array
 *                 means contiguous [B, H, L, D].  Every stride is in elements,
 *                 positive and a multiple of 8 (16 bytes; the TMA loads and the
 *                 16-byte row stores need it), at most 2^38.  The rows of o must
 *                 not overlap; q, k and v may (e.g. slices of one packed QKV
 *                 tensor, or [B, L, H, D] storage viewed as [B, H, L, D]).
 *   lse           fp32 [B, H, Lq] contiguous.
 *   window        -1: none; w >= 0: causal sliding window, query i sees keys
 *                 i - w .. i (requires causal and Lq <= Lk, as fa2_fwd_window).
 *   workspace     optional, as fa2_fwd_ws (used by non-causal calls without a
 *                 window; 256-byte aligned when given).
 *   (other arguments as for fa2_fwd)
 *
 * Errors as fa2_fwd, plus FA2_ERR_INVALID_ARG for a stride that breaks the
 * rules above, a bad window or a misaligned workspace.
 */
fa2_status fa2_fwd_ex(const void *q, const void *k, const void *v, void *o,
                      float *lse, int B, int H, int Lq, int Lk, int D,
                      const long long *q_strides, const long long *k_strides,
                      const long long *v_strides, const long long *o_strides,
                      int causal, int window, float scale, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * fa2_fwd_window -- fa2_fwd for causal attention restricted to a sliding
 * window: query i sees keys i - window <= j <= i ("Flash Attention:
 * principles and implementation" (tbr8.org), section 6.3, window_size =
 * (window, 0) with causal=True: `window` keys to the left, none to the right).
 * K/V tiles entirely left of a query tile's band are never visited, so the
 * work grows as Lq * window instead of Lq * Lk / 2.
 *
 *   window   >= 0 (0: each query sees only its own key; >= Lk: plain causal).
 *   Lq <= Lk is required (every row keeps key i).
 *   (other arguments as for fa2_fwd)
 *
 * Errors: as fa2_fwd; FA2_ERR_INVALID_ARG for window < 0 or Lq > Lk.
 */
fa2_status fa2_fwd_window(const void *q, const void *k, const void *v, void *o,
                          float *lse, int B, int H, int Lq, int Lk, int D,
                          int window, float scale, void *stream);

/*
 * fa2_workspace_size -- bytes of device workspace fa2_fwd_ws needs for this
 * problem on `device` (its SM count sets the schedule).  *bytes = 0 when the
 * pass uses none: causal passes, Lq == 0, and non-causal shapes for which
 * dealing out whole query tiles already keeps the SMs evenly busy (the cut
 * ranges are only used when they are estimated to save at least 5 %).  The
 * environment variable FA2_SPLIT=always (or =never) overrides that estimate
 * for this call and for the fa2_fwd_ws calls that follow; it must not change
 * between sizing a workspace and the calls that use it.
 *
 *   B .. causal  as for fa2_fwd.
 *   device       CUDA device ordinal the pass will run on.
 *   bytes        out: required size in bytes.
 *
 * Returns FA2_OK; FA2_ERR_INVALID_ARG / FA2_ERR_UNSUPPORTED as fa2_fwd;
 * FA2_ERR_CUDA if the device cannot be queried.
 */
fa2_status fa2_workspace_size(int B, int H, int Lq, int Lk, int D, int causal,
                              int device, size_t *bytes);

/*
 * fa2_fwd_ws -- fa2_fwd with a caller-owned device workspace, which lets a
 * non-causal pass balance the work evenly over the SMs: the key-tile
 * iterations of all query tiles are cut into one range per SM, the ranges
 * balanced in tiles plus a fixed cost per query tile they touch, and a
 * query tile whose keys straddle two ranges is computed in parts that are
 * merged afterwards: each part's O and log-sum-exp are combined exactly as
 * the online softmax merges two key blocks (Olowookere, "FlashAttention-2
 * from scratch with a custom Triton kernel", section "Running max m_i and
 * running normaliser"; "Chapter 08: Flash Attention -- blocked attention",
 * section 2).  Causal passes ignore the workspace (they balance whole tiles,
 * heaviest first).
 *
 *   workspace        device pointer, 256-byte aligned, at least
 *                    fa2_workspace_size() bytes, ZERO-FILLED before its first
 *                    use; every completed call leaves it ready for the next
 *                    (the arrival counters at its start, the only part that
 *                    must start at zero, are zero again).
 *   workspace_bytes  its size.
 *   (other arguments as for fa2_fwd)
 *
 * A NULL workspace (allowed when fa2_workspace_size reports 0) runs the pass
 * as fa2_fwd does.  Calls that may run at the same time (different streams)
 * must not share a workspace.  Errors: as fa2_fwd, plus FA2_ERR_INVALID_ARG
 * for a misaligned workspace or one smaller than the pass needs.
 */
fa2_status fa2_fwd_ws(const void *q, const void *k, const void *v, void *o,
                      float *lse, int B, int H, int Lq, int Lk, int D,
                      int causal, float scale, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * fa2_fwd_noalloc -- fa2_fwd_ws for callers that may not allocate device
 * memory, with the workspace taken from a fixed scratch buffer that lives in
 * the library itself (FA2_NOALLOC_SCRATCH_BYTES per device).  The FlashAttention
 * write-ups this library follows have no counterpart to this entry point.
 *
 * Who cannot allocate: code hosted inside a framework that owns every byte of
 * device memory through its own pool and budget (a plug-in may only use the
 * pointers it is handed, since a side cudaMalloc would escape that budget),
 * and latency-critical loops that rule out cudaMalloc / cudaFree because
 * either can synchronise the device and take unbounded time.  This entry point
 * calls neither, nor any routine that allocates.
 *
 * Same arguments, outputs, schedule and results (bit for bit) as fa2_fwd_ws
 * given a workspace of fa2_workspace_size() bytes.
 *
 *   - The first call on a device does the set-up: it looks up the scratch's
 *     device address with that device current (and the CUDA module holding it
 *     is loaded then).  Make that first call before any stream capture.
 *   - Each call clears the arrival counters at the start of the scratch (the
 *     only part that must start at zero) with a memset enqueued on `stream`,
 *     ahead of the kernel.
 *   - The scratch is one buffer per device, shared by every call: calls that
 *     overlap on the GPU (e.g. enqueued on different streams without ordering
 *     between them) race on it and their outputs are undefined.  Order them
 *     on one stream, or use fa2_fwd_ws with a workspace per stream.
 *
 * Errors: as fa2_fwd_ws; FA2_ERR_UNSUPPORTED when the pass needs more than
 * FA2_NOALLOC_SCRATCH_BYTES of workspace (fa2_workspace_size() tells how much
 * it needs; no shape does on a GPU with at most 152 SMs); FA2_ERR_CUDA if the
 * scratch cannot be looked up or cleared.
 */
#define FA2_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)

fa2_status fa2_fwd_noalloc(const void *q, const void *k, const void *v, void *o,
                           float *lse, int B, int H, int Lq, int Lk, int D,
                           int causal, float scale, void *stream);

/*
 * fa2_fwd_fp8 -- the forward pass on e4m3 inputs: the FP8 mode of
 * FlashAttention-3 that "Flash Attention: principles and implementation"
 * (tbr8.org), section 4.3, names.  The page fixes no format; this library's
 * reading: Q, K and V are stored as e4m3 (OCP FP8 E4M3: bias 7, largest finite
 * 448, no infinities) with one fp32 descale per (batch, head) each, the real
 * input being the stored value times its descale.  The pass computes
 *
 *     s_ij = scale * dq[b,h] * dk[b,h] * sum_d Q8[b,h,i,d] * K8[b,h,j,d]
 *     O[b,h,i,:] = dv[b,h] * sum_j P~_ij V8[b,h,j,:] / sum_j P~_ij
 *     LSE[b,h,i] = ln sum_j exp(s_ij)                       (natural log)
 *
 * where the products accumulate in fp32 on the tensor cores (kind::f8f6f4)
 * and P~ are the softmax weights (relative to the running row max, at most
 * 2^8) rounded to e4m3 for the P V product; O is divided by the sum of those
 * rounded weights and LSE comes from the unrounded fp32 sum.
 *
 *   q, k, v     device pointers, e4m3 bytes [B, H, Lq|Lk, D], contiguous.
 *   descale_q, descale_k, descale_v
 *               device pointers, fp32 [B, H] (4-byte aligned), read only.
 *   o, lse      as fa2_fwd (bf16 O, fp32 natural-log LSE of the real scores).
 *   D           must be 128.
 *   workspace, workspace_bytes
 *               optional, as fa2_fwd_ws; the size is fa2_workspace_size() of
 *               the same problem with D = 128 (NULL: whole query tiles).
 *
 * Errors: as fa2_fwd_ws; FA2_ERR_INVALID_ARG also for a missing or misaligned
 * descale pointer; FA2_ERR_UNSUPPORTED for D != 128.
 */
fa2_status fa2_fwd_fp8(const void *q, const void *k, const void *v,
                       const float *descale_q, const float *descale_k,
                       const float *descale_v, void *o, float *lse, int B,
                       int H, int Lq, int Lk, int D, int causal, float scale,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * fa2_bwd_workspace_size -- bytes of device workspace fa2_bwd needs: two fp32
 * per query row (-lse * log2 e and -Delta), rows padded to a multiple of 64
 * per head.  Returns FA2_OK; FA2_ERR_INVALID_ARG for bad sizes;
 * FA2_ERR_UNSUPPORTED for D other than 64, 128 or 256.
 */
fa2_status fa2_bwd_workspace_size(int B, int H, int Lq, int Lk, int D, size_t *bytes);

/*
 * fa2_bwd -- the backward pass of the same attention ("Chapter 08: Flash
 * Attention -- blocked attention", section 6): given dout = dL/dO, writes
 *
 *     Delta_i = sum_d dout_id * o_id                 (into the workspace)
 *     dS      = P * (dout V^T - Delta)               (P recomputed from lse)
 *     dv = P^T dout,   dk = scale * dS^T q,   dq = scale * dS k
 *
 * with the same scores, scale and causal rule as fa2_fwd; o and lse must be
 * that call's outputs for the same q, k, v.  Three kernels run in order on
 * `stream`: Delta, dq (query tiles resident), dk and dv (key tiles resident).
 *
 *   q, k, v, o   device bf16 inputs (layouts as fa2_fwd); lse fp32 [B, H, Lq].
 *   dout         device bf16 [B, H, Lq, D].
 *   dq           device bf16 [B, H, Lq, D] output.
 *   dk, dv       device bf16 [B, H, Lk, D] outputs (zero rows for keys no
 *                query sees, e.g. causal keys beyond the last query).
 *   D            64, 128 or 256 (FA2_ERR_UNSUPPORTED otherwise).  At 256 two CTAs
 *                share each resident tile, each accumulating half of the
 *                gradient columns.
 *   workspace    device pointer, 16-byte aligned, at least
 *                fa2_bwd_workspace_size() bytes; overwritten (may be NULL
 *                when Lq == 0, where dk and dv are simply zeroed).
 *   (other arguments as for fa2_fwd)
 *
 * Errors as fa2_fwd, plus FA2_ERR_INVALID_ARG for a missing or misaligned
 * dout/dq/dk/dv/workspace or a workspace that is too small.
 */
fa2_status fa2_bwd(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dout, void *dq, void *dk,
                   void *dv, int B, int H, int Lq, int Lk, int D, int causal,
                   float scale, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * fa2_bwd_window -- the backward pass of fa2_fwd_window's sliding-window
 * attention ("Flash Attention: principles and implementation", section 6.3,
 * window_size = (window, 0) with causal): query i sees keys
 * max(0, i - window) .. i only, so P, dS and the gradients are those of that
 * mask.  o and lse must be fa2_fwd_window's outputs for the same window.
 * dk and dv rows of keys that no query sees are zero.
 *
 *   window       >= 0; Lq <= Lk (as fa2_fwd_window).
 *   (other arguments, workspace and errors as fa2_bwd; FA2_ERR_INVALID_ARG for
 *   window < 0 or Lq > Lk)
 */
fa2_status fa2_bwd_window(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, void *dq, void *dk,
                          void *dv, int B, int H, int Lq, int Lk, int D, int window,
                          float scale, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * fa2_bwd_ex -- the backward pass on strided views, the counterpart of
 * fa2_fwd_ex: the same computation as fa2_bwd (causal flag) or fa2_bwd_window
 * (window >= 0, which requires causal and Lq <= Lk), with every [B, H, L, D]
 * tensor given as a view whose rows of D elements are contiguous.
 *
 *   q, k, v, o, dout   bf16 inputs; dq, dk, dv bf16 outputs.  Element
 *                      (b, h, i, d) of x is at x + b*x_strides[0] +
 *                      h*x_strides[1] + i*x_strides[2] + d.  A NULL stride
 *                      array means contiguous [B, H, L, D].  Every stride is in
 *                      elements, positive, a multiple of 8 (16 bytes) and at
 *                      most 2^38.  The rows of dq, dk and dv must not overlap
 *                      one another; the inputs may.
 *   lse                fp32 [B, H, Lq] contiguous (fa2_fwd_ex's output).
 *   window             -1: none; w >= 0: as fa2_bwd_window.
 *   (other arguments and the workspace as fa2_bwd)
 *
 * Errors as fa2_bwd, plus FA2_ERR_INVALID_ARG for a stride that breaks the
 * rules above or a bad window.
 */
fa2_status fa2_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, void *dq, void *dk, void *dv,
                      int B, int H, int Lq, int Lk, int D,
                      const long long *q_strides, const long long *k_strides,
                      const long long *v_strides, const long long *o_strides,
                      const long long *do_strides, const long long *dq_strides,
                      const long long *dk_strides, const long long *dv_strides,
                      int causal, int window, float scale, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * fa2_fwd_from_host -- the same pass starting from, and ending in, HOST
 * memory: copies q, k, v from the host into the caller's device staging
 * buffers, runs the pass, and copies O and LSE back into the caller's host
 * buffers.  Host buffers should be pinned (page-locked) for the copies to be
 * asynchronous.
 *
 * The work is cut into up to 8 chunks of whole heads and overlapped: chunk c's
 * kernel runs while chunk c+1's inputs arrive and chunk c-1's outputs leave.
 * Copies and kernels run on three streams of the library's own (per device,
 * created by the first call), ordered after all work already enqueued on
 * `stream`, and `stream` waits for them: once `stream` has been synchronised,
 * o_host and lse_host hold the results.  Calls from several host threads
 * enqueue one at a time.
 *
 *   q_host .. lse_host   host pointers (same layouts as fa2_fwd).
 *   q_dev  .. lse_dev    caller-owned device buffers of the same sizes.
 *
 * Errors: as fa2_fwd; FA2_ERR_CUDA if a copy cannot be enqueued or the
 * library's streams cannot be created.
 */
fa2_status fa2_fwd_from_host(const void *q_host, const void *k_host,
                             const void *v_host, void *o_host, float *lse_host,
                             void *q_dev, void *k_dev, void *v_dev, void *o_dev,
                             float *lse_dev, int B, int H, int Lq, int Lk,
                             int D, int causal, float scale, void *stream);

/*
 * fa2_get_device_error -- synchronises `stream`, then reads and clears the
 * library's device-side error word on the current device.  Every inter-warp
 * wait inside the kernels is bounded (one second; FA2_WAIT_LIMIT_MS in the
 * environment changes it); a wait that runs out records a code here, the
 * kernel winds down without hanging the GPU (each CTA first waits for the
 * copies and MMAs it has issued), and the outputs of that call are undefined
 * (a workspace it used must be zero-filled again before reuse).
 *
 * The word is one per device, shared by every stream and every call of this
 * library on that device: the first fa2_get_device_error to read it after a
 * time-out reports and clears it, whichever stream that call names.  `stream`
 * only selects what is synchronised before the read, so to attribute a
 * time-out to one stream's calls, read the word with every other stream of
 * this library idle.
 *
 * For tests only, two environment variables (read on every call) exercise
 * this path in the forward kernel: FA2_TEST_STALL=1 makes its softmax warps
 * first wait on a barrier nothing completes (that wait runs out, then the
 * other roles' waits on them), and FA2_TEST_WAIT_LIMIT_NS (nanoseconds)
 * shortens its inter-warp waits so the test ends quickly; the waits for a
 * CTA's own copies and MMAs keep the full bound.
 *
 *   detail   optional (may be NULL): receives the raw code (0 = none): the
 *            waiting role in bits 8-11 (forward: 1 TMA producer, 2 MMA
 *            issuer, 3 softmax, 4 a CTA's final wait for its own work;
 *            backward: 5 producer, 6 MMA issuer, 7 elementwise warps) and the
 *            barrier in the low byte.
 *
 * Returns FA2_OK, FA2_ERR_TIMEOUT, or FA2_ERR_CUDA if the synchronisation or
 * the read fails.
 */
fa2_status fa2_get_device_error(void *stream, int *detail);

/* Static human-readable name of a status code (never NULL). */
const char *fa2_status_string(fa2_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int fa2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA2_GB300_H */

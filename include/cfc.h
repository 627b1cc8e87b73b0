/*
 * cfc.h -- C ABI of the batched CfC K-loop library for one NVIDIA GB300 (sm_103a).
 *
 * The three operations of the method:
 *
 *   cfc_kloop_forward   the three-head closed-form continuous-time (CfC) cell
 *                       run over K steps for B independent samples;
 *   cfc_kloop_backward  backward through time: parameter gradients summed over
 *                       the batch, grad_h0 and (optionally) grad_x;
 *   reduce_axis0        deterministic, atomic-free column sum [B, N] -> [N];
 *
 * and around them:
 *
 *   reduce_axis0_multi  reduce_axis0 for a list of matrices in few launches;
 *   cfc_tau_kloop_*     the pages' single-head tau-cell K loop (FP32);
 *   cfc_grn_*           the multi-horizon GRN heads on every K position (FP32);
 *   cfc_kloop_forward_backward_static
 *                       forward + backward for callers that cannot allocate
 *                       device memory (fixed workspace inside the library);
 *   helpers             workspace sizes, status strings, the device error
 *                       word and its self-test, per-kernel event tracing.
 *
 * Cell (per sample, step k = 0..K-1, heads c = f, g, h~ in that order):
 *   A_c    = b[c] + W_in[c] x_k + W_rec[c] h_k
 *   g      = tanh(A_g),  hh = tanh(A_h~),  gate = sigmoid(-A_f * dt) = 1/(1+exp(A_f dt))
 *   h_{k+1} = gate * g + (1 - gate) * hh,   h_seq[:, k] = h_{k+1}
 * The per-sample pre-activation over row-major [n_hid, n_in] / [n_hid, n_hid]
 * weights, tanh as the squashing function, the argument order of the backward,
 * overwrite-vs-accumulate rules and the optional grad_x follow "K-loop
 * Parallelization Implementation Plan", Tasks 2 and 3 (cfc_step_batched and
 * cfc_step_backward_batched).  The reducer follows Task 1 of that page
 * (reduce_axis0: argument order, overwrite, summation order).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     every buffer.  Nothing is allocated, freed or synchronised inside a call.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and runs asynchronously in stream order.
 *   - A non-zero return value means the arguments were rejected (nothing was
 *     launched) or a launch failed; cfc_status_string() names the reason.
 *   - Results are bit-identical from run to run for the same inputs,
 *     configuration and GPU model: no atomics, fixed summation orders.
 *   - Layouts are dense row-major with the last index fastest.
 *
 * Precision modes (`math`):
 *   CFC_MATH_FP32  x, h0, W_in, W_rec, h_seq are float; all arithmetic fp32.
 *   CFC_MATH_TF32  same storage as FP32; every operand of the projections and
 *                  gradient contractions (x, h, W, dA) is rounded to TF32 (10
 *                  mantissa bits, nearest, ties away from zero), products are
 *                  accumulated in fp32.  Activations and state stay fp32.
 *   CFC_MATH_BF16  x, h0, W_in, W_rec and h_seq are bfloat16 (raw 16-bit);
 *                  b, dt, y, grad inputs and all gradient outputs are float.
 *                  h_{k+1} is rounded to bf16 (nearest even) and that value is
 *                  stored and carried; dA is rounded to bf16 before the
 *                  gradient contractions; accumulation is fp32.
 */
#ifndef CFC_H_
#define CFC_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CFC_OK = 0,
  CFC_ERR_NULL = -1,      /* a required pointer is NULL                        */
  CFC_ERR_SHAPE = -2,     /* a size is negative, zero where not allowed, or too large */
  CFC_ERR_ALIGN = -3,     /* a pointer is not aligned to its element size      */
  CFC_ERR_WORKSPACE = -4, /* workspace NULL or smaller than cfc_kloop_workspace_bytes() */
  CFC_ERR_MODE = -5,      /* unknown math mode or gradient path                */
  CFC_ERR_LAUNCH = -6,    /* a kernel launch failed (cudaGetLastError != 0)    */
  CFC_ERR_DEVICE = -7,    /* no usable CUDA device / unsupported architecture  */
  CFC_ERR_TOO_LARGE = -8  /* sizes need more than CFC_STATIC_WORKSPACE_BYTES   */
} cfc_status;

typedef enum { CFC_MATH_FP32 = 0, CFC_MATH_TF32 = 1, CFC_MATH_BF16 = 2 } cfc_math;

/* How the per-sample parameter gradients are summed over the batch.
 *   CFC_GRAD_SCRATCH: each sample's packed gradient row (length N, below) is
 *     written once to a caller-provided per_sample_scratch[B, N] (overwrite;
 *     the K steps are summed on chip), then reduce_axis0 sums the B rows.
 *     This is the pages' per-batch scratch + reducer scheme ("K-loop
 *     Parallelization Implementation Plan", Tasks 3-5).
 *   CFC_GRAD_GEMM: the gradients are contracted directly over all B*K rows
 *     (dW = dA^T [x; h; 1]) as one batch-dimension GEMM with a fixed split
 *     over row blocks; the split partials live in the workspace and are summed
 *     by reduce_axis0 ("kernel-optimization" plan, Task 2 Step 3: weight
 *     gradient as a batch-dimension GEMM).
 * Packed per-sample layout, N = 3*(n_in + n_hid + 1)*n_hid floats:
 *   [ gW_in (c, i, j) : 3*n_hid*n_in | gW_rec (c, i, j) : 3*n_hid*n_hid | gb (c, i) : 3*n_hid ] */
typedef enum { CFC_GRAD_SCRATCH = 0, CFC_GRAD_GEMM = 1 } cfc_grad_path;

/* Human-readable name of a status code (static string, never NULL). */
const char* cfc_status_string(int status);

/* N = 3*(n_in + n_hid + 1)*n_hid, or 0 for invalid sizes. Host-only. */
long long cfc_per_sample_length(int n_in, int n_hid);

/* Bytes of device workspace that cfc_kloop_forward and cfc_kloop_backward
 * need for these sizes (the same value for both calls).  Host-only; returns 0
 * for invalid arguments.  The forward stores the activations of every step
 * there and the backward reads them, so the same workspace, untouched, must be
 * passed to the backward of the same inputs. */
size_t cfc_kloop_workspace_bytes(int B, int K, int n_in, int n_hid, int math, int grad_path);

/* Number of rows S of the gradient partials [S, N] that the backward sums with
 * reduce_axis0 (B for CFC_GRAD_SCRATCH; a fixed split of the B*K rows for
 * CFC_GRAD_GEMM).  Host-only; 0 for invalid arguments. */
int cfc_kloop_grad_splits(int B, int K, int n_in, int n_hid, int math, int grad_path);

/* Device-side error word of the library (host-blocking diagnostic: waits for
 * all work on the device).  Returns 0 if no kernel has reported an error,
 * 1 if a tensor-core kernel gave up a bounded wait (its outputs are then not
 * valid), or CFC_ERR_DEVICE if the word cannot be read.  clear != 0 resets it. */
int cfc_device_error(int clear);

/* Diagnostic of the timeout path: launches one kernel whose bounded mbarrier
 * wait (the wait helper of the K-loop kernels) runs out after max_polls polls
 * (1 .. 2^20) because nothing completes the barrier; the kernel then sets the
 * device error word and returns, so cfc_device_error reports 1 afterwards.  No
 * other state changes; the context stays usable.  CFC_ERR_SHAPE for max_polls
 * out of range. */
int cfc_selftest_timeout(int max_polls, void* stream);

/* Forward K-loop.
 *   x      [B, K, n_in]      (float or bf16 by `math`)
 *   h0     [B, n_hid]        (float or bf16)
 *   W_in   [3, n_hid, n_in]  heads f, g, h~ (float or bf16)
 *   W_rec  [3, n_hid, n_hid] (float or bf16)
 *   b      [3, n_hid]        float
 *   dt     [B] float if dt_stride == 1, or one float broadcast if dt_stride == 0
 *   h_seq  [B, K, n_hid]     OUTPUT, overwrite: h_seq[:, k] = h_{k+1}
 *   workspace / workspace_bytes: see cfc_kloop_workspace_bytes.
 * Requirements: B >= 1, K >= 1, 1 <= n_in, 1 <= n_hid <= 1024, n_in + n_hid <= 1024;
 * every pointer aligned to 16 bytes. */
int cfc_kloop_forward(const void* x, const void* h0, const void* W_in, const void* W_rec,
                      const float* b, const float* dt, int dt_stride,
                      int B, int K, int n_in, int n_hid, int math,
                      void* h_seq, void* workspace, size_t workspace_bytes, void* stream);

/* Backward through the K loop of the forward that wrote `workspace`.
 * Inputs as in the forward, plus
 *   h_seq        [B, K, n_hid] as written by that forward
 *   grad_h_seq   [B, K, n_hid] float or NULL: upstream gradient of every h_seq[:, k]
 *   grad_h_last  [B, n_hid] float or NULL: extra upstream gradient of h_K
 *   y            [B, n_hid] float or NULL: target of the loss 0.5*||h_K - y||^2;
 *                adds h_K - y to the gradient of h_K
 * Outputs (all overwrite; the three parameter gradients are summed over B):
 *   grad_W_in [3, n_hid, n_in], grad_W_rec [3, n_hid, n_hid], grad_b [3, n_hid]
 *   grad_h0   [B, n_hid] or NULL
 *   grad_x    [B, K, n_in] or NULL (as in the pages' backward, grad_x is optional)
 *   per_sample_scratch [B, N] float: required for CFC_GRAD_SCRATCH (it then
 *                holds each sample's packed gradient), ignored (may be NULL)
 *                for CFC_GRAD_GEMM.
 * At least one upstream gradient (grad_h_seq, grad_h_last or y) must be given. */
int cfc_kloop_backward(const void* x, const void* h0, const void* W_in, const void* W_rec,
                       const float* b, const float* dt, int dt_stride,
                       int B, int K, int n_in, int n_hid, int math,
                       const void* h_seq, const float* grad_h_seq, const float* grad_h_last,
                       const float* y,
                       float* grad_W_in, float* grad_W_rec, float* grad_b,
                       float* grad_h0, float* grad_x,
                       float* per_sample_scratch, int grad_path,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Column sum of a row-major [n_batch, n_tail] float matrix into out[n_tail]
 * (overwrite), atomic-free, in a fixed association order that is bit-identical
 * to the pages' reference reducer ("K-loop Parallelization Implementation
 * Plan", Task 1): with 256 partial sums,
 *   p[t] = ((0.0f + in[t]) + in[t+256]) + in[t+512] + ...,  t = 0..255,
 * then p[t] += p[t+s] for s = 128, 64, ..., 1 and t < s;  out[j] = p[0].
 * n_batch == 0 writes +0.0f.  n_batch >= 0, 0 <= n_tail <= 2^35; per_batch and
 * out must be 4-byte aligned and must not overlap (16-byte alignment and
 * n_tail % 4 == 0 select the float4 path; otherwise scalar, same order). */
int reduce_axis0(const float* per_batch, int n_batch, long long n_tail, float* out, void* stream);

/* ---------------------------------------------------------------------------
 * The pages' single-head tau-cell ("K-loop Parallelization Implementation
 * Plan", Task 2: cfc_step_batched, Task 3: cfc_step_backward_batched), FP32:
 *   pre = b + W_in x_k + W_rec h_k,  s = tanh(pre),
 *   decay_i = exp(-dt / max(tau_i, 1e-6)),  h_{k+1} = h_k * decay + (1 - decay) * s,
 *   h_seq[:, k] = h_{k+1}.
 * Backward (dh = gradient reaching h_{k+1}): d_pre = dh (1 - decay)(1 - s^2);
 * gb += d_pre, gW_in += d_pre (x) x_k, gW_rec += d_pre (x) h_k,
 * gtau += dh (h_k - s) decay dt / max(tau, 1e-6)^2 where tau > 1e-6 (else 0);
 * grad h_k = W_rec^T d_pre + dh decay, grad x_k = W_in^T d_pre.
 * Shapes: x [B, K, n_in], h0 [B, n_hid], W_in [n_hid, n_in], W_rec [n_hid, n_hid],
 * b [n_hid], tau [n_hid], dt [B] (dt_stride 1) or [1] (dt_stride 0).  Every
 * pointer 16-byte aligned.  Sizes: 1 <= n_in, n_hid <= 1024 and the sample's
 * weights and gradient, 2 n_hid ((n_in + n_hid) | 1) floats, within one SM's
 * shared memory (about 28 K floats each; n_in = 64, n_hid = 128 fits) —
 * otherwise CFC_ERR_SHAPE. */

/* Packed per-sample gradient length (n_in + n_hid + 2) * n_hid, layout
 * [gW_in (i, j) | gW_rec (i, j) | gb (i) | gtau (i)]; 0 if unsupported. */
long long cfc_tau_per_sample_length(int n_in, int n_hid);

/* Workspace bytes of the tau-cell forward/backward pair (the saved s values),
 * 0 for unsupported sizes. */
size_t cfc_tau_kloop_workspace_bytes(int B, int K, int n_in, int n_hid);

/* Forward K loop: h_seq [B, K, n_hid] (overwrite) and s in the workspace. */
int cfc_tau_kloop_forward(const float* x, const float* h0, const float* W_in, const float* W_rec, const float* b,
                          const float* tau, const float* dt, int dt_stride, int B, int K, int n_in, int n_hid,
                          float* h_seq, void* workspace, size_t workspace_bytes, void* stream);

/* Backward through the K loop of the forward that filled `workspace`.
 * Upstream gradients as for cfc_kloop_backward (at least one of grad_h_seq
 * [B, K, n_hid], grad_h_last [B, n_hid], y [B, n_hid]).  Outputs (overwrite):
 * grad_W_in [n_hid, n_in], grad_W_rec [n_hid, n_hid], grad_b [n_hid],
 * grad_tau [n_hid] summed over the batch by reduce_axis0 from
 * per_sample_scratch [B, cfc_tau_per_sample_length] (written, required);
 * grad_h0 [B, n_hid] and grad_x [B, K, n_in] optional (NULL). */
int cfc_tau_kloop_backward(const float* x, const float* h0, const float* W_in, const float* W_rec,
                           const float* b, const float* tau, const float* dt, int dt_stride, int B, int K,
                           int n_in, int n_hid, const float* h_seq, const float* grad_h_seq,
                           const float* grad_h_last, const float* y, float* grad_W_in, float* grad_W_rec,
                           float* grad_b, float* grad_tau, float* grad_h0, float* grad_x,
                           float* per_sample_scratch, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Multi-horizon GRN heads on every K position of the trunk state, FP32.
 * Forward per horizon j of a row h (the ml-alpha commit history, commit "wire
 * TFT GRN heads into PerceptionTrainer (Phase 1.7)"):
 *   z1 = W1[j] h + b1[j],  a1 = GELU(z1) (exact: z Phi(z)),  z2 = W2[j] a1 + b2[j],
 *   gate = w_gate[j].z2 + b_gate[j],  main = w_main[j].z2 + b_main[j],
 *   skip = w_skip[j].h + b_skip[j],   p[j] = sigmoid(skip + sigmoid(gate) main).
 * Backward ("K-loop Parallelization Implementation Plan", Commit 2 / Task 11):
 * the chain rule of that forward from dL/dp, with
 *   grad_h = grad_h_carry + sum_j lambda[j] (W1[j]^T dz1_j + dskip_j w_skip[j])
 * (lambda scales the trunk gradient only) and every parameter gradient summed
 * per sample over its K rows (k = K-1 .. 0), then over the batch by
 * reduce_axis0.
 * Sizes: hidden (Hd) a multiple of 4 in [4, 256], head_mid (M) a multiple of 4
 * in [4, 64], n_horizons (J) in [1, 8]; otherwise CFC_ERR_SHAPE.  Rows are
 * r = b*K + k, so h may be the K loop's h_seq [B, K, Hd] and grad_h its
 * grad_h_seq.  Parameters (and gradients) are one packed vector of
 * cfc_grn_param_length floats, the ten tensors in this order, horizon-major:
 * [W1 (J,M,Hd) | b1 (J,M) | W2 (J,M,M) | b2 (J,M) | w_gate (J,M) | b_gate (J) |
 *  w_main (J,M) | b_main (J) | w_skip (J,Hd) | b_skip (J)].
 * Every pointer 16-byte aligned (CFC_ERR_ALIGN). */

/* Packed parameter / per-sample gradient length; 0 if unsupported. */
long long cfc_grn_param_length(int hidden, int head_mid, int n_horizons);

/* Floats per row of the forward's saved intermediates (z1, a1, z2 [J, M],
 * gate, main [J]): J (3 M + 2); 0 if unsupported. */
long long cfc_grn_saved_per_row(int head_mid, int n_horizons);

/* Workspace bytes of cfc_grn_backward for B*K rows; 0 if unsupported. */
size_t cfc_grn_workspace_bytes(int B, int K, int hidden, int head_mid, int n_horizons);

/* Forward over `rows` rows: probs [rows, J] and saved [rows, saved_per_row]
 * (both overwrite).  rows = 0 is a no-op. */
int cfc_grn_forward(const float* h, long long rows, int hidden, int head_mid, int n_horizons,
                    const float* params, float* probs, float* saved, void* stream);

/* Backward of the forward that wrote probs and saved for h [B*K, Hd]:
 * grad_probs [B*K, J] = dL/dp, lambda [J], grad_h_carry [B*K, Hd] (optional,
 * NULL = zero).  Outputs (overwrite): grad_h [B*K, Hd], per_sample_scratch
 * [B, cfc_grn_param_length] (each sample's gradient), grad_params
 * [cfc_grn_param_length] (their sum in reduce_axis0's order). */
int cfc_grn_backward(const float* h, int B, int K, int hidden, int head_mid, int n_horizons, const float* params,
                     const float* probs, const float* saved, const float* grad_probs, const float* lambda,
                     const float* grad_h_carry, float* grad_h, float* per_sample_scratch, float* grad_params,
                     void* workspace, size_t workspace_bytes, void* stream);

/* reduce_axis0 for `count` independent matrices with one launch per kernel
 * configuration (the pages' training step calls the reducer 17 times, once per
 * scratch buffer: "K-loop Parallelization Implementation Plan", Self-Review).
 * per_batch, n_batch, n_tail and out are HOST arrays of `count` entries; entry
 * i is a device matrix [n_batch[i], n_tail[i]] and its device output
 * out[i][n_tail[i]] (overwrite), with the rules of reduce_axis0.  Every out[i]
 * receives exactly the bits reduce_axis0 would write.  0 <= count <= 4096;
 * entries with n_tail 0 are skipped; matrices and outputs must not overlap.
 * All entries are checked before anything is launched. */
int reduce_axis0_multi(const float* const* per_batch, const int* n_batch, const long long* n_tail,
                       float* const* out, int count, void* stream);

/* Forward + backward without allocation.  This entry point has no counterpart
 * in the pages; it exists for callers that cannot allocate device memory
 * when they run the K loop (code running under an allocator it does not own,
 * plugins barred from cudaMalloc, real-time loops where an allocation would
 * stall).  It computes what cfc_kloop_forward followed by cfc_kloop_backward
 * with CFC_GRAD_GEMM computes, but keeps the whole workspace in a fixed device
 * array inside the library and always runs the CUDA-core (SIMT) kernels: the
 * SIMT forward and backward K loops, the SIMT weight-gradient tiles and
 * reduce_axis0, in every precision mode.  The regular entry points choose
 * cluster or tensor-core kernels, which sum in other orders, so the two
 * agree within the parity tolerances (fp32: 1e-4 relative; TF32 / bf16:
 * 2e-3 normwise), not bit for bit; each is run-to-run bit-identical.
 *   - The array holds CFC_STATIC_WORKSPACE_BYTES bytes on every device that
 *     loads the library, until the process exits.  Sizes whose SIMT workspace
 *     (the W_cat^T copy, the [B,K,3H] activations and dA, and the weight
 *     gradient's split partials) is larger are rejected with
 *     CFC_ERR_TOO_LARGE before anything is launched.
 *   - The caller passes all inputs and outputs (same meaning, layout and
 *     overwrite rules as the two calls it replaces); nothing is allocated or
 *     freed by the call.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  The address is kept for the life of the process: a
 *     device reset after that first call is not supported.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Nothing in it has to start at zero (every part that is read is written
 *     earlier in the same call), but calls whose work overlaps on the GPU
 *     (for example on two streams) race on it and must be serialised. */
#define CFC_STATIC_WORKSPACE_BYTES (16u << 20)
int cfc_kloop_forward_backward_static(const void* x, const void* h0, const void* W_in,
                                      const void* W_rec, const float* b, const float* dt,
                                      int dt_stride, int B, int K, int n_in, int n_hid, int math,
                                      const float* grad_h_seq, const float* grad_h_last,
                                      const float* y,
                                      void* h_seq, float* grad_W_in, float* grad_W_rec,
                                      float* grad_b, float* grad_h0, float* grad_x, void* stream);

/* Kernel tracing (diagnostics, off by default).  While enabled, every kernel
 * that this library launches is bracketed by two CUDA events recorded on its
 * launch stream, so per-kernel device time can be read back afterwards.
 * Host-side state, not thread-safe; the events are created by the library
 * (the only resources it creates), so do not enable tracing inside CUDA-graph
 * capture.
 *   cfc_trace_enable(on): clears all records; on != 0 starts recording.
 *   cfc_trace_count():    number of recorded launches.
 *   cfc_trace_get(i, &name, &ms): kernel name (static string) and device time
 *                         in milliseconds of record i; waits for that record's
 *                         stop event.  Returns CFC_OK or CFC_ERR_SHAPE for a
 *                         bad index. */
int cfc_trace_enable(int on);
int cfc_trace_count(void);
int cfc_trace_get(int i, const char** name, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* CFC_H_ */

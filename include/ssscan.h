/*
 * ssscan.h — C ABI of libssscan.so: the Mamba selective-scan forward and
 * backward, the depthwise causal conv1d backward and the RMSNorm backward,
 * written for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a caller-owned DEVICE pointer to a dense,
 *   row-major (C-contiguous) buffer; strided views are not accepted (the
 *   rustytorch backward_cuda commit message reports a GPU matmul that read a
 *   strided view's storage as if it were dense).  The library never allocates or frees memory
 *   in these calls; scratch comes from the caller's `workspace`, sized by the
 *   matching *_workspace_size() query.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls only enqueue work on it and return; device-side failures
 *   surface at the caller's next synchronisation or through ss_device_status().
 * - Return value: SS_OK (0) or a negative SS_ERR_* code.  Arguments are
 *   validated on the host before anything is launched; on an error nothing
 *   is launched and no output is touched.  ss_strerror() gives the text.
 * - Activations (x, delta, z, dy, y, Bm, Cm of the scan; x of conv1d; x, dy of
 *   RMSNorm) are fp32 (SS_F32) or bf16 (SS_BF16) as given by `dtype`; states,
 *   checkpoints, A, D, weights and every gradient are fp32.
 * - Gradients of parameters ACCUMULATE (+=): dA, dD, dw, db, dscale.
 *   Gradients of activations are OVERWRITTEN (=): dx, ddelta, dz, dB, dC,
 *   dh0 — the convention of mamba-rs backward_ops.rs ("accumulated" weight,
 *   bias and scale gradients; "overwritten" input gradients).
 * - Reductions are deterministic: fixed-order trees over per-block partials,
 *   no atomics.  Two identical calls give bitwise-identical results.
 */
#ifndef SSSCAN_H
#define SSSCAN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SS_OK 0
#define SS_ERR_NULL (-1)        /* a required pointer is NULL */
#define SS_ERR_DIM (-2)         /* a size is <= 0, or out of the supported range */
#define SS_ERR_UNSUPPORTED (-3) /* N not in {4,8,16}, unknown dtype, d_conv not in 1..4, chunk not 8 or a multiple of 16 */
#define SS_ERR_ALIGN (-4)       /* a pointer is not 16-byte aligned, or D / dim not a multiple of 8 */
#define SS_ERR_WORKSPACE (-5)   /* workspace NULL or smaller than the *_workspace_size() query */
#define SS_ERR_CUDA (-6)        /* a CUDA runtime call or kernel launch failed */
#define SS_ERR_DEVICE (-7)      /* a kernel gave up on a bounded wait (ss_device_status) */

/* activation dtypes */
#define SS_F32 0
#define SS_BF16 1

/* Human-readable text of a status code (static storage, never NULL). */
const char* ss_strerror(int code);

/*
 * Number of checkpoints the forward writes: ceil(L / chunk).
 */
int ss_scan_num_chunks(int L, int chunk);

/*
 * Workspace bytes ss_scan_fwd needs for these sizes (0 on invalid sizes, and
 * 0 when the layer has enough (batch row, channel) parallelism by itself).
 */
size_t ss_scan_fwd_workspace_size(int B, int L, int D, int N, int chunk, int dtype);

/*
 * ss_scan_fwd — selective-scan forward.
 *
 * The diagonal selective SSM trained by backpropagation through time in the
 * rustytorch MambaBlock (whose scan runs step by step) and mamba-rs
 * (backpropagation through time through the state); per batch b, channel d,
 * state n, step t:
 *     a_t   = exp(delta_t[d] * A[d,n])
 *     h_t   = a_t * h_{t-1} + delta_t[d] * B_t[n] * x_t[d]        (h_{-1} = h0, or 0)
 *     y_t[d] = (sum_n C_t[n] * h_t[d,n] + D[d] * x_t[d]) * silu(z_t[d])
 *
 *   x, delta, z : [B, L, D]  activations (dtype); delta is already positive (post-softplus)
 *   A           : [D, N]     fp32 (negative for a decaying state)
 *   Bm, Cm      : [B, L, N]  activations (dtype), shared by all D channels
 *   Dv          : [D]        fp32 skip weight
 *   h0          : [B, D, N]  fp32 initial state, or NULL for zeros
 *   y           : [B, L, D]  output (dtype; bf16 is rounded to nearest even)
 *   ckpt        : [B, ceil(L/chunk), D, N] fp32 output: ckpt[b,c,d,:] is the
 *                 state entering step c*chunk (c = 0 holds h0 or zeros).  The
 *                 backward rebuilds every other state from these.
 *   h_last      : [B, D, N]  fp32 final state h_{L-1}, or NULL
 *   chunk       : checkpoint interval: 8, or a multiple of 16.  chunk = 8
 *                 lets the backward skip its recompute pass at the price of
 *                 N*4 bytes of checkpoint per 8 steps and channel.
 *   N           : 4, 8 or 16;  D: a multiple of 8
 *   dt_bias, delta_softplus : the discretisation of delta fused in front of
 *                 the scan (the Mamba layer's delta = softplus(raw + dt_bias)):
 *                 the recurrence uses f(delta + dt_bias[d]) with f = softplus
 *                 when delta_softplus != 0 (softplus(v) = log(1 + e^v)), else
 *                 the identity; dt_bias is [D] fp32 or NULL (zero).  With
 *                 dt_bias NULL and delta_softplus 0, delta is used as given.
 *   workspace   : device scratch of at least ss_scan_fwd_workspace_size()
 *                 bytes (NULL allowed when that is 0), 16-byte aligned,
 *                 contents need not be initialised.  When B*D is small the
 *                 sequence is cut into segments; the scratch holds each
 *                 segment's zero-start end state and its sum of delta, from
 *                 which every segment composes the state it starts from.
 * Alignment: every pointer 16-byte aligned.
 */
int ss_scan_fwd(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                const float* Dv, const void* z, const float* h0,
                void* y, float* ckpt, float* h_last,
                int B, int L, int D, int N, int chunk, int dtype,
                const float* dt_bias, int delta_softplus,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * Workspace bytes ss_scan_bwd needs for these sizes (0 on invalid sizes).
 */
size_t ss_scan_bwd_workspace_size(int B, int L, int D, int N, int chunk, int dtype);

/*
 * ss_scan_bwd — reverse-mode gradient of  sum(y * dy) + sum(h_last * dh_last)
 * through ss_scan_fwd (backpropagation through time through the SSM state).
 *
 * Inputs are those of the forward plus
 *   ckpt     : [B, ceil(L/chunk), D, N] the forward's checkpoints, same chunk (at most 512)
 *   dy       : [B, L, D] activations (dtype): dL/dy
 *   dh_last  : [B, D, N] fp32 gradient arriving on the final state, or NULL (zero)
 * Outputs (fp32):
 *   dx, ddelta, dz : [B, L, D]   overwritten
 *   dB, dC         : [B, L, N]   overwritten (summed over the D channels)
 *   dA             : [D, N]      accumulated (+=, summed over batch and time)
 *   dD             : [D]         accumulated (+=)
 *   dh0            : [B, D, N]   overwritten, or NULL to skip
 * with, for G_t = dL/dh_t = ds_t*C_t + a_{t+1}*G_{t+1},  ds_t = dy_t*silu(z_t):
 *   q_t = G_t*a_t*h_{t-1};  ddelta_t = sum_n (q_t*A + G_t*B_t*x_t);
 *   dx_t = ds_t*D + delta_t*sum_n G_t*B_t;  dz_t = dy_t*s_t*silu'(z_t);
 *   dA += sum q_t*delta_t;  dB_t = sum_d G_t*delta_t*x_t;  dC_t = sum_d ds_t*h_t;
 *   dD += sum ds_t*x_t;  dh0 = a_0*G_0.
 * With the fused discretisation (dt_bias / delta_softplus as in ss_scan_fwd,
 * which must have been called with the same values), ddelta is the gradient
 * with respect to the raw delta: the above times softplus'(v) = sigmoid(v)
 * (evaluated as 1 - exp(-delta)) when delta_softplus, and
 *   d_dt_bias : [D] fp32, accumulated (+=) with sum_{b,t} of that ddelta, or NULL.
 * The states are rebuilt chunk by chunk from `ckpt`, never stored in full.
 * workspace: device scratch of at least ss_scan_bwd_workspace_size() bytes,
 *   16-byte aligned, contents need not be initialised.
 */
int ss_scan_bwd(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                const float* Dv, const void* z, const float* ckpt, const void* dy, const float* dh_last,
                float* dx, float* ddelta, float* dz, float* dA, float* dB, float* dC, float* dD, float* dh0,
                int B, int L, int D, int N, int chunk, int dtype,
                const float* dt_bias, int delta_softplus, float* d_dt_bias,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * Sequence sharding.  The recurrence of ss_scan_fwd over steps t0 .. t1-1 of a
 * channel is an affine map of the state entering the piece,
 *     h -> exp(A * sum_t delta_t) * h + h_end,
 * where h_end is the state the piece reaches from a zero start: the product
 * of the a_t over the piece is the exponential of A times the piece's sum of
 * delta.  The adjoint of ss_scan_bwd is the same map run the other way,
 *     g -> exp(A * sum_t delta_t) * g + g_start,
 * from the carry arriving at the piece's end to the adjoint it sends out of its
 * first step (g_start: that adjoint when nothing arrives, i.e. a_0 * G_0 of the
 * piece with dh_last = 0).  Composing these maps over the pieces in order
 * (ss_scan_carries) gives every piece the state (forward) or carry (backward)
 * it starts from; ss_scan_fwd with h0 = that state and ss_scan_bwd with
 * dh_last = that carry then give each piece exactly its part of the scan over
 * the whole sequence (up to rounding order), so that a sequence cut along
 * time over P ranks needs one exchange of [B, D, N] + [B, D] per pass.
 *
 * ss_scan_fwd_summary — one piece's forward summary:
 *   x, delta : [B, L, D];  Bm : [B, L, N]  (dtype; the piece's steps only)
 *   A        : [D, N] fp32
 *   h_end    : [B, D, N] fp32 output, the state after the piece's last step from h = 0
 *   delta_sum: [B, D]    fp32 output, sum over the piece of delta (after the
 *              fused discretisation dt_bias / delta_softplus, as in ss_scan_fwd)
 * Sizes, dtypes and alignment as ss_scan_fwd; no workspace.
 */
int ss_scan_fwd_summary(const void* x, const void* delta, const float* A, const void* Bm,
                        float* h_end, float* delta_sum, int B, int L, int D, int N, int dtype,
                        const float* dt_bias, int delta_softplus, void* stream);

/*
 * ss_scan_bwd_summary — one piece's backward summary:
 *   delta, z, dy : [B, L, D];  Cm : [B, L, N]  (dtype; the piece's steps only)
 *   A        : [D, N] fp32
 *   g_start  : [B, D, N] fp32 output, what ss_scan_bwd would give as dh0 for
 *              the piece with dh_last NULL
 *   delta_sum: [B, D] fp32 output, as in ss_scan_fwd_summary
 * Sizes, dtypes and alignment as ss_scan_bwd; no workspace.
 */
int ss_scan_bwd_summary(const void* delta, const float* A, const void* Cm, const void* z, const void* dy,
                        float* g_start, float* delta_sum, int B, int L, int D, int N, int dtype,
                        const float* dt_bias, int delta_softplus, void* stream);

/*
 * ss_scan_carries — composes the P pieces' maps (piece-major arrays, as an
 * all-gather over ranks delivers them):
 *   delta_sum : [P, B, D]    fp32, summ : [P, B, D, N] fp32 (h_end or g_start)
 *   init      : [B, D, N]    fp32 carry entering the whole scan (h0 forward,
 *               dh_last backward), or NULL for zeros
 *   carry     : [P, B, D, N] fp32 output
 *   reverse 0 (forward):  carry[0] = init,   carry[p+1] = exp(A*delta_sum[p]) * carry[p] + summ[p]
 *   reverse 1 (backward): carry[P-1] = init, carry[p-1] = exp(A*delta_sum[p]) * carry[p] + summ[p]
 * so carry[p] is the state entering piece p (forward) or the carry arriving at
 * its end (backward); summ[P-1] (forward) and summ[0] (backward) are not read.
 * The maps are composed by an associative scan in the kernel.
 * 1 <= P <= 64 (else SS_ERR_UNSUPPORTED); B < 65536; pointers 4-byte aligned.
 */
int ss_scan_carries(const float* A, const float* delta_sum, const float* summ, const float* init, float* carry,
                    int P, int B, int D, int N, int reverse, void* stream);

/*
 * Workspace bytes conv1d_causal_bwd needs (0 on invalid sizes).
 */
size_t conv1d_causal_bwd_workspace_size(int B, int L, int D, int d_conv);

/*
 * conv1d_causal_bwd — backward of the depthwise causal conv1d
 *     out[b,t,d] = bias[d] + sum_k w[d,k] * x[b, t-(d_conv-1)+k, d]      (x at t<0 is 0)
 * whose per-channel shift register holds the newest input at tap d_conv-1
 * (mamba-rs backward_ops.rs, backward_conv1d_step).  Full-sequence gradient:
 *   dout : [B, L, D] fp32, dL/dout (the gradient after the SiLU backward)
 *   x    : [B, L, D] conv input (x_dtype: SS_F32 or SS_BF16)
 *   w    : [D, d_conv] fp32
 *   dx   : [B, L, D] fp32, overwritten: dx[s] = sum_k dout[s+d_conv-1-k] * w[k]
 *   dw   : [D, d_conv] fp32, accumulated: += sum_{b,t} dout[t] * x[t-(d_conv-1)+k]
 *   db   : [D] fp32, accumulated: += sum_{b,t} dout[t]
 * d_conv in 1..4; D a multiple of 8; pointers 16-byte aligned.  dw and db
 * equal the pages' per-step contributions summed over every step.
 */
int conv1d_causal_bwd(const float* dout, const void* x, const float* w,
                      float* dx, float* dw, float* db,
                      int B, int L, int D, int d_conv, int x_dtype,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * conv1d_causal_silu_bwd — conv1d_causal_bwd fused with the SiLU backward of
 * the conv -> SiLU branch (see conv1d_causal_fwd with silu = 1): given
 *   dact : [B, L, D] fp32, dL/d(silu(pre)),
 * it forms g = dact * silu'(pre) with pre = bias + sum_k w[k] x[t-(d_conv-1)+k]
 * recomputed from x, w and bias (NULL: zero), silu'(v) = s (1 + v (1 - s)),
 * s = sigmoid(v), and then writes / accumulates dx, dw, db exactly as
 * conv1d_causal_bwd does with dout = g (db is the bias gradient).  Same
 * workspace (conv1d_causal_bwd_workspace_size), sizes and alignment rules;
 * bias 16-byte aligned when given.
 */
int conv1d_causal_silu_bwd(const float* dact, const void* x, const float* w, const float* bias,
                           float* dx, float* dw, float* db, int B, int L, int D, int d_conv, int x_dtype,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * Workspace bytes rmsnorm_bwd needs (0 on invalid sizes).
 */
size_t rmsnorm_bwd_workspace_size(int rows, int dim);

/*
 * rmsnorm_bwd — backward of y[r,i] = x[r,i] * scale[i] / rms[r]
 * (mamba-rs backward_ops.rs, backward_rms_norm):
 *   inv = 1/rms[r];  dot = inv^2 * sum_i dy*scale*x
 *   dx[r,i]    = inv * (scale[i]*dy[r,i] - x[r,i]*dot/dim)     overwritten
 *   dscale[i] += sum_r dy[r,i]*x[r,i]*inv                        accumulated
 *   dy, x : [rows, dim] (dtype);  scale : [dim] fp32;  rms : [rows] fp32, the
 *   root mean square saved by the forward (not its inverse; eps already inside);
 *   dx : [rows, dim] fp32;  dscale : [dim] fp32.
 * dim a multiple of 8 and at most 32768; pointers 16-byte aligned.
 */
int rmsnorm_bwd(const void* dy, const void* x, const float* scale, const float* rms,
                float* dx, float* dscale, int rows, int dim, int dtype,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * rmsnorm_bwd_noalloc — rmsnorm_bwd for callers that cannot allocate device
 * memory: code that runs under an allocator it does not own (a host
 * framework's operator or plugin interface that hands over only inputs and
 * outputs), or that cannot pay the device-wide synchronisation a cudaMalloc /
 * cudaFree may cause in a latency-critical loop.  The pages have no
 * counterpart of this entry point; it computes exactly what rmsnorm_bwd
 * computes, with the same argument meaning, layout and errors, minus the
 * workspace arguments.
 *   - Scratch: a fixed array inside the library (4 MiB per GPU that loads the
 *     library, held until the process exits) takes the per-block dscale
 *     partials; nothing is allocated or freed by the call.
 *   - Limit: dim <= 8192; larger dim returns SS_ERR_DIM before any launch.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array: calls that may overlap on the GPU
 *     (other streams, other host threads) race on it and must be serialised
 *     by the caller.  Each call overwrites every partial it reads, so no
 *     clearing is needed.
 *   - dscale partials are summed over a different number of blocks than in
 *     rmsnorm_bwd, so dscale can differ from rmsnorm_bwd's in the last bits;
 *     dx is identical.
 */
int rmsnorm_bwd_noalloc(const void* dy, const void* x, const float* scale, const float* rms,
                        float* dx, float* dscale, int rows, int dim, int dtype, void* stream);

/*
 * conv1d_causal_fwd — the depthwise causal conv1d that conv1d_causal_bwd
 * differentiates, with an optional SiLU on its output (the conv -> SiLU branch
 * in front of the scan).  The pages give only the backward (mamba-rs
 * backward_ops.rs, backward_conv1d_step, whose shift register fixes the tap
 * order: newest input at tap d_conv-1); this is the operation it inverts:
 *   pre[b,t,d] = bias[d] + sum_k w[d,k] * x[b, t-(d_conv-1)+k, d]      (x at t<0 is 0)
 *   out[b,t,d] = silu ? pre * sigmoid(pre) : pre
 *   x    : [B, L, D] (x_dtype: SS_F32 or SS_BF16)
 *   out  : [B, L, D] same dtype, overwritten (bf16 rounded to nearest even)
 *   w    : [D, d_conv] fp32;  bias : [D] fp32, or NULL for zero
 * d_conv in 1..4; D a multiple of 8; x, out and bias 16-byte aligned.
 */
int conv1d_causal_fwd(const void* x, const float* w, const float* bias, void* out,
                      int B, int L, int D, int d_conv, int silu, int x_dtype, void* stream);

/*
 * rmsnorm_fwd — RMSNorm forward, producing the root mean square that
 * rmsnorm_bwd takes (mamba-rs backward_ops.rs, backward_rms_norm receives the
 * saved rms itself):
 *   rms[r]   = sqrt(mean_i x[r,i]^2 + eps)
 *   y[r,i]   = x[r,i] * scale[i] / rms[r]
 *   x, y  : [rows, dim] (dtype; y overwritten, bf16 rounded to nearest even)
 *   scale : [dim] fp32;  rms : [rows] fp32 output, or NULL
 * dim a multiple of 8 and at most 32768; eps >= 0 (else SS_ERR_DIM);
 * x, y, scale and rms 16-byte aligned.
 */
int rmsnorm_fwd(const void* x, const float* scale, float eps, void* y, float* rms,
                int rows, int dim, int dtype, void* stream);

/*
 * ss_scan_step — one recurrent step of the selective SSM for B independent
 * sequences (decode): the recurrence of ss_scan_fwd at a single t, with the
 * state carried in place.  Running it L times from h equals ss_scan_fwd over
 * those L steps from h0 = h (up to rounding order): the rustytorch
 * rtx-transformers tests listing (mamba_step_equivalence.rs) exposes the
 * recurrent state as a single-step updater pinned by that equivalence.
 *   x, delta, z : [B, D] (dtype);  Bm, Cm : [B, N] (dtype)
 *   A : [D, N] fp32;  Dv : [D] fp32
 *   h : [B, D, N] fp32, read and overwritten with the new state
 *   y : [B, D] (dtype) output: (sum_n Cm[n] h[d,n] + Dv[d] x[d]) * silu(z[d])
 * N in {4, 8, 16}; A and h 16-byte aligned.
 */
int ss_scan_step(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                 const float* Dv, const void* z, float* h, void* y, int B, int D, int N, int dtype,
                 void* stream);

/*
 * conv1d_causal_step — one step of the depthwise causal conv1d (+ optional
 * SiLU) for B sequences, with the shift register carried in place (mamba-rs
 * backward_ops.rs, backward_conv1d_step: the current input enters at tap
 * d_conv-1):
 *   conv_state : [B, D, d_conv] fp32, newest input at index d_conv-1; every
 *                tap moves one place towards 0 and x enters at d_conv-1
 *   out[b,d]   = act(bias[d] + sum_k w[d,k] * conv_state[b,d,k])   (after the shift)
 *   x, out : [B, D] (dtype);  w : [D, d_conv] fp32;  bias : [D] fp32 or NULL
 * Running it L times from a zero state equals conv1d_causal_fwd over L steps.
 */
int conv1d_causal_step(const void* x, float* conv_state, const float* w, const float* bias, void* out,
                       int B, int D, int d_conv, int silu, int dtype, void* stream);

/*
 * ss_count_nonfinite — failure detection: writes to `count` (a device
 * uint64) the number of NaN and +-Inf values among the n elements of `p`
 * (dtype SS_F32 or SS_BF16; a value counts when its exponent field is all
 * ones).  A caller checks a step's gradients with it and drops the step when
 * the count is nonzero.  The count is exact and independent of the launch
 * (two fixed-order integer passes, no atomics).
 *   p         : device buffer, 16-byte aligned (NULL allowed when n == 0)
 *   count     : device, 8-byte aligned, overwritten
 *   workspace : ss_count_nonfinite_workspace_size() bytes, 16-byte aligned
 */
size_t ss_count_nonfinite_workspace_size(void);
int ss_count_nonfinite(const void* p, size_t n, int dtype, unsigned long long* count, void* workspace,
                       size_t ws_bytes, void* stream);

/*
 * ss_device_status — synchronises `stream`, then reads and clears the
 * library's device-side error word.  Returns SS_OK, or SS_ERR_DEVICE when a
 * kernel gave up on a bounded wait for its own asynchronous copies since the
 * last call (its overwritten outputs are then invalid; the CTAs that gave up
 * add zero to the accumulated gradients dA, dD, d_dt_bias, dw, db, dscale),
 * or SS_ERR_CUDA.
 */
int ss_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSSCAN_H */

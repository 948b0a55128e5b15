/*
 * falcon.h -- C ABI of the GB300 (sm_103a) Falcon fast-weight attention
 * library: chunk-parallel forward of Falcon-1 and Falcon-1A and its backward
 * pass, the forward of Falcon-2 and Falcon-2A (per-column step sizes) and of
 * Falcon-3A (sliding window) in token-recurrent and chunk form, and the
 * single-token recurrent decode step.
 *
 * The operations are defined on the page hyper.ai/fr/papers/2608.27763
 * ("Fast Weight Attention for Continual Learning"):
 *   - causal write pair x_t = phi(k_{t-1}), y_t = v_t, boundary x_1 = 0 with
 *     eta_1 = 0, and the read after write o_t = S_t^T phi(q_t): Section 4,
 *     "Naming and formula summary", and Section 3 "Indexing and causality
 *     conventions";
 *   - Falcon-1: S_t = (1 - eta_t lambda_t) S_{t-1} + eta_t x_t r_t^T with
 *     r_t = v_t - S_{t-1}^T x_t: Section 3.1, Eq. (3.3);
 *   - Falcon-1A: S_t = (1 - eta_t lambda_t) S_{t-1} + eta_t x_t v_t^T:
 *     Section 4.3, Eq. (4.6);
 *   - step size eta_t = beta_t / (||x_t||^2 + lambda_t + eps), 0 when the
 *     denominator is 0: Section 3.1, Eq. (3.4) and Section 4.3, Eq. (4.8);
 *   - decay clamp alpha_t = min(eta_t lambda_t, 1 - eps_gamma),
 *     gamma_t = 1 - alpha_t, evaluated in log space: Section 4.3, "Decay
 *     positivity", and Section 4.4, Eq. (4.15)-(4.16).
 * phi is the identity or the l2 map u / max(||u||_2, 1e-12) ("QK-l2" of the
 * experiments).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers owned by the caller.  The library keeps
 *     no pointer after a call returns and allocates no memory; scratch space,
 *     where needed, is the caller's `workspace`.
 *   - Every call is asynchronous on the caller's `stream` (0 = legacy default
 *     stream) and returns before the GPU work ends.  A nonzero return means
 *     nothing was launched (argument errors) or a launch failed (FALCON_ERR_CUDA).
 *   - A chunked call with few heads and many chunks runs part of its work on a
 *     second stream the library creates once per device (with its events):
 *     the call forks from the caller's stream and joins back to it by events,
 *     so later work on the caller's stream sees the call complete, and a
 *     stream capture of the call captures the fork and the join.
 *   - The chunked forwards launch their kernels as programmatic dependent
 *     launches, and their last kernel lets the next such launch on the
 *     stream begin early.  Each of the library's kernels waits for the grid
 *     before it (griddepcontrol.wait) before it reads or writes memory, so
 *     stream order holds for the library's own calls and for ordinary
 *     launches.  A kernel of the caller's that is launched right after one of
 *     these calls with programmatic stream serialization may start before the
 *     call ends, and must wait for it (cudaGridDependencySynchronize) before it
 *     reads the call's outputs, as every such launch must.
 *   - Tensors are dense, row-major, contiguous; [B,H,T,m] means element
 *     (b,h,t,i) is at ((b*H + h)*T + t)*m + i.
 *   - Every pointer must be 16-byte aligned (FALCON_ERR_MISALIGNED otherwise).
 *   - The library never prints, exits or traps.
 */
#ifndef FALCON_GB300_H
#define FALCON_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define FALCON_OK 0
#define FALCON_ERR_NULL_PTR (-1)   /* a required pointer is NULL */
#define FALCON_ERR_BAD_SHAPE (-2)  /* unsupported size (see each call) */
#define FALCON_ERR_BAD_DTYPE (-3)  /* dtype or phi code out of range */
#define FALCON_ERR_MISALIGNED (-4) /* a pointer is not 16-byte aligned */
#define FALCON_ERR_WORKSPACE (-5)  /* workspace NULL or smaller than required */
#define FALCON_ERR_CUDA (-6)       /* a CUDA launch or query failed */
#define FALCON_ERR_TIMEOUT (-7)    /* a device-side wait hit its limit */
#define FALCON_ERR_BAD_ARG (-8)    /* eps/eps_gamma (or another scalar argument) out of range */
#define FALCON_ERR_DEVICE (-9)     /* the current device is not sm_103 */
#define FALCON_ERR_SCRATCH_LIMIT (-10) /* needs more than FALCON_FIXED_SCRATCH_BYTES */

/* Size of the scratch array built into the library for
 * falcon1_fwd_chunked_fixed_scratch (held on every GPU that loads it). */
#define FALCON_FIXED_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Element type of q, k, v and o.  beta, lambda, states and features are
 * always float32. */
#define FALCON_BF16 0
#define FALCON_F32 1

/* Feature map phi applied to q and k: the identity, the l2 map
 * u / max(||u||_2, 1e-12), or RMSNorm(u) = u / sqrt(||u||_2^2 / d + eps_rms)
 * with eps_rms = 1e-6 (Section 4.1, "Scaled features": the pages' default
 * feature map; they name eps_rms without a value). */
#define FALCON_PHI_IDENTITY 0
#define FALCON_PHI_L2 1
#define FALCON_PHI_RMS 2

/* Ridge parameterisation (Section 4.1, "Scaled DeltaNet and the common ridge
 * parameterization"): lambda as given, or a base ridge lambda_bar from which
 * the recurrence takes lambda_t = lambda_bar_t * ||x_t||^2. */
#define FALCON_RIDGE_GIVEN 0
#define FALCON_RIDGE_SCALED 1

/* Problem description for the chunked forward calls.
 *   B, H   batch and heads; the B*H heads are independent.
 *   T      tokens per head, T >= 0; T need not be a multiple of `chunk`
 *          (the last chunk is partial).
 *   m      feature dimension of q, k (and of the state's rows): 16, 32, 64
 *          or 128.
 *   dv     value dimension: 16, 32, 64 or 128.
 *   chunk  chunk length C used by the chunk-parallel form: 16, 32 or 64.  It
 *          changes only the rounding, never the result in exact arithmetic.
 *   dtype  FALCON_BF16 or FALCON_F32 (q, k, v, o).
 *   phi    FALCON_PHI_IDENTITY, FALCON_PHI_L2 or FALCON_PHI_RMS.
 *   eps    >= 0, the step-size stabiliser of Eq. (3.4).
 *   eps_gamma in (0, 1), the clamp margin: gamma_t >= eps_gamma.
 *   ridge  FALCON_RIDGE_GIVEN (lambda is lambda_t) or FALCON_RIDGE_SCALED
 *          (lambda is the base ridge; lambda_t = lambda_t(input) * ||x_t||^2). */
typedef struct {
  int64_t B, H, T;
  int32_t m, dv, chunk;
  int32_t dtype;
  int32_t phi;
  float eps;
  float eps_gamma;
  int32_t ridge;
} falcon_shape;

/* Bytes of device workspace a chunked forward call with this shape needs
 * (0 means the call accepts workspace = NULL).  Returns 0 for an invalid
 * shape as well; the forward call then reports the shape error. */
size_t falcon_workspace_bytes(const falcon_shape *shape);

/* Falcon-1 chunk-parallel forward (Section 3.1 Eq. (3.3) with Eq. (3.4)).
 *   q, k    [B,H,T,m]  dtype
 *   v       [B,H,T,dv] dtype
 *   beta    [B,H,T]    f32, the gain beta_t (the pages use beta in (0,2))
 *   lambda  [B,H,T]    f32, the ridge coefficient lambda_t >= 0
 *   S0      [B,H,m,dv] f32, state entering token 1; NULL means zeros
 *   x_prev  [B,H,m]    f32, write feature of token 1 (phi(k) of the token
 *           before this segment); NULL means a fresh sequence, where the
 *           boundary sentinel applies (x_1 = 0, eta_1 = 0)
 *   o       [B,H,T,dv] dtype, out: o_t = S_t^T phi(q_t)
 *   S_out   [B,H,m,dv] f32, out: S_T.  May alias S0.
 *   x_last  [B,H,m]    f32, out, nullable: phi(k_T) (x_prev of the next
 *           segment; left untouched when T = 0 and x_prev is NULL, copied
 *           from x_prev when T = 0 otherwise)
 *   workspace, workspace_bytes: device scratch of at least
 *           falcon_workspace_bytes(shape) bytes, 256-byte aligned; contents
 *           are overwritten.  Concurrent calls need separate workspaces.
 * Errors: FALCON_ERR_NULL_PTR, _BAD_SHAPE, _BAD_DTYPE, _MISALIGNED,
 * _WORKSPACE, _BAD_ARG, _DEVICE (nothing launched); _CUDA (launch failed). */
int falcon1_fwd_chunked(const falcon_shape *shape, const void *q, const void *k,
                        const void *v, const float *beta, const float *lambda,
                        const float *S0, const float *x_prev, void *o,
                        float *S_out, float *x_last, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* falcon1_fwd_chunked for callers that cannot allocate device memory: the
 * paper has no counterpart; this is a library convenience.  It computes
 * exactly what falcon1_fwd_chunked computes, but takes no workspace: its
 * scratch is a fixed array of FALCON_FIXED_SCRATCH_BYTES inside the library
 * (held on every GPU that loads the library until the process exits), so the
 * call allocates nothing.  It serves callers that are handed only input and
 * output buffers (a C host program, a plugin interface), whose allocator is
 * out of reach at the call site, or that forbid allocation after start-up.
 *   - Shapes with falcon_workspace_bytes(shape) > FALCON_FIXED_SCRATCH_BYTES
 *     are rejected with FALCON_ERR_SCRATCH_LIMIT (nothing launched).
 *   - The first call on each device, with that device current, resolves the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture on the device.  A tensor-core shape with
 *     few heads and many chunks (the chunk-range pieces described above)
 *     also creates, on its first use on the device, the library's second
 *     stream and its events, as falcon1_fwd_chunked does; a warm-up call of
 *     such a shape does that set-up too.
 *   - All calls on a device share the array, which keeps the previous call's
 *     contents (nothing needs clearing: every scratch element read is written
 *     first by the same call).  Calls whose GPU work overlaps race on it: issue
 *     them on one stream.
 * Other arguments, layouts, ownership and errors are those of
 * falcon1_fwd_chunked. */
int falcon1_fwd_chunked_fixed_scratch(const falcon_shape *shape, const void *q,
                                      const void *k, const void *v,
                                      const float *beta, const float *lambda,
                                      const float *S0, const float *x_prev,
                                      void *o, float *S_out, float *x_last,
                                      cudaStream_t stream);

/* Falcon-1A chunk-parallel forward (Section 4.3 Eq. (4.6), step size
 * Eq. (4.8) with E_t = ||x_t||^2).  Arguments, layouts, ownership and errors
 * are those of falcon1_fwd_chunked. */
int falcon1a_fwd_chunked(const falcon_shape *shape, const void *q,
                         const void *k, const void *v, const float *beta,
                         const float *lambda, const float *S0,
                         const float *x_prev, void *o, float *S_out,
                         float *x_last, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* Falcon-1A with the normalised read (Section 2.2, Eq. (2.1)-(2.3): the
 * normaliser z_t of linear attention on the shifted write stream):
 *     o_t = S_t^T phi(q_t) / (z_t^T phi(q_t) + eps_attn),
 *     z_t = gamma_t z_{t-1} + eta_t x_t,
 * with S_t the Falcon-1A state and z taking the same step size eta_t and
 * clamped decay gamma_t as the numerator.  The pages define z for plain linear
 * attention (lambda = 0, unit gain, where this is their Eq. (2.3) exactly) and
 * defer the Falcon-1A version to an appendix they do not include; this is the
 * plainest reading.  The denominator is not clamped away from zero (the pages
 * note that the normalised read is attention-like only for a nonnegative
 * normaliser): callers with signed features choose eps_attn accordingly.
 *   z0      [B,H,m] f32, normaliser entering token 1; NULL means zeros
 *   z_out   [B,H,m] f32, out, nullable: z_T (may alias z0)
 *   eps_attn >= 0 and finite (FALCON_ERR_BAD_ARG otherwise)
 *   workspace: at least falcon_normalized_workspace_bytes(shape) bytes.
 * Other arguments, layouts, ownership and errors are those of
 * falcon1a_fwd_chunked (o holds the normalised read).  The call runs the
 * Falcon-1A forward and then one to three plain kernels for the denominator
 * (ordinary launches: they start after the forward's kernels complete); on the
 * tensor-core path with m = 64 the forward's map launch also writes the
 * denominator's per-chunk terms to the workspace. */
size_t falcon_normalized_workspace_bytes(const falcon_shape *shape);
int falcon1a_fwd_chunked_normalized(const falcon_shape *shape, const void *q,
                                    const void *k, const void *v,
                                    const float *beta, const float *lambda,
                                    const float *S0, const float *z0,
                                    const float *x_prev, float eps_attn,
                                    void *o, float *S_out, float *z_out,
                                    float *x_last, void *workspace,
                                    size_t workspace_bytes,
                                    cudaStream_t stream);

/* Bytes of device workspace falcon1_bwd_chunked / falcon1a_bwd_chunked need
 * for this shape (0 for an invalid shape; the call then reports the error). */
size_t falcon_bwd_workspace_bytes(const falcon_shape *shape);
/* Backward pass of the Falcon-1 chunk-parallel forward: the gradient of
 *   L = <dO, o> + <dS_T, S_T> + <dx_last, x_last>
 * with respect to every input of falcon1_fwd_chunked.  The pages state that
 * training differentiates through the update, so that the slow weights that
 * produce q, k, v, beta and lambda learn (Section 3, "Implicit fast-memory
 * objective"), through the log-decay renormalisation and the normalised step
 * size (Section 4.6, "Backward pass"); this is the exact gradient of the
 * forward as computed, with two conventions: on the clamped branch of the
 * decay (eta_t lambda_t >= 1 - eps_gamma) gamma_t = eps_gamma is a constant,
 * and the boundary sentinel (eta_1 = 0) passes no gradient to beta_1,
 * lambda_1.  The call recomputes the forward (chunk maps and the state
 * entering every chunk) in its workspace; it needs none of the forward's
 * outputs.
 *   shape, q, k, v, beta, lambda, S0, x_prev: the forward's arguments
 *           (S0 and x_prev nullable as there)
 *   dO      [B,H,T,dv] dtype, the cotangent of o
 *   dS_T    [B,H,m,dv] f32, nullable (zero), the cotangent of S_T
 *   dx_last [B,H,m] f32, nullable (zero), the cotangent of x_last
 *   dq, dk  [B,H,T,m] dtype, out;   dv [B,H,T,dv] dtype, out
 *   dbeta, dlambda [B,H,T] f32, out (with FALCON_RIDGE_SCALED, dlambda is
 *           the gradient for the lambda input, the base ridge)
 *   dS0     [B,H,m,dv] f32, out, nullable (not written); may alias dS_T
 *   dx_prev [B,H,m] f32, out, nullable (not written); zeros when x_prev is
 *           NULL (the sentinel feature is a constant)
 *   workspace, workspace_bytes: at least falcon_bwd_workspace_bytes(shape)
 *           bytes, 256-byte aligned; contents are overwritten.
 * Every shape and dtype of falcon1_fwd_chunked is accepted (fp32 arithmetic
 * on CUDA cores).  Errors as for falcon1_fwd_chunked. */
int falcon1_bwd_chunked(const falcon_shape *shape, const void *q, const void *k,
                        const void *v, const float *beta, const float *lambda,
                        const float *S0, const float *x_prev, const void *dO,
                        const float *dS_T, const float *dx_last, void *dq, void *dk,
                        void *dv, float *dbeta, float *dlambda, float *dS0,
                        float *dx_prev, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream);
/* The backward pass of falcon1a_fwd_chunked (Section 4.3 Eq. (4.6)).
 * Arguments, layouts, ownership and errors are those of falcon1_bwd_chunked. */
int falcon1a_bwd_chunked(const falcon_shape *shape, const void *q, const void *k,
                         const void *v, const float *beta, const float *lambda,
                         const float *S0, const float *x_prev, const void *dO,
                         const float *dS_T, const float *dx_last, void *dq, void *dk,
                         void *dv, float *dbeta, float *dlambda, float *dS0,
                         float *dx_prev, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);
/* Falcon-2 forward (per-column step sizes), token-recurrent form: every
 * column j of the state follows its own step size and clamped decay,
 *   eta_{j,t} = beta_{j,t} / (||x_t||^2 + lambda_t + eps)  (0 at the sentinel
 *   and when the denominator is 0), gamma_{j,t} = 1 - min(eta_{j,t} lambda_t,
 *   1 - eps_gamma), S_t[:, j] = gamma_{j,t} S_{t-1}[:, j] + eta_{j,t} x_t r_{t,j},
 *   r_t = v_t - S_{t-1}^T x_t,  o_t = S_t^T phi(q_t);
 * page hyper.ai/fr/papers/2608.27763, the regression-family display of
 * Section 3.1 and the per-column NLMS step sizes of Section 4.2.
 * Arguments, layouts, ownership and errors are those of falcon1_fwd_chunked
 * except:
 *   beta    [B,H,T,dv] f32: one gain per value column and token
 *   shape->chunk is checked (16, 32 or 64) but not used: the call runs the
 *           recurrence token by token, and needs no workspace.
 * One CTA per head and 32 value columns runs the tokens in order; the state
 * stays in registers. */
int falcon2_fwd_recurrent(const falcon_shape *shape, const void *q,
                          const void *k, const void *v, const float *beta,
                          const float *lambda, const float *S0,
                          const float *x_prev, void *o, float *S_out,
                          float *x_last, cudaStream_t stream);

/* Falcon-2A, the per-column inner-product rule (Section 4.3, "Falcon-2A:
 * per-column inner-product write"): as falcon2_fwd_recurrent with r_t
 * replaced by v_t and E_t = ||x_t||^2 in the step size. */
int falcon2a_fwd_recurrent(const falcon_shape *shape, const void *q,
                           const void *k, const void *v, const float *beta,
                           const float *lambda, const float *S0,
                           const float *x_prev, void *o, float *S_out,
                           float *x_last, cudaStream_t stream);

/* Falcon-3A forward, the sliding-window inner-product rule (Section 4.5),
 * token-recurrent form, for fresh sequences:
 *   for t >= 2 the window I_t of the last `window` write pairs (x_j, v_j),
 *   j >= 2, B_t = |I_t|: N_bar_t = (1/B_t) sum x_j v_j^T, E_bar_t =
 *   (1/B_t) sum ||x_j||^2, eta_t = beta_t / (E_bar_t + lambda_t + eps)
 *   (lambda_t = lambda_bar_t * E_bar_t with FALCON_RIDGE_SCALED), gamma_t =
 *   1 - min(eta_t lambda_t, 1 - eps_gamma), S_t = gamma_t S_{t-1} +
 *   eta_t N_bar_t; token 1 is the boundary (no update); o_t = S_t^T phi(q_t).
 *   window  1 .. 32 (window 1 is Falcon-1A); FALCON_ERR_BAD_ARG otherwise.
 * Arguments, layouts, ownership and errors are those of falcon1_fwd_chunked
 * except: no x_prev (the window does not reach into a previous segment: exact
 * continuation would need the last window - 1 pairs), no workspace, and
 * shape->chunk is checked but not used. */
int falcon3a_fwd_recurrent(const falcon_shape *shape, int32_t window,
                           const void *q, const void *k, const void *v,
                           const float *beta, const float *lambda,
                           const float *S0, void *o, float *S_out,
                           float *x_last, cudaStream_t stream);

/* Falcon-2A forward in chunk form: the same result as falcon2a_fwd_recurrent
 * (up to rounding).  Every value column j has its own step sizes and
 * decays, so within a chunk of 64 tokens o_{t,j} = e^{G_{j,t}} (Q S)_{t,j} +
 * sum_{s<=t} <phi(q_t), x_s> e^{G_{j,t} - G_{j,s}} eta_{j,s} v_{s,j} and the
 * state leaving it is S o e^{G_C} + X^T V' (G_{j,.} the chunk-local log
 * prefix of column j; no triangular solve: the inner-product rule writes the
 * target itself).  For bf16 q, k, v with m = dv = 64 and shape->chunk = 64
 * this runs on the tensor cores and needs a workspace of
 * falcon_workspace_bytes(shape) bytes (256-byte aligned); for every other
 * shape it runs falcon2a_fwd_recurrent and ignores the workspace.
 * Arguments, layouts and errors are those of falcon2a_fwd_recurrent, plus
 * workspace / workspace_bytes as in falcon1_fwd_chunked. */
/* Falcon-2 forward in chunk form: the same result as falcon2_fwd_recurrent
 * (up to rounding).  Every value column j runs its own scalar-step delta
 * rule on the shared write features (Section 3.1, regression display; Section
 * 4.2, per-column step sizes), so inside a chunk of 64 tokens the written
 * residuals u_{t,j} = eta_{j,t} r_{t,j} of column j solve a unit-lower system
 * built from the shared Gram <x_t, x_l> and the column's own decays: one
 * batched per-column triangular solve per chunk.  With E_{t,j} the product of
 * column j's gammas over the chunk up to token t and w = u / E, the solve is
 * u_t = eta_t v_t - eta_t E_{t-1} ((X S)_t + sum_{l<t} <x_t, x_l> w_l), the
 * output o_t = E_t ((Q S)_t + sum_{l<=t} <q_t, x_l> w_l) and the state leaving
 * the chunk E_C (S + X^T W); a chunk whose decay product falls below e^{-60}
 * in some column (clamped gammas) runs token by token instead.  The chunks of
 * a head are sequential (the per-column systems depend on the entering
 * state): one CTA per head.  For bf16 q, k, v with m = dv = 64 and
 * shape->chunk = 64 this runs on the tensor cores; for every other shape it
 * runs falcon2_fwd_recurrent.  Arguments, layouts, ownership and errors are
 * those of falcon2_fwd_recurrent; no workspace is needed. */
int falcon2_fwd_chunked(const falcon_shape *shape, const void *q,
                        const void *k, const void *v, const float *beta,
                        const float *lambda, const float *S0,
                        const float *x_prev, void *o, float *S_out,
                        float *x_last, cudaStream_t stream);
int falcon2a_fwd_chunked(const falcon_shape *shape, const void *q,
                         const void *k, const void *v, const float *beta,
                         const float *lambda, const float *S0,
                         const float *x_prev, void *o, float *S_out,
                         float *x_last, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);
/* Falcon-3A forward in chunk form: the same result as falcon3a_fwd_recurrent
 * (up to rounding), computed as the masked-attention form of Section 4.6:
 * within a chunk of 64 tokens the state after token t is e^{g_t} S plus the
 * write pairs of the chunk and of the B - 1 pairs before it, each weighted by
 * w_{t,j} = sum over the chunk's tokens s <= t whose window holds pair j of
 * e^{g_t - g_s} eta_s / B_s; the chunk maps are composed across chunks by the
 * tensor-core scan.  For bf16 q, k, v with m = dv = 64 and shape->chunk = 64
 * this runs on the tensor cores and needs a workspace of
 * falcon_workspace_bytes(shape) bytes (256-byte aligned); for every other
 * shape it runs falcon3a_fwd_recurrent and ignores the workspace.
 * Arguments, layouts and errors are those of falcon3a_fwd_recurrent, plus
 * workspace / workspace_bytes as in falcon1_fwd_chunked. */
int falcon3a_fwd_chunked(const falcon_shape *shape, int32_t window,
                         const void *q, const void *k, const void *v,
                         const float *beta, const float *lambda,
                         const float *S0, void *o, float *S_out,
                         float *x_last, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);
/* One recurrent token (read after write) for N independent states: the
 * Falcon-1 update of Section 3.1 Eq. (3.3), as in the one-step listing of page
 * rcap.io/posts/fast-weight-attention-for-continual-learning-2026-08-27.
 *   q, k    [N,m]  dtype;  v, o [N,dv] dtype;  beta, lambda [N] f32
 *   S       [N,m,dv] f32, updated in place to S_t
 *   x_prev  [N,m] f32: read as this token's write feature x_t, then
 *           overwritten with phi(k_t) for the next token
 *   fresh   [N] bytes, nullable: nonzero marks a state whose sequence starts
 *           at this token (sentinel: x_t = 0, eta_t = 0, so S is not
 *           decayed and o = S^T phi(q)); NULL means no state is fresh
 * phi and ridge as in falcon_shape.
 * m, dv in {16, 32, 64, 128}.  N >= 0 (N = 0 launches nothing).
 * Errors as for falcon1_fwd_chunked (no workspace). */
int falcon1_decode_step(int64_t N, int32_t m, int32_t dv, int32_t dtype,
                        int32_t phi, int32_t ridge, float eps, float eps_gamma,
                        const void *q,
                        const void *k, const void *v, const float *beta,
                        const float *lambda, float *S, float *x_prev,
                        const uint8_t *fresh, void *o, cudaStream_t stream);

/* The same single-token step for Falcon-1A (Section 4.3 Eq. (4.6)). */
int falcon1a_decode_step(int64_t N, int32_t m, int32_t dv, int32_t dtype,
                         int32_t phi, int32_t ridge, float eps, float eps_gamma,
                         const void *q,
                         const void *k, const void *v, const float *beta,
                         const float *lambda, float *S, float *x_prev,
                         const uint8_t *fresh, void *o, cudaStream_t stream);

/* Waits for `stream`, then reads and clears the library's device error word
 * (set by a kernel whose bounded wait ran out).  Returns FALCON_OK,
 * FALCON_ERR_TIMEOUT, or FALCON_ERR_CUDA if the stream itself failed.
 * The error word is one per device, not one per call: every call on the
 * device writes the same word, so with calls in flight on several streams a
 * timeout in any of them is reported to whichever caller reads the word
 * first (and cleared for the others).  Callers that need a per-call status
 * synchronise their streams one at a time. */
int falcon_sync_check(cudaStream_t stream);

/* Diagnostic of the failure path (no counterpart in the paper): launches a
 * kernel whose threads wait on a barrier that nothing completes.  The wait
 * gives up after limit_us microseconds (1 .. 10^7) and records the expiry in
 * the device error word, exactly as the chunked kernels do when a wait is
 * lost; nothing traps and the CUDA context stays usable.  A following
 * falcon_sync_check(stream) returns FALCON_ERR_TIMEOUT (and clears the word).
 * Returns FALCON_ERR_BAD_ARG for limit_us out of range. */
int falcon_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/* Static description of a return code. */
const char *falcon_strerror(int code);

/* Library version, major*10000 + minor*100 + patch. */
int falcon_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FALCON_GB300_H */

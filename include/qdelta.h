/*
 * qdelta.h -- C ABI of the GB300 (sm_103a) Q-Delta / QED / EDA forwards, the
 * Q-Delta backward and the decode steps.
 *
 * Every entry point takes plain device pointers and sizes; no C++ or framework
 * types cross this boundary.  All device buffers are owned by the caller.  Every
 * compute call is asynchronous on the caller's stream and does not synchronise.
 * No call throws; each returns a qd_status and, on error, records a message
 * retrievable with qd_last_error() (per host thread).
 *
 * Layouts (row-major, dense, no padding):
 *   tokens    q, k        [B][T][H][dk]      in the call's dtype
 *             v, o        [B][T][H][dv]      in the call's dtype
 *   Q-Delta   alpha, beta, lam  [B][T][H]    in the call's dtype
 *   QED       g, b        [B][T][H][dk], w [B][T][H][dv] in the call's dtype;
 *             lam_h [H] fp32
 *   state     S0, S_final, S    [B][H][dv][dk] fp32 (decode: [N][H][dv][dk])
 *             Q-Delta's state is d_v x d_k (o = S q); QED's state is K x V
 *             (o = S^T q) and is stored transposed, so both share this format.
 * Every pointer must be 16-byte aligned.  S0 may alias S_final (in-place carry).
 *
 * Supported: dk, dv in {16, 32, 64, 128}; chunk = 64; any T >= 0 (a ragged last
 * chunk is handled); dtype QD_F32 or QD_BF16 (math in fp32, state in fp32).
 */
#ifndef QDELTA_GB300_H
#define QDELTA_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define QD_API __attribute__((visibility("default")))
#else
#define QD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QD_OK = 0,
    QD_ERR_ARG = 1,          /* null / misaligned pointer, negative or overflowing size */
    QD_ERR_UNSUPPORTED = 2,  /* valid but unsupported: head dim, chunk size, dtype */
    QD_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    QD_ERR_TIMEOUT = 4,      /* a kernel's bounded wait gave up (see qd_device_status) */
    QD_ERR_WORKSPACE = 5     /* workspace missing or smaller than *_workspace_bytes() */
} qd_status;

typedef enum { QD_F32 = 0, QD_BF16 = 1 } qd_dtype;

/*
 * qdelta_fwd -- chunkwise-parallel forward of the gated Q-Delta recurrence.
 *
 * Defines (reading notes "Q-Delta: Beyond Key-Value Associative State
 * Evolution", Sec. 3.3.1, Eqs. 17-20, the boxed gated form), per (b, h), for
 * t = 1..T, starting from S_0 = S0 (or 0):
 *     x_t = k_t + lambda_t q_t
 *     S_t = alpha_t S_{t-1} (I - beta_t x_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t
 * computed chunk by chunk (Sec. 3.3.2, Eqs. 20-27: WY / UT-transform form, with
 * the notes' corrections of the v1 transposes and decay factors).
 * alpha == NULL means alpha = 1 and lam == NULL means lambda = 0: lam == NULL
 * is Gated DeltaNet, both NULL is DeltaNet.  beta must not be NULL.
 * S0 == NULL starts from zero; S_final == NULL skips writing the final state.
 * o receives o_t in the call's dtype.
 *
 * workspace: device scratch of at least qdelta_workspace_bytes(...) bytes
 * (may be NULL when that returns 0).  Calls that share a workspace must be
 * ordered on one stream.  A workspace is needed when few (b, h) streams carry a
 * long sequence (bf16, dk = dv = 128): each sequence is then cut into segments
 * that run in parallel (the chunk map S -> S Phi + Psi is linear in the state)
 * and are stitched together in fp32; the workspace holds three d_v x d_k fp32
 * states per segment.
 */
QD_API qd_status qdelta_fwd(const void *q, const void *k, const void *v,
                     const void *alpha, const void *beta, const void *lam,
                     const float *S0, void *o, float *S_final,
                     int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace qdelta_fwd needs for these sizes (0 if none). */
QD_API size_t qdelta_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype);

/*
 * qed_fwd -- chunked forward of QED over GDN-2 (reading notes "The Query Knows
 * What to Forget", Sec. 2.1-2.2: GDN-2 update of Eqs. 4/8, erase vector of
 * Eq. 6).  With the paper's K x V state S (stored transposed, see above):
 *     Sbar_t = Diag(exp g_t) S_{t-1}
 *     u_t = b_t * q_t;  d_t = u_t - k_t (k_t^T u_t);  a_t = b_t * k_t + lam_h[h] d_t
 *     S_t = Sbar_t + k_t (w_t * v_t - Sbar_t^T a_t)^T
 *     o_t = S_t^T q_t
 * g is the per-key-channel log-decay (g <= 0 expected).  The chunked kernel
 * factors exp(G_t - G_i) into exp(G_t) exp(-G_i) within a chunk, G the in-chunk
 * cumulative log-decay; it stays accurate while every channel's log-decay summed
 * over one 64-token chunk is >= -80 (fp32 range).  lam_h must not be NULL.
 */
QD_API qd_status qed_fwd(const void *q, const void *k, const void *v,
                  const void *g, const void *b, const void *w, const float *lam_h,
                  const float *S0, void *o, float *S_final,
                  int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * qed_fwd_variant -- qed_fwd for one of the ablation arms of the QED notes
 * ("The Query Knows What to Forget", Sec. 3.2, Table 1).  Each arm changes only
 * the term added to the base erase vector b_t * k_t, with P(u) = u - k (k^T u):
 *     QD_QED_FULL           lam_h P(b_t * q_t)   (qed_fwd)
 *     QD_QED_NOGATE         lam_h P(q_t)         (b removed from the new term only)
 *     QD_QED_NOGATE_NOPROJ  lam_h q_t            (no gate, no projection)
 *     QD_QED_RAND           lam_h P(b_t * z_h)   (z_h: a fixed vector per head)
 * z_h [H][dk] fp32 is required for QD_QED_RAND and ignored otherwise.  Every
 * other argument, layout and the workspace rule are those of qed_fwd.
 */
typedef enum { QD_QED_FULL = 0, QD_QED_NOGATE = 1, QD_QED_NOGATE_NOPROJ = 2, QD_QED_RAND = 3 } qd_qed_variant;

QD_API qd_status qed_fwd_variant(const void *q, const void *k, const void *v,
                                 const void *g, const void *b, const void *w, const float *lam_h,
                                 const float *S0, void *o, float *S_final,
                                 int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                                 qd_qed_variant variant, const float *z_h,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * qed_step -- one decode step of QED (T = 1), state in place.  With the state
 * stored transposed (S^ = S^T, [dv][dk]) and e = exp(g_t), per row i:
 *     S^_i <- S^_i Diag(e) + (w_i v_i - (S^_i Diag(e)) . a_t) k_t,   o_i = S^_i q_t
 * (the QED notes' Eqs. 4, 6, 8 for one token; a_t of the chosen arm, as in
 * qed_fwd_variant).  Each state row is read once and written once.
 *   S  [N][H][dv][dk] fp32, updated in place
 *   q, k, g, b [N][H][dk]; v, w, o [N][H][dv] in the call's dtype; lam_h [H] fp32;
 *   z_h [H][dk] fp32 (QD_QED_RAND only)
 */
QD_API qd_status qed_step(float *S, const void *q, const void *k, const void *v,
                          const void *g, const void *b, const void *w, const float *lam_h, void *o,
                          int N, int H, int dk, int dv, qd_dtype dtype,
                          qd_qed_variant variant, const float *z_h, cudaStream_t stream);

/* Bytes of device workspace qed_fwd needs for these sizes (0 if none).  The
 * tensor-core path (bf16, dk = dv = 128) derives each chunk's decay-folded operands
 * (a*e^G, q*e^G, k*e^-G, w*v as bf16 [B][T][H][128], and e^{G_C} per chunk and
 * channel in fp32) into the workspace, 8 * B * T * H * 128 bytes and a little more
 * (one hand-over counter per chunk and stream); the other paths need none.  While
 * B * H leaves at least 8 SMs free, the derive step runs on those SMs beside the
 * per-stream chains, in one cooperative launch, and hands each chunk over through its
 * counter; otherwise it is a launch of its own before the chains.  As for qdelta_fwd,
 * very few (b, h) streams (at most 16) carrying a long sequence are further cut into
 * segments that run in parallel (QED's per-chunk map of the transposed state is
 * linear, S^ -> S^ Phi + Psi) and are stitched together in fp32, with three d_v x d_k
 * fp32 states per segment after the derived operands.  Calls sharing a workspace must
 * be ordered on one stream. */
QD_API size_t qed_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype);

/*
 * qdelta_step -- one decode step of the same recurrence (T = 1), state in place.
 * Uses the single-pass output form of the Q-Delta notes, Sec. 2.4:
 *     o_t = alpha_t S_{t-1} q_t + beta_t (v_t - alpha_t S_{t-1} x_t)(k_t^T q_t)
 * so each state row is read once and written once.
 *   S  [N][H][dv][dk] fp32, updated in place from S_{t-1} to S_t
 *   q, k [N][H][dk]; v, o [N][H][dv]; alpha, beta, lam [N][H] (alpha, lam nullable)
 */
QD_API qd_status qdelta_step(float *S, const void *q, const void *k, const void *v,
                      const void *alpha, const void *beta, const void *lam, void *o,
                      int N, int H, int dk, int dv, qd_dtype dtype, cudaStream_t stream);

/*
 * qdelta_fwd_prologue -- qdelta_fwd from the layer's projections: the feature map
 * and the gates are computed inside the forward, with no separate pass over HBM.
 * Per token-head, before the recurrence:
 *     q = SiLU(q_raw) / |SiLU(q_raw)|_2,  k = SiLU(k_raw) / |SiLU(k_raw)|_2
 *         ("Parallelizing Linear Transformers with the Delta Rule over Sequence
 *          Length", sec. 3.8; an all-zero SiLU row stays zero)
 *     beta = sigmoid(b_logit)             (same section)
 *     lambda = sigmoid(l_logit)           (Q-Delta notes, sec. 2.5 / App. B; the bias
 *                                          is part of the logit)
 *     alpha = exp(-softplus(a_logit))     (the decay parameterisation of the workloads)
 * a_logit == NULL means alpha = 1 and l_logit == NULL means lambda = 0.  Arguments,
 * layouts and the workspace rule are those of qdelta_fwd, with q_raw, k_raw in place
 * of q, k and the logits in place of the gates.  The bf16 tensor-core path evaluates
 * sigmoid through the hardware tanh (relative error ~2^-11, below the bf16 rounding
 * of q and k); the fp32 path uses the accurate functions.
 */
QD_API qd_status qdelta_fwd_prologue(const void *q_raw, const void *k_raw, const void *v,
                                     const void *a_logit, const void *b_logit, const void *l_logit,
                                     const float *S0, void *o, float *S_final,
                                     int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* qdelta_step with the same prologue (q_raw, k_raw [N][H][dk], logits [N][H]). */
QD_API qd_status qdelta_step_prologue(float *S, const void *q_raw, const void *k_raw, const void *v,
                                      const void *a_logit, const void *b_logit, const void *l_logit, void *o,
                                      int N, int H, int dk, int dv, qd_dtype dtype, cudaStream_t stream);

/*
 * qdelta_bwd -- backward of qdelta_fwd: the gradients of
 *     L = sum_{b,t,h} <dO_t, o_t> + sum_{b,h} <dS_final, S_T>
 * with respect to q, k, v, alpha, beta, lam and S0, i.e. the adjoint of the
 * recurrence qdelta_fwd computes (Sec. 3.3.1 of the Q-Delta notes, chunked as in
 * Sec. 3.3.2).  The pages train the layer end to end ("Parallelizing Linear
 * Transformers with the Delta Rule over Sequence Length", sec. 3) but state no
 * backward; this is the derivative of the stated forward.
 *
 * Inputs: q, k, v, alpha, beta, lam, S0, dtype, sizes exactly as passed to
 * qdelta_fwd (alpha NULL = 1, lam NULL = 0, S0 NULL = 0); dO [B][T][H][dv] in the
 * call's dtype; dS_final [B][H][dv][dk] fp32 or NULL (= 0).
 * Outputs, each overwritten, in the call's dtype unless stated:
 *   dq, dk [B][T][H][dk]; dv [B][T][H][dv]; dbeta [B][T][H]   (required)
 *   dalpha [B][T][H]: written when alpha and dalpha are both non-NULL
 *   dlam [B][T][H]:   written when lam and dlam are both non-NULL
 *   dS0 [B][H][dv][dk] fp32: written when non-NULL (also when S0 is NULL)
 * No output may alias an input.  workspace: at least qdelta_bwd_workspace_bytes(...)
 * bytes (two checkpoint arrays: the state entering, and the gradient reaching the
 * state leaving, every chunk of 64 tokens; fp32, or fp16 tiles in half of that space
 * on the tensor-core path).  T = 0 writes dS0 = dS_final (or 0) and nothing else.
 * Precision: fp32 inputs, and head dims other than 128, run in fp32 on CUDA cores.
 * bf16 inputs at dk = dv = 128 run on the tensor cores with fp32 accumulation, and
 * the state and its gradient carried across chunks in fp32: the checkpoint forward is
 * the bf16 forward, the reverse sweep of the state gradient takes bf16 operands, and
 * the per-chunk gradients take fp16 operands (10-bit mantissa; their intermediates
 * stay far inside fp16's range at unit-scale inputs), the two checkpoints among them,
 * stored as fp16; the elementwise work is fp32.
 * Errors as for qdelta_fwd.
 */
QD_API qd_status qdelta_bwd(const void *q, const void *k, const void *v,
                            const void *alpha, const void *beta, const void *lam, const float *S0,
                            const void *dO, const float *dS_final,
                            void *dq, void *dk_out, void *dv_out, void *dalpha, void *dbeta, void *dlam,
                            float *dS0, int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace qdelta_bwd needs for these sizes (never 0 when T > 0). */
QD_API size_t qdelta_bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype);

/*
 * qdelta_bwd_prologue -- backward of qdelta_fwd_prologue: the gradients of the same L
 * as qdelta_bwd with respect to the projections q_raw, k_raw, v, the gate logits and
 * S0.  The inputs go through the prologue's maps (see qdelta_fwd_prologue; fp32
 * arithmetic, stored in the call's dtype), the recurrence's backward runs on them
 * (qdelta_bwd), and the chain rule takes the gradients back through the maps:
 *     with s = SiLU(x), n = |s|, y = s / n:  dx = ((dy - y (y . dy)) / n) * SiLU'(x)
 *     d b_logit = dbeta beta (1 - beta),  d l_logit = dlam lam (1 - lam),
 *     d a_logit = -dalpha alpha (1 - alpha)          (alpha = exp(-softplus) = sigmoid(-a))
 * An all-zero SiLU row (left zero by the forward) passes no gradient.  Arguments and
 * outputs as qdelta_bwd with the raw inputs and the logits' gradients in place of the
 * mapped ones (dq_raw, dk_raw [B][T][H][dk]; da_logit, db_logit, dl_logit [B][T][H]).
 * workspace: at least qdelta_bwd_prologue_workspace_bytes(...) bytes.
 */
QD_API qd_status qdelta_bwd_prologue(const void *q_raw, const void *k_raw, const void *v,
                                     const void *a_logit, const void *b_logit, const void *l_logit,
                                     const float *S0, const void *dO, const float *dS_final,
                                     void *dq_raw, void *dk_raw, void *dv_out, void *da_logit, void *db_logit,
                                     void *dl_logit, float *dS0, int B, int T, int H, int dk, int dv, int chunk,
                                     qd_dtype dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace qdelta_bwd_prologue needs for these sizes. */
QD_API size_t qdelta_bwd_prologue_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype);

/*
 * eda_fwd -- erase-then-delta forward ("Erase-then-Delta Attention", core method:
 * a targeted erase along a direction e, then the Delta write along the key).  Per
 * (b, h), with the memory M (d_k x d_v), stored as S = M^T in the state layout:
 *     M <- M - e_t (e_t^T M)                       erase (the page's "(e^T M) e" read as
 *                                                   the outer product that fits the shapes)
 *     M <- M - beta_t k_t (k_t^T M - v_t^T)         Delta write (the page's unit step: beta = 1)
 *     o_t = M^T q_t                                 read-out after both steps
 * e [B][T][H][dk] in the call's dtype, used as given (the page's default is
 * e = q/|q|; pass that to get it).  beta [B][T][H] or NULL (= 1).  Other arguments,
 * layouts, state convention and errors as for qdelta_fwd.
 * bf16 with dk = dv = 128 runs on the tensor cores: o_t = S_{t-1} r_t + beta_t (k_t.q_t) v_t
 * with r_t = (I - e e^T)(q_t - beta_t (k_t.q_t) k_t) formed in fp32 per token (the
 * read-out's cancellation at e = q done before any rounding), then the Delta rule over
 * 2T+1 sub-tokens (erase e_t, write k_t) in fp16 operands with fp32 accumulation and an
 * fp32 state; inputs and states must lie inside fp16's range (|x| < 65504).  That path
 * needs eda_workspace_bytes() of workspace (QD_ERR_WORKSPACE without it); fp32 inputs and
 * other head dims run a recurrence in fp32 and need none (workspace may then be NULL).
 */
QD_API qd_status eda_fwd(const void *q, const void *k, const void *v, const void *e, const void *beta,
                         const float *S0, void *o, float *S_final, int B, int T, int H, int dk, int dv,
                         int chunk, qd_dtype dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace eda_fwd needs for these sizes: for bf16 at dk = dv = 128 the
 * fp16 sub-token keys ([B][2T+1][H][128]), the fp16 queries r_t, values and sub-token
 * outputs ([B][T][H][128] each), the sub-tokens' bf16 strengths and one fp32 scalar per
 * token-head, each rounded up to 256 bytes; 0 otherwise. */
QD_API size_t eda_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype);

/*
 * qdelta_fwd_static_scratch -- qdelta_fwd for callers that cannot allocate device
 * memory at call time.  The pages have no counterpart: this is a property of the
 * library, not of the method.
 *
 * Some callers cannot pass a workspace: plain C code that holds only the input and
 * output pointers and no device allocator, or a serving loop whose device memory is
 * reserved up front and that must not call cudaMalloc (which can synchronise the
 * device and can fail under memory pressure) during a step.  This entry point takes
 * no workspace and allocates nothing.  Arguments and results are those of
 * qdelta_fwd.  When the segment scan needs scratch it uses a fixed 24 MiB array in
 * the library's device image (room for 128 segment-heads, B * G * H, of three
 * 128 x 128 fp32 states), which every GPU that loads the library holds until the
 * process exits.  Sizes needing more return QD_ERR_WORKSPACE.
 * The array's device address is looked up on the first call made on each device,
 * so make that first call before any stream capture.  All calls share the array:
 * calls whose work overlaps on the GPU race on it.
 */
QD_API qd_status qdelta_fwd_static_scratch(const void *q, const void *k, const void *v,
                                           const void *alpha, const void *beta, const void *lam,
                                           const float *S0, void *o, float *S_final,
                                           int B, int T, int H, int dk, int dv, int chunk,
                                           qd_dtype dtype, cudaStream_t stream);

/*
 * qd_device_status -- synchronises `stream`, then reports whether any kernel of
 * this library gave up a bounded wait since the last call (QD_ERR_TIMEOUT) or the
 * stream holds a CUDA error (QD_ERR_CUDA).  Clears the timeout flag.
 */
QD_API qd_status qd_device_status(cudaStream_t stream);

/*
 * qd_selftest_bounded_wait -- test hook for the failure path above, not part of any
 * computation.  Launches one CTA on `stream` whose only mbarrier wait can never
 * complete (nothing arrives on it); the wait is the library's bounded wait with a
 * limit of limit_us microseconds (1 .. 1000000), after which the CTA records the
 * timeout exactly as a library kernel does and exits: no trap, no fault, no hang.
 * The next qd_device_status(stream) then returns QD_ERR_TIMEOUT (and clears it);
 * the context stays usable.  QD_ERR_ARG for a limit out of range.
 */
QD_API qd_status qd_selftest_bounded_wait(unsigned limit_us, cudaStream_t stream);

/* Message of the last failed call on this host thread ("" if none). */
QD_API const char *qd_last_error(void);

/* Number of kernels the last successful compute call on this thread launched. */
QD_API int qd_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* QDELTA_GB300_H */

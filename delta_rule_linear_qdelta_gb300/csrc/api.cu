// The C ABI of include/qdelta.h: argument validation, kernel selection and
// error reporting.  No allocation happens here; all buffers belong to the caller.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "../../include/qdelta.h"
#include "qd_internal.cuh"

namespace {

thread_local char g_err[512] = "";
thread_local int g_launches = 0;

qd_status fail(qd_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

qd_status cuda_fail(cudaError_t e, const char *what) {
    return fail(QD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool head_dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Common checks for the chunked forwards.  Returns QD_OK or an error with message.
qd_status check_fwd(const char *fn, const void *const *req, int nreq, const void *const *opt, int nopt,
                    int B, int T, int H, int dk, int dv, int chunk, qd_dtype dt) {
    if (B < 0 || T < 0 || H < 0) return fail(QD_ERR_ARG, "%s: negative size B=%d T=%d H=%d", fn, B, T, H);
    if (dt != QD_F32 && dt != QD_BF16) return fail(QD_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dt);
    if (!head_dim_ok(dk) || !head_dim_ok(dv))
        return fail(QD_ERR_UNSUPPORTED, "%s: head dims dk=%d dv=%d not in {16,32,64,128}", fn, dk, dv);
    if (chunk != 64) return fail(QD_ERR_UNSUPPORTED, "%s: chunk=%d (only 64 is supported)", fn, chunk);
    const double elems = (double)B * T * H * (dk > dv ? dk : dv);
    if (elems > 9.0e15) return fail(QD_ERR_ARG, "%s: sizes overflow", fn);
    if ((double)B * H > 2147483647.0) return fail(QD_ERR_ARG, "%s: B*H exceeds the grid limit", fn);
    const bool empty = (B == 0 || H == 0 || T == 0);
    for (int i = 0; i < nreq; ++i) {
        if (!req[i] && !empty) return fail(QD_ERR_ARG, "%s: required pointer argument #%d is NULL", fn, i);
        if (!aligned16(req[i])) return fail(QD_ERR_ARG, "%s: pointer argument #%d not 16-byte aligned", fn, i);
    }
    for (int i = 0; i < nopt; ++i)
        if (!aligned16(opt[i])) return fail(QD_ERR_ARG, "%s: optional pointer #%d not 16-byte aligned", fn, i);
    return QD_OK;
}

// T == 0: the final state is the initial state.
qd_status empty_sequence(const float *S0, float *S_final, int B, int H, int dk, int dv, cudaStream_t s) {
    if (!S_final || B == 0 || H == 0) return QD_OK;
    const size_t bytes = (size_t)B * H * dk * dv * sizeof(float);
    cudaError_t e = cudaSuccess;
    if (!S0) e = cudaMemsetAsync(S_final, 0, bytes, s);
    else if (S0 != S_final) e = cudaMemcpyAsync(S_final, S0, bytes, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? QD_OK : cuda_fail(e, "state copy for T=0");
}

}  // namespace

namespace qd {
qd_status report_error(qd_status status, const char *msg) { return fail(status, "%s", msg); }

qd_status check_qdelta_fwd_args(const char *fn, const void *q, const void *k, const void *v, const void *alpha,
                                const void *beta, const void *lam, const float *S0, void *o, float *S_final,
                                int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype) {
    g_err[0] = 0;
    const void *req[] = {q, k, v, beta, o};
    const void *opt[] = {alpha, lam, S0, S_final};
    return check_fwd(fn, req, 5, opt, 4, B, T, H, dk, dv, chunk, dtype);
}
}  // namespace qd

extern "C" {

const char *qd_last_error(void) { return g_err; }

int qd_last_launch_count(void) { return g_launches; }

size_t qdelta_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk != 64) return 0;
    return qd::qdelta_segment_workspace(B, H, qd::qdelta_segments(B, T, H, dk, dv, dtype));
}

size_t qed_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk != 64) return 0;
    qd::QedArgs a{};
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    if (!qd::qed_tc_supported(a, dtype)) return 0;     // the CUDA-core path needs none
    return qd::qed_tc_workspace(B, T, H, qd::qed_segments(B, T, H, dk, dv, dtype));
}

size_t qdelta_bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype) {
    (void)dtype;
    if (B <= 0 || T <= 0 || H <= 0 || chunk != 64 || !head_dim_ok(dk) || !head_dim_ok(dv)) return 0;
    return qd::qdelta_bwd_workspace(B, T, H, dk, dv);
}

qd_status qdelta_bwd(const void *q, const void *k, const void *v, const void *alpha, const void *beta,
                     const void *lam, const float *S0, const void *dO, const float *dS_final, void *dq,
                     void *dk_out, void *dv_out, void *dalpha, void *dbeta, void *dlam, float *dS0, int B, int T,
                     int H, int dk, int dv, int chunk, qd_dtype dtype, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    g_err[0] = 0;
    const void *req[] = {q, k, v, beta, dO, dq, dk_out, dv_out, dbeta};
    const void *opt[] = {alpha, lam, S0, dS_final, dalpha, dlam, dS0, workspace};
    qd_status st = check_fwd("qdelta_bwd", req, 9, opt, 8, B, T, H, dk, dv, chunk, dtype);
    if (st != QD_OK) return st;
    if ((double)B * H * ((T + 63) / 64) > 2147483647.0) return fail(QD_ERR_ARG, "qdelta_bwd: B*H*chunks exceeds the grid limit");
    if (B == 0 || H == 0) { g_launches = 0; return QD_OK; }
    if (T == 0) { g_launches = 0; return empty_sequence(dS_final, dS0, B, H, dk, dv, stream); }
    const size_t need = qdelta_bwd_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
    if (!workspace || workspace_bytes < need)
        return fail(QD_ERR_WORKSPACE, "qdelta_bwd: workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    float *chk = static_cast<float *>(workspace);
    const size_t half = need / 2 / sizeof(float);
    qd::QDeltaBwdArgs a{q, k, v, alpha, beta, lam, S0, dO, dS_final, dq, dk_out, dv_out, dalpha, dbeta, dlam,
                        dS0, B, T, H, dk, dv, chk, chk + half};
    int n = 0;
    cudaError_t e = qd::launch_qdelta_bwd(a, dtype, stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "qdelta_bwd launch");
    g_launches = n;
    return QD_OK;
}

}  // extern "C"

namespace {

// The chunked forward: tensor-core kernel (single pass or segment scan) where it
// applies, else the CUDA-core kernel.
cudaError_t run_forward(const qd::QDeltaArgs &a, qd_dtype dtype, cudaStream_t stream, int *n) {
    if (qd::qdelta_tc_supported(a, dtype)) {
        const int G = qd::qdelta_segments(a.B, a.T, a.H, a.dk, a.dv, dtype);
        return G > 1 ? qd::launch_qdelta_segmented(a, G, stream, n) : qd::launch_qdelta_chunk_tc(a, stream, n);
    }
    return qd::launch_qdelta_chunk_simt(a, dtype, stream, n);
}

qd_status qdelta_fwd_impl(const char *fn, int prologue, const void *q, const void *k, const void *v,
                          const void *alpha, const void *beta, const void *lam, const float *S0, void *o,
                          float *S_final, int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    g_err[0] = 0;
    const void *req[] = {q, k, v, beta, o};
    const void *opt[] = {alpha, lam, S0, S_final, workspace};
    qd_status st = check_fwd(fn, req, 5, opt, 5, B, T, H, dk, dv, chunk, dtype);
    if (st != QD_OK) return st;
    const size_t need = qdelta_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
    if (need && (!workspace || workspace_bytes < need))
        return fail(QD_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need, workspace_bytes);
    int n = 0;
    if (B == 0 || H == 0) { g_launches = 0; return QD_OK; }
    if (T == 0) { g_launches = 0; return empty_sequence(S0, S_final, B, H, dk, dv, stream); }
    qd::QDeltaArgs a{q, k, v, alpha, beta, lam, S0, o, S_final, B, T, H, dk, dv, workspace, workspace_bytes,
                     prologue};
    cudaError_t e = run_forward(a, dtype, stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "qdelta_fwd launch");
    g_launches = n;
    return QD_OK;
}

qd_status qdelta_step_impl(const char *fn, int prologue, float *S, const void *q, const void *k,
                           const void *v, const void *alpha, const void *beta, const void *lam, void *o, int N,
                           int H, int dk, int dv, qd_dtype dtype, cudaStream_t stream) {
    g_err[0] = 0;
    if (N < 0 || H < 0) return fail(QD_ERR_ARG, "%s: negative size N=%d H=%d", fn, N, H);
    if (dtype != QD_F32 && dtype != QD_BF16) return fail(QD_ERR_UNSUPPORTED, "%s: unknown dtype", fn);
    if (!head_dim_ok(dk) || !head_dim_ok(dv))
        return fail(QD_ERR_UNSUPPORTED, "%s: head dims dk=%d dv=%d not in {16,32,64,128}", fn, dk, dv);
    if ((double)N * H > 2147483647.0) return fail(QD_ERR_ARG, "%s: N*H exceeds the grid limit", fn);
    const bool empty = (N == 0 || H == 0);
    const void *req[] = {S, q, k, v, beta, o};
    for (int i = 0; i < 6; ++i) {
        if (!req[i] && !empty) return fail(QD_ERR_ARG, "%s: required pointer argument #%d is NULL", fn, i);
        if (!aligned16(req[i])) return fail(QD_ERR_ARG, "%s: pointer argument #%d not 16-byte aligned", fn, i);
    }
    if (!aligned16(alpha) || !aligned16(lam)) return fail(QD_ERR_ARG, "%s: gate pointer not 16-byte aligned", fn);
    g_launches = 0;
    if (empty) return QD_OK;
    int n = 0;
    qd::StepArgs a{S, q, k, v, alpha, beta, lam, o, N, H, dk, dv, prologue};
    cudaError_t e = qd::launch_qdelta_step(a, dtype, stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "qdelta_step launch");
    g_launches = n;
    return QD_OK;
}

}  // namespace

extern "C" {

qd_status qdelta_fwd(const void *q, const void *k, const void *v, const void *alpha, const void *beta,
                     const void *lam, const float *S0, void *o, float *S_final, int B, int T, int H,
                     int dk, int dv, int chunk, qd_dtype dtype, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    return qdelta_fwd_impl("qdelta_fwd", 0, q, k, v, alpha, beta, lam, S0, o, S_final, B, T, H, dk, dv, chunk,
                           dtype, workspace, workspace_bytes, stream);
}

size_t qdelta_bwd_prologue_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk != 64 || !head_dim_ok(dk) || !head_dim_ok(dv)) return 0;
    return qd::prologue_bwd_buffers(B, T, H, dk, dtype).bwd + qdelta_bwd_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
}

qd_status qdelta_bwd_prologue(const void *q_raw, const void *k_raw, const void *v, const void *a_logit,
                              const void *b_logit, const void *l_logit, const float *S0, const void *dO,
                              const float *dS_final, void *dq_raw, void *dk_raw, void *dv_out, void *da_logit,
                              void *db_logit, void *dl_logit, float *dS0, int B, int T, int H, int dk, int dv,
                              int chunk, qd_dtype dtype, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    g_err[0] = 0;
    const void *req[] = {q_raw, k_raw, v, b_logit, dO, dq_raw, dk_raw, dv_out, db_logit};
    const void *opt[] = {a_logit, l_logit, S0, dS_final, da_logit, dl_logit, dS0, workspace};
    qd_status st = check_fwd("qdelta_bwd_prologue", req, 9, opt, 8, B, T, H, dk, dv, chunk, dtype);
    if (st != QD_OK) return st;
    if ((double)B * H * ((T + 63) / 64) > 2147483647.0)
        return fail(QD_ERR_ARG, "qdelta_bwd_prologue: B*H*chunks exceeds the grid limit");
    if (B == 0 || H == 0) { g_launches = 0; return QD_OK; }
    if (T == 0) { g_launches = 0; return empty_sequence(dS_final, dS0, B, H, dk, dv, stream); }
    const size_t need = qdelta_bwd_prologue_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
    if (!workspace || workspace_bytes < need)
        return fail(QD_ERR_WORKSPACE, "qdelta_bwd_prologue: workspace of %zu bytes needed, %zu given", need,
                    workspace_bytes);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const qd::PrologueBwdBuffers w = qd::prologue_bwd_buffers(B, T, H, dk, dtype);
    qd::QDeltaBwdArgs raw{q_raw, k_raw, v, a_logit, b_logit, l_logit, S0, dO, dS_final, dq_raw, dk_raw, dv_out,
                          da_logit, db_logit, dl_logit, dS0, B, T, H, dk, dv, nullptr, nullptr};
    int n = 0;
    cudaError_t e = qd::launch_prologue_map(raw, dtype, ws, stream, &n);
    if (e == cudaSuccess) {
        float *chk = reinterpret_cast<float *>(ws + w.bwd);
        const size_t half = qdelta_bwd_workspace_bytes(B, T, H, dk, dv, chunk, dtype) / 2 / sizeof(float);
        qd::QDeltaBwdArgs m{ws + w.q, ws + w.k, v, a_logit ? ws + w.a : nullptr, ws + w.b,
                            l_logit ? ws + w.l : nullptr, S0, dO, dS_final, ws + w.dq, ws + w.dk, dv_out,
                            a_logit ? ws + w.da : nullptr, ws + w.db, l_logit ? ws + w.dl : nullptr, dS0,
                            B, T, H, dk, dv, chk, chk + half, 1, 1, q_raw, k_raw, a_logit, b_logit, l_logit};
        e = qd::launch_qdelta_bwd(m, dtype, stream, &n);
    }
    if (e == cudaSuccess) e = qd::launch_prologue_chain(raw, dtype, ws, stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "qdelta_bwd_prologue launch");
    g_launches = n;
    return QD_OK;
}

size_t eda_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk != 64) return 0;
    qd::EdaArgs a{};
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv;
    if (!qd::eda_tc_supported(a, dtype)) return 0;     // the recurrent kernel needs none
    return qd::eda_tc_workspace(B, T, H);
}

qd_status eda_fwd(const void *q, const void *k, const void *v, const void *e, const void *beta, const float *S0,
                  void *o, float *S_final, int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    g_err[0] = 0;
    const void *req[] = {q, k, v, e, o};
    const void *opt[] = {beta, S0, S_final, workspace};
    qd_status st = check_fwd("eda_fwd", req, 5, opt, 4, B, T, H, dk, dv, chunk, dtype);
    if (st != QD_OK) return st;
    if (B == 0 || H == 0) { g_launches = 0; return QD_OK; }
    if (T == 0) { g_launches = 0; return empty_sequence(S0, S_final, B, H, dk, dv, stream); }
    qd::EdaArgs a{q, k, v, e, beta, S0, o, S_final, B, T, H, dk, dv};
    const size_t need = eda_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
    if (need && (!workspace || workspace_bytes < need))
        return fail(QD_ERR_WORKSPACE, "eda_fwd: workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    int n = 0;
    cudaError_t err = need ? qd::launch_eda_tc(a, workspace, stream, &n) : qd::launch_eda(a, dtype, stream, &n);
    if (err != cudaSuccess) return cuda_fail(err, "eda_fwd launch");
    g_launches = n;
    return QD_OK;
}

qd_status qdelta_fwd_prologue(const void *q_raw, const void *k_raw, const void *v, const void *a_logit,
                              const void *b_logit, const void *l_logit, const float *S0, void *o, float *S_final,
                              int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    return qdelta_fwd_impl("qdelta_fwd_prologue", 1, q_raw, k_raw, v, a_logit, b_logit, l_logit, S0, o, S_final,
                           B, T, H, dk, dv, chunk, dtype, workspace, workspace_bytes, stream);
}

qd_status qed_fwd_variant(const void *q, const void *k, const void *v, const void *g, const void *b,
                          const void *w, const float *lam_h, const float *S0, void *o, float *S_final, int B,
                          int T, int H, int dk, int dv, int chunk, qd_dtype dtype, qd_qed_variant variant,
                          const float *z_h, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    g_err[0] = 0;
    if (variant < QD_QED_FULL || variant > QD_QED_RAND)
        return fail(QD_ERR_ARG, "qed_fwd_variant: unknown variant %d", (int)variant);
    const void *req[] = {q, k, v, g, b, w, lam_h, o};
    const void *opt[] = {S0, S_final, workspace, z_h};
    qd_status st = check_fwd("qed_fwd", req, 8, opt, 4, B, T, H, dk, dv, chunk, dtype);
    if (st != QD_OK) return st;
    if (variant == QD_QED_RAND && !z_h && B > 0 && H > 0 && T > 0)
        return fail(QD_ERR_ARG, "qed_fwd_variant: the rand arm needs z_h [H][dk]");
    const size_t need = qed_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
    if (need && (!workspace || workspace_bytes < need))
        return fail(QD_ERR_WORKSPACE, "qed_fwd: workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    int n = 0;
    if (B == 0 || H == 0) { g_launches = 0; return QD_OK; }
    if (T == 0) { g_launches = 0; return empty_sequence(S0, S_final, B, H, dk, dv, stream); }
    qd::QedArgs a{q, k, v, g, b, w, lam_h, S0, o, S_final, B, T, H, dk, dv, workspace, workspace_bytes,
                  (int)variant, z_h};
    cudaError_t e;
    if (qd::qed_tc_supported(a, dtype)) {
        const int G = qd::qed_segments(B, T, H, dk, dv, dtype);
        e = qd::launch_qed_tc(a, G, stream, &n);
    } else {
        e = qd::launch_qed_chunk_simt(a, dtype, stream, &n);
    }
    if (e != cudaSuccess) return cuda_fail(e, "qed_fwd launch");
    g_launches = n;
    return QD_OK;
}

qd_status qed_fwd(const void *q, const void *k, const void *v, const void *g, const void *b, const void *w,
                  const float *lam_h, const float *S0, void *o, float *S_final, int B, int T, int H, int dk,
                  int dv, int chunk, qd_dtype dtype, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
    return qed_fwd_variant(q, k, v, g, b, w, lam_h, S0, o, S_final, B, T, H, dk, dv, chunk, dtype, QD_QED_FULL,
                           nullptr, workspace, workspace_bytes, stream);
}

qd_status qed_step(float *S, const void *q, const void *k, const void *v, const void *g, const void *b,
                   const void *w, const float *lam_h, void *o, int N, int H, int dk, int dv, qd_dtype dtype,
                   qd_qed_variant variant, const float *z_h, cudaStream_t stream) {
    g_err[0] = 0;
    if (N < 0 || H < 0) return fail(QD_ERR_ARG, "qed_step: negative size N=%d H=%d", N, H);
    if (dtype != QD_F32 && dtype != QD_BF16) return fail(QD_ERR_UNSUPPORTED, "qed_step: unknown dtype");
    if (variant < QD_QED_FULL || variant > QD_QED_RAND)
        return fail(QD_ERR_ARG, "qed_step: unknown variant %d", (int)variant);
    if (!head_dim_ok(dk) || !head_dim_ok(dv))
        return fail(QD_ERR_UNSUPPORTED, "qed_step: head dims dk=%d dv=%d not in {16,32,64,128}", dk, dv);
    if ((double)N * H > 2147483647.0) return fail(QD_ERR_ARG, "qed_step: N*H exceeds the grid limit");
    const bool empty = (N == 0 || H == 0);
    const void *req[] = {S, q, k, v, g, b, w, lam_h, o};
    for (int i = 0; i < 9; ++i) {
        if (!req[i] && !empty) return fail(QD_ERR_ARG, "qed_step: required pointer argument #%d is NULL", i);
        if (!aligned16(req[i])) return fail(QD_ERR_ARG, "qed_step: pointer argument #%d not 16-byte aligned", i);
    }
    if (!aligned16(z_h)) return fail(QD_ERR_ARG, "qed_step: z_h not 16-byte aligned");
    if (variant == QD_QED_RAND && !z_h && !empty) return fail(QD_ERR_ARG, "qed_step: the rand arm needs z_h [H][dk]");
    g_launches = 0;
    if (empty) return QD_OK;
    int n = 0;
    qd::QedStepArgs a{S, q, k, v, g, b, w, lam_h, o, N, H, dk, dv, (int)variant, z_h};
    cudaError_t e = qd::launch_qed_step(a, dtype, stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "qed_step launch");
    g_launches = n;
    return QD_OK;
}

qd_status qdelta_step(float *S, const void *q, const void *k, const void *v, const void *alpha,
                      const void *beta, const void *lam, void *o, int N, int H, int dk, int dv,
                      qd_dtype dtype, cudaStream_t stream) {
    return qdelta_step_impl("qdelta_step", 0, S, q, k, v, alpha, beta, lam, o, N, H, dk, dv, dtype, stream);
}

qd_status qdelta_step_prologue(float *S, const void *q_raw, const void *k_raw, const void *v,
                               const void *a_logit, const void *b_logit, const void *l_logit, void *o, int N,
                               int H, int dk, int dv, qd_dtype dtype, cudaStream_t stream) {
    return qdelta_step_impl("qdelta_step_prologue", 1, S, q_raw, k_raw, v, a_logit, b_logit, l_logit, o, N, H, dk,
                            dv, dtype, stream);
}

qd_status qd_selftest_bounded_wait(unsigned limit_us, cudaStream_t stream) {
    g_err[0] = 0;
    if (limit_us < 1 || limit_us > 1000000)
        return fail(QD_ERR_ARG, "qd_selftest_bounded_wait: limit_us=%u not in [1, 1000000]", limit_us);
    cudaError_t e = qd::launch_wait_selftest((uint64_t)limit_us * 1000ull, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qd_selftest_bounded_wait launch");
    g_launches = 1;
    return QD_OK;
}

qd_status qd_device_status(cudaStream_t stream) {
    g_err[0] = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "qd_device_status");
    const bool t1 = qd::tc_read_and_clear_timeout(), t2 = qd::bwd_tc_read_and_clear_timeout();
    const bool t3 = qd::selftest_read_and_clear_timeout(), t4 = qd::grad_tc_read_and_clear_timeout();
    if (t1 || t2 || t3 || t4)
        return fail(QD_ERR_TIMEOUT, "a tensor-core kernel gave up a bounded wait (results of that call are invalid)");
    return QD_OK;
}

}  // extern "C"

// Internal declarations shared by the library's translation units (not part of
// the C ABI).  Device helpers for dtype conversion and the launcher signatures.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qdelta.h"

namespace qd {

enum { kF32 = 0, kBF16 = 1 };

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// The prologue computed from the layer's projections ("Parallelizing Linear
// Transformers with the Delta Rule over Sequence Length", sec. 3.8: q, k =
// SiLU(x)/|SiLU(x)|_2, beta = sigmoid; Q-Delta notes sec. 2.5: lambda = sigmoid; the
// decay alpha = exp(-softplus(x)), log alpha = -softplus(x)).  Accurate forms for the
// fp32 paths; the tensor-core path uses the hardware tanh (sigmoid(x) =
// (1 + tanh(x/2))/2), whose error is below the bf16 rounding its results get.
__device__ __forceinline__ float silu_acc(float x) { return x / (1.f + expf(-x)); }
__device__ __forceinline__ float sigmoid_acc(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float neg_softplus(float x) { return -(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)))); }
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sigmoid_fast(float x) { return fmaf(0.5f, tanh_fast(0.5f * x), 0.5f); }
__device__ __forceinline__ float silu_fast(float x) { return x * sigmoid_fast(x); }

// Arguments of one Q-Delta forward (layouts as in include/qdelta.h).
struct QDeltaArgs {
    const void *q, *k, *v, *alpha, *beta, *lam;
    const float *S0;
    void *o;
    float *S_final;
    int B, T, H, dk, dv;
    void *ws;
    size_t ws_bytes;
    int prologue;     // q, k, alpha, beta, lam are projections and logits (qdelta_fwd_prologue)
    float *S_chk;     // if set, the state entering every chunk of 64 tokens (the backward's
                      // checkpoints), per (b*H + h, chunk): an [dv][dk] fp32 array from the
                      // CUDA-core kernel, a 32 KB fp16 operand tile (tc::chk_tile_off) from
                      // the tensor-core kernel
};

// Arguments of one Q-Delta backward (layouts as in include/qdelta.h); nk, nv are
// d_k, d_v.  S_chk and dS_chk are the two checkpoint arrays in the workspace, one entry
// per (b*H + h, chunk of 64): the state entering each chunk and the gradient reaching
// the state leaving it -- [dv][dk] fp32 for the CUDA-core kernels, a 32 KB fp16 tile in
// the 128-byte-swizzled operand layout (tc::chk_tile_off) for the tensor-core ones
// (qdelta_bwd_tc_supported decides both the format and the forward that writes it).
struct QDeltaBwdArgs {
    const void *q, *k, *v, *alpha, *beta, *lam;
    const float *S0;
    const void *dO;
    const float *dS_final;
    void *dq, *dk, *dv, *dalpha, *dbeta, *dlam;
    float *dS0;
    int B, T, H, nk, nv;
    float *S_chk, *dS_chk;
    int grad_f32;     // dq, dk, dalpha, dbeta, dlam written as fp32 whatever the dtype (for the
                      // prologue's chain rule, which would otherwise see them rounded)
    int gates_f32;    // alpha, beta, lam are fp32 arrays whatever the dtype (gates mapped from
                      // logits: alpha near 1 rounded to bf16 would lose most of log alpha)
    // backward from projections: the raw inputs, from which the checkpoint forward runs
    // with the prologue (null otherwise)
    const void *raw_q, *raw_k, *raw_a, *raw_b, *raw_l;
};

// A gate value of token `tok`: fp32 when f32, else the call's dtype.
template <typename TIn>
__device__ __forceinline__ float gate_val(const void *p, size_t tok, int f32) {
    return f32 ? static_cast<const float *>(p)[tok] : to_f(static_cast<const TIn *>(p)[tok]);
}

// Arguments of one EDA forward (erase along e, then the Delta write): q, k, e
// [B][T][H][dk], v, o [B][T][H][dv], beta [B][T][H] or NULL (= 1).
struct EdaArgs {
    const void *q, *k, *v, *e, *beta;
    const float *S0;
    void *o;
    float *S_final;
    int B, T, H, dk, dv;
};
// The EDA forward: a recurrent fp32 kernel, one CTA per (b, h), dv <= 128.
cudaError_t launch_eda(const EdaArgs &a, int dtype, cudaStream_t s, int *nlaunch);
// The EDA forward on the tensor cores (bf16, dk = dv = 128): a sub-token pass, the fp16
// instance of the Q-Delta tensor-core forward over 2T+1 sub-tokens and a read-out pass,
// in eda_tc_workspace(B, T, H) bytes of workspace.
bool eda_tc_supported(const EdaArgs &a, int dtype);
size_t eda_tc_workspace(int B, int T, int H);
cudaError_t launch_eda_tc(const EdaArgs &a, void *ws, cudaStream_t s, int *nlaunch);

// QED ablation arms ("The Query Knows What to Forget", Table 1): the term added to
// the base erase vector b*k, P(u) = u - k (k^T u):
//   full lambda_h P(b*q); nogate lambda_h P(q); nogate-noproj lambda_h q;
//   rand lambda_h P(b*z_h) with z_h [H][dk] fp32.  Values match qd_qed_variant.
enum { kQedFull = 0, kQedNogate = 1, kQedNogateNoproj = 2, kQedRand = 3 };

// Arguments of one QED forward.
struct QedArgs {
    const void *q, *k, *v, *g, *b, *w;
    const float *lam_h, *S0;
    void *o;
    float *S_final;
    int B, T, H, dk, dv;
    void *ws;
    size_t ws_bytes;
    int variant;          // kQed*
    const float *z;       // [H][dk] for kQedRand, else unused
};

// Arguments of one QED decode step.
struct QedStepArgs {
    float *S;
    const void *q, *k, *v, *g, *b, *w;
    const float *lam_h;
    void *o;
    int N, H, dk, dv;
    int variant;
    const float *z;
};

// Arguments of one decode step.
struct StepArgs {
    float *S;
    const void *q, *k, *v, *alpha, *beta, *lam;
    void *o;
    int N, H, dk, dv;
    int prologue;     // as in QDeltaArgs
};

// Launchers.  Each returns the first CUDA error and adds its launches to *nlaunch.
cudaError_t launch_qdelta_chunk_simt(const QDeltaArgs &a, int dtype, cudaStream_t s, int *nlaunch);
// Backward of the chunked forward: checkpoint forward, reverse state-gradient sweep and
// the per-chunk gradient kernel.  qdelta_bwd_workspace is the workspace it needs.
size_t qdelta_bwd_workspace(int B, int T, int H, int dk, int dv);
cudaError_t launch_qdelta_bwd(const QDeltaBwdArgs &a, int dtype, cudaStream_t s, int *nlaunch);
// Backward from projections: byte offsets in its workspace (the mapped inputs q, k,
// alpha, beta, lambda; their gradients; the recurrence backward's own workspace from
// `bwd` on), and the two kernels around qdelta_bwd.  `raw` carries the projections and
// logits in q, k, alpha, beta, lam and the caller's outputs in dq, dk, dalpha, dbeta, dlam.
struct PrologueBwdBuffers {
    size_t q, k, a, b, l, dq, dk, da, db, dl, bwd;
};
PrologueBwdBuffers prologue_bwd_buffers(int B, int T, int H, int dk, int dtype);
cudaError_t launch_prologue_map(const QDeltaBwdArgs &raw, int dtype, uint8_t *ws, cudaStream_t s, int *nlaunch);
cudaError_t launch_prologue_chain(const QDeltaBwdArgs &raw, int dtype, const uint8_t *ws, cudaStream_t s,
                                  int *nlaunch);
// The reverse sweep and the per-chunk gradients on the tcgen05 tensor cores (bf16,
// dk = dv = 128: qdelta_bwd_tc_supported) and their timeout words.
bool qdelta_bwd_tc_supported(const QDeltaBwdArgs &a, int dtype);
cudaError_t launch_qdelta_bwd_dstate_tc(const QDeltaBwdArgs &a, cudaStream_t s);
cudaError_t launch_qdelta_bwd_grad_tc(const QDeltaBwdArgs &a, cudaStream_t s);
bool bwd_tc_read_and_clear_timeout();
bool grad_tc_read_and_clear_timeout();
cudaError_t launch_qed_chunk_simt(const QedArgs &a, int dtype, cudaStream_t s, int *nlaunch);
cudaError_t launch_qdelta_step(const StepArgs &a, int dtype, cudaStream_t s, int *nlaunch);
cudaError_t launch_qed_step(const QedStepArgs &a, int dtype, cudaStream_t s, int *nlaunch);

// Tensor-core (tcgen05) chunked Q-Delta forward: bf16, dk = dv = 128.  flags select the
// segment-scan passes: kTcNoV (v taken as 0, v not read), kTcS0Identity (S0 = I per
// head, needs dk = dv), kTcNoO (o not written); kTcF16 takes q, k, v, o as fp16 and forms
// every operand in fp16 (alpha null, no prologue, no checkpoints).
enum { kTcNoV = 1, kTcS0Identity = 2, kTcNoO = 4, kTcF16 = 8 };
bool qdelta_tc_supported(const QDeltaArgs &a, int dtype);
cudaError_t launch_qdelta_chunk_tc(const QDeltaArgs &a, cudaStream_t s, int *nlaunch, int flags = 0);
// Tensor-core (tcgen05) chunked QED forward: bf16, dk = dv = 128; flags as above.  The
// state-independent per-chunk operands are derived first (qed_derive_kernel) into the
// workspace, over the same [B][T] view the chain kernel then runs on (a segment view
// when segmented): Ae, Qe, Ke, W*V as [B][T][H][128] bf16 and e^{G_C} as
// [B][H][nchunks][128] fp32.
struct QedDerived {
    void *Ae, *Qe, *Ke, *WV;
    float *ecg;
};
bool qed_tc_supported(const QedArgs &a, int dtype);
size_t qed_derived_bytes(int B, int T, int H, int G);
QedDerived qed_derived_buffers(int B, int T, int H, void *ws);
cudaError_t launch_qed_derive(const QedArgs &a, const QedDerived &d, int no_v, cudaStream_t s, int *nlaunch);
// One pass of the chain kernel over derived operands (the QED instance of the Q-Delta
// tensor-core kernel); a carries the view's sizes, S0, o and S_final.
cudaError_t launch_qed_chain_tc(const QedArgs &a, const QedDerived &d, cudaStream_t s, int *nlaunch, int flags = 0);
// Derive and chain in one cooperative launch: the chains of the B*H streams on B*H SMs,
// the derive step on the rest, handing each chunk over through `done` (B*H*ceil(T/64)
// counters in device memory, cleared by the launch).  Needs B*H below the SM count.
cudaError_t launch_qed_fused_tc(const QedArgs &a, const QedDerived &d, unsigned int *done, cudaStream_t s,
                                int *nlaunch);
// SMs of the current device (0 if unknown).
int sm_count();
// Segment scan of the tensor-core forward for long sequences over few (b, h)
// streams: the number of segments for these sizes (1 = a single pass), its
// workspace, and the launch (three passes of the forward kernel and a combine).
int qdelta_segments(int B, int T, int H, int dk, int dv, int dtype);
size_t qdelta_segment_workspace(int B, int H, int G);
cudaError_t launch_qdelta_segmented(const QDeltaArgs &a, int G, cudaStream_t s, int *nlaunch);
// The same for QED, whose per-chunk state map is also a right-multiplication of the
// [dv][dk] state (S_out = S_in Phi + Psi); qed_segments is its own policy.
int qed_segments(int B, int T, int H, int dk, int dv, int dtype);
cudaError_t launch_qed_segmented(const QedArgs &a, int G, const QedDerived &d, cudaStream_t s, int *nlaunch);
// The whole tensor-core QED forward: derive over the (segment) view, then one chain pass
// or the segment scan; in one pass with the derive beside the chains (launch_qed_fused_tc)
// when B*H leaves at least 8 SMs to the derive step.  Workspace: qed_tc_workspace(B, T,
// H, G) bytes at a.ws (the derived operands, then the segment states, then the hand-over
// counters).
size_t qed_tc_workspace(int B, int T, int H, int G);
cudaError_t launch_qed_tc(const QedArgs &a, int G, cudaStream_t s, int *nlaunch);
// Reads and clears the device word the tensor-core kernels set when a bounded wait runs out.
bool tc_read_and_clear_timeout();
// One CTA whose only mbarrier wait can never complete, bounded by limit_ns: sets its own
// timeout word, read and cleared like the kernels' by selftest_read_and_clear_timeout.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s);
bool selftest_read_and_clear_timeout();

// Records `msg` as this host thread's last error (qd_last_error) and returns `status`.
qd_status report_error(qd_status status, const char *msg);
// The host-side argument checks of qdelta_fwd (pointers, alignment, sizes, head
// dims, chunk, dtype), without the workspace check; no CUDA call.
qd_status check_qdelta_fwd_args(const char *fn, const void *q, const void *k, const void *v, const void *alpha,
                                const void *beta, const void *lam, const float *S0, void *o, float *S_final,
                                int B, int T, int H, int dk, int dv, int chunk, qd_dtype dtype);

}  // namespace qd

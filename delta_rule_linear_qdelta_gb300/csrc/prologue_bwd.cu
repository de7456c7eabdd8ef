// Backward of the forward from projections (qdelta_bwd_prologue): the layer's input
// maps ("Parallelizing Linear Transformers with the Delta Rule over Sequence Length",
// sec. 3.8: q, k = SiLU(x)/|SiLU(x)|, beta = sigmoid; Q-Delta notes sec. 2.5: lambda =
// sigmoid; the decay alpha = exp(-softplus(x)) = sigmoid(-x)) around the recurrence's
// backward, by the chain rule.  Two kernels, one warp per token-head row:
//   map:    q, k (fp32 arithmetic, stored in the call's dtype) and alpha, beta, lambda (kept
//           in fp32: alpha near 1 rounded to bf16 would lose most of log alpha) from the
//           projections and logits; the checkpoint forward runs the prologue forward on
//           the raw inputs, and the backward kernels return the mapped inputs' gradients in
//           fp32 (the chain rule's projection below cancels part of dy);
//   chain:  with s = SiLU(x), n = |s|, y = s / n and the incoming dy,
//           dx = ((dy - y (y . dy)) / n) * SiLU'(x),  SiLU'(x) = sig(x) (1 + x (1 - sig(x)))
//           (an all-zero s, which the forward leaves at y = 0, passes no gradient), and
//           d b = dbeta beta (1 - beta), d l = dlam lam (1 - lam), d a = -dalpha alpha (1 - alpha).
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kWarps = 8;    // rows per CTA

template <typename TIn>
__global__ void __launch_bounds__(32 * kWarps) prologue_map_kernel(QDeltaBwdArgs raw, int d, TIn *qm, TIn *km,
                                                                   float *am, float *bm, float *lm) {
    const size_t rows = (size_t)raw.B * raw.T * raw.H;
    const size_t row = (size_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    for (int which = 0; which < 2; ++which) {
        const TIn *x = (const TIn *)(which ? raw.k : raw.q) + row * d;
        TIn *y = (which ? km : qm) + row * d;
        float s[4], ss = 0.f;                         // d <= 128: at most four elements per lane
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            s[i] = j < d ? silu_acc(to_f(x[j])) : 0.f;
            ss = fmaf(s[i], s[i], ss);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = ss > 0.f ? 1.f / sqrtf(ss) : 1.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (lane + 32 * i < d) y[lane + 32 * i] = from_f<TIn>(s[i] * inv);
    }
    if (lane == 0) {
        if (raw.alpha) am[row] = expf(neg_softplus(to_f(((const TIn *)raw.alpha)[row])));
        bm[row] = sigmoid_acc(to_f(((const TIn *)raw.beta)[row]));
        if (raw.lam) lm[row] = sigmoid_acc(to_f(((const TIn *)raw.lam)[row]));
    }
}

template <typename TIn>
__global__ void __launch_bounds__(32 * kWarps) prologue_chain_kernel(QDeltaBwdArgs raw, int d, const float *dq,
                                                                     const float *dk, const float *da,
                                                                     const float *db, const float *dl) {
    const size_t rows = (size_t)raw.B * raw.T * raw.H;
    const size_t row = (size_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    for (int which = 0; which < 2; ++which) {
        const TIn *x = (const TIn *)(which ? raw.k : raw.q) + row * d;
        const float *dy = (which ? dk : dq) + row * d;
        TIn *dx = (TIn *)(which ? raw.dk : raw.dq) + row * d;
        float xv[4], s[4], g[4], ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            xv[i] = j < d ? to_f(x[j]) : 0.f;
            g[i] = j < d ? dy[j] : 0.f;
            s[i] = xv[i] * sigmoid_acc(xv[i]);
            ss = fmaf(s[i], s[i], ss);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (!(ss > 0.f)) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (lane + 32 * i < d) dx[lane + 32 * i] = from_f<TIn>(0.f);
            continue;
        }
        const float n = sqrtf(ss), inv = 1.f / n;
        float ydy = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) ydy = fmaf(s[i] * inv, g[i], ydy);
#pragma unroll
        for (int off = 16; off; off >>= 1) ydy += __shfl_xor_sync(0xffffffffu, ydy, off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            if (j < d) {
                const float sg = sigmoid_acc(xv[i]);
                dx[j] = from_f<TIn>((g[i] - s[i] * inv * ydy) * inv * (sg * (1.f + xv[i] * (1.f - sg))));
            }
        }
    }
    if (lane == 0) {
        const float bt = sigmoid_acc(to_f(((const TIn *)raw.beta)[row]));
        ((TIn *)raw.dbeta)[row] = from_f<TIn>(db[row] * bt * (1.f - bt));
        if (raw.alpha && raw.dalpha) {
            const float al = expf(neg_softplus(to_f(((const TIn *)raw.alpha)[row])));
            ((TIn *)raw.dalpha)[row] = from_f<TIn>(-da[row] * al * (1.f - al));
        }
        if (raw.lam && raw.dlam) {
            const float lm = sigmoid_acc(to_f(((const TIn *)raw.lam)[row]));
            ((TIn *)raw.dlam)[row] = from_f<TIn>(dl[row] * lm * (1.f - lm));
        }
    }
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

PrologueBwdBuffers prologue_bwd_buffers(int B, int T, int H, int dk, int dtype) {
    const size_t el = dtype == kBF16 ? 2 : 4, rows = (size_t)B * T * H;
    PrologueBwdBuffers w{};
    size_t off = 0;
    w.q = off; off += up256(rows * dk * el);
    w.k = off; off += up256(rows * dk * el);
    w.a = off; off += up256(rows * 4);                // mapped gates: fp32
    w.b = off; off += up256(rows * 4);
    w.l = off; off += up256(rows * 4);
    w.dq = off; off += up256(rows * dk * 4);          // the mapped inputs' gradients: fp32
    w.dk = off; off += up256(rows * dk * 4);
    w.da = off; off += up256(rows * 4);
    w.db = off; off += up256(rows * 4);
    w.dl = off; off += up256(rows * 4);
    w.bwd = off;
    return w;
}

cudaError_t launch_prologue_map(const QDeltaBwdArgs &raw, int dtype, uint8_t *ws, cudaStream_t s, int *nlaunch) {
    const PrologueBwdBuffers w = prologue_bwd_buffers(raw.B, raw.T, raw.H, raw.nk, dtype);
    const size_t rows = (size_t)raw.B * raw.T * raw.H;
    const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
    if (dtype == kBF16) {
        using T = __nv_bfloat16;
        prologue_map_kernel<T><<<grid, 32 * kWarps, 0, s>>>(raw, raw.nk, (T *)(ws + w.q), (T *)(ws + w.k),
                                                            (float *)(ws + w.a), (float *)(ws + w.b),
                                                            (float *)(ws + w.l));
    } else {
        prologue_map_kernel<float><<<grid, 32 * kWarps, 0, s>>>(raw, raw.nk, (float *)(ws + w.q), (float *)(ws + w.k),
                                                                (float *)(ws + w.a), (float *)(ws + w.b),
                                                                (float *)(ws + w.l));
    }
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

cudaError_t launch_prologue_chain(const QDeltaBwdArgs &raw, int dtype, const uint8_t *ws, cudaStream_t s,
                                  int *nlaunch) {
    const PrologueBwdBuffers w = prologue_bwd_buffers(raw.B, raw.T, raw.H, raw.nk, dtype);
    const size_t rows = (size_t)raw.B * raw.T * raw.H;
    const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
    if (dtype == kBF16) {
        using T = __nv_bfloat16;
        prologue_chain_kernel<T><<<grid, 32 * kWarps, 0, s>>>(raw, raw.nk, (const float *)(ws + w.dq),
                                                              (const float *)(ws + w.dk), (const float *)(ws + w.da),
                                                              (const float *)(ws + w.db), (const float *)(ws + w.dl));
    } else {
        prologue_chain_kernel<float><<<grid, 32 * kWarps, 0, s>>>(raw, raw.nk, (const float *)(ws + w.dq),
                                                                  (const float *)(ws + w.dk), (const float *)(ws + w.da),
                                                                  (const float *)(ws + w.db), (const float *)(ws + w.dl));
    }
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

}  // namespace qd

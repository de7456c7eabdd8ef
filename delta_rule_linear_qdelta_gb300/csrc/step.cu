// Decode steps: one token of the gated Q-Delta recurrence, or of QED, per
// (sequence, head), state updated in place.  Memory bound: the fp32 state is read once and
// written once; everything else is a few hundred bytes per head.
//
// Per state row s (length dk), with x = k + lambda q and kq = k . q
// ("Q-Delta: Beyond Key-Value Associative State Evolution", Sec. 3.3.1 Eq. 19 and
// the single-pass output form derived in the notes' Sec. 2.4):
//   p = s . x,  r = s . q,  e = v_row - alpha p
//   s' = alpha s + beta e k,  o_row = alpha r + beta e kq
//
// Layout: a group of LANES lanes owns one row, VEC consecutive floats per lane
// (a 16-byte access for dk = 128), so a warp's access to a row is one fully
// coalesced 512-byte line.  Each warp keeps UNROLL rows in flight.  One CTA of
// 4 warps per (sequence, head).
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kStepThreads = 128;
constexpr int kUnroll = 4;

template <int VEC> struct Vec;
template <> struct Vec<1> { using T = float; };
template <> struct Vec<2> { using T = float2; };
template <> struct Vec<4> { using T = float4; };

template <int VEC> __device__ __forceinline__ void vload(const float *p, float (&r)[VEC]) {
    typename Vec<VEC>::T x = *reinterpret_cast<const typename Vec<VEC>::T *>(p);
    const float *f = reinterpret_cast<const float *>(&x);
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e] = f[e];
}
template <int VEC> __device__ __forceinline__ void vstore(float *p, const float (&r)[VEC]) {
    typename Vec<VEC>::T x;
    float *f = reinterpret_cast<float *>(&x);
#pragma unroll
    for (int e = 0; e < VEC; ++e) f[e] = r[e];
    *reinterpret_cast<typename Vec<VEC>::T *>(p) = x;
}

template <int LANES> __device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LANES / 2; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off, LANES);
    return x;
}

template <typename TIn, int DK>
__global__ void __launch_bounds__(kStepThreads) qdelta_step_kernel(StepArgs a) {
    constexpr int VEC = DK >= 128 ? 4 : (DK >= 64 ? 2 : 1);
    constexpr int LANES = DK / VEC;             // 32, or 16 when dk = 16
    constexpr int RPW = 32 / LANES;             // rows per warp per pass
    constexpr int NW = kStepThreads / 32;
    const int head = blockIdx.x;                // n * H + h
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LANES, l = lane % LANES;
    const int dv = a.dv;

    const TIn *q = (const TIn *)a.q + (size_t)head * DK;
    const TIn *k = (const TIn *)a.k + (size_t)head * DK;
    const TIn *v = (const TIn *)a.v + (size_t)head * dv;
    float alpha = a.alpha ? to_f(((const TIn *)a.alpha)[head]) : 1.f;
    float beta = to_f(((const TIn *)a.beta)[head]);
    float lam = a.lam ? to_f(((const TIn *)a.lam)[head]) : 0.f;
    TIn *o = (TIn *)a.o + (size_t)head * dv;
    float *S = a.S + (size_t)head * dv * DK;

    float qv[VEC], kv[VEC], xv[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        qv[e] = to_f(q[l * VEC + e]);
        kv[e] = to_f(k[l * VEC + e]);
    }
    if (a.prologue) {                           // the feature map and gates from projections/logits
        if (a.alpha) alpha = expf(neg_softplus(alpha));
        beta = sigmoid_acc(beta);
        if (a.lam) lam = sigmoid_acc(lam);
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            qv[e] = silu_acc(qv[e]);
            kv[e] = silu_acc(kv[e]);
            sq = fmaf(qv[e], qv[e], sq);
            sk = fmaf(kv[e], kv[e], sk);
        }
        sq = group_sum<LANES>(sq);
        sk = group_sum<LANES>(sk);
        const float iq = sq > 0.f ? 1.f / sqrtf(sq) : 1.f, ik = sk > 0.f ? 1.f / sqrtf(sk) : 1.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            qv[e] *= iq;
            kv[e] *= ik;
        }
    }
    float kq = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        xv[e] = kv[e] + lam * qv[e];
        kq = fmaf(kv[e], qv[e], kq);
    }
    kq = group_sum<LANES>(kq);

    const int row_step = NW * RPW;              // rows covered by one pass of the CTA
    for (int base = warp * RPW; base < dv; base += row_step * kUnroll) {   // warp-uniform
        const int r0 = base + sub;
        float s[kUnroll][VEC] = {};
        float vr[kUnroll] = {};
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int row = r0 + u * row_step;
            if (row < dv) {
                vload<VEC>(S + (size_t)row * DK + l * VEC, s[u]);
                vr[u] = to_f(v[row]);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int row = r0 + u * row_step;
            float p = 0.f, r = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                p = fmaf(s[u][e], xv[e], p);
                r = fmaf(s[u][e], qv[e], r);
            }
            p = group_sum<LANES>(p);
            r = group_sum<LANES>(r);
            if (row < dv) {
                const float err = vr[u] - alpha * p;
                const float be = beta * err;
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[u][e] = fmaf(alpha, s[u][e], be * kv[e]);
                vstore<VEC>(S + (size_t)row * DK + l * VEC, s[u]);
                if (l == 0) o[row] = from_f<TIn>(fmaf(alpha, r, be * kq));
            }
        }
    }
}

// QED decode step ("The Query Knows What to Forget", Eqs. 4/6/8), state S^ = S^T
// ([dv][dk]) in place.  With eg = e^{g}, the erase vector a (or an ablation arm's),
// ea = eg*a, eq = eg*q and kq = k . q, per state row s (a d_v index i):
//   p = s . ea,  sq = s . eq,  r = w_i v_i - p
//   s' = eg*s + r k,  o_i = sq + r kq            (o = S^_new q in one pass)
// Same layout and row pipelining as the Q-Delta step above.
template <typename TIn, int DK>
__global__ void __launch_bounds__(kStepThreads) qed_step_kernel(QedStepArgs a) {
    constexpr int VEC = DK >= 128 ? 4 : (DK >= 64 ? 2 : 1);
    constexpr int LANES = DK / VEC;
    constexpr int RPW = 32 / LANES;
    constexpr int NW = kStepThreads / 32;
    const int head = blockIdx.x;                // n * H + h
    const int h = head % a.H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LANES, l = lane % LANES;
    const int dv = a.dv;

    const TIn *q = (const TIn *)a.q + (size_t)head * DK;
    const TIn *k = (const TIn *)a.k + (size_t)head * DK;
    const TIn *g = (const TIn *)a.g + (size_t)head * DK;
    const TIn *bg = (const TIn *)a.b + (size_t)head * DK;
    const TIn *v = (const TIn *)a.v + (size_t)head * dv;
    const TIn *w = (const TIn *)a.w + (size_t)head * dv;
    const float lam_h = a.lam_h[h];
    const bool gate = a.variant == kQedFull || a.variant == kQedRand;
    const bool proj = a.variant != kQedNogateNoproj;
    const float *zh = a.variant == kQedRand ? a.z + (size_t)h * DK : nullptr;
    TIn *o = (TIn *)a.o + (size_t)head * dv;
    float *S = a.S + (size_t)head * dv * DK;

    float qv[VEC], kv[VEC], bv[VEC], eg[VEC], u[VEC];
    float kq = 0.f, ku = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const int j = l * VEC + e;
        qv[e] = to_f(q[j]);
        kv[e] = to_f(k[j]);
        bv[e] = to_f(bg[j]);
        eg[e] = __expf(to_f(g[j]));
        const float x = zh ? zh[j] : qv[e];
        u[e] = gate ? bv[e] * x : x;
        kq = fmaf(kv[e], qv[e], kq);
        ku = fmaf(kv[e], u[e], ku);
    }
    kq = group_sum<LANES>(kq);
    ku = proj ? group_sum<LANES>(ku) : 0.f;
    float ea[VEC], eq[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        ea[e] = eg[e] * (bv[e] * kv[e] + lam_h * (u[e] - kv[e] * ku));
        eq[e] = eg[e] * qv[e];
    }

    const int row_step = NW * RPW;
    for (int base = warp * RPW; base < dv; base += row_step * kUnroll) {   // warp-uniform
        const int r0 = base + sub;
        float s[kUnroll][VEC] = {};
        float wv[kUnroll] = {};
#pragma unroll
        for (int uu = 0; uu < kUnroll; ++uu) {
            const int row = r0 + uu * row_step;
            if (row < dv) {
                vload<VEC>(S + (size_t)row * DK + l * VEC, s[uu]);
                wv[uu] = to_f(w[row]) * to_f(v[row]);
            }
        }
#pragma unroll
        for (int uu = 0; uu < kUnroll; ++uu) {
            const int row = r0 + uu * row_step;
            float p = 0.f, sq = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                p = fmaf(s[uu][e], ea[e], p);
                sq = fmaf(s[uu][e], eq[e], sq);
            }
            p = group_sum<LANES>(p);
            sq = group_sum<LANES>(sq);
            if (row < dv) {
                const float r = wv[uu] - p;
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[uu][e] = fmaf(eg[e], s[uu][e], r * kv[e]);
                vstore<VEC>(S + (size_t)row * DK + l * VEC, s[uu]);
                if (l == 0) o[row] = from_f<TIn>(fmaf(r, kq, sq));
            }
        }
    }
}

template <typename TIn>
cudaError_t run_qed_step(const QedStepArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)((size_t)a.N * a.H);
    switch (a.dk) {
        case 16: qed_step_kernel<TIn, 16><<<grid, kStepThreads, 0, s>>>(a); break;
        case 32: qed_step_kernel<TIn, 32><<<grid, kStepThreads, 0, s>>>(a); break;
        case 64: qed_step_kernel<TIn, 64><<<grid, kStepThreads, 0, s>>>(a); break;
        case 128: qed_step_kernel<TIn, 128><<<grid, kStepThreads, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t run_step(const StepArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)((size_t)a.N * a.H);
    switch (a.dk) {
        case 16: qdelta_step_kernel<TIn, 16><<<grid, kStepThreads, 0, s>>>(a); break;
        case 32: qdelta_step_kernel<TIn, 32><<<grid, kStepThreads, 0, s>>>(a); break;
        case 64: qdelta_step_kernel<TIn, 64><<<grid, kStepThreads, 0, s>>>(a); break;
        case 128: qdelta_step_kernel<TIn, 128><<<grid, kStepThreads, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qed_step(const QedStepArgs &a, int dtype, cudaStream_t s, int *nlaunch) {
    cudaError_t e = dtype == kBF16 ? run_qed_step<__nv_bfloat16>(a, s) : run_qed_step<float>(a, s);
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

cudaError_t launch_qdelta_step(const StepArgs &a, int dtype, cudaStream_t s, int *nlaunch) {
    cudaError_t e = dtype == kBF16 ? run_step<__nv_bfloat16>(a, s) : run_step<float>(a, s);
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

}  // namespace qd

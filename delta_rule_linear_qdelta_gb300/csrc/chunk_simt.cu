// Chunked forward on CUDA cores in fp32 (SIMT): the fp32 path of qdelta_fwd and
// qed_fwd, and the path for head dims the tensor-core kernel does not take.
//
// One CTA per (b, h, d_v tile of DVT columns) walks the chunks of its sequence in
// order, holding its DVT x dk slice of the state in shared memory (fp32) for the
// whole sequence.  Every matrix lives in shared memory with an odd row stride so
// that row walks by consecutive threads are bank-conflict free.
//
// Q-Delta per chunk ("Q-Delta: Beyond Key-Value Associative State Evolution",
// Sec. 3.3.2, Eqs. 20-27, with the corrected transposes and gamma_r/gamma_i decay;
// the notes' two UT solves folded into one, since
// (I + L_gamma)^{-1} = D_gamma (I + L)^{-1} D_gamma^{-1}):
//   l_i = sum_{j<=i} log alpha_j,  X = K + diag(lambda) Q,  H_ij = exp(l_i - l_j) (j <= i)
//   A = strictly_lower(diag(beta)(H * X K^T))
//   (I + A) Z = diag(beta) V - diag(beta gamma) X S^T          forward substitution
//   O = diag(gamma) Q S^T + (H * Q K^T) Z                       (H includes the diagonal)
//   S <- gamma_C S + Z^T diag(exp(l_C - l_i)) K
// QED per chunk ("The Query Knows What to Forget", Eq. 6 and the GDN-2 update of
// Eqs. 4/8), state held as S^ = S^T (V x K), G_i = sum_{j<=i} g_j per key channel:
//   a_i = b_i*k_i + lam_h (u_i - k_i (k_i^T u_i)),  u_i = b_i*q_i
//   At_ti = sum_c a_tc k_ic exp(G_tc - G_ic)  (i < t);  P_ti = same with q_t (i <= t)
//   (I + At) Z = W*V - (A*e^G) S^^T;  O = (Q*e^G) S^^T + P Z
//   S^ <- S^ diag(e^{G_C}) + Z^T (K*e^{G_C - G})
// Here the decay inside the Grams is applied per term as exp(G_t - G_i) <= 1, so
// this path is exact for any g <= 0.
//
// A ragged last chunk is padded with alpha = 1, beta = 0, b = 0, g = 0 and zero
// tokens, which leaves state and outputs of the valid rows unchanged.
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kC = 64;      // chunk length
constexpr int kNT = 256;    // threads per CTA

__device__ __forceinline__ void chunk_log_prefix(float *ell) {
    // inclusive prefix sum of ell[0..63] by warp 0 (two values per lane)
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        float a = ell[2 * l], b = ell[2 * l + 1];
        float s = a + b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            float n = __shfl_up_sync(0xffffffffu, s, off);
            if (l >= off) s += n;
        }
        const float excl = s - (a + b);
        ell[2 * l] = excl + a;
        ell[2 * l + 1] = s;
    }
}

template <int DVT>
__device__ __forceinline__ void forward_substitute(const float *Am, float *Zs) {
    // (I + A) Z = R in place (Zs holds R), A strictly lower [C][C+1]; one thread per column
    constexpr int LC = kC + 1, LV = DVT + 1;
    if (threadIdx.x < DVT) {
        const int d = threadIdx.x;
        for (int i = 1; i < kC; ++i) {
            float acc = Zs[i * LV + d];
            const float *Ai = Am + i * LC;
            for (int m = 0; m < i; ++m) acc -= Ai[m] * Zs[m * LV + d];
            Zs[i * LV + d] = acc;
        }
    }
}

template <typename TIn, int DK, int DVT>
__global__ void __launch_bounds__(kNT) qdelta_chunk_simt_kernel(QDeltaArgs a) {
    constexpr int C = kC, LK = DK + 1, LV = DVT + 1, LC = C + 1;
    extern __shared__ float sm[];
    float *Qs = sm;                 // [C][LK]
    float *Ks = Qs + C * LK;        // [C][LK]
    float *Xs = Ks + C * LK;        // [C][LK]
    float *Ss = Xs + C * LK;        // [DVT][LK]  state rows d0 .. d0+DVT-1
    float *Zs = Ss + DVT * LK;      // [C][LV]    V -> R -> Z -> Z*exp(l_C - l_i)
    float *Ws = Zs + C * LV;        // [C][LV]    gamma Q S^T
    float *Am = Ws + C * LV;        // [C][LC]
    float *Pm = Am + C * LC;        // [C][LC]
    float *ell = Pm + C * LC;       // [C]
    float *bet = ell + C;           // [C]
    float *lmb = bet + C;           // [C]

    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v;
    const TIn *alpha = (const TIn *)a.alpha, *beta = (const TIn *)a.beta, *lam = (const TIn *)a.lam;
    TIn *o = (TIn *)a.o;
    const int T = a.T, H = a.H, dv = a.dv;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int d0 = blockIdx.y * DVT;
    const int tid = threadIdx.x;
    const size_t s_base = (size_t)bh * dv * DK + (size_t)d0 * DK;

    for (int idx = tid; idx < DVT * DK; idx += kNT) {
        const int d = idx / DK, j = idx % DK;
        Ss[d * LK + j] = a.S0 ? a.S0[s_base + (size_t)d * DK + j] : 0.f;
    }

    const int nchunk = (T + C - 1) / C;
    for (int c0 = 0; c0 < T; c0 += C) {
        const int n = min(C, T - c0);
        __syncthreads();
        if (a.S_chk) {                                    // checkpoint: the state entering this chunk
            float *chk = a.S_chk + ((size_t)bh * nchunk + c0 / C) * dv * DK + (size_t)d0 * DK;
            for (int idx = tid; idx < DVT * DK; idx += kNT) chk[idx] = Ss[(idx / DK) * LK + idx % DK];
        }
        for (int idx = tid; idx < C * DK; idx += kNT) {
            const int t = idx / DK, j = idx % DK;
            const size_t tok = ((size_t)b * T + c0 + t) * H + h;
            const bool ok = t < n;
            Qs[t * LK + j] = ok ? to_f(q[tok * DK + j]) : 0.f;
            Ks[t * LK + j] = ok ? to_f(k[tok * DK + j]) : 0.f;
        }
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int t = idx / DVT, d = idx % DVT;
            const size_t tok = ((size_t)b * T + c0 + t) * H + h;
            Zs[t * LV + d] = t < n ? to_f(v[tok * dv + d0 + d]) : 0.f;
        }
        if (tid < C) {
            const int t = tid;
            const size_t tok = ((size_t)b * T + c0 + t) * H + h;
            const bool ok = t < n;
            if (a.prologue) {                             // gates from their logits
                ell[t] = (ok && alpha) ? neg_softplus(to_f(alpha[tok])) : 0.f;
                bet[t] = ok ? sigmoid_acc(to_f(beta[tok])) : 0.f;
                lmb[t] = (ok && lam) ? sigmoid_acc(to_f(lam[tok])) : 0.f;
            } else {
                ell[t] = (ok && alpha) ? logf(to_f(alpha[tok])) : 0.f;
                bet[t] = ok ? to_f(beta[tok]) : 0.f;
                lmb[t] = (ok && lam) ? to_f(lam[tok]) : 0.f;
            }
        }
        __syncthreads();
        if (a.prologue) {                                 // q, k = SiLU(x)/|SiLU(x)|, a warp per row
            const int lane = tid & 31, warp = tid >> 5;
            for (int r = warp; r < 2 * C; r += kNT / 32) {
                float *row = (r < C ? Qs : Ks) + (r % C) * LK;
                float ss = 0.f;
                for (int j = lane; j < DK; j += 32) {
                    const float y = silu_acc(row[j]);
                    row[j] = y;
                    ss = fmaf(y, y, ss);
                }
#pragma unroll
                for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = ss > 0.f ? 1.f / sqrtf(ss) : 1.f;   // padding rows stay zero
                for (int j = lane; j < DK; j += 32) row[j] *= inv;
            }
            __syncthreads();
        }
        chunk_log_prefix(ell);
        for (int idx = tid; idx < C * DK; idx += kNT) {
            const int t = idx / DK, j = idx % DK;
            Xs[t * LK + j] = Ks[t * LK + j] + lmb[t] * Qs[t * LK + j];
        }
        __syncthreads();
        // Grams with decay and masks
        for (int idx = tid; idx < C * C; idx += kNT) {
            const int t = idx / C, i = idx % C;
            float am = 0.f, pm = 0.f;
            if (i <= t) {
                const float *xt = Xs + t * LK, *qt = Qs + t * LK, *ki = Ks + i * LK;
                float gx = 0.f, gq = 0.f;
#pragma unroll 8
                for (int j = 0; j < DK; ++j) {
                    gx = fmaf(xt[j], ki[j], gx);
                    gq = fmaf(qt[j], ki[j], gq);
                }
                const float dec = expf(ell[t] - ell[i]);
                am = (i < t) ? bet[t] * dec * gx : 0.f;
                pm = dec * gq;
            }
            Am[t * LC + i] = am;
            Pm[t * LC + i] = pm;
        }
        // R = beta (V - gamma X S^T), W = gamma Q S^T
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int t = idx / DVT, d = idx % DVT;
            const float *xt = Xs + t * LK, *qt = Qs + t * LK, *sd = Ss + d * LK;
            float xs = 0.f, qs = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) {
                xs = fmaf(xt[j], sd[j], xs);
                qs = fmaf(qt[j], sd[j], qs);
            }
            const float gam = expf(ell[t]);
            Zs[t * LV + d] = bet[t] * (Zs[t * LV + d] - gam * xs);
            Ws[t * LV + d] = gam * qs;
        }
        __syncthreads();
        forward_substitute<DVT>(Am, Zs);
        __syncthreads();
        // O = gamma Q S^T + P Z  (skipped when only the states are wanted)
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int t = idx / DVT, d = idx % DVT;
            if (t < n && o) {
                float acc = Ws[t * LV + d];
                const float *pt = Pm + t * LC;
                for (int i = 0; i <= t; ++i) acc = fmaf(pt[i], Zs[i * LV + d], acc);
                const size_t tok = ((size_t)b * T + c0 + t) * H + h;
                o[tok * dv + d0 + d] = from_f<TIn>(acc);
            }
        }
        __syncthreads();
        const float lC = ell[C - 1];
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int i = idx / DVT, d = idx % DVT;
            Zs[i * LV + d] *= expf(lC - ell[i]);
        }
        __syncthreads();
        const float gC = expf(lC);
        for (int idx = tid; idx < DVT * DK; idx += kNT) {
            const int d = idx / DK, j = idx % DK;
            float acc = gC * Ss[d * LK + j];
#pragma unroll 8
            for (int i = 0; i < C; ++i) acc = fmaf(Zs[i * LV + d], Ks[i * LK + j], acc);
            Ss[d * LK + j] = acc;
        }
    }
    __syncthreads();
    if (a.S_final)
        for (int idx = tid; idx < DVT * DK; idx += kNT) {
            const int d = idx / DK, j = idx % DK;
            a.S_final[s_base + (size_t)d * DK + j] = Ss[d * LK + j];
        }
}

template <typename TIn, int DK, int DVT>
__global__ void __launch_bounds__(kNT) qed_chunk_simt_kernel(QedArgs a) {
    constexpr int C = kC, LK = DK + 1, LV = DVT + 1, LC = C + 1;
    extern __shared__ float sm[];
    float *Qs = sm;                 // [C][LK]  q -> q*e^G
    float *Ks = Qs + C * LK;        // [C][LK]  k -> k*e^{G_C - G}
    float *Gs = Ks + C * LK;        // [C][LK]  G (in-chunk cumulative log-decay)
    float *As = Gs + C * LK;        // [C][LK]  b -> a -> a*e^G
    float *Ss = As + C * LK;        // [DVT][LK]
    float *Zs = Ss + DVT * LK;      // [C][LV]  w*v -> R -> Z
    float *Ws = Zs + C * LV;        // [C][LV]  (q*e^G) S^^T
    float *Am = Ws + C * LV;        // [C][LC]
    float *Pm = Am + C * LC;        // [C][LC]

    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v;
    const TIn *g = (const TIn *)a.g, *bg = (const TIn *)a.b, *w = (const TIn *)a.w;
    TIn *o = (TIn *)a.o;
    const int T = a.T, H = a.H, dv = a.dv;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int d0 = blockIdx.y * DVT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float lam_h = a.lam_h[h];
    const size_t s_base = (size_t)bh * dv * DK + (size_t)d0 * DK;
    const bool gate = a.variant == kQedFull || a.variant == kQedRand;   // the new term keeps b
    const bool proj = a.variant != kQedNogateNoproj;                    // ... and the projection
    const float *zh = a.variant == kQedRand ? a.z + (size_t)h * DK : nullptr;

    for (int idx = tid; idx < DVT * DK; idx += kNT) {
        const int d = idx / DK, j = idx % DK;
        Ss[d * LK + j] = a.S0 ? a.S0[s_base + (size_t)d * DK + j] : 0.f;
    }

    for (int c0 = 0; c0 < T; c0 += C) {
        const int n = min(C, T - c0);
        __syncthreads();
        for (int idx = tid; idx < C * DK; idx += kNT) {
            const int t = idx / DK, j = idx % DK;
            const size_t e = (((size_t)b * T + c0 + t) * H + h) * DK + j;
            const bool ok = t < n;
            Qs[t * LK + j] = ok ? to_f(q[e]) : 0.f;
            Ks[t * LK + j] = ok ? to_f(k[e]) : 0.f;
            Gs[t * LK + j] = ok ? to_f(g[e]) : 0.f;
            As[t * LK + j] = ok ? to_f(bg[e]) : 0.f;
        }
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int t = idx / DVT, d = idx % DVT;
            const size_t e = (((size_t)b * T + c0 + t) * H + h) * (size_t)dv + d0 + d;
            Zs[t * LV + d] = t < n ? to_f(w[e]) * to_f(v[e]) : 0.f;
        }
        __syncthreads();
        if (tid < DK)
            for (int t = 1; t < C; ++t) Gs[t * LK + tid] += Gs[(t - 1) * LK + tid];
        // erase vector a_t = b*k + lam_h P(u) (full: u = b*q), one warp per token; the
        // ablation arms take u = q (nogate), u = q without P (nogate-noproj), u = b*z_h (rand)
        for (int t = warp; t < C; t += kNT / 32) {
            auto u_of = [&](int j) {
                const float x = zh ? zh[j] : Qs[t * LK + j];
                return gate ? As[t * LK + j] * x : x;
            };
            float ku = 0.f;
            if (proj) {
                for (int j = lane; j < DK; j += 32) ku += Ks[t * LK + j] * u_of(j);
#pragma unroll
                for (int off = 16; off; off >>= 1) ku += __shfl_xor_sync(0xffffffffu, ku, off);
            }
            for (int j = lane; j < DK; j += 32) {
                const float bj = As[t * LK + j], kj = Ks[t * LK + j];
                const float u = u_of(j);
                As[t * LK + j] = bj * kj + lam_h * (u - kj * ku);
            }
        }
        __syncthreads();
        for (int idx = tid; idx < C * C; idx += kNT) {
            const int t = idx / C, i = idx % C;
            float am = 0.f, pm = 0.f;
            if (i <= t) {
                const float *at = As + t * LK, *qt = Qs + t * LK, *ki = Ks + i * LK;
                const float *gt = Gs + t * LK, *gi = Gs + i * LK;
                for (int j = 0; j < DK; ++j) {
                    const float kd = ki[j] * expf(gt[j] - gi[j]);
                    am = fmaf(at[j], kd, am);
                    pm = fmaf(qt[j], kd, pm);
                }
                if (i == t) am = 0.f;
            }
            Am[t * LC + i] = am;
            Pm[t * LC + i] = pm;
        }
        __syncthreads();
        for (int idx = tid; idx < C * DK; idx += kNT) {
            const int t = idx / DK, j = idx % DK;
            const float G = Gs[t * LK + j];
            const float eg = expf(G);
            Qs[t * LK + j] *= eg;
            As[t * LK + j] *= eg;
            Ks[t * LK + j] *= expf(Gs[(C - 1) * LK + j] - G);
        }
        __syncthreads();
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int t = idx / DVT, d = idx % DVT;
            const float *at = As + t * LK, *qt = Qs + t * LK, *sd = Ss + d * LK;
            float as = 0.f, qs = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) {
                as = fmaf(at[j], sd[j], as);
                qs = fmaf(qt[j], sd[j], qs);
            }
            Zs[t * LV + d] -= as;
            Ws[t * LV + d] = qs;
        }
        __syncthreads();
        forward_substitute<DVT>(Am, Zs);
        __syncthreads();
        for (int idx = tid; idx < C * DVT; idx += kNT) {
            const int t = idx / DVT, d = idx % DVT;
            if (t < n) {
                float acc = Ws[t * LV + d];
                const float *pt = Pm + t * LC;
                for (int i = 0; i <= t; ++i) acc = fmaf(pt[i], Zs[i * LV + d], acc);
                const size_t e = (((size_t)b * T + c0 + t) * H + h) * (size_t)dv + d0 + d;
                o[e] = from_f<TIn>(acc);
            }
        }
        for (int idx = tid; idx < DVT * DK; idx += kNT) {
            const int d = idx / DK, j = idx % DK;
            float acc = expf(Gs[(C - 1) * LK + j]) * Ss[d * LK + j];
#pragma unroll 8
            for (int i = 0; i < C; ++i) acc = fmaf(Zs[i * LV + d], Ks[i * LK + j], acc);
            Ss[d * LK + j] = acc;
        }
    }
    __syncthreads();
    if (a.S_final)
        for (int idx = tid; idx < DVT * DK; idx += kNT) {
            const int d = idx / DK, j = idx % DK;
            a.S_final[s_base + (size_t)d * DK + j] = Ss[d * LK + j];
        }
}

template <int DK, int DVT>
constexpr size_t qdelta_smem() {
    return sizeof(float) * (3 * kC * (DK + 1) + DVT * (DK + 1) + 2 * kC * (DVT + 1) +
                            2 * kC * (kC + 1) + 3 * kC);
}
template <int DK, int DVT>
constexpr size_t qed_smem() {
    return sizeof(float) * (4 * kC * (DK + 1) + DVT * (DK + 1) + 2 * kC * (DVT + 1) +
                            2 * kC * (kC + 1));
}

template <typename TIn, int DK, int DVT>
cudaError_t run_qdelta(const QDeltaArgs &a, cudaStream_t s) {
    auto kern = qdelta_chunk_simt_kernel<TIn, DK, DVT>;
    constexpr size_t smem = qdelta_smem<DK, DVT>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, a.dv / DVT);
    kern<<<grid, kNT, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename TIn, int DK, int DVT>
cudaError_t run_qed(const QedArgs &a, cudaStream_t s) {
    auto kern = qed_chunk_simt_kernel<TIn, DK, DVT>;
    constexpr size_t smem = qed_smem<DK, DVT>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, a.dv / DVT);
    kern<<<grid, kNT, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_qdelta(const QDeltaArgs &a, cudaStream_t s) {
    const bool wide = a.dv >= 32;
    switch (a.dk) {
        case 16: return wide ? run_qdelta<TIn, 16, 32>(a, s) : run_qdelta<TIn, 16, 16>(a, s);
        case 32: return wide ? run_qdelta<TIn, 32, 32>(a, s) : run_qdelta<TIn, 32, 16>(a, s);
        case 64: return wide ? run_qdelta<TIn, 64, 32>(a, s) : run_qdelta<TIn, 64, 16>(a, s);
        case 128: return wide ? run_qdelta<TIn, 128, 32>(a, s) : run_qdelta<TIn, 128, 16>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <typename TIn>
cudaError_t dispatch_qed(const QedArgs &a, cudaStream_t s) {
    const bool wide = a.dv >= 32;
    switch (a.dk) {
        case 16: return wide ? run_qed<TIn, 16, 32>(a, s) : run_qed<TIn, 16, 16>(a, s);
        case 32: return wide ? run_qed<TIn, 32, 32>(a, s) : run_qed<TIn, 32, 16>(a, s);
        case 64: return wide ? run_qed<TIn, 64, 32>(a, s) : run_qed<TIn, 64, 16>(a, s);
        case 128: return wide ? run_qed<TIn, 128, 32>(a, s) : run_qed<TIn, 128, 16>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_qdelta_chunk_simt(const QDeltaArgs &a, int dtype, cudaStream_t s, int *nlaunch) {
    cudaError_t e = dtype == kBF16 ? dispatch_qdelta<__nv_bfloat16>(a, s) : dispatch_qdelta<float>(a, s);
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

cudaError_t launch_qed_chunk_simt(const QedArgs &a, int dtype, cudaStream_t s, int *nlaunch) {
    cudaError_t e = dtype == kBF16 ? dispatch_qed<__nv_bfloat16>(a, s) : dispatch_qed<float>(a, s);
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

}  // namespace qd

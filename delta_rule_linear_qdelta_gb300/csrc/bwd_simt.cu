// Backward of the chunked Q-Delta forward on CUDA cores (fp32 arithmetic).
//
// The gradients are those of L = sum_t <dO_t, o_t> + <dS_final, S_T> with respect to
// q, k, v, alpha, beta, lambda and S0: the adjoint of the chunked form of the gated
// recurrence ("Q-Delta: Beyond Key-Value Associative State Evolution", Sec. 3.3.2,
// with the corrected transposes and decay; the single solve
// (I + L_gamma)^{-1} = D_gamma (I + L)^{-1} D_gamma^{-1}).  Per chunk of C = 64 tokens,
// l_i = sum_{j<=i} log alpha_j, gamma_i = e^{l_i}, w_i = e^{l_C - l_i}, X = K + diag(lambda) Q,
// H_ij = e^{l_i - l_j} (j <= i), P = H * Q K^T, M = strictly_lower(H * X K^T),
// T = (I + diag(beta) M)^{-1}, XS = diag(gamma) X S_in^T, QS = diag(gamma) Q S_in^T,
// Z = T diag(beta) (V - XS), the forward is O = QS + P Z, S_out = gamma_C S_in + Z^T diag(w) K,
// and its adjoint, given dO and dS_out:
//   dZ = P^T dO + diag(w) K dS_out^T      dR = T^T dZ          dXS = -diag(beta) dR
//   dA = -strictly_lower(dR Z^T)           dM = diag(beta) dA    dP = lower(dO Z^T)
//   dS_in = gamma_C dS_out + (gamma dO)^T Q + (gamma dXS)^T X
//   dX = (gamma dXS) S_in + (H * dM) K
//   dQ = (gamma dO) S_in + (H * dP) K + diag(lambda) dX
//   dK = (H * dP)^T Q + (H * dM)^T X + diag(w) Z dS_out + dX
//   dV = diag(beta) dR,  dbeta = rowsum(dA * M) + rowsum(dR * (V - XS)),  dlambda = rowsum(dX * Q)
//   dl = rowsum(dO * QS) + rowsum(dXS * XS) + rowsum(E) - colsum(E) - wz,
//        E = dP * P + dM * M,  wz_i = w_i (Z dS_out)_i . K_i,
//        plus gamma_C <dS_out, S_in> + sum_i wz_i on the chunk's last token,
//   d log alpha = reverse cumulative sum of dl within the chunk, dalpha = d log alpha / alpha.
//
// Three launches:
//   1. the chunk forward without its output, storing the state entering each chunk
//      (S_chk): the tcgen05 kernel for bf16 at d = 128, else the fp32 CUDA-core one;
//   2. the reverse sweep of dS over the chunks (qdelta_bwd_dstate_kernel here, one CTA
//      per (b, h, d_v tile), since rows of dS evolve independently as rows of S do; the
//      tcgen05 sweep of bwd_tc.cu for bf16 at d = 128), storing the
//      gradient reaching the state leaving each chunk (dS_chk) and dS0.  It needs no
//      forward state: dS_in depends only on dS_out, dO, q, k and the gates;
//   3. qdelta_bwd_grad_kernel (or its tcgen05 version in bwd_grad_tc.cu for bf16
//      at d = 128): every input gradient, one CTA per (b, h, chunk), all chunks in
//      parallel, from the two checkpoints of its chunk.
// A ragged last chunk is padded with alpha = 1, beta = 0, lambda = 0 and zero tokens and
// zero dO, which adds nothing to any gradient of a valid token.
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kC = 64;       // chunk length (checkpoint spacing)
constexpr int kNTs = 256;    // threads of the reverse sweep
constexpr int kNTg = 512;    // threads of the gradient kernel
constexpr int kDVS = 16;     // d_v columns per pass of the gradient kernel

// inclusive prefix sum of x[0..63] by warp 0 (two values per lane)
__device__ __forceinline__ void prefix64(float *x) {
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        const float a = x[2 * l], b = x[2 * l + 1];
        float s = a + b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, s, off);
            if (l >= off) s += n;
        }
        x[2 * l] = s - b;
        x[2 * l + 1] = s;
    }
}

// reverse (suffix) cumulative sum of x[0..63] by warp 0
__device__ __forceinline__ void suffix64(float *x) {
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        const float a = x[2 * l], b = x[2 * l + 1];
        float s = a + b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float n = __shfl_down_sync(0xffffffffu, s, off);
            if (l + off < 32) s += n;
        }
        x[2 * l] = s;
        x[2 * l + 1] = s - a;
    }
}

// Gates of tokens c0 .. c0+63 of stream (b, h) by threads 0..63: log alpha, beta,
// lambda, with the padding of a ragged chunk.
template <typename TIn>
__device__ __forceinline__ void load_gates(const QDeltaBwdArgs &a, int b, int h, int c0, int n, float *la,
                                           float *bet, float *lmb) {
    if (threadIdx.x < kC) {
        const int t = threadIdx.x;
        const bool ok = t < n;
        const size_t tok = ((size_t)b * a.T + c0 + (ok ? t : 0)) * a.H + h;
        la[t] = (ok && a.alpha) ? logf(gate_val<TIn>(a.alpha, tok, a.gates_f32)) : 0.f;
        bet[t] = ok ? gate_val<TIn>(a.beta, tok, a.gates_f32) : 0.f;
        lmb[t] = (ok && a.lam) ? gate_val<TIn>(a.lam, tok, a.gates_f32) : 0.f;
    }
}

// Reverse sweep: dS over the chunks of one (b, h), rows d0 .. d0+DVT-1 of dS.
template <typename TIn, int DK, int DVT>
__global__ void __launch_bounds__(kNTs) qdelta_bwd_dstate_kernel(QDeltaBwdArgs a) {
    constexpr int C = kC, LK = DK + 1, LV = DVT + 1, LC = C + 1;
    extern __shared__ float sm[];
    float *Qs = sm;                 // [C][LK]
    float *Ks = Qs + C * LK;        // [C][LK]
    float *Xs = Ks + C * LK;        // [C][LK]
    float *dSs = Xs + C * LK;       // [DVT][LK]   dS rows d0 ..
    float *dOt = dSs + DVT * LK;    // [C][LV]
    float *dZt = dOt + C * LV;      // [C][LV]     dZ -> dR
    float *Am = dZt + C * LV;       // [C][LC]     diag(beta) M
    float *Pm = Am + C * LC;        // [C][LC]
    float *ell = Pm + C * LC;       // [C]
    float *bet = ell + C;
    float *lmb = bet + C;
    float *gam = lmb + C;

    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *dO = (const TIn *)a.dO;
    const int T = a.T, H = a.H, dv = a.nv, nchunk = (T + C - 1) / C;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int d0 = blockIdx.y * DVT;
    const int tid = threadIdx.x;
    const size_t s_base = (size_t)bh * dv * DK + (size_t)d0 * DK;

    for (int idx = tid; idx < DVT * DK; idx += kNTs)
        dSs[(idx / DK) * LK + idx % DK] = a.dS_final ? a.dS_final[s_base + idx] : 0.f;

    for (int c = nchunk - 1; c >= 0; --c) {
        const int c0 = c * C, n = min(C, T - c0);
        __syncthreads();
        float *chk = a.dS_chk + ((size_t)bh * nchunk + c) * dv * DK + (size_t)d0 * DK;
        for (int idx = tid; idx < DVT * DK; idx += kNTs) chk[idx] = dSs[(idx / DK) * LK + idx % DK];
        for (int idx = tid; idx < C * DK; idx += kNTs) {
            const int t = idx / DK, j = idx % DK;
            const size_t tok = ((size_t)b * T + c0 + t) * H + h;
            const bool ok = t < n;
            Qs[t * LK + j] = ok ? to_f(q[tok * DK + j]) : 0.f;
            Ks[t * LK + j] = ok ? to_f(k[tok * DK + j]) : 0.f;
        }
        for (int idx = tid; idx < C * DVT; idx += kNTs) {
            const int t = idx / DVT, d = idx % DVT;
            const size_t tok = ((size_t)b * T + c0 + t) * H + h;
            dOt[t * LV + d] = t < n ? to_f(dO[tok * dv + d0 + d]) : 0.f;
        }
        load_gates<TIn>(a, b, h, c0, n, ell, bet, lmb);
        __syncthreads();
        prefix64(ell);
        for (int idx = tid; idx < C * DK; idx += kNTs) {
            const int t = idx / DK, j = idx % DK;
            Xs[t * LK + j] = Ks[t * LK + j] + lmb[t] * Qs[t * LK + j];
        }
        __syncthreads();
        if (tid < C) gam[tid] = expf(ell[tid]);
        for (int idx = tid; idx < C * C; idx += kNTs) {
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
                am = i < t ? bet[t] * dec * gx : 0.f;
                pm = dec * gq;
            }
            Am[t * LC + i] = am;
            Pm[t * LC + i] = pm;
        }
        // dZ, state part: diag(w) K dS^T
        const float lC = ell[C - 1];
        for (int idx = tid; idx < C * DVT; idx += kNTs) {
            const int t = idx / DVT, d = idx % DVT;
            const float *kt = Ks + t * LK, *sd = dSs + d * LK;
            float acc = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) acc = fmaf(kt[j], sd[j], acc);
            dZt[t * LV + d] = expf(lC - ell[t]) * acc;
        }
        __syncthreads();
        // dZ += P^T dO
        for (int idx = tid; idx < C * DVT; idx += kNTs) {
            const int t = idx / DVT, d = idx % DVT;
            float acc = dZt[t * LV + d];
            for (int i = t; i < C; ++i) acc = fmaf(Pm[i * LC + t], dOt[i * LV + d], acc);
            dZt[t * LV + d] = acc;
        }
        __syncthreads();
        // (I + A)^T dR = dZ by back substitution, one thread per column
        if (tid < DVT) {
            const int d = tid;
            for (int t = C - 2; t >= 0; --t) {
                float acc = dZt[t * LV + d];
                for (int i = t + 1; i < C; ++i) acc -= Am[i * LC + t] * dZt[i * LV + d];
                dZt[t * LV + d] = acc;
            }
        }
        __syncthreads();
        // dS <- gamma_C dS + (gamma dO)^T Q - (gamma beta dR)^T X
        const float gC = gam[C - 1];
        for (int idx = tid; idx < DVT * DK; idx += kNTs) {
            const int d = idx / DK, j = idx % DK;
            float acc = gC * dSs[d * LK + j];
#pragma unroll 8
            for (int t = 0; t < C; ++t) {
                const float g = gam[t];
                acc = fmaf(g * dOt[t * LV + d], Qs[t * LK + j], acc);
                acc = fmaf(-g * bet[t] * dZt[t * LV + d], Xs[t * LK + j], acc);
            }
            dSs[d * LK + j] = acc;
        }
    }
    __syncthreads();
    if (a.dS0)
        for (int idx = tid; idx < DVT * DK; idx += kNTs) a.dS0[s_base + idx] = dSs[(idx / DK) * LK + idx % DK];
}

// Every input gradient of chunk c of stream (b, h); blockIdx.x = bh * nchunk + c.
// Thread (r, jc) = (tid / 8, tid % 8) owns row r and columns jc + 8m of the n x dk
// results, accumulated in registers over the passes through d_v.
template <typename TIn, int DK>
__global__ void __launch_bounds__(kNTg) qdelta_bwd_grad_kernel(QDeltaBwdArgs a) {
    constexpr int C = kC, LK = DK + 1, DV = kDVS, LV = DV + 1, LC = C + 1, JN = DK / 8;
    static_assert(kNTg == 8 * C, "one row of 8 threads per token");
    extern __shared__ float sm[];
    float *Qs = sm;                 // [C][LK]
    float *Ks = Qs + C * LK;        // [C][LK]
    float *Pm = Ks + C * LK;        // [C][LC]  P               -> E
    float *Mm = Pm + C * LC;        // [C][LC]  M               -> dA * M
    float *Tm = Mm + C * LC;        // [C][LC]  (I + diag(beta) M)^{-1}
    float *dAm = Tm + C * LC;       // [C][LC]  sum dR Z^T      -> H * dM
    float *dPm = dAm + C * LC;      // [C][LC]  sum dO Z^T      -> H * dP
    float *Ss = dPm + C * LC;       // [DV][LK] S_in rows of this pass
    float *dSs = Ss + DV * LK;      // [DV][LK] dS_out rows of this pass
    float *Rt = dSs + DV * LK;      // [C][LV]  V -> V - XS
    float *dOt = Rt + C * LV;       // [C][LV]
    float *XSt = dOt + C * LV;      // [C][LV]
    float *QSt = XSt + C * LV;      // [C][LV]
    float *Zt = QSt + C * LV;       // [C][LV]
    float *dZt = Zt + C * LV;       // [C][LV]
    float *dRt = dZt + C * LV;      // [C][LV]
    float *ell = dRt + C * LV;      // [C] log alpha -> prefix l
    float *la = ell + C;            // [C] log alpha
    float *bet = la + C;
    float *lmb = bet + C;
    float *gam = lmb + C;
    float *wC = gam + C;
    float *sq = wC + C;             // rowsum(dO * QS)
    float *sx = sq + C;             // rowsum(dXS * XS)
    float *sb = sx + C;             // rowsum(dR * (V - XS))
    float *wz = sb + C;
    float *red = wz + C;            // [kNTg / 32]

    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v, *dO = (const TIn *)a.dO;
    const int T = a.T, H = a.H, dv = a.nv, nchunk = (T + C - 1) / C;
    const int c = blockIdx.x % nchunk, bh = blockIdx.x / nchunk, b = bh / H, h = bh % H;
    const int c0 = c * C, n = min(C, T - c0);
    const int tid = threadIdx.x, r = tid >> 3, jc = tid & 7;
    const size_t chk_base = ((size_t)bh * nchunk + c) * dv * DK;

    for (int idx = tid; idx < C * DK; idx += kNTg) {
        const int t = idx / DK, j = idx % DK;
        const size_t tok = ((size_t)b * T + c0 + t) * H + h;
        const bool ok = t < n;
        Qs[t * LK + j] = ok ? to_f(q[tok * DK + j]) : 0.f;
        Ks[t * LK + j] = ok ? to_f(k[tok * DK + j]) : 0.f;
    }
    load_gates<TIn>(a, b, h, c0, n, la, bet, lmb);
    if (tid < C) {
        sq[tid] = sx[tid] = sb[tid] = 0.f;
    }
    __syncthreads();
    if (tid < C) ell[tid] = la[tid];
    __syncthreads();
    prefix64(ell);
    __syncthreads();
    if (tid < C) {
        gam[tid] = expf(ell[tid]);
        wC[tid] = expf(ell[C - 1] - ell[tid]);
    }
    for (int idx = tid; idx < C * C; idx += kNTg) {
        const int t = idx / C, i = idx % C;
        float mm = 0.f, pm = 0.f;
        if (i <= t) {
            const float *qt = Qs + t * LK, *kt = Ks + t * LK, *ki = Ks + i * LK;
            const float lt = lmb[t];
            float gx = 0.f, gq = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) {
                gx = fmaf(fmaf(lt, qt[j], kt[j]), ki[j], gx);
                gq = fmaf(qt[j], ki[j], gq);
            }
            const float dec = expf(ell[t] - ell[i]);
            mm = i < t ? dec * gx : 0.f;
            pm = dec * gq;
        }
        Mm[t * LC + i] = mm;
        Pm[t * LC + i] = pm;
        dAm[t * LC + i] = bet[t] * mm;                    // A, scratch for the inverse
    }
    __syncthreads();
    // T = (I + A)^{-1}, one column per thread by forward substitution
    if (tid < C) {
        const int j = tid;
        for (int i = 0; i < C; ++i) {
            float acc = i == j ? 1.f : 0.f;
            if (i > j)
                for (int m = j; m < i; ++m) acc -= dAm[i * LC + m] * Tm[m * LC + j];
            Tm[i * LC + j] = acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += kNTg) dAm[(idx / C) * LC + idx % C] = dPm[(idx / C) * LC + idx % C] = 0.f;

    float accX[JN], accQ[JN], accK[JN];
#pragma unroll
    for (int m = 0; m < JN; ++m) accX[m] = accQ[m] = accK[m] = 0.f;
    float gS = 0.f;

    for (int e0 = 0; e0 < dv; e0 += DV) {
        __syncthreads();
        for (int idx = tid; idx < DV * DK; idx += kNTg) {
            const int d = idx / DK, j = idx % DK;
            const float s = a.S_chk[chk_base + (size_t)(e0 + d) * DK + j];
            const float g = a.dS_chk[chk_base + (size_t)(e0 + d) * DK + j];
            Ss[d * LK + j] = s;
            dSs[d * LK + j] = g;
            gS = fmaf(s, g, gS);
        }
        for (int idx = tid; idx < C * DV; idx += kNTg) {
            const int t = idx / DV, d = idx % DV;
            const size_t tok = ((size_t)b * T + c0 + t) * H + h;
            const bool ok = t < n;
            Rt[t * LV + d] = ok ? to_f(v[tok * dv + e0 + d]) : 0.f;
            dOt[t * LV + d] = ok ? to_f(dO[tok * dv + e0 + d]) : 0.f;
        }
        __syncthreads();
        // XS, QS, V - XS and the state part of dZ
        for (int idx = tid; idx < C * DV; idx += kNTg) {
            const int t = idx / DV, d = idx % DV;
            const float *qt = Qs + t * LK, *kt = Ks + t * LK, *sd = Ss + d * LK, *gd = dSs + d * LK;
            const float lt = lmb[t];
            float xs = 0.f, qs = 0.f, kd = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) {
                xs = fmaf(fmaf(lt, qt[j], kt[j]), sd[j], xs);
                qs = fmaf(qt[j], sd[j], qs);
                kd = fmaf(kt[j], gd[j], kd);
            }
            XSt[t * LV + d] = gam[t] * xs;
            QSt[t * LV + d] = gam[t] * qs;
            Rt[t * LV + d] -= gam[t] * xs;
            dZt[t * LV + d] = wC[t] * kd;
        }
        __syncthreads();
        // Z = T diag(beta) (V - XS);  dZ += P^T dO
        for (int idx = tid; idx < C * DV; idx += kNTg) {
            const int t = idx / DV, d = idx % DV;
            float z = 0.f;
            for (int i = 0; i <= t; ++i) z = fmaf(Tm[t * LC + i] * bet[i], Rt[i * LV + d], z);
            Zt[t * LV + d] = z;
            float dz = dZt[t * LV + d];
            for (int i = t; i < C; ++i) dz = fmaf(Pm[i * LC + t], dOt[i * LV + d], dz);
            dZt[t * LV + d] = dz;
        }
        __syncthreads();
        // dR = T^T dZ
        for (int idx = tid; idx < C * DV; idx += kNTg) {
            const int t = idx / DV, d = idx % DV;
            float acc = 0.f;
            for (int i = t; i < C; ++i) acc = fmaf(Tm[i * LC + t], dZt[i * LV + d], acc);
            dRt[t * LV + d] = acc;
        }
        __syncthreads();
        // sum dR Z^T (strictly lower) and dO Z^T (lower) over this pass's columns
        for (int idx = tid; idx < C * C; idx += kNTg) {
            const int t = idx / C, i = idx % C;
            if (i <= t) {
                float ra = 0.f, pa = 0.f;
#pragma unroll
                for (int d = 0; d < DV; ++d) {
                    const float z = Zt[i * LV + d];
                    ra = fmaf(dRt[t * LV + d], z, ra);
                    pa = fmaf(dOt[t * LV + d], z, pa);
                }
                if (i < t) dAm[t * LC + i] += ra;
                dPm[t * LC + i] += pa;
            }
        }
        // dV = diag(beta) dR
        for (int idx = tid; idx < C * DV; idx += kNTg) {
            const int t = idx / DV, d = idx % DV;
            if (t < n) {
                const size_t tok = ((size_t)b * T + c0 + t) * H + h;
                ((TIn *)a.dv)[tok * dv + e0 + d] = from_f<TIn>(bet[t] * dRt[t * LV + d]);
            }
        }
        if (tid < C) {
            const int t = tid;
            float s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int d = 0; d < DV; ++d) {
                const float dr = dRt[t * LV + d];
                s1 = fmaf(dOt[t * LV + d], QSt[t * LV + d], s1);
                s2 = fmaf(-bet[t] * dr, XSt[t * LV + d], s2);
                s3 = fmaf(dr, Rt[t * LV + d], s3);
            }
            sq[t] += s1;
            sx[t] += s2;
            sb[t] += s3;
        }
        // (gamma dXS) S_in, (gamma dO) S_in, Z dS_out for row r
        {
            const float gr = gam[r], fxr = -bet[r] * gam[r];
#pragma unroll 4
            for (int d = 0; d < DV; ++d) {
                const float fx = fxr * dRt[r * LV + d], fq = gr * dOt[r * LV + d], fz = Zt[r * LV + d];
                const float *sd = Ss + d * LK + jc, *gd = dSs + d * LK + jc;
#pragma unroll
                for (int m = 0; m < JN; ++m) {
                    accX[m] = fmaf(fx, sd[8 * m], accX[m]);
                    accQ[m] = fmaf(fq, sd[8 * m], accQ[m]);
                    accK[m] = fmaf(fz, gd[8 * m], accK[m]);
                }
            }
        }
    }
    // <dS_out, S_in>
#pragma unroll
    for (int off = 16; off; off >>= 1) gS += __shfl_xor_sync(0xffffffffu, gS, off);
    if ((tid & 31) == 0) red[tid >> 5] = gS;
    __syncthreads();
    // dA = -sum dR Z^T; dM = beta dA; E = dP * P + dM * M; keep dA * M for dbeta and
    // H * dM, H * dP for the n x dk products
    for (int idx = tid; idx < C * C; idx += kNTg) {
        const int t = idx / C, i = idx % C;
        const int o = t * LC + i;
        float hdm = 0.f, hdp = 0.f, e = 0.f, am = 0.f;
        if (i <= t) {
            const float hti = expf(ell[t] - ell[i]);
            const float da = i < t ? -dAm[o] : 0.f, dm = bet[t] * da, dp = dPm[o];
            e = dp * Pm[o] + dm * Mm[o];
            am = da * Mm[o];
            hdm = hti * dm;
            hdp = hti * dp;
        }
        Pm[o] = e;
        Mm[o] = am;
        dAm[o] = hdm;
        dPm[o] = hdp;
    }
    __syncthreads();
    if (tid < C) {
        const int t = tid;
        float rowE = 0.f, colE = 0.f, dbm = 0.f;
        for (int i = 0; i < C; ++i) {
            rowE += Pm[t * LC + i];
            colE += Pm[i * LC + t];
            dbm += Mm[t * LC + i];
        }
        sq[t] += sx[t] + rowE - colE;                     // dl without the wz and last-token terms
        sb[t] += dbm;                                     // dbeta
    }
    {
        const float lr = lmb[r];
        float dl_p = 0.f, wz_p = 0.f;
        const size_t tok = ((size_t)b * T + c0 + r) * H + h;
#pragma unroll
        for (int m = 0; m < JN; ++m) {
            const int j = jc + 8 * m;
            float dx = accX[m], dq = accQ[m], dkk = 0.f;
            for (int i = 0; i < C; ++i) {
                const float kij = Ks[i * LK + j], qij = Qs[i * LK + j];
                dx = fmaf(dAm[r * LC + i], kij, dx);
                dq = fmaf(dPm[r * LC + i], kij, dq);
                dkk = fmaf(dPm[i * LC + r], qij, dkk);
                dkk = fmaf(dAm[i * LC + r], fmaf(lmb[i], qij, kij), dkk);
            }
            dq = fmaf(lr, dx, dq);
            dkk += fmaf(wC[r], accK[m], dx);
            dl_p = fmaf(dx, Qs[r * LK + j], dl_p);
            wz_p = fmaf(accK[m], Ks[r * LK + j], wz_p);
            if (r < n) {
                if (a.grad_f32) {
                    ((float *)a.dq)[tok * DK + j] = dq;
                    ((float *)a.dk)[tok * DK + j] = dkk;
                } else {
                    ((TIn *)a.dq)[tok * DK + j] = from_f<TIn>(dq);
                    ((TIn *)a.dk)[tok * DK + j] = from_f<TIn>(dkk);
                }
            }
        }
#pragma unroll
        for (int off = 4; off; off >>= 1) {
            dl_p += __shfl_xor_sync(0xffffffffu, dl_p, off);
            wz_p += __shfl_xor_sync(0xffffffffu, wz_p, off);
        }
        if (jc == 0) {
            wz[r] = wC[r] * wz_p;
            if (r < n && a.dlam && a.lam) {
                if (a.grad_f32) ((float *)a.dlam)[tok] = dl_p;
                else ((TIn *)a.dlam)[tok] = from_f<TIn>(dl_p);
            }
        }
    }
    __syncthreads();
    if (tid < 32) {
        float tot = 0.f, wsum = wz[2 * tid] + wz[2 * tid + 1];
        for (int w = 0; w < kNTg / 32; ++w) tot += red[w];
#pragma unroll
        for (int off = 16; off; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
        sq[2 * tid] -= wz[2 * tid];
        sq[2 * tid + 1] -= wz[2 * tid + 1];
        if (tid == 31) sq[C - 1] += gam[C - 1] * tot + wsum;
    }
    __syncwarp();
    suffix64(sq);                                         // d log alpha
    __syncthreads();
    if (tid < n) {
        const size_t tok = ((size_t)b * T + c0 + tid) * H + h;
        const float dal = sq[tid] / expf(la[tid]);
        if (a.grad_f32) {
            ((float *)a.dbeta)[tok] = sb[tid];
            if (a.dalpha && a.alpha) ((float *)a.dalpha)[tok] = dal;
        } else {
            ((TIn *)a.dbeta)[tok] = from_f<TIn>(sb[tid]);
            if (a.dalpha && a.alpha) ((TIn *)a.dalpha)[tok] = from_f<TIn>(dal);
        }
    }
}

template <int DK, int DVT>
constexpr size_t dstate_smem() {
    return sizeof(float) * (3 * kC * (DK + 1) + DVT * (DK + 1) + 2 * kC * (DVT + 1) + 2 * kC * (kC + 1) + 4 * kC);
}
template <int DK>
constexpr size_t grad_smem() {
    return sizeof(float) * (2 * kC * (DK + 1) + 5 * kC * (kC + 1) + 2 * kDVS * (DK + 1) + 7 * kC * (kDVS + 1) +
                            10 * kC + kNTg / 32);
}

template <typename TIn, int DK, int DVT>
cudaError_t run_bwd(const QDeltaBwdArgs &a, cudaStream_t s, bool tc) {
    cudaError_t e;
    if (tc) {
        e = launch_qdelta_bwd_dstate_tc(a, s);
    } else {
        auto ks = qdelta_bwd_dstate_kernel<TIn, DK, DVT>;
        constexpr size_t sm_s = dstate_smem<DK, DVT>();
        e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_s);
        if (e != cudaSuccess) return e;
        ks<<<dim3(a.B * a.H, a.nv / DVT), kNTs, sm_s, s>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    if (tc) return launch_qdelta_bwd_grad_tc(a, s);
    auto kg = qdelta_bwd_grad_kernel<TIn, DK>;
    constexpr size_t sm_g = grad_smem<DK>();
    e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_g);
    if (e != cudaSuccess) return e;
    const int nchunk = (a.T + kC - 1) / kC;
    kg<<<(unsigned)(a.B * a.H * nchunk), kNTg, sm_g, s>>>(a);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_bwd(const QDeltaBwdArgs &a, cudaStream_t s, bool m) {
    const bool wide = a.nv >= 32;
    switch (a.nk) {
        case 16: return wide ? run_bwd<TIn, 16, 32>(a, s, m) : run_bwd<TIn, 16, 16>(a, s, m);
        case 32: return wide ? run_bwd<TIn, 32, 32>(a, s, m) : run_bwd<TIn, 32, 16>(a, s, m);
        case 64: return wide ? run_bwd<TIn, 64, 32>(a, s, m) : run_bwd<TIn, 64, 16>(a, s, m);
        case 128: return wide ? run_bwd<TIn, 128, 32>(a, s, m) : run_bwd<TIn, 128, 16>(a, s, m);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

size_t qdelta_bwd_workspace(int B, int T, int H, int dk, int dv) {
    const size_t nchunk = (size_t)((T + kC - 1) / kC);
    return 2 * (size_t)B * H * nchunk * dv * dk * sizeof(float);
}

cudaError_t launch_qdelta_bwd(const QDeltaBwdArgs &a, int dtype, cudaStream_t s, int *nlaunch) {
    // 1. forward over the chunks, keeping the state entering each (the tensor-core
    //    kernel where it applies, without its output)
    const bool pro = a.raw_q != nullptr;              // from projections: the prologue forward
    QDeltaArgs f{pro ? a.raw_q : a.q, pro ? a.raw_k : a.k, a.v, pro ? a.raw_a : a.alpha, pro ? a.raw_b : a.beta,
                 pro ? a.raw_l : a.lam, a.S0, nullptr, nullptr, a.B, a.T, a.H, a.nk, a.nv, nullptr, 0, pro ? 1 : 0,
                 a.S_chk};
    //    The checkpoint format follows the backward kernels: fp16 operand tiles for the
    //    tensor-core ones (whose conditions include the tensor-core forward's), fp32 rows
    //    for the CUDA-core ones.
    const bool m = qdelta_bwd_tc_supported(a, dtype);
    cudaError_t e = m ? launch_qdelta_chunk_tc(f, s, nlaunch, kTcNoO) : launch_qdelta_chunk_simt(f, dtype, s, nlaunch);
    if (e != cudaSuccess) return e;
    // 2. reverse sweep of dS and 3. the per-chunk gradients
    e = dtype == kBF16 ? dispatch_bwd<__nv_bfloat16>(a, s, m) : dispatch_bwd<float>(a, s, m);
    if (e == cudaSuccess) *nlaunch += 2;
    return e;
}

}  // namespace qd

// Per-chunk gradients of the Q-Delta backward on the warp tensor cores (TF32 mma.sync,
// fp32 accumulation): bf16 inputs, d_k = d_v = 128.  (The reverse sweep of the state
// gradient that precedes it runs on tcgen05, bwd_tc.cu.)
//
// The adjoint of the WY form ("Q-Delta: Beyond Key-Value Associative State Evolution",
// Sec. 3.3.2; the formulas are in bwd_simt.cu's header), one CTA per (b, h, chunk) from
// the two checkpoints of its chunk.  TF32 operands (unit roundoff 2^-11) with fp32
// accumulation.
#include "qd_internal.cuh"
#include "tc_common.cuh"

namespace qd {
namespace {

using tc::mma_tf32;
using tc::to_tf32;

constexpr int kC = 64, kD = 128, kNT = 512;
constexpr int LQ = kD + 8;      // bf16 token rows (272 B): conflict-free fragment loads
constexpr int LS = kD + 4;      // dS rows (fp32)
constexpr int LA = kC + 8;      // A, P rows (fp32)

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// d[n] (16 x 8 tiles n = 0..NT-1 of a 16 x 8NT strip) += A (16 x K) B (K x 8NT) on the
// TF32 m16n8k8 MMA; fa(r, k), fb(k, n) give the operand entries in fp32.  Fragment
// layout (lane = 4 g + t): A rows g, g+8 / columns t, t+4; B rows t, t+4 / column g;
// d[n] = (g, 8n+2t), (g, 8n+2t+1), (g+8, 8n+2t), (g+8, 8n+2t+1).
template <int K, int NT, class FA, class FB>
__device__ __forceinline__ void mma_strip(float (&d)[NT][4], int k_begin, FA fa, FB fb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
    for (int k0 = k_begin; k0 < K; k0 += 8) {
        const uint32_t a[4] = {to_tf32(fa(g, k0 + t)), to_tf32(fa(g + 8, k0 + t)), to_tf32(fa(g, k0 + t + 4)),
                               to_tf32(fa(g + 8, k0 + t + 4))};
#pragma unroll
        for (int n = 0; n < NT; ++n)
            mma_tf32(d[n], a, to_tf32(fb(k0 + t, 8 * n + g)), to_tf32(fb(k0 + t + 4, 8 * n + g)));
    }
}

// ---------------------------------------------------------------------------------
// Per-chunk gradients on the warp tensor cores: one CTA per (b, h, chunk), the adjoint
// of bwd_simt.cu's header.  T = (I + diag(beta) M)^{-1} is formed once per chunk (a
// blocked substitution on the identity); d_v is taken in four quarters of 32 rows of
// S_in / dS_out (fp32 in shared memory), with Z, dR of the quarter from single
// products with T, and the three n x d_k products (gamma dXS) S_in, (gamma dO) S_in and
// Z dS_out accumulated in registers across quarters.  The row sums come from them:
// rowsum(dO * QS) = Q . (gamma dO) S_in,  rowsum(dXS * XS) = X . (gamma dXS) S_in,
// and w_i (Z dS_out)_i . K_i.

constexpr int kQV = 32;         // d_v rows per quarter
constexpr int LV4 = kQV + 8;    // bf16 rows of the quarter's v / dO
constexpr int LR = kQV + 8;     // fp32 rows of R, Z, dZ -> dR

__global__ void __launch_bounds__(kNT, 1) qdelta_bwd_grad_mma_kernel(QDeltaBwdArgs a) {
    extern __shared__ __align__(16) uint8_t smb[];
    __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(smb);      // [C][LQ]
    __nv_bfloat16 *Ks = Qs + kC * LQ;                                 // [C][LQ]
    __nv_bfloat16 *Vq = Ks + kC * LQ;                                 // [C][LV4]
    __nv_bfloat16 *dOq = Vq + kC * LV4;                               // [C][LV4]
    float *Sq = reinterpret_cast<float *>(dOq + kC * LV4);            // [kQV][LS]  S_in rows
    float *dSq = Sq + kQV * LS;                                       // [kQV][LS]  dS_out rows
    float *Rq = dSq + kQV * LS;                                       // [C][LR]    V - XS
    float *Zq = Rq + kC * LR;                                         // [C][LR]
    float *dRq = Zq + kC * LR;                                        // [C][LR]    dR
    float *dZq = dRq + kC * LR;                                       // [C][LR]    dZ
    float *Mm = dZq + kC * LR;                                        // [C][LA]    M -> dA * M
    float *Pm = Mm + kC * LA;                                         // [C][LA]    P -> E
    float *Tm = Pm + kC * LA;                                         // [C][LA]    T, then dR scratch
    float *dAm = Tm + kC * LA;                                        // [C][LA]    sum dR Z^T -> H * dM
    float *dPm = dAm + kC * LA;                                       // [C][LA]    sum dO Z^T -> H * dP
    float *ell = dPm + kC * LA, *la = ell + kC, *bet = la + kC, *lmb = bet + kC, *gam = lmb + kC;
    float *wgt = gam + kC, *sb = wgt + kC, *srow = sb + kC, *red = srow + kC;
    // per-token partial sums of the four warps that share a row block (column group cg),
    // added in a fixed order at the end so that results are run-to-run identical
    float *part_s = red + kNT / 32, *part_z = part_s + 4 * kC, *part_l = part_z + 4 * kC;   // [4][kC] each

    const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q, *k = (const __nv_bfloat16 *)a.k;
    const __nv_bfloat16 *v = (const __nv_bfloat16 *)a.v, *dO = (const __nv_bfloat16 *)a.dO;
    const int T = a.T, H = a.H, nchunk = (T + kC - 1) / kC;
    const int c = blockIdx.x % nchunk, bh = blockIdx.x / nchunk, b = bh / H, h = bh % H;
    const int c0 = c * kC, n = min(kC, T - c0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
    const size_t chk_base = ((size_t)bh * nchunk + c) * kD * kD;
    auto tok_of = [&](int t) { return ((size_t)b * T + c0 + t) * H + h; };

    for (int i = tid; i < 2 * kC * (kD / 8); i += kNT) {
        const int which = i / (kC * kD / 8), r = (i / (kD / 8)) % kC, col = 8 * (i % (kD / 8));
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) x = *reinterpret_cast<const uint4 *>((which ? k : q) + tok_of(r) * kD + col);
        *reinterpret_cast<uint4 *>((which ? Ks : Qs) + r * LQ + col) = x;
    }
    if (tid < kC) {
        const int t = tid;
        const bool ok = t < n;
        const size_t tok = tok_of(ok ? t : 0);
        la[t] = (ok && a.alpha) ? logf(gate_val<__nv_bfloat16>(a.alpha, tok, a.gates_f32)) : 0.f;
        bet[t] = ok ? gate_val<__nv_bfloat16>(a.beta, tok, a.gates_f32) : 0.f;
        lmb[t] = (ok && a.lam) ? gate_val<__nv_bfloat16>(a.lam, tok, a.gates_f32) : 0.f;
        ell[t] = la[t];
        sb[t] = srow[t] = 0.f;
    }
    for (int i = tid; i < kC * LA; i += kNT) dAm[i] = dPm[i] = 0.f;
    __syncthreads();
    if (tid < 32) {
        const float x0 = ell[2 * tid], x1 = ell[2 * tid + 1];
        float s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, off);
            if (tid >= off) s += y;
        }
        ell[2 * tid] = s - x1;
        ell[2 * tid + 1] = s;
    }
    __syncthreads();
    if (tid < kC) {
        gam[tid] = expf(ell[tid]);
        wgt[tid] = expf(ell[kC - 1] - ell[tid]);
    }
    auto xval = [&](int t, int j) { return fmaf(lmb[t], bf(Qs + t * LQ + j), bf(Ks + t * LQ + j)); };
    // M = H * X K^T (strict) on warps 0-7, P = H * Q K^T on warps 8-15
    {
        const bool isx = warp < 8;
        const int rb = (warp & 7) >> 1, cb = 32 * (warp & 1);
        float acc[4][4] = {};
        if (cb <= 16 * rb + 15) {
            auto fa = [&](int r, int kk) { return isx ? xval(16 * rb + r, kk) : bf(Qs + (16 * rb + r) * LQ + kk); };
            mma_strip<kD, 4>(acc, 0, fa, [&](int kk, int nn) { return bf(Ks + (cb + nn) * LQ + kk); });
        }
        float *dst = isx ? Mm : Pm;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 16 * rb + g + 8 * (e >> 1), i = cb + 8 * nt + 2 * tq + (e & 1);
                dst[t * LA + i] = (isx ? i < t : i <= t) ? expf(ell[t] - ell[i]) * acc[nt][e] : 0.f;
            }
    }
    __syncthreads();
    // T = (I + diag(beta) M)^{-1}: block row jb = I_jb - A(jb, <jb) T(<jb), then the
    // 16 x 16 diagonal block by substitution, one column per thread
    for (int jb = 0; jb < 4; ++jb) {
        if (jb > 0 && warp < 2 * jb) {                    // columns 8 warp .. of block row jb
            const int col = 8 * warp, t = 16 * jb + g, cc = col + 2 * tq;
            float acc[1][4] = {};
            mma_strip<kC, 1>(acc, 0, [&](int r, int kk) {
                const int row = 16 * jb + r;
                return kk < 16 * jb ? -bet[row] * Mm[row * LA + kk] : 0.f;
            }, [&](int kk, int nn) { return kk < 16 * jb ? Tm[kk * LA + col + nn] : 0.f; });
            *reinterpret_cast<float2 *>(Tm + t * LA + cc) = make_float2(acc[0][0], acc[0][1]);
            *reinterpret_cast<float2 *>(Tm + (t + 8) * LA + cc) = make_float2(acc[0][2], acc[0][3]);
        }
        __syncthreads();
        if (tid < 16 * (jb + 1)) {
            const int col = tid, t0 = 16 * jb;
            float r[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float x = col < t0 ? Tm[(t0 + t) * LA + col] : (col == t0 + t ? 1.f : 0.f);
#pragma unroll
                for (int i = 0; i < t; ++i) x = fmaf(-bet[t0 + t] * Mm[(t0 + t) * LA + t0 + i], r[i], x);
                r[t] = x;
            }
#pragma unroll
            for (int t = 0; t < 16; ++t) Tm[(t0 + t) * LA + col] = r[t];
        }
        if (tid >= 16 * (jb + 1) && tid < kC)             // the zero upper part of block row jb
            for (int t = 0; t < 16; ++t) Tm[(16 * jb + t) * LA + tid] = 0.f;
        __syncthreads();
    }

    // register accumulators of this warp: rows 16 rb.., columns 32 cb.. of the n x d_k results
    const int rb = warp >> 2, cb = 32 * (warp & 3);
    float aX[4][4] = {}, aQ[4][4] = {}, aK[4][4] = {};
    float gS = 0.f;
    for (int e0 = 0; e0 < kD; e0 += kQV) {
        __syncthreads();
        for (int i = tid; i < kQV * kD / 4; i += kNT) {
            const int d = (4 * i) / kD, j = (4 * i) % kD;
            const float4 sv = *reinterpret_cast<const float4 *>(a.S_chk + chk_base + (size_t)(e0 + d) * kD + j);
            const float4 gv = *reinterpret_cast<const float4 *>(a.dS_chk + chk_base + (size_t)(e0 + d) * kD + j);
            *reinterpret_cast<float4 *>(Sq + d * LS + j) = sv;
            *reinterpret_cast<float4 *>(dSq + d * LS + j) = gv;
            gS += sv.x * gv.x + sv.y * gv.y + sv.z * gv.z + sv.w * gv.w;
        }
        for (int i = tid; i < 2 * kC * (kQV / 8); i += kNT) {
            const int which = i / (kC * kQV / 8), r = (i / (kQV / 8)) % kC, col = 8 * (i % (kQV / 8));
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (r < n) x = *reinterpret_cast<const uint4 *>((which ? dO : v) + tok_of(r) * kD + e0 + col);
            *reinterpret_cast<uint4 *>((which ? dOq : Vq) + r * LV4 + col) = x;
        }
        __syncthreads();
        // warps 0-7: R = V - gamma X S^T; warps 8-15: dZ = diag(w) K dS^T + P^T dO (16 x 16 each)
        {
            const int w8 = warp & 7, r0 = 16 * (w8 >> 1), n0 = 16 * (w8 & 1);
            float acc[2][4] = {};
            if (warp < 8) {
                mma_strip<kD, 2>(acc, 0, [&](int r, int kk) { return xval(r0 + r, kk); },
                                 [&](int kk, int nn) { return Sq[(n0 + nn) * LS + kk]; });
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = r0 + g + 8 * (e >> 1), d = n0 + 8 * nt + 2 * tq + (e & 1);
                        Rq[t * LR + d] = bf(Vq + t * LV4 + d) - gam[t] * acc[nt][e];
                    }
            } else {
                mma_strip<kD, 2>(acc, 0, [&](int r, int kk) { return wgt[r0 + r] * bf(Ks + (r0 + r) * LQ + kk); },
                                 [&](int kk, int nn) { return dSq[(n0 + nn) * LS + kk]; });
                mma_strip<kC, 2>(acc, r0, [&](int r, int kk) { return Pm[kk * LA + r0 + r]; },
                                 [&](int kk, int nn) { return bf(dOq + kk * LV4 + n0 + nn); });
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = r0 + g + 8 * (e >> 1), d = n0 + 8 * nt + 2 * tq + (e & 1);
                        dZq[t * LR + d] = acc[nt][e];
                    }
            }
        }
        __syncthreads();
        // warps 0-7: Z = T diag(beta) R; warps 8-15: dR = T^T dZ (separate buffers: no barrier between)
        {
            const int w8 = warp & 7, r0 = 16 * (w8 >> 1), n0 = 16 * (w8 & 1);
            float acc[2][4] = {};
            if (warp < 8)
                mma_strip<kC, 2>(acc, 0, [&](int r, int kk) { return kk <= r0 + 15 ? Tm[(r0 + r) * LA + kk] : 0.f; },
                                 [&](int kk, int nn) { return bet[kk] * Rq[kk * LR + n0 + nn]; });
            else
                mma_strip<kC, 2>(acc, r0, [&](int r, int kk) { return Tm[kk * LA + r0 + r]; },
                                 [&](int kk, int nn) { return dZq[kk * LR + n0 + nn]; });
            float *dst = warp < 8 ? Zq : dRq;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t = r0 + g, d = n0 + 8 * nt + 2 * tq;
                *reinterpret_cast<float2 *>(dst + t * LR + d) = make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2 *>(dst + (t + 8) * LR + d) = make_float2(acc[nt][2], acc[nt][3]);
            }
        }
        __syncthreads();
        // sum dR Z^T (warps 0-7) and dO Z^T (warps 8-15) over this quarter
        {
            const bool isa = warp < 8;
            const int r0 = 16 * ((warp & 7) >> 1), n0 = 32 * (warp & 1);
            if (n0 <= r0 + 15) {
                float *acc_m = isa ? dAm : dPm;
                float acc[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int t = r0 + g, i = n0 + 8 * nt + 2 * tq;
                    acc[nt][0] = acc_m[t * LA + i];
                    acc[nt][1] = acc_m[t * LA + i + 1];
                    acc[nt][2] = acc_m[(t + 8) * LA + i];
                    acc[nt][3] = acc_m[(t + 8) * LA + i + 1];
                }
                if (isa)
                    mma_strip<kQV, 4>(acc, 0, [&](int r, int kk) { return dRq[(r0 + r) * LR + kk]; },
                                      [&](int kk, int nn) { return Zq[(n0 + nn) * LR + kk]; });
                else
                    mma_strip<kQV, 4>(acc, 0, [&](int r, int kk) { return bf(dOq + (r0 + r) * LV4 + kk); },
                                      [&](int kk, int nn) { return Zq[(n0 + nn) * LR + kk]; });
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int t = r0 + g, i = n0 + 8 * nt + 2 * tq;
                    *reinterpret_cast<float2 *>(acc_m + t * LA + i) = make_float2(acc[nt][0], acc[nt][1]);
                    *reinterpret_cast<float2 *>(acc_m + (t + 8) * LA + i) = make_float2(acc[nt][2], acc[nt][3]);
                }
            }
        }
        // n x d_k accumulators: (gamma dXS) S_in, (gamma dO) S_in, Z dS_out over this quarter
        mma_strip<kQV, 4>(aX, 0, [&](int r, int kk) { const int t = 16 * rb + r; return -gam[t] * bet[t] * dRq[t * LR + kk]; },
                          [&](int kk, int nn) { return Sq[kk * LS + cb + nn]; });
        mma_strip<kQV, 4>(aQ, 0, [&](int r, int kk) { const int t = 16 * rb + r; return gam[t] * bf(dOq + t * LV4 + kk); },
                          [&](int kk, int nn) { return Sq[kk * LS + cb + nn]; });
        mma_strip<kQV, 4>(aK, 0, [&](int r, int kk) { return Zq[(16 * rb + r) * LR + kk]; },
                          [&](int kk, int nn) { return dSq[kk * LS + cb + nn]; });
        // dV = diag(beta) dR and rowsum(dR * R)
        for (int i = tid; i < kC * kQV / 2; i += kNT) {
            const int t = i / (kQV / 2), d = 2 * (i % (kQV / 2));
            if (t < n) {
                __nv_bfloat162 pr = __floats2bfloat162_rn(bet[t] * dRq[t * LR + d], bet[t] * dRq[t * LR + d + 1]);
                *reinterpret_cast<__nv_bfloat162 *>((__nv_bfloat16 *)a.dv + tok_of(t) * kD + e0 + d) = pr;
            }
        }
        if (tid < kC) {
            float s = 0.f;
#pragma unroll 8
            for (int d = 0; d < kQV; ++d) s = fmaf(dRq[tid * LR + d], Rq[tid * LR + d], s);
            sb[tid] += s;
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) gS += __shfl_xor_sync(0xffffffffu, gS, off);
    if (lane == 0) red[warp] = gS;
    __syncthreads();
    // dA = -sum dR Z^T, dM = beta dA, E = dP * P + dM * M, dA * M, H * dM, H * dP
    for (int idx = tid; idx < kC * kC; idx += kNT) {
        const int t = idx / kC, i = idx % kC, o = t * LA + i;
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
    if (tid < kC) {
        const int t = tid;
        float rowE = 0.f, colE = 0.f, dbm = 0.f;
        for (int i = 0; i < kC; ++i) {
            rowE += Pm[t * LA + i];
            colE += Pm[i * LA + t];
            dbm += Mm[t * LA + i];
        }
        srow[t] = rowE - colE;
        sb[t] += dbm;                                     // dbeta
    }
    {
        // row sums from the accumulators before the masked products join them:
        // Q . (gamma dO) S_in + X . (gamma dXS) S_in, and K . Z dS_out
        float s_lo = 0.f, s_hi = 0.f, z_lo = 0.f, z_hi = 0.f;
        const int t_lo = 16 * rb + g, t_hi = t_lo + 8;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = e < 2 ? t_lo : t_hi, j = cb + 8 * nt + 2 * tq + (e & 1);
                const float sv = bf(Qs + t * LQ + j) * aQ[nt][e] + xval(t, j) * aX[nt][e];
                const float zv = bf(Ks + t * LQ + j) * aK[nt][e];
                if (e < 2) { s_lo += sv; z_lo += zv; } else { s_hi += sv; z_hi += zv; }
            }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            s_lo += __shfl_xor_sync(0xffffffffu, s_lo, off);
            s_hi += __shfl_xor_sync(0xffffffffu, s_hi, off);
            z_lo += __shfl_xor_sync(0xffffffffu, z_lo, off);
            z_hi += __shfl_xor_sync(0xffffffffu, z_hi, off);
        }
        if (tq == 0) {
            const int cg = warp & 3;
            part_s[cg * kC + t_lo] = s_lo;
            part_s[cg * kC + t_hi] = s_hi;
            part_z[cg * kC + t_lo] = wgt[t_lo] * z_lo;
            part_z[cg * kC + t_hi] = wgt[t_hi] * z_hi;
        }
        // dX = (gamma dXS) S_in + (H * dM) K;  dQ = (gamma dO) S_in + (H * dP) K + lambda dX
        mma_strip<kC, 4>(aX, 0, [&](int r, int kk) { return dAm[(16 * rb + r) * LA + kk]; },
                         [&](int kk, int nn) { return bf(Ks + kk * LQ + cb + nn); });
        mma_strip<kC, 4>(aQ, 0, [&](int r, int kk) { return dPm[(16 * rb + r) * LA + kk]; },
                         [&](int kk, int nn) { return bf(Ks + kk * LQ + cb + nn); });
        // dK = (H * dP)^T Q + (H * dM)^T X + diag(w) Z dS_out + dX
        float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = e < 2 ? t_lo : t_hi, j = cb + 8 * nt + 2 * tq + (e & 1);
                const float dx = aX[nt][e];
                aK[nt][e] = fmaf(wgt[t], aK[nt][e], dx);
                aQ[nt][e] = fmaf(lmb[t], dx, aQ[nt][e]);
                if (e < 2) l_lo = fmaf(dx, bf(Qs + t * LQ + j), l_lo);
                else l_hi = fmaf(dx, bf(Qs + t * LQ + j), l_hi);
            }
        mma_strip<kC, 4>(aK, 16 * rb, [&](int r, int kk) { return dPm[kk * LA + 16 * rb + r]; },
                         [&](int kk, int nn) { return bf(Qs + kk * LQ + cb + nn); });
        mma_strip<kC, 4>(aK, 16 * rb, [&](int r, int kk) { return dAm[kk * LA + 16 * rb + r]; },
                         [&](int kk, int nn) { return xval(kk, cb + nn); });
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
        }
        if (tq == 0) {
            part_l[(warp & 3) * kC + t_lo] = l_lo;
            part_l[(warp & 3) * kC + t_hi] = l_hi;
        }
        auto put2 = [&](void *base, size_t idx, float x0, float x1) {   // two adjacent gradient entries
            if (a.grad_f32) *reinterpret_cast<float2 *>((float *)base + idx) = make_float2(x0, x1);
            else *reinterpret_cast<__nv_bfloat162 *>((__nv_bfloat16 *)base + idx) = __floats2bfloat162_rn(x0, x1);
        };
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int j = cb + 8 * nt + 2 * tq;
            if (t_lo < n) {
                put2(a.dq, tok_of(t_lo) * kD + j, aQ[nt][0], aQ[nt][1]);
                put2(a.dk, tok_of(t_lo) * kD + j, aK[nt][0], aK[nt][1]);
            }
            if (t_hi < n) {
                put2(a.dq, tok_of(t_hi) * kD + j, aQ[nt][2], aQ[nt][3]);
                put2(a.dk, tok_of(t_hi) * kD + j, aK[nt][2], aK[nt][3]);
            }
        }
    }
    __syncthreads();
    if (tid < 32) {                                       // dl, then d log alpha by a suffix sum
        float tot = 0.f;
        for (int w = 0; w < kNT / 32; ++w) tot += red[w];
        auto sum4 = [&](const float *pp, int t) { return ((pp[t] + pp[kC + t]) + pp[2 * kC + t]) + pp[3 * kC + t]; };
        const float z0 = sum4(part_z, 2 * tid), z1 = sum4(part_z, 2 * tid + 1);
        float x0 = srow[2 * tid] + sum4(part_s, 2 * tid) - z0, x1 = srow[2 * tid + 1] + sum4(part_s, 2 * tid + 1) - z1;
        float wsum = z0 + z1;
#pragma unroll
        for (int off = 16; off; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
        if (tid == 31) x1 += gam[kC - 1] * tot + wsum;
        float s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, s, off);
            if (tid + off < 32) s += y;
        }
        srow[2 * tid] = s;
        srow[2 * tid + 1] = s - x0;
    }
    __syncthreads();
    if (tid < n) {
        const size_t tok = tok_of(tid);
        auto put1 = [&](void *base, float x) {
            if (a.grad_f32) ((float *)base)[tok] = x;
            else ((__nv_bfloat16 *)base)[tok] = __float2bfloat16_rn(x);
        };
        put1(a.dbeta, sb[tid]);
        if (a.dalpha && a.alpha) put1(a.dalpha, srow[tid] / expf(la[tid]));
        if (a.dlam && a.lam) put1(a.dlam, ((part_l[tid] + part_l[kC + tid]) + part_l[2 * kC + tid]) + part_l[3 * kC + tid]);
    }
}

constexpr size_t kGradSmem = (2 * kC * LQ + 2 * kC * LV4) * sizeof(__nv_bfloat16) +
                             sizeof(float) * (2 * kQV * LS + 4 * kC * LR + 5 * kC * LA + 8 * kC + kNT / 32 + 12 * kC);

}  // namespace

bool qdelta_bwd_mma_supported(const QDeltaBwdArgs &a, int dtype) {
    return dtype == kBF16 && a.nk == kD && a.nv == kD;
}

cudaError_t launch_qdelta_bwd_grad_mma(const QDeltaBwdArgs &a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(qdelta_bwd_grad_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kGradSmem);
    if (e != cudaSuccess) return e;
    const int nchunk = (a.T + kC - 1) / kC;
    qdelta_bwd_grad_mma_kernel<<<(unsigned)(a.B * a.H * nchunk), kNT, kGradSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qd

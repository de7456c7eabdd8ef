// Reverse state-gradient sweep of the Q-Delta backward on the warp tensor cores
// (TF32 mma.sync, fp32 accumulation): bf16 inputs, d_k = d_v = 128.
//
// The same recurrence as qdelta_bwd_dstate_kernel (bwd_simt.cu), per chunk of 64
// tokens in reverse ("Q-Delta: Beyond Key-Value Associative State Evolution",
// Sec. 3.3.2, adjoint of the WY form):
//   A = strictly_lower(diag(beta)(H * X K^T)),  P = H * Q K^T (diagonal included)
//   dZ = diag(w) K dS^T + P^T dO,   (I + A)^T dR = dZ
//   dS <- gamma_C dS + (gamma dO)^T Q - (gamma beta dR)^T X
// with one CTA per (b, h) holding all of dS (128 x 128 fp32) in shared memory.  The
// triangular solve runs in 16-token blocks from the last: the coupling to later
// blocks is a tensor-core product, the 16 x 16 diagonal block a per-column
// substitution.  TF32 operands (unit roundoff 2^-11) with fp32 accumulation; the
// state gradient itself stays fp32 across chunks.
#include "qd_internal.cuh"
#include "tc_common.cuh"

namespace qd {
namespace {

using tc::mma_tf32;
using tc::to_tf32;

constexpr int kC = 64, kD = 128, kNT = 512;
constexpr int LQ = kD + 8;      // bf16 token rows (272 B): conflict-free fragment loads
constexpr int LS = kD + 4;      // dS rows (fp32)
constexpr int LZ = kD + 8;      // dZ / dR rows (fp32)
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

__global__ void __launch_bounds__(kNT, 1) qdelta_bwd_dstate_mma_kernel(QDeltaBwdArgs a) {
    extern __shared__ __align__(16) uint8_t smb[];
    __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(smb);      // [C][LQ]
    __nv_bfloat16 *Ks = Qs + kC * LQ;                                 // [C][LQ]
    __nv_bfloat16 *dOs = Ks + kC * LQ;                                // [C][LQ]
    float *dS = reinterpret_cast<float *>(dOs + kC * LQ);             // [D][LS]   dS rows d, columns j
    float *dZ = dS + kD * LS;                                         // [C][LZ]   dZ -> dR
    float *Am = dZ + kC * LZ;                                         // [C][LA]
    float *Pm = Am + kC * LA;                                         // [C][LA]
    float *ell = Pm + kC * LA, *bet = ell + kC, *lmb = bet + kC, *gam = lmb + kC, *wgt = gam + kC;

    const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q, *k = (const __nv_bfloat16 *)a.k;
    const __nv_bfloat16 *dO = (const __nv_bfloat16 *)a.dO;
    const int T = a.T, H = a.H, nchunk = (T + kC - 1) / kC;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
    const size_t s_base = (size_t)bh * kD * kD;

    for (int i = tid; i < kD * kD / 4; i += kNT) {
        const int d = (4 * i) / kD, j = (4 * i) % kD;
        const float4 v = a.dS_final ? reinterpret_cast<const float4 *>(a.dS_final + s_base)[i]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(dS + d * LS + j) = v;
    }

    for (int c = nchunk - 1; c >= 0; --c) {
        const int c0 = c * kC, n = min(kC, T - c0);
        __syncthreads();
        // checkpoint: the gradient reaching the state that leaves chunk c
        float *chk = a.dS_chk + ((size_t)bh * nchunk + c) * kD * kD;
        for (int i = tid; i < kD * kD / 4; i += kNT) {
            const int d = (4 * i) / kD, j = (4 * i) % kD;
            reinterpret_cast<float4 *>(chk)[i] = *reinterpret_cast<const float4 *>(dS + d * LS + j);
        }
        // q, k, dO of the chunk (16-byte loads; rows past T are zero)
        for (int i = tid; i < 3 * kC * (kD / 8); i += kNT) {
            const int which = i / (kC * kD / 8), r = (i / (kD / 8)) % kC, col = 8 * (i % (kD / 8));
            const __nv_bfloat16 *src = which == 0 ? q : which == 1 ? k : dO;
            __nv_bfloat16 *dst = which == 0 ? Qs : which == 1 ? Ks : dOs;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < n) v = *reinterpret_cast<const uint4 *>(src + (((size_t)b * T + c0 + r) * H + h) * kD + col);
            *reinterpret_cast<uint4 *>(dst + r * LQ + col) = v;
        }
        if (tid < kC) {
            const int t = tid;
            const bool ok = t < n;
            const size_t tok = ((size_t)b * T + c0 + (ok ? t : 0)) * H + h;
            ell[t] = (ok && a.alpha) ? logf(__bfloat162float(((const __nv_bfloat16 *)a.alpha)[tok])) : 0.f;
            bet[t] = ok ? __bfloat162float(((const __nv_bfloat16 *)a.beta)[tok]) : 0.f;
            lmb[t] = (ok && a.lam) ? __bfloat162float(((const __nv_bfloat16 *)a.lam)[tok]) : 0.f;
        }
        __syncthreads();
        if (tid < 32) {                                   // inclusive prefix of log alpha
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
        // Grams X K^T (warps 0-7) and Q K^T (warps 8-15): rows 16 rb.., columns 32 cb..
        {
            const bool isx = warp < 8;
            const int rb = (warp & 7) >> 1, cb = 32 * (warp & 1);
            float acc[4][4] = {};
            if (cb <= 16 * rb + 15) {
                auto fa = [&](int r, int kk) {
                    const int t = 16 * rb + r;
                    const float qv = bf(Qs + t * LQ + kk);
                    return isx ? fmaf(lmb[t], qv, bf(Ks + t * LQ + kk)) : qv;
                };
                auto fb = [&](int kk, int nn) { return bf(Ks + (cb + nn) * LQ + kk); };
                mma_strip<kD, 4>(acc, 0, fa, fb);
            }
            float *dst = isx ? Am : Pm;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 16 * rb + g + 8 * (e >> 1), i = cb + 8 * nt + 2 * tq + (e & 1);
                    float v = 0.f;
                    if (isx ? i < t : i <= t) v = expf(ell[t] - ell[i]) * acc[nt][e] * (isx ? bet[t] : 1.f);
                    dst[t * LA + i] = v;
                }
        }
        __syncthreads();
        // dZ = diag(w) K dS^T + P^T dO: rows 16 rb.., columns 32 cb..
        {
            const int rb = warp >> 2, cb = 32 * (warp & 3);
            float acc[4][4] = {};
            mma_strip<kD, 4>(acc, 0, [&](int r, int kk) { return wgt[16 * rb + r] * bf(Ks + (16 * rb + r) * LQ + kk); },
                             [&](int kk, int nn) { return dS[(cb + nn) * LS + kk]; });
            mma_strip<kC, 4>(acc, 16 * rb, [&](int r, int kk) { return Pm[kk * LA + 16 * rb + r]; },
                             [&](int kk, int nn) { return bf(dOs + kk * LQ + cb + nn); });
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int t = 16 * rb + g, col = cb + 8 * nt + 2 * tq;
                *reinterpret_cast<float2 *>(dZ + t * LZ + col) = make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2 *>(dZ + (t + 8) * LZ + col) = make_float2(acc[nt][2], acc[nt][3]);
            }
        }
        __syncthreads();
        // (I + A)^T dR = dZ, in place, 16-token blocks from the last
        for (int jb = 3; jb >= 0; --jb) {
            if (jb < 3) {                                 // dZ_jb -= A(later, jb)^T dR(later)
                const int kb = 16 * (jb + 1), col = 8 * warp;
                float acc[1][4];
                const int t = 16 * jb + g, cc = col + 2 * tq;
                acc[0][0] = dZ[t * LZ + cc];
                acc[0][1] = dZ[t * LZ + cc + 1];
                acc[0][2] = dZ[(t + 8) * LZ + cc];
                acc[0][3] = dZ[(t + 8) * LZ + cc + 1];
                mma_strip<kC, 1>(acc, kb, [&](int r, int kk) { return -Am[kk * LA + 16 * jb + r]; },
                                 [&](int kk, int nn) { return dZ[kk * LZ + col + nn]; });
                __syncthreads();                          // every read of dZ_jb done
                *reinterpret_cast<float2 *>(dZ + t * LZ + cc) = make_float2(acc[0][0], acc[0][1]);
                *reinterpret_cast<float2 *>(dZ + (t + 8) * LZ + cc) = make_float2(acc[0][2], acc[0][3]);
                __syncthreads();
            }
            if (tid < kD) {                               // the diagonal block, one column per thread
                const int d = tid, t0 = 16 * jb;
                float r[16];
#pragma unroll
                for (int t = 15; t >= 0; --t) {
                    float v = dZ[(t0 + t) * LZ + d];
#pragma unroll
                    for (int i = t + 1; i < 16; ++i) v = fmaf(-Am[(t0 + i) * LA + t0 + t], r[i], v);
                    r[t] = v;
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) dZ[(t0 + t) * LZ + d] = r[t];
            }
            __syncthreads();
        }
        // dS <- gamma_C dS + (gamma dO)^T Q - (gamma beta dR)^T X: rows 16 rb.., columns 64 cb..
        {
            const int rb = warp >> 1, cb = 64 * (warp & 1);
            const float gC = gam[kC - 1];
            float acc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int d = 16 * rb + g, col = cb + 8 * nt + 2 * tq;
                acc[nt][0] = gC * dS[d * LS + col];
                acc[nt][1] = gC * dS[d * LS + col + 1];
                acc[nt][2] = gC * dS[(d + 8) * LS + col];
                acc[nt][3] = gC * dS[(d + 8) * LS + col + 1];
            }
            mma_strip<kC, 8>(acc, 0, [&](int r, int kk) { return gam[kk] * bf(dOs + kk * LQ + 16 * rb + r); },
                             [&](int kk, int nn) { return bf(Qs + kk * LQ + cb + nn); });
            mma_strip<kC, 8>(acc, 0, [&](int r, int kk) { return -gam[kk] * bet[kk] * dZ[kk * LZ + 16 * rb + r]; },
                             [&](int kk, int nn) {
                                 return fmaf(lmb[kk], bf(Qs + kk * LQ + cb + nn), bf(Ks + kk * LQ + cb + nn));
                             });
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int d = 16 * rb + g, col = cb + 8 * nt + 2 * tq;
                *reinterpret_cast<float2 *>(dS + d * LS + col) = make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2 *>(dS + (d + 8) * LS + col) = make_float2(acc[nt][2], acc[nt][3]);
            }
        }
    }
    __syncthreads();
    if (a.dS0)
        for (int i = tid; i < kD * kD / 4; i += kNT) {
            const int d = (4 * i) / kD, j = (4 * i) % kD;
            reinterpret_cast<float4 *>(a.dS0 + s_base)[i] = *reinterpret_cast<const float4 *>(dS + d * LS + j);
        }
}

constexpr size_t kDstateSmem = 3 * kC * LQ * sizeof(__nv_bfloat16) +
                               sizeof(float) * (kD * LS + kC * LZ + 2 * kC * LA + 5 * kC);

}  // namespace

bool qdelta_bwd_mma_supported(const QDeltaBwdArgs &a, int dtype) {
    return dtype == kBF16 && a.nk == kD && a.nv == kD;
}

cudaError_t launch_qdelta_bwd_dstate_mma(const QDeltaBwdArgs &a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(qdelta_bwd_dstate_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kDstateSmem);
    if (e != cudaSuccess) return e;
    qdelta_bwd_dstate_mma_kernel<<<a.B * a.H, kNT, kDstateSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qd

// The QED derive step on CUDA cores, shared by its own kernel (chunk_tc_qed.cu) and the
// fused QED kernel (chunk_tc.cu): for one 32-token half of one chunk of one (b, h), the
// decay-folded operands Ae = a*e^G, Qe = q*e^G, Ke = k*e^-G, W*V (bf16, token layout) and,
// from the second half, e^{G_C} per channel (fp32).  "The Query Knows What to Forget",
// Sec. 2.1-2.2 (Eqs. 4, 6, 8); the chunk algebra is in chunk_tc_qed.cu's header.
#pragma once

#include <cuda_bf16.h>

#include "qd_internal.cuh"
#include "tc_common.cuh"

namespace qd {
namespace tc {

constexpr int kDeriveThreads = 256;

struct QedDeriveParams {
    const __nv_bfloat16 *q, *k, *v, *g, *b, *w;
    const float *lam_h, *z;
    __nv_bfloat16 *Ae, *Qe, *Ke, *WV;
    float *ecg;          // [B][H][nchunks][128]: e^{G_C} per chunk and channel
    int B, T, H;
    int variant;
    int no_v;            // v is not read and W*V not written
};

// One 32-token half of a chunk, on threads 0..255 of the calling CTA (sync() synchronises
// exactly those); s_part is 2 x 16 x 128 floats of shared memory.
// Thread (cg, rg): channels 8 cg .. 8 cg + 7 (one 16-byte vector of each input) of the
// half's tokens 2 rg and 2 rg + 1.  A token row's sixteen channel groups sit in one
// half-warp, so k.u is reduced there by shuffles.  The per-channel prefix of g runs over
// a thread's two tokens, then across the sixteen token groups through shared memory;
// the second half also reads g of the first (its own prefix starts there, and it writes
// e^{G_C}).  Every input vector is loaded before any arithmetic (14 loads of 16 bytes
// in flight per thread).
constexpr int kTokPerThread = 2, kGroups = 16;

// A thread's inputs of one half: its 16-byte pieces of q, k, b, g, g of the first half
// (second half only), v, w for its two tokens (zero past T).
constexpr int kDeriveIn = 7;
struct QedDeriveIn {
    uint4 x[kDeriveIn][kTokPerThread];   // q, k, b, g, g0, v, w
};
// The global source of piece (x, i) of this thread, or null where it is zero.
__device__ __forceinline__ const __nv_bfloat16 *qed_derive_src(const QedDeriveParams &p, int chunk, int half,
                                                               int bh, int x, int i) {
    const int tid = threadIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int t0 = chunk * kC, nt = min(kC, p.T - t0);
    const int rg = tid >> 4, j0 = 8 * (tid & 15);
    const int t = x == 4 ? kTokPerThread * rg + i : 32 * half + kTokPerThread * rg + i;
    const bool ok = x == 4 ? (half && t < nt) : (x >= 5 ? (t < nt && !p.no_v) : t < nt);
    const __nv_bfloat16 *src = x == 0 ? p.q : x == 1 ? p.k : x == 2 ? p.b : x == 3 || x == 4 ? p.g : x == 5 ? p.v : p.w;
    return ok ? src + (((size_t)b * p.T + t0 + t) * p.H + h) * kD + j0 : nullptr;
}
__device__ __forceinline__ void qed_derive_load(const QedDeriveParams &p, int chunk, int half, int bh,
                                                QedDeriveIn &in) {
#pragma unroll
    for (int x = 0; x < kDeriveIn; ++x)
#pragma unroll
        for (int i = 0; i < kTokPerThread; ++i) {
            const __nv_bfloat16 *src = qed_derive_src(p, chunk, half, bh, x, i);
            in.x[x][i] = src ? *reinterpret_cast<const uint4 *>(src) : make_uint4(0u, 0u, 0u, 0u);
        }
}
// The rest of one half from its loaded inputs.
template <typename Sync>
__device__ __forceinline__ void qed_derive_finish(const QedDeriveParams &p, int chunk, int half, int bh,
                                                  const QedDeriveIn &in, float (*s_part)[kGroups][kD], Sync sync) {
    const int tid = threadIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int t0 = chunk * kC, nt = min(kC, p.T - t0);
    const int nchunks = (p.T + kC - 1) / kC;
    const bool gate = p.variant == kQedFull || p.variant == kQedRand;
    const bool proj = p.variant != kQedNogateNoproj;
    const float *zrow = p.variant == kQedRand ? p.z + (size_t)h * kD : nullptr;
    const float lam = p.lam_h[h];
    const int cg = tid & 15, rg = tid >> 4, j0 = 8 * cg;
    auto off = [&](int t) { return (((size_t)b * p.T + t0 + t) * p.H + h) * kD + j0; };
    const uint4 *rq = in.x[0], *rk = in.x[1], *rb = in.x[2], *rgv = in.x[3], *rg0 = in.x[4];
    const uint4 *rv = in.x[5], *rw = in.x[6];
    float zf[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) zf[e] = zrow ? zrow[j0 + e] : 0.f;
    // per-channel sums of g over this thread's tokens (own half, and the first half)
    float gs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, g0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
        float gf[8], hf8[8];
        unpack8(rgv[i], gf);
        unpack8(rg0[i], hf8);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            gs[e] += gf[e];
            g0[e] += hf8[e];
        }
    }
    *reinterpret_cast<float4 *>(&s_part[1][rg][j0]) = make_float4(gs[0], gs[1], gs[2], gs[3]);
    *reinterpret_cast<float4 *>(&s_part[1][rg][j0 + 4]) = make_float4(gs[4], gs[5], gs[6], gs[7]);
    *reinterpret_cast<float4 *>(&s_part[0][rg][j0]) = make_float4(g0[0], g0[1], g0[2], g0[3]);
    *reinterpret_cast<float4 *>(&s_part[0][rg][j0 + 4]) = make_float4(g0[4], g0[5], g0[6], g0[7]);
    // k.u per token, reduced over the sixteen channel groups of the half-warp
    float ku[kTokPerThread];
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
        float kf[8], bf8[8], xf[8];
        unpack8(rk[i], kf);
        unpack8(rb[i], bf8);
        unpack8(rq[i], xf);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x = zrow ? zf[e] : xf[e];
            acc = fmaf(kf[e], gate ? bf8[e] * x : x, acc);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        ku[i] = proj ? acc : 0.f;
    }
    sync();
    // G before this thread's first token: the first half's total (second half only),
    // then the own half's groups before rg
    float G[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < kGroups + rg; ++r) {
        if (r < kGroups && !half) continue;
        const float *src = r < kGroups ? &s_part[0][r][j0] : &s_part[1][r - kGroups][j0];
        const float4 x = *reinterpret_cast<const float4 *>(src);
        const float4 y = *reinterpret_cast<const float4 *>(src + 4);
        G[0] += x.x; G[1] += x.y; G[2] += x.z; G[3] += x.w;
        G[4] += y.x; G[5] += y.y; G[6] += y.z; G[7] += y.w;
    }
    if (half && rg == kGroups - 1) {                   // e^{G_C}: G over the whole chunk
        float ec[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ec[e] = __expf(G[e] + gs[e]);
        float4 *dst = reinterpret_cast<float4 *>(p.ecg + ((size_t)bh * nchunks + chunk) * kD + j0);
        dst[0] = make_float4(ec[0], ec[1], ec[2], ec[3]);
        dst[1] = make_float4(ec[4], ec[5], ec[6], ec[7]);
    }
    // per token: G_t, the erase vector a_t, and the operands
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
        const int t = 32 * half + kTokPerThread * rg + i;
        float qf[8], kf[8], bf8[8], gf[8], ae[8], qe[8], ke[8];
        unpack8(rq[i], qf);
        unpack8(rk[i], kf);
        unpack8(rb[i], bf8);
        unpack8(rgv[i], gf);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            G[e] += gf[e];
            const float x = zrow ? zf[e] : qf[e];
            const float u = gate ? bf8[e] * x : x;
            const float a = bf8[e] * kf[e] + lam * (proj ? u - kf[e] * ku[i] : u);
            const float eg = __expf(G[e]), ig = __expf(-G[e]);
            ae[e] = a * eg;
            qe[e] = qf[e] * eg;
            ke[e] = kf[e] * ig;
        }
        if (t < nt) {
            const size_t o = off(t);
            *reinterpret_cast<uint4 *>(p.Ae + o) = pack8(ae);
            *reinterpret_cast<uint4 *>(p.Qe + o) = pack8(qe);
            *reinterpret_cast<uint4 *>(p.Ke + o) = pack8(ke);
            if (!p.no_v) {
                float vf[8], wf[8];
                unpack8(rv[i], vf);
                unpack8(rw[i], wf);
#pragma unroll
                for (int e = 0; e < 8; ++e) vf[e] *= wf[e];
                *reinterpret_cast<uint4 *>(p.WV + o) = pack8(vf);
            }
        }
    }
}

// One half: its loads, then the rest.
template <typename Sync>
__device__ __forceinline__ void qed_derive_half(const QedDeriveParams &p, int chunk, int half, int bh,
                                                float (*s_part)[kGroups][kD], Sync sync) {
    QedDeriveIn in;
    qed_derive_load(p, chunk, half, bh, in);
    qed_derive_finish(p, chunk, half, bh, in, s_part, sync);
}

}  // namespace tc
}  // namespace qd

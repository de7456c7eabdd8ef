// Chunked QED forward on the sm_103a tensor cores, bf16, dk = dv = 128, chunk C = 64.
//
// Recurrence ("The Query Knows What to Forget", Sec. 2.1-2.2: GDN-2 update of
// Eqs. 4/8, erase vector of Eq. 6), with the state kept as S^ = S^T ([dv][dk]):
//   S^_t = S^_{t-1} D_t (I - a_t k_t^T) + (w_t * v_t) k_t^T,   o_t = S^_t q_t,
//   D_t = Diag(e^{g_t}),  a_t = b_t*k_t + lam_h (u_t - k_t (k_t^T u_t)),  u_t = b_t*q_t
//   (the ablation arms of Table 1 take u_t = q_t, u_t = q_t without the projection,
//   or u_t = b_t*z_h; see qd_internal.cuh).
// Per chunk, with the in-chunk cumulative log-decay G_t = sum_{j<=t} g_j (a vector
// over the dk channels, anchored at the chunk start):
//   Ae = A*e^G, Qe = Q*e^G, Ke = K*e^-G                  (elementwise, per channel)
//   G  = [Ae; Qe] Ke^T                 -> At = strictly_lower, P = incl_lower
//   Tinv = (I + At)^{-1}
//   U^T = (W*V)^T Tinv^T,  W^T = Ae^T Tinv^T,  Z^T = U^T - S^ W^T
//   O^T = S^ Qe^T + Z^T P^T
//   S^ <- S^ diag(e^{G_C}) + Z^T (K*e^{G_C - G}) = (S^ + Z^T Ke) diag(e^{G_C})
// The last form reads the same Ke tile as the Gram and applies the chunk's
// per-channel decay once, to the fp32 state, in the epilogue.  The factored decay
// stays in fp32 range while every channel's log-decay summed over one chunk is >= -80.
//
// Two kernels:
//   qed_derive_kernel (this file, CUDA cores): every chunk independently, in parallel
//     over all chunks: k.u per token, the erase vector a, the per-channel prefix G and
//     the operands Ae, Qe, Ke, W*V (bf16, the [B][T][H][128] token layout) and e^{G_C}
//     per chunk (fp32) into the workspace.  It is bandwidth bound: it reads the six
//     input vectors once and writes four.
//   the chain: the warp-specialised tensor-core chunk kernel of chunk_tc.cu in its QED
//     instance, which takes Ae, Qe, Ke, W*V where the Q-Delta instance takes X, Q, K, V,
//     runs with unit gates and multiplies the state by e^{G_C} per channel in its
//     epilogue.  With the state-independent operands prepared, its per-chunk critical
//     path is that of the Q-Delta kernel.
#include <cuda_bf16.h>
#include <math.h>

#include "qd_internal.cuh"
#include "tc_common.cuh"

namespace qd {
namespace {

using namespace tc;

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

// Two CTAs per (chunk, b*H + h), one per 32-token half (blockIdx.x = 2 chunk + half).
// Thread (cg, rg): channels 8 cg .. 8 cg + 7 (one 16-byte vector of each input) of the
// half's tokens 2 rg and 2 rg + 1.  A token row's sixteen channel groups sit in one
// half-warp, so k.u is reduced there by shuffles.  The per-channel prefix of g runs over
// a thread's two tokens, then across the sixteen token groups through shared memory;
// the second half also reads g of the first (its own prefix starts there, and it writes
// e^{G_C}).  Every input vector is loaded before any arithmetic (12 loads of 16 bytes
// in flight per thread); at most 128 registers a thread, so two CTAs share an SM.
constexpr int kTokPerThread = 2, kGroups = 16;
__global__ void __launch_bounds__(kDeriveThreads, 2) qed_derive_kernel(const QedDeriveParams p) {
    __shared__ __align__(16) float s_part[2][kGroups][kD];   // [first half, own half][group][channel]
    const int tid = threadIdx.x;
    const int chunk = blockIdx.x >> 1, half = blockIdx.x & 1, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    const int t0 = chunk * kC, nt = min(kC, p.T - t0);
    const int nchunks = (p.T + kC - 1) / kC;
    const bool gate = p.variant == kQedFull || p.variant == kQedRand;
    const bool proj = p.variant != kQedNogateNoproj;
    const float *zrow = p.variant == kQedRand ? p.z + (size_t)h * kD : nullptr;
    const float lam = p.lam_h[h];
    const int cg = tid & 15, rg = tid >> 4, j0 = 8 * cg;
    auto off = [&](int t) { return (((size_t)b * p.T + t0 + t) * p.H + h) * kD + j0; };
    auto ld8 = [&](const __nv_bfloat16 *src, int t) {
        return *reinterpret_cast<const uint4 *>(src + off(t));
    };
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 rq[kTokPerThread], rk[kTokPerThread], rb[kTokPerThread], rgv[kTokPerThread], rg0[kTokPerThread];
    uint4 rv[kTokPerThread], rw[kTokPerThread];
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {          // all loads first
        const int t = 32 * half + kTokPerThread * rg + i, t_first = kTokPerThread * rg + i;
        const bool ok = t < nt;
        rq[i] = ok ? ld8(p.q, t) : zero;
        rk[i] = ok ? ld8(p.k, t) : zero;
        rb[i] = ok ? ld8(p.b, t) : zero;
        rgv[i] = ok ? ld8(p.g, t) : zero;
        rg0[i] = (half && t_first < nt) ? ld8(p.g, t_first) : zero;
        rv[i] = (ok && !p.no_v) ? ld8(p.v, t) : zero;
        rw[i] = (ok && !p.no_v) ? ld8(p.w, t) : zero;
    }
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
    __syncthreads();
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

}  // namespace

bool qed_tc_supported(const QedArgs &a, int dtype) {
    return dtype == kBF16 && a.dk == kD && a.dv == kD && (long long)a.T * a.H * kD * 2 < (1ll << 40) &&
           (long long)a.B * a.H <= 65535;
}

QedDerived qed_derived_buffers(int B, int T, int H, void *ws) {
    const size_t tok = (size_t)B * T * H * kD;             // elements of one token tensor
    __nv_bfloat16 *base = static_cast<__nv_bfloat16 *>(ws);
    QedDerived d;
    d.Ae = base;
    d.Qe = base + tok;
    d.Ke = base + 2 * tok;
    d.WV = base + 3 * tok;
    d.ecg = reinterpret_cast<float *>(base + 4 * tok);
    return d;
}

size_t qed_derived_bytes(int B, int T, int H, int G) {
    const int Tg = T / G;
    const size_t nchunks = (size_t)(Tg + kC - 1) / kC;
    return 4 * (size_t)B * T * H * kD * 2 + (size_t)B * G * H * nchunks * kD * sizeof(float);
}

cudaError_t launch_qed_derive(const QedArgs &a, const QedDerived &d, int no_v, cudaStream_t s, int *nlaunch) {
    QedDeriveParams p{(const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v,
                      (const __nv_bfloat16 *)a.g, (const __nv_bfloat16 *)a.b, (const __nv_bfloat16 *)a.w,
                      a.lam_h, a.z, (__nv_bfloat16 *)d.Ae, (__nv_bfloat16 *)d.Qe, (__nv_bfloat16 *)d.Ke,
                      (__nv_bfloat16 *)d.WV, d.ecg, a.B, a.T, a.H, a.variant, no_v};
    const dim3 grid(2 * ((a.T + kC - 1) / kC), a.B * a.H);  // B * H <= 65535 (qed_tc_supported)
    qed_derive_kernel<<<grid, kDeriveThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

size_t qed_tc_workspace(int B, int T, int H, int G) {
    return qed_derived_bytes(B, T, H, G) + qdelta_segment_workspace(B, H, G);
}

cudaError_t launch_qed_tc(const QedArgs &a, int G, cudaStream_t s, int *nlaunch) {
    QedArgs view = a;                                 // the segment view [B*G][T/G]
    view.B = a.B * G;
    view.T = a.T / G;
    const QedDerived d = qed_derived_buffers(view.B, view.T, a.H, a.ws);
    cudaError_t e = launch_qed_derive(view, d, 0, s, nlaunch);
    if (e != cudaSuccess) return e;
    if (G == 1) return launch_qed_chain_tc(a, d, s, nlaunch, 0);
    QedArgs seg = a;                                  // the segment states follow the derived operands
    seg.ws = static_cast<uint8_t *>(a.ws) + qed_derived_bytes(a.B, a.T, a.H, G);
    return launch_qed_segmented(seg, G, d, s, nlaunch);
}

}  // namespace qd

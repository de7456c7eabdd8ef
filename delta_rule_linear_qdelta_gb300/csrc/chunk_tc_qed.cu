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
//   U^T = (W*V)^T Tinv^T,  Z^T = U^T - (S^ Ae^T) Tinv^T      (= U^T - S^ W^T, W = Tinv Ae)
//   O^T = S^ Qe^T + Z^T P^T
//   S^ <- S^ diag(e^{G_C}) + Z^T (K*e^{G_C - G}) = (S^ + Z^T Ke) diag(e^{G_C})
// The last form reads the same Ke tile as the Gram and applies the chunk's
// per-channel decay once, to the fp32 state, in the epilogue.  The factored decay
// stays in fp32 range while every channel's log-decay summed over one chunk is >= -80.
//
// Two steps:
//   the derive step (qed_derive.cuh, CUDA cores): every chunk independently: k.u per
//     token, the erase vector a, the per-channel prefix G and the operands Ae, Qe, Ke,
//     W*V (bf16, the [B][T][H][128] token layout) and e^{G_C} per chunk (fp32) into the
//     workspace.  It reads the six input vectors once and writes four.
//   the chain: the warp-specialised tensor-core chunk kernel of chunk_tc.cu in its QED
//     instance, which takes Ae, Qe, Ke, W*V where the Q-Delta instance takes X, Q, K, V,
//     runs with unit gates and multiplies the state by e^{G_C} per channel in its
//     epilogue.  With the state-independent operands prepared, its per-chunk critical
//     path is that of the Q-Delta kernel.
// They run in one cooperative launch (launch_qed_fused_tc: the derive step on the SMs the
// B*H chains leave free, handing chunks over through counters) while B*H leaves at least
// 8 SMs, else as qed_derive_kernel (this file) and then the chain kernel.
#include <cuda_bf16.h>
#include <math.h>

#include "qd_internal.cuh"
#include "qed_derive.cuh"
#include "tc_common.cuh"

namespace qd {
namespace {

using namespace tc;

// Two CTAs per (chunk, b*H + h), one per 32-token half (blockIdx.x = 2 chunk + half),
// two CTAs per SM (at most 128 registers a thread).
__global__ void __launch_bounds__(kDeriveThreads, 2) qed_derive_kernel(const QedDeriveParams p) {
    __shared__ __align__(16) float s_part[2][kGroups][kD];   // [first half, own half][group][channel]
    qed_derive_half(p, blockIdx.x >> 1, blockIdx.x & 1, blockIdx.y, s_part, []() { __syncthreads(); });
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

namespace {
size_t qed_done_bytes(int B, int T, int H) {          // the fused launch's hand-over counters
    return ((size_t)B * H * ((T + kC - 1) / kC) * sizeof(unsigned int) + 255) & ~(size_t)255;
}
}  // namespace

size_t qed_tc_workspace(int B, int T, int H, int G) {
    return qed_derived_bytes(B, T, H, G) + qdelta_segment_workspace(B, H, G) + qed_done_bytes(B, T, H);
}

cudaError_t launch_qed_tc(const QedArgs &a, int G, cudaStream_t s, int *nlaunch) {
    QedArgs view = a;                                 // the segment view [B*G][T/G]
    view.B = a.B * G;
    view.T = a.T / G;
    const QedDerived d = qed_derived_buffers(view.B, view.T, a.H, a.ws);
    if (G == 1 && (long long)a.B * a.H + 8 <= sm_count()) {
        unsigned int *done = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(a.ws) +
                                                              qed_derived_bytes(a.B, a.T, a.H, 1) +
                                                              qdelta_segment_workspace(a.B, a.H, 1));
        return launch_qed_fused_tc(a, d, done, s, nlaunch);
    }
    cudaError_t e = launch_qed_derive(view, d, 0, s, nlaunch);
    if (e != cudaSuccess) return e;
    if (G == 1) return launch_qed_chain_tc(a, d, s, nlaunch, 0);
    QedArgs seg = a;                                  // the segment states follow the derived operands
    seg.ws = static_cast<uint8_t *>(a.ws) + qed_derived_bytes(a.B, a.T, a.H, G);
    return launch_qed_segmented(seg, G, d, s, nlaunch);
}

}  // namespace qd

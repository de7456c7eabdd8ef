// EDA, erase-then-delta ("Erase-then-Delta Attention", core method), on the tensor cores:
// bf16 inputs, dk = dv = 128.  Per token, with the state S = M^T ([dv][dk], fp32),
//   S <- S (I - e e^T)                      erase along e
//   S <- S (I - beta k k^T) + beta v k^T    Delta write along k
//   o  = S q                                read-out after both steps,
// so that, with c = beta (k.q),
//   o_t = S_{t-1} (I - e e^T) (q - c k) + c v = S_{t-1} r_t + c_t v_t,
//   r_t = y - (e.y) e,  y = q - c k.
// Both steps are Delta-rule steps (key e, value 0, strength 1; key k, value v, strength
// beta), and S_{t-1} r_t is a read-out taken after the step before the erase of token t.
// So the forward is the Delta rule (no decay) over 2T+1 sub-tokens s with a query each,
// in the read-after-write form of the chunked Q-Delta kernel:
//   s = 0       key 0,    value 0,   strength 0        query r_0
//   s = 2t + 1  key e_t,  value 0,   strength 1        query 0
//   s = 2t + 2  key k_t,  value v_t, strength beta_t   query r_{t+1} (0 after the last token)
// which gives o'_{2t} = S_{t-1} r_t and the final state; then o_t = o'_{2t} + c_t v_t.
//
// Why this form: with the page's e = q/|q| the read-out after both steps, S_t q, cancels
// most of S q (the erase removes that direction) down to |o| of about a tenth of |S q|,
// and the 16-bit operands of a chunked read-out of S_t q would carry the rounding error of
// the large terms.  r_t is that cancellation done first, in fp32 on the token vectors:
// it is small exactly when o is, and the read S_{t-1} r_t has nothing left to cancel.
// The sub-token operands and the kernel's intermediates are fp16 (11 significant bits;
// the bf16 inputs convert exactly): an fp64 emulation of the kernel's roundings at
// T = 150 and 2048 (tests/test_eda_rounding_model.py) gives 1.7e-3 relative L2 on o (most
// of it the final bf16 rounding) and 4e-4 on S, against 4.6e-3 with bf16 intermediates.
// Inputs and states must stay inside fp16's range (|x| < 65504).
//
// Three launches on the caller's stream: eda_subtoken_kernel (r_t, c_t and the sub-token
// arrays), the fp16 instance of the Q-Delta tensor-core forward (chunk_tc.cu) over the
// [B][2T+1] sub-token sequence, and eda_readout_kernel (o_t = o'_{2t} + c_t v_t).  Only the
// keys are stored per sub-token; queries, values and outputs are nonzero (needed) on one
// sub-token of each pair, so they are compact [B][T][H][128] arrays (r_t, v_t, o'_{2t})
// that the kernel reads and writes through pair maps, the other rows coming from the
// maps' zero fill.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qd_internal.cuh"
#include "tc_common.cuh"

namespace qd {
namespace {

using tc::kD;
using tc::pack8hp;
using tc::pack8p;
using tc::unpack8;
using tc::unpack8h;

constexpr int kThreads = 256;                       // 16 token-heads of 16 threads per block

// The workspace: Ks fp16 [B][2T+1][H][128] (the sub-token keys); Vc, Rc, Oc fp16
// [B][T][H][128] (v_t, r_t, o'_{2t}); beta_s bf16 [B][2T+1][H]; c fp32 [B][T][H]; each
// region 256-byte aligned.
struct EdaTcBuffers {
    __half *Ks, *Vc, *Rc, *Oc;
    __nv_bfloat16 *bs;
    float *c;
};
size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }
size_t eda_keys_bytes(int B, int T, int H) { return round256((size_t)B * (2 * (size_t)T + 1) * H * kD * 2); }
size_t eda_rows_bytes(int B, int T, int H) { return round256((size_t)B * T * H * kD * 2); }
EdaTcBuffers eda_tc_buffers(int B, int T, int H, void *ws) {
    uint8_t *p = static_cast<uint8_t *>(ws);
    const size_t keys = eda_keys_bytes(B, T, H), rows = eda_rows_bytes(B, T, H);
    EdaTcBuffers w;
    w.Ks = reinterpret_cast<__half *>(p);
    w.Vc = reinterpret_cast<__half *>(p + keys);
    w.Rc = reinterpret_cast<__half *>(p + keys + rows);
    w.Oc = reinterpret_cast<__half *>(p + keys + 2 * rows);
    w.bs = reinterpret_cast<__nv_bfloat16 *>(p + keys + 3 * rows);
    w.c = reinterpret_cast<float *>(p + keys + 3 * rows + round256((size_t)B * (2 * (size_t)T + 1) * H * 2));
    return w;
}

// Thread (token-head th, channel group cg): channels 8 cg .. 8 cg + 7 of token-head
// th = (b T + t) H + h; the sixteen threads of a token-head are one half-warp, so its
// three dot products (k.q, e.q, e.k) are reduced by shuffles within it.  Every thread of
// the block takes part in the shuffles; those past the last token-head load zeros and
// store nothing.
__global__ void __launch_bounds__(kThreads)
eda_subtoken_kernel(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                    const __nv_bfloat16 *e, const __nv_bfloat16 *beta, EdaTcBuffers w, int B, int T, int H) {
    const long long n = (long long)B * T * H;
    const long long th = (long long)blockIdx.x * (kThreads / 16) + (threadIdx.x >> 4);
    const int cg = threadIdx.x & 15, j0 = 8 * cg;
    const bool ok = th < n;
    float qf[8], kf[8], vf[8], ef[8];
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const size_t src = (size_t)(ok ? th : 0) * kD + j0;
    unpack8(ok ? *reinterpret_cast<const uint4 *>(q + src) : zero, qf);
    unpack8(ok ? *reinterpret_cast<const uint4 *>(k + src) : zero, kf);
    unpack8(ok ? *reinterpret_cast<const uint4 *>(v + src) : zero, vf);
    unpack8(ok ? *reinterpret_cast<const uint4 *>(e + src) : zero, ef);
    const float bt = (ok && beta) ? __bfloat162float(beta[th]) : 1.f;
    float kq = 0.f, eq = 0.f, ek = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        kq = fmaf(kf[i], qf[i], kq);
        eq = fmaf(ef[i], qf[i], eq);
        ek = fmaf(ef[i], kf[i], ek);
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
        kq += __shfl_xor_sync(0xffffffffu, kq, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
        ek += __shfl_xor_sync(0xffffffffu, ek, o);
    }
    if (!ok) return;
    const float c = bt * kq;                        // y = q - c k
    const float ey = eq - c * ek;                   // e.y
    float rf[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) rf[i] = qf[i] - c * kf[i] - ey * ef[i];
    const int Tp = 2 * T + 1;
    const long long bt_ = th / H;                   // b T + t
    const int h = (int)(th - bt_ * H), t = (int)(bt_ % T);
    const long long b = bt_ / T;
    auto row = [&](int s) { return ((size_t)(b * Tp + s) * H + h); };   // sub-token row index
    auto put = [&](__half *dst, int s, const float *f) {
        *reinterpret_cast<uint4 *>(dst + row(s) * kD + j0) = pack8hp(f);
    };
    const float zf[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    *reinterpret_cast<uint4 *>(w.Rc + (size_t)th * kD + j0) = pack8hp(rf);
    *reinterpret_cast<uint4 *>(w.Vc + (size_t)th * kD + j0) = pack8hp(vf);
    put(w.Ks, 2 * t + 1, ef);
    put(w.Ks, 2 * t + 2, kf);
    if (t == 0) put(w.Ks, 0, zf);                   // the leading sub-token changes nothing
    if (cg == 0) {
        w.bs[row(2 * t + 1)] = __float2bfloat16_rn(1.f);
        w.bs[row(2 * t + 2)] = __float2bfloat16_rn(bt);   // exact: a bf16 input or 1
        if (t == 0) w.bs[row(0)] = __float2bfloat16_rn(0.f);
        w.c[th] = c;
    }
}

// o_t = o'_{2t} + c_t v_t, rounded once to bf16; same thread layout as above.
__global__ void __launch_bounds__(kThreads)
eda_readout_kernel(const __nv_bfloat16 *v, EdaTcBuffers w, __nv_bfloat16 *o, int B, int T, int H) {
    const long long n = (long long)B * T * H;
    const long long th = (long long)blockIdx.x * (kThreads / 16) + (threadIdx.x >> 4);
    if (th >= n) return;
    const int j0 = 8 * (threadIdx.x & 15);
    float of[8], vf[8];
    unpack8h(*reinterpret_cast<const uint4 *>(w.Oc + (size_t)th * kD + j0), of);
    unpack8(*reinterpret_cast<const uint4 *>(v + (size_t)th * kD + j0), vf);
    const float c = w.c[th];
#pragma unroll
    for (int i = 0; i < 8; ++i) of[i] = fmaf(c, vf[i], of[i]);
    *reinterpret_cast<uint4 *>(o + (size_t)th * kD + j0) = pack8p(of);
}

}  // namespace

bool eda_tc_supported(const EdaArgs &a, int dtype) {
    return dtype == kBF16 && a.dk == kD && a.dv == kD && a.T > 0 &&
           (2 * (long long)a.T + 1) * a.H * kD * 2 < (1ll << 40);
}

size_t eda_tc_workspace(int B, int T, int H) {
    return eda_keys_bytes(B, T, H) + 3 * eda_rows_bytes(B, T, H) +
           round256((size_t)B * (2 * (size_t)T + 1) * H * 2) + round256((size_t)B * T * H * 4);
}

cudaError_t launch_eda_tc(const EdaArgs &a, void *ws, cudaStream_t s, int *nlaunch) {
    const EdaTcBuffers w = eda_tc_buffers(a.B, a.T, a.H, ws);
    const long long n = (long long)a.B * a.T * a.H;
    const unsigned grid = (unsigned)((n + kThreads / 16 - 1) / (kThreads / 16));
    eda_subtoken_kernel<<<grid, kThreads, 0, s>>>(
        (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v,
        (const __nv_bfloat16 *)a.e, (const __nv_bfloat16 *)a.beta, w, a.B, a.T, a.H);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *nlaunch += 1;
    QDeltaArgs sub{};
    sub.q = w.Rc;                                     // compact: the kernel's pair maps
    sub.k = w.Ks;
    sub.v = w.Vc;
    sub.beta = w.bs;
    sub.S0 = a.S0;
    sub.o = w.Oc;
    sub.S_final = a.S_final;
    sub.B = a.B;
    sub.T = 2 * a.T + 1;
    sub.H = a.H;
    sub.dk = kD;
    sub.dv = kD;
    e = launch_qdelta_chunk_tc(sub, s, nlaunch, kTcF16);
    if (e != cudaSuccess) return e;
    eda_readout_kernel<<<grid, kThreads, 0, s>>>((const __nv_bfloat16 *)a.v, w, (__nv_bfloat16 *)a.o, a.B, a.T,
                                                 a.H);
    e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

}  // namespace qd

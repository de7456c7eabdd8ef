// Per-chunk gradients of the Q-Delta backward on the sm_103a tensor cores (tcgen05 +
// TMEM + TMA): bf16 inputs, dk = dv = 128, chunk C = 64.  One CTA of 8 warps per
// (b, h, chunk), all chunks in parallel, from the two checkpoints of its chunk: the
// state entering it (S = S_chk) and the gradient reaching the state leaving it
// (dS = dS_chk), each an fp16 [dv][dk] tile already in the operand layout (written so by
// the forward's checkpoint instance and the reverse sweep), copied in with one bulk copy
// each beside the q, k, v, dO tiles.
//
// The adjoint of the WY form ("Q-Delta: Beyond Key-Value Associative State Evolution",
// Sec. 3.3.2; the formulas are in bwd_simt.cu's header).  Per chunk, with H the decay
// mask, M = strictly_lower(H * X K^T), P = H * Q K^T, T = (I + diag(beta) M)^{-1}:
//   R = V - diag(gamma) X S^T,  Z = T diag(beta) R
//   dZ = P^T dO + diag(w) K dS^T,  dR = T^T dZ
//   dA = -strictly_lower(dR Z^T),  dM = diag(beta) dA,  dP = lower(dO Z^T)
//   dX = -diag(gamma beta) dR S + (H * dM) K
//   dQ = diag(gamma) dO S + (H * dP) K + diag(lambda) dX
//   dK = (H * dP)^T Q + (H * dM)^T X + diag(w) Z dS + dX,   dV = diag(beta) dR
// and the gate gradients from row sums of these (see bwd_simt.cu).
//
// Every product has M = 128 with the TMEM lanes indexing a head dimension:
//   G   = [X; Q] K^T                       lanes: X rows | Q rows   (masks, inverse)
//   D1  = S X^T,  dSK = dS K^T,  B = dO^T P      lanes: d_v
//   Z^T = R^T (T diag beta)^T,  dR^T = dZ^T T     lanes: d_v  (A operands packed in TMEM)
//   D5  = [dR; dO] Z^T                     lanes: dR rows | dO rows  (dA, dP)
//   D6  = S^T [-gamma beta dR; gamma dO]^T  (+= K^T [H*dM; H*dP]^T)   lanes: d_k  (dX^T | dQ^T)
//   D7  = dS^T Z^T,  D8 = [X; Q]^T [H*dM; H*dP]                        lanes: d_k  (dK^T)
// The operands are fp16 (kind::f16 with both sides f16): the bf16 inputs convert
// exactly, and the intermediates (the state and its gradient, R, Z, dZ, dR, the inverse,
// the masked matrices) keep 11 significant bits instead of bf16's 8 -- in fp64 emulation of
// this kernel's roundings the relative error of dlambda, the gradient with the most
// cancellation, is 5e-4 with fp16 operands against 4e-3 with bf16 ones.  These values stay
// far inside fp16's range (|x| < 65504) at the workloads' scales.
// S X^T, dS K^T and dO^T P need neither the inverse nor each other: they are issued as
// soon as the masks are written, and the warps the solve's first phases leave idle form
// R^T and dZ^T from them while the inverse runs, so the Z and dR products start as soon
// as it ends.
// Operands that a product needs transposed are written transposed from TMEM (16x256b
// loads, stmatrix.trans) in the 128-byte swizzle.  Sums over a head dimension (the row
// sums of the gate gradients) are a butterfly over the warp's 32 lanes, each lane ending
// with two tokens' totals, then over the warps through shared memory.
//
// Shared memory, by phase (offsets from a 1024-aligned base):
//   XQ  0       32 KB  X rows 0-63 | Q rows 64-127 (two 64-column panels; bf16 from TMA, fp16 after)
//   RO  32768   32 KB  dO rows 64-127 (TMA, then fp16); dR rows 0-63 later; then E (fp32)
//   Sb  65536   32 KB  S as fp16 [dv][dk];  dSb 98304  32 KB  dS as fp16 (bulk copies)
//   K   131072  16 KB
//   V   147456  16 KB  | T 163840 8 KB | T1 172032 8 KB;  all three later RS (32 KB:
//                       -gamma beta dR rows 0-63 | gamma dO rows 64-127), then dq/dk rows
//   MP  180224  16 KB  M rows 0-63 | P rows 64-127 (fp16), then H*dM | H*dP in place
//   R1  196608  17 KB  A = beta M (fp32) for the solve, then Z as [t][dv] (fp16)
//   Y   214016  4.5 KB the solve's scratch
// TMEM (512 columns): G 0-63 (then dS K^T, then D5), A 64-127 (D1 -> R^T, then D7),
// RP 128-159 (packed R^T), Z 160-223, B 224-287 (dO^T P, then D8), DR 288-351,
// D6 352-479, ZP 480-511 (packed dZ^T).
//
// Every wait is bounded; on a timeout the kernel sets its error word, waits (bounded)
// for its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "qd_internal.cuh"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace qd {

__device__ unsigned int g_grad_tc_timeout = 0;

namespace {

using namespace ptx;
using namespace tc;

constexpr int kNT = 256;
constexpr uint32_t OFF_XQ = 0, OFF_RO = 32768, OFF_SB = 65536, OFF_DSB = 98304, OFF_K = 131072;
constexpr uint32_t OFF_V = 147456, OFF_TT = 163840, OFF_T1 = 172032, OFF_RS = OFF_V;
constexpr uint32_t OFF_MP = 180224, OFF_R1 = 196608, OFF_Y = 214016, OFF_ZR = OFF_R1;
constexpr uint32_t kSmemUsed = OFF_Y + 32 * LY * 4;   // 218624
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
static_assert(OFF_MP % 1024 == 0 && OFF_R1 % 1024 == 0 && OFF_Y >= OFF_R1 + 64 * LA * 4, "tile placement");
constexpr uint32_t kTmaBytes = 4 * kC * kD * 2 + 2 * kChkTileBytes;   // q, k, v, dO tiles; S, dS
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t TM_G = 0, TM_A = 64, TM_RP = 128, TM_Z = 160, TM_B = 224, TM_DR = 288, TM_D6 = 352, TM_ZP = 480;

struct GradTcParams {
    const void *alpha, *beta, *lam;
    const uint8_t *S_chk, *dS_chk;                    // fp16 checkpoint tiles (chk_tile_off)
    void *dq, *dk, *dv, *dalpha, *dbeta, *dlam;
    int B, T, H;
    int grad_f32, gates_f32;
};

// The 64 values x[0..63] of every lane of the warp summed over the lanes: lane l
// returns the totals of entries 2l and 2l + 1.
__device__ __forceinline__ float2 warp_sum64(float (&x)[64]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 32; ++i) {                    // 64 -> 32 (offset 16)
        const bool hi = lane & 16;
        const float send = hi ? x[i] : x[32 + i];
        const float keep = hi ? x[32 + i] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {                    // 32 -> 16 (offset 8)
        const bool hi = lane & 8;
        const float send = hi ? x[i] : x[16 + i];
        const float keep = hi ? x[16 + i] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {                     // 16 -> 8 (offset 4)
        const bool hi = lane & 4;
        const float send = hi ? x[i] : x[8 + i];
        const float keep = hi ? x[8 + i] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {                     // 8 -> 4 (offset 2)
        const bool hi = lane & 2;
        const float send = hi ? x[i] : x[4 + i];
        const float keep = hi ? x[4 + i] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {                     // 4 -> 2 (offset 1)
        const bool hi = lane & 1;
        const float send = hi ? x[i] : x[2 + i];
        const float keep = hi ? x[2 + i] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
    return make_float2(x[0], x[1]);
}
// The same for 32 values: lane l returns the total of entry l.
__device__ __forceinline__ float warp_sum32(float (&x)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {               // 32 -> 16 -> ... -> 1 entries a lane
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const bool hi = lane & w;
            const float send = hi ? x[i] : x[w + i];
            const float keep = hi ? x[w + i] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return x[0];
}

__global__ void __launch_bounds__(kNT, 1)
qdelta_bwd_grad_tc_kernel(const GradTcParams p, const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmDQ,
                          const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_ld, bar_mma, bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ __align__(16) float g_ell[kC], g_beta[kC], g_lam[kC], g_gam[kC], g_w[kC], g_ig[kC], g_la[kC];
    __shared__ float red[8][kC];                       // per-warp partial sums over a head dimension
    __shared__ float sdot[8];                          // <dS, S> partials
    __shared__ float s_db[kC], s_dl[kC];               // dbeta, dl per token

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    const int T = p.T, H = p.H, nchunks = (T + kC - 1) / kC;
    const int c = blockIdx.x % nchunks, bh = blockIdx.x / nchunks, b = bh / H, h = bh % H;
    const int c0 = c * kC, n = min(kC, T - c0);
    const size_t chk = ((size_t)bh * nchunks + c) * kChkTileBytes;
    const bool issuer = (tid == 0);
    const uint32_t sbase = smem_u32(sm);
    auto tok_of = [&](int t) { return ((size_t)b * T + c0 + t) * H + h; };

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_drain, 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    for (int i = tid; i < 16384 / 16; i += kNT)        // T, T1: zeros above the diagonal blocks
        reinterpret_cast<uint4 *>(sm + OFF_TT)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_ld, kTmaBytes);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
            tma_load_4d(sm + OFF_XQ + pnl * 16384 + 8192, &tmQ, &bar_ld, 64 * pnl, h, c0, b);
            tma_load_4d(sm + OFF_K + pnl * 8192, &tmK, &bar_ld, 64 * pnl, h, c0, b);
            tma_load_4d(sm + OFF_V + pnl * 8192, &tmV, &bar_ld, 64 * pnl, h, c0, b);
            tma_load_4d(sm + OFF_RO + pnl * 16384 + 8192, &tmD, &bar_ld, 64 * pnl, h, c0, b);
        }
        bulk_load(sm + OFF_SB, p.S_chk + chk, kChkTileBytes, &bar_ld);
        bulk_load(sm + OFF_DSB, p.dS_chk + chk, kChkTileBytes, &bar_ld);
    }
    // gates (tokens past T: alpha 1, beta 0, lambda 0)
    if (tid < kC) {
        const bool ok = tid < n;
        const size_t tok = tok_of(ok ? tid : 0);
        const float a = (ok && p.alpha) ? gate_val<__nv_bfloat16>(p.alpha, tok, p.gates_f32) : 1.f;
        g_la[tid] = logf(a);
        g_beta[tid] = ok ? gate_val<__nv_bfloat16>(p.beta, tok, p.gates_f32) : 0.f;
        g_lam[tid] = (ok && p.lam) ? gate_val<__nv_bfloat16>(p.lam, tok, p.gates_f32) : 0.f;
    }
    __syncthreads();
    if (warp == 0) {                                   // l = inclusive prefix of log alpha; gamma, w, e^{-l}
        const float x0 = g_la[2 * lane], x1 = g_la[2 * lane + 1];
        float s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        const float e1 = s, e0 = s - x1, eC = __shfl_sync(0xffffffffu, s, 31);
        g_ell[2 * lane] = e0;
        g_ell[2 * lane + 1] = e1;
        g_gam[2 * lane] = __expf(e0);
        g_gam[2 * lane + 1] = __expf(e1);
        g_w[2 * lane] = __expf(eC - e0);
        g_w[2 * lane + 1] = __expf(eC - e1);
        g_ig[2 * lane] = eC > -80.f ? __expf(-e0) : 0.f;
        g_ig[2 * lane + 1] = eC > -80.f ? __expf(-e1) : 0.f;
    }
    bool ok = true;
    if (!mbar_wait(&bar_ld, 0, kWaitNs)) { ok = false; abort_flag = 1; }
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);
    const int row = 32 * q4 + lane;                    // this thread's TMEM lane
    uint32_t mma_phase = 0;
    auto commit_wait = [&]() {                         // the issuer's products so far have run
        if (issuer) umma_commit(&bar_mma);
        if (!mbar_wait(&bar_mma, mma_phase, kWaitNs)) { ok = false; abort_flag = 1; }
        mma_phase ^= 1;
        tc_fence_after();
    };
    auto sync_mma = [&]() {                            // smem and TMEM writes before the next products
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    // e^{l_t - l_i} for i <= t (the decay mask H), factored while l_C > -80
    const bool split = g_ell[kC - 1] > -80.f;
    // H[t][32 hf + cc] for cc < 32 into f (above the diagonal too; callers mask), the
    // branch taken once for the whole row
    auto hrow = [&](int t, float (&f)[32]) {
        if (split) {
            const float gt = g_gam[t];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 x = *reinterpret_cast<const float4 *>(g_ig + 32 * hf + 4 * c4);
                f[4 * c4] = gt * x.x; f[4 * c4 + 1] = gt * x.y; f[4 * c4 + 2] = gt * x.z; f[4 * c4 + 3] = gt * x.w;
            }
        } else {
            const float lt = g_ell[t];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 x = *reinterpret_cast<const float4 *>(g_ell + 32 * hf + 4 * c4);
                f[4 * c4] = __expf(lt - x.x); f[4 * c4 + 1] = __expf(lt - x.y);
                f[4 * c4 + 2] = __expf(lt - x.z); f[4 * c4 + 3] = __expf(lt - x.w);
            }
        }
    };

    // ------------------------------------------------------------- X and the Gram
    // K, Q and dO from bf16 to fp16 in place, X = K + lambda Q (fp16)
    {
        uint4 kr[4], qr[4], dr[4];
        float lm[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int u = tid + kNT * r, pnl = u >> 9;
            const uint32_t off = (uint32_t)(u & 511) << 4;
            kr[r] = *reinterpret_cast<const uint4 *>(sm + OFF_K + pnl * 8192 + off);
            qr[r] = *reinterpret_cast<const uint4 *>(sm + OFF_XQ + pnl * 16384 + 8192 + off);
            dr[r] = *reinterpret_cast<const uint4 *>(sm + OFF_RO + pnl * 16384 + 8192 + off);
            lm[r] = g_lam[off >> 7];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int u = tid + kNT * r, pnl = u >> 9;
            const uint32_t off = (uint32_t)(u & 511) << 4;
            float kf[8], qf[8], xf[8], df[8];
            unpack8(kr[r], kf);
            unpack8(qr[r], qf);
            unpack8(dr[r], df);
#pragma unroll
            for (int e = 0; e < 8; ++e) xf[e] = fmaf(lm[r], qf[e], kf[e]);
            *reinterpret_cast<uint4 *>(sm + OFF_XQ + pnl * 16384 + off) = pack8hp(xf);
            *reinterpret_cast<uint4 *>(sm + OFF_XQ + pnl * 16384 + 8192 + off) = pack8hp(qf);
            *reinterpret_cast<uint4 *>(sm + OFF_K + pnl * 8192 + off) = pack8hp(kf);
            *reinterpret_cast<uint4 *>(sm + OFF_RO + pnl * 16384 + 8192 + off) = pack8hp(df);
        }
    }
    sync_mma();
    if (issuer) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_G, smem_desc(sbase + OFF_XQ + ko, 16, 1024),
                      smem_desc(sbase + OFF_K + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                      idesc_f16(128, 64, false, false), k > 0);
        }
    }
    // <dS, S> over the two checkpoint tiles (one layout: an elementwise product) while the
    // Gram runs
    {
        float dot = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint32_t off = (uint32_t)(tid + kNT * r) << 4;
            float sf[8], df[8];
            unpack8h(*reinterpret_cast<const uint4 *>(sm + OFF_SB + off), sf);
            unpack8h(*reinterpret_cast<const uint4 *>(sm + OFF_DSB + off), df);
#pragma unroll
            for (int e = 0; e < 8; ++e) dot = fmaf(sf[e], df[e], dot);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) sdot[warp] = dot;
    }
    commit_wait();
    // masks: A = beta M (fp32, R1) for the solve; M (rows 0-63) and P (rows 64-127) fp16 in MP
    {
        float g[32];
        tmem_ld32(tl + TM_G + 32 * hf, g);
        tmem_ld_wait();
        const bool arow = q4 < 2;
        const int t = 32 * (arow ? q4 : q4 - 2) + lane;
        float hf32[32];
        hrow(t, hf32);
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) {
            const int i = 32 * hf + cc;
            g[cc] = (arow ? i < t : i <= t) ? hf32[cc] * g[cc] : 0.f;
        }
        uint8_t *mp = sm + OFF_MP + (arow ? 0 : 8192);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            *reinterpret_cast<uint4 *>(mp + sw128_off(t, 32 * hf + 8 * ch)) = pack8hp(g + 8 * ch);
        if (arow) {
            const float bt = g_beta[t];
            float *Arow = reinterpret_cast<float *>(sm + OFF_R1) + t * LA + 32 * hf;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *reinterpret_cast<float4 *>(Arow + 4 * c4) =
                    make_float4(bt * g[4 * c4], bt * g[4 * c4 + 1], bt * g[4 * c4 + 2], bt * g[4 * c4 + 3]);
        }
    }
    sync_mma();                                        // M, P (and A) written; TM_G read
    // S X^T (into A), dS K^T (into G), dO^T P (into B), lanes d_v: they need neither the
    // inverse nor each other, so they run while the solve does
    if (issuer) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_A, smem_desc(sbase + OFF_SB + ko, 16, 1024), smem_desc(sbase + OFF_XQ + ko, 16, 1024),
                          idesc_f16(128, 64, false, false), k > 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_G, smem_desc(sbase + OFF_DSB + ko, 16, 1024),
                          smem_desc(sbase + OFF_K + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                          idesc_f16(128, 64, false, false), k > 0);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16(tm + TM_B, smem_desc(sbase + OFF_RO + 8192 + k * 2048, 16384, 1024),
                          smem_desc(sbase + OFF_MP + 8192 + k * 2048, 8192, 1024), idesc_f16(128, 64, true, true), k > 0);
        umma_commit(&bar_mma);
    }
    // R^T = V^T - (S X^T) diag(gamma) (fp32 back into A, packed into RP) and
    // dZ^T = dO^T P + (dS K^T) diag(w) (packed into ZP), for this warp's lane quarter, by
    // the warps the solve's first phases leave idle (4-7)
    auto form_r_dz = [&]() {
        if (!mbar_wait(&bar_mma, mma_phase, kWaitNs)) { ok = false; abort_flag = 1; }
        tc_fence_after();
        const int vp = row >> 6, vc = row & 63;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
            float d1[32], gk[32], bb[32];
            tmem_ld32(tl + TM_A + 32 * h2, d1);
            tmem_ld32(tl + TM_G + 32 * h2, gk);
            tmem_ld32(tl + TM_B + 32 * h2, bb);
            tmem_ld_wait();
            uint32_t rp[16], zp[16];
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) {
                const int t = 32 * h2 + cc;
                const float vv = bf(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_V + vp * 8192 + sw128_off(t, vc)));
                d1[cc] = vv - g_gam[t] * d1[cc];
                bb[cc] = fmaf(g_w[t], gk[cc], bb[cc]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                rp[j] = pack_half2(d1[2 * j], d1[2 * j + 1]);
                zp[j] = pack_half2(bb[2 * j], bb[2 * j + 1]);
            }
            tmem_st32(tl + TM_A + 32 * h2, d1);
            tmem_st16(tl + TM_RP + 16 * h2, rp);
            tmem_st16(tl + TM_ZP + 16 * h2, zp);
        }
        tmem_st_wait();
        tc_fence_before();
    };
    // T = (I + beta M)^{-1} (fp16, zero above the diagonal blocks) and T1 = T diag(beta)
    unit_lower_inverse<false, true>(reinterpret_cast<float *>(sm + OFF_R1), reinterpret_cast<float *>(sm + OFF_Y),
                                    sm + OFF_TT, sm + OFF_T1, nullptr, g_beta, form_r_dz,
                                    []() { __syncthreads(); });
    mma_phase ^= 1;                                    // the phase warps 4-7 waited on
    sync_mma();
    // Z^T = R^T T1^T, dR^T = dZ^T T (A operands packed in TMEM)
    if (issuer) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16_ta(tm + TM_Z, tm + TM_RP + 8 * k, smem_desc(sbase + OFF_T1 + k * 32, 16, 1024),
                         idesc_f16(128, 64, false, false), k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16_ta(tm + TM_DR, tm + TM_ZP + 8 * k, smem_desc(sbase + OFF_TT + k * 2048, 8192, 1024),
                         idesc_f16(128, 64, false, true), k > 0);
    }
    commit_wait();

    // ---------------------------------------------------------- transposed operands
    // 64 TMEM columns (tokens) of the 16 lanes L.. -> a [token][d_v] fp16 tile at dst
    // (64-column panels pstride apart), each token scaled by f(t); warps 0-3 take lanes
    // 32 q4 .. + 15, warps 4-7 lanes 32 q4 + 16 .. + 31.
    auto tstore = [&](uint32_t col, uint32_t dst, uint32_t pstride, auto f) {
        const int L = 32 * q4 + 16 * hf, t4 = lane & 3;
        float ov[32];
        tmem_ld16x256_x8(tm + col + ((uint32_t)L << 16), ov);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float f0 = f(8 * j + 2 * t4), f1 = f(8 * j + 2 * t4 + 1);
            pk[2 * j] = pack_half2(ov[4 * j] * f0, ov[4 * j + 1] * f1);
            pk[2 * j + 1] = pack_half2(ov[4 * j + 2] * f0, ov[4 * j + 3] * f1);
        }
        const int m = lane >> 3, cl = L + 8 * (m & 1);
        const uint32_t base = dst + (uint32_t)(cl >> 6) * pstride;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const int tok = 8 * (j + (m >> 1)) + (lane & 7);
            stmatrix_x4_trans(base + sw128_off(tok, cl & 63), pk[2 * j], pk[2 * j + 1], pk[2 * j + 2], pk[2 * j + 3]);
        }
    };
    // Z -> [t][dv] (R1's place); dR -> rows 0-63 of RO; -gamma beta dR -> rows 0-63 of RS
    tstore(TM_Z, sbase + OFF_ZR, 8192, [](int) { return 1.f; });
    tstore(TM_DR, sbase + OFF_RO, 16384, [](int) { return 1.f; });
    tstore(TM_DR, sbase + OFF_RS, 16384, [&](int t) { return -g_gam[t] * g_beta[t]; });
    // gamma dO -> rows 64-127 of RS (from rows 64-127 of RO)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int u = tid + kNT * r, pnl = u >> 9;
        const uint32_t off = (uint32_t)(u & 511) << 4;
        float f[8];
        unpack8h(*reinterpret_cast<const uint4 *>(sm + OFF_RO + pnl * 16384 + 8192 + off), f);
        const float gt = g_gam[off >> 7];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= gt;
        *reinterpret_cast<uint4 *>(sm + OFF_RS + pnl * 16384 + 8192 + off) = pack8hp(f);
    }
    // sum_v dR R (dbeta, second term; row = d_v, 32 tokens from 32 hf)
    {
        float dr[32], rr[32];
        tmem_ld32(tl + TM_DR + 32 * hf, dr);
        tmem_ld32(tl + TM_A + 32 * hf, rr);
        tmem_ld_wait();
        float pr[32];
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) pr[cc] = dr[cc] * rr[cc];
        red[warp][32 * hf + lane] = warp_sum32(pr);       // token 32 hf + lane
    }
    sync_mma();
    if (tid < kC) {                                    // sum over the four lane quarters of the half
        const int hh = tid >> 5;
        s_db[tid] = (red[4 * hh][tid] + red[4 * hh + 1][tid]) + (red[4 * hh + 2][tid] + red[4 * hh + 3][tid]);
    }
    // D5 = [dR; dO] Z^T (lanes: dR rows | dO rows), D6 = S^T [-gamma beta dR; gamma dO]^T,
    // D7 = dS^T Z^T (lanes: d_k)
    if (issuer) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_G, smem_desc(sbase + OFF_RO + ko, 16, 1024),
                      smem_desc(sbase + OFF_ZR + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                      idesc_f16(128, 64, false, false), k > 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_D6, smem_desc(sbase + OFF_SB + k * 2048, 16384, 1024),
                      smem_desc(sbase + OFF_RS + ko, 16, 1024), idesc_f16(128, 128, true, false), k > 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            umma_bf16(tm + TM_A, smem_desc(sbase + OFF_DSB + k * 2048, 16384, 1024),
                      smem_desc(sbase + OFF_ZR + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                      idesc_f16(128, 64, true, false), k > 0);
    }
    commit_wait();

    // ---------------------------------------- dA, dP: E = dP * P + dM * M, H * dM, H * dP
    float *E = reinterpret_cast<float *>(sm + OFF_RO);  // [64][LA] fp32 (RO is consumed)
    {
        float d5[32];
        tmem_ld32(tl + TM_G + 32 * hf, d5);
        tmem_ld_wait();
        const bool arow = q4 < 2;
        const int t = 32 * (arow ? q4 : q4 - 2) + lane;
        uint8_t *mp = sm + OFF_MP + (arow ? 0 : 8192);
        float mv[32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            float f[8];
            unpack8h(*reinterpret_cast<const uint4 *>(mp + sw128_off(t, 32 * hf + 8 * ch)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) mv[8 * ch + e] = f[e];
        }
        float hd[32], ev[32], dam = 0.f;
        const float bt = g_beta[t];
        float hf32[32];
        hrow(t, hf32);
        // A rows: dA = -(dR Z^T) strictly lower, dM = beta dA;  P rows: dP = dO Z^T, lower.
        // One loop for both (warp-uniform lim and f): x = the kept D5 entry, dM | dP = f x.
        const int lim = arow ? t : t + 1;
        const float f = arow ? -bt : 1.f;
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) {
            const int i = 32 * hf + cc;
            const float x = i < lim ? d5[cc] : 0.f;
            dam = fmaf(x, mv[cc], dam);                   // -rowsum(dA * M) on A rows
            const float dm = f * x;
            ev[cc] = dm * mv[cc];
            hd[cc] = (i <= t ? hf32[cc] : 0.f) * dm;
        }
        dam = -dam;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)                    // H * dM | H * dP over M | P
            *reinterpret_cast<uint4 *>(mp + sw128_off(t, 32 * hf + 8 * ch)) = pack8hp(hd + 8 * ch);
        float *er = E + t * LA + 32 * hf;
        if (!arow)
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *reinterpret_cast<float4 *>(er + 4 * c4) = make_float4(ev[4 * c4], ev[4 * c4 + 1], ev[4 * c4 + 2], ev[4 * c4 + 3]);
        __syncthreads();
        if (arow) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                float4 x = *reinterpret_cast<const float4 *>(er + 4 * c4);
                x.x += ev[4 * c4]; x.y += ev[4 * c4 + 1]; x.z += ev[4 * c4 + 2]; x.w += ev[4 * c4 + 3];
                *reinterpret_cast<float4 *>(er + 4 * c4) = x;
            }
            red[warp][t] = dam;                           // rowsum(dA * M) of this column half
        }
    }
    // row sums of D6 (the un-masked parts) against X and Q: X . aX^T + Q . aQ^T per token
    float D6x[64];                                        // this thread's half of D6: aX^T (hf 0) | aQ^T (hf 1)
    {
        tmem_ld32(tl + TM_D6 + 64 * hf, *reinterpret_cast<float(*)[32]>(D6x));
        tmem_ld32(tl + TM_D6 + 64 * hf + 32, *reinterpret_cast<float(*)[32]>(D6x + 32));
        tmem_ld_wait();
    }
    sync_mma();                                           // H*dM, H*dP and E written; red[] for dA*M
    if (tid < kC) {                                       // dbeta = rowsum(dA * M) + sum_v dR R
        s_db[tid] += red[tid >> 5][tid] + red[4 + (tid >> 5)][tid];
        float re = 0.f, ce = 0.f;
#pragma unroll 8
        for (int i = 0; i < kC; ++i) {
            re += E[tid * LA + i];
            ce += E[i * LA + tid];
        }
        s_dl[tid] = re - ce;                              // rowsum(E) - colsum(E)
    }
    {
        const int jp = row >> 6, jc = row & 63;           // this thread's d_k column j = row
        float pr[64];
#pragma unroll
        for (int t = 0; t < kC; ++t) {
            const uint32_t o = jp * 16384 + sw128_off(t, jc);
            const float xv = __half2float(*reinterpret_cast<const __half *>(sm + OFF_XQ + o + (hf ? 8192 : 0)));
            pr[t] = xv * D6x[t];                          // X[t][j] aX^T[j][t]  or  Q[t][j] aQ^T[j][t]
        }
        const float2 s2 = warp_sum64(pr);
        __syncthreads();                                  // red[] reads above are done
        red[warp][2 * lane] = s2.x;
        red[warp][2 * lane + 1] = s2.y;
    }
    // dX^T, dQ^T: D6 += K^T [H*dM; H*dP]^T;  D8 = [X; Q]^T [H*dM; H*dP] (into B)
    if (issuer) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16(tm + TM_D6, smem_desc(sbase + OFF_K + k * 2048, 8192, 1024),
                      smem_desc(sbase + OFF_MP + k * 32, 16, 1024), idesc_f16(128, 128, true, false), 1);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            umma_bf16(tm + TM_B, smem_desc(sbase + OFF_XQ + k * 2048, 16384, 1024),
                      smem_desc(sbase + OFF_MP + k * 2048, 8192, 1024), idesc_f16(128, 64, true, true), k > 0);
    }
    sync_mma();                                           // red[] of the row sums complete
    if (tid < kC) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w][tid];
        s_dl[tid] += s;                                   // + rowsum(dO * QS) + rowsum(dXS * XS)
    }
    commit_wait();
    __syncthreads();                                      // red[] is read above before it is refilled

    // ------------------------------------------------------ dq, dk, dlambda, w z
    {
        const int j = row, jp = j >> 6, jc = j & 63;
        // one loop for both halves (warp-uniform operands):
        //   hf 0: dK^T = w (Z dS)^T + D8 + dX^T,   row-sum term w_t K[t][j] (Z dS)[t][j]
        //   hf 1: dQ^T = lambda dX^T + dQ^T',       row-sum term dX[t][j] Q[t][j]
        // with a = (Z dS)^T (D7) or dX^T, b = D8 + dX^T or dQ^T' (D6 without lambda dX^T)
        const bool kside = hf == 0;
        float a[64], bb[64];
        tmem_ld32(tl + (kside ? TM_A : TM_D6), *reinterpret_cast<float(*)[32]>(a));
        tmem_ld32(tl + (kside ? TM_A : TM_D6) + 32, *reinterpret_cast<float(*)[32]>(a + 32));
        tmem_ld32(tl + (kside ? TM_B : TM_D6 + 64), *reinterpret_cast<float(*)[32]>(bb));
        tmem_ld32(tl + (kside ? TM_B : TM_D6 + 64) + 32, *reinterpret_cast<float(*)[32]>(bb + 32));
        tmem_ld_wait();
        if (kside) {
            float dx[64];
            tmem_ld32(tl + TM_D6, *reinterpret_cast<float(*)[32]>(dx));
            tmem_ld32(tl + TM_D6 + 32, *reinterpret_cast<float(*)[32]>(dx + 32));
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < kC; ++t) bb[t] += dx[t];
        }
        const float *cf = kside ? g_w : g_lam;
        const uint8_t *tile = kside ? sm + OFF_K + jp * 8192 : sm + OFF_XQ + jp * 16384 + 8192;
        float ps[64], dd[64];                             // the row-sum terms; dK^T or dQ^T
#pragma unroll
        for (int t = 0; t < kC; ++t) {
            const float m = __half2float(*reinterpret_cast<const __half *>(tile + sw128_off(t, jc)));
            const float c = cf[t];
            ps[t] = (kside ? c * m : m) * a[t];
            dd[t] = fmaf(c, a[t], bb[t]);
        }
        {
            const float2 s2 = warp_sum64(ps);
            red[warp][2 * lane] = s2.x;
            red[warp][2 * lane + 1] = s2.y;
        }
        // dk (hf 0) or dq (hf 1) column j: fp32 straight to global memory, bf16 into a
        // [t][dk] tile (Sb's place: dk panels, then dq panels) for the TMA store
        if (p.grad_f32) {                                 // token t at dst + t H kD
            float *dst = static_cast<float *>(hf ? p.dq : p.dk) + tok_of(0) * kD + j;
            const int step = H * kD;
#pragma unroll
            for (int t = 0; t < kC; ++t)
                if (t < n) dst[t * step] = dd[t];
        } else {
            uint8_t *st = sm + OFF_SB + (hf ? 16384 : 0) + jp * 8192;
#pragma unroll
            for (int t = 0; t < kC; ++t)
                *reinterpret_cast<__nv_bfloat16 *>(st + sw128_off(t, jc)) = __float2bfloat16_rn(dd[t]);
        }
    }
    // dV = diag(beta) dR (row = d_v, 32 tokens from 32 hf; always bf16) -> [t][dv] tile in dSb's place
    {
        float dr[32];
        tmem_ld32(tl + TM_DR + 32 * hf, dr);
        tmem_ld_wait();
        uint8_t *st = sm + OFF_DSB + (row >> 6) * 8192;
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) {
            const int t = 32 * hf + cc;
            *reinterpret_cast<__nv_bfloat16 *>(st + sw128_off(t, row & 63)) = __float2bfloat16_rn(g_beta[t] * dr[cc]);
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (issuer && !abort_flag) {                          // rows past T are clipped by the copies
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
            tma_store_4d(&tmDV, sm + OFF_DSB + pnl * 8192, 64 * pnl, h, c0, b);
            if (!p.grad_f32) {
                tma_store_4d(&tmDK, sm + OFF_SB + pnl * 8192, 64 * pnl, h, c0, b);
                tma_store_4d(&tmDQ, sm + OFF_SB + 16384 + pnl * 8192, 64 * pnl, h, c0, b);
            }
        }
        tma_store_commit();
    }
    // gate gradients: dlambda = rowsum(dX * Q); dl = (row sums) - w z (+ the last token's
    // gamma_C <dS, S> + sum w z); d log alpha its suffix sum; dalpha = d log alpha / alpha
    if (warp == 0) {
        float wz2[2], dl2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = 2 * lane + u;
            const float wzt = (red[0][t] + red[1][t]) + (red[2][t] + red[3][t]);
            const float dlam = (red[4][t] + red[5][t]) + (red[6][t] + red[7][t]);
            wz2[u] = wzt;
            dl2[u] = s_dl[t] - wzt;
            if (t < n) {
                const size_t tok = tok_of(t);
                if (p.lam && p.dlam) {
                    if (p.grad_f32) static_cast<float *>(p.dlam)[tok] = dlam;
                    else static_cast<__nv_bfloat16 *>(p.dlam)[tok] = __float2bfloat16_rn(dlam);
                }
                const float db = s_db[t];
                if (p.grad_f32) static_cast<float *>(p.dbeta)[tok] = db;
                else static_cast<__nv_bfloat16 *>(p.dbeta)[tok] = __float2bfloat16_rn(db);
            }
        }
        float wsum = wz2[0] + wz2[1];
#pragma unroll
        for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
        if (lane == 31) {
            float dot = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) dot += sdot[w];
            dl2[1] += g_gam[kC - 1] * dot + wsum;
        }
        float s = dl2[0] + dl2[1];                        // suffix sums within the chunk
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, s, off);
            if (lane + off < 32) s += y;
        }
        const float sl[2] = {s, s - dl2[0]};
        if (p.alpha && p.dalpha)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 2 * lane + u;
                if (t < n) {
                    const float da = sl[u] / __expf(g_la[t]);
                    const size_t tok = tok_of(t);
                    if (p.grad_f32) static_cast<float *>(p.dalpha)[tok] = da;
                    else static_cast<__nv_bfloat16 *>(p.dalpha)[tok] = __float2bfloat16_rn(da);
                }
            }
    }

    if (abort_flag) {
        if (issuer) {
            mbar_wait(&bar_ld, 0, kWaitNs);
            umma_commit(&bar_drain);
            mbar_wait(&bar_drain, 0, kWaitNs);
        }
        if (lane == 0) atomicExch(&g_grad_tc_timeout, 1u);
    }
    if (issuer) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
    (void)ok;
}

}  // namespace

cudaError_t launch_qdelta_bwd_grad_tc(const QDeltaBwdArgs &a, cudaStream_t s) {
    CUtensorMap mq, mk, mv, md, mdq, mdk, mdv;
    if (!make_token_map(&mq, a.q, a.B, a.T, a.H) || !make_token_map(&mk, a.k, a.B, a.T, a.H) ||
        !make_token_map(&mv, a.v, a.B, a.T, a.H) || !make_token_map(&md, a.dO, a.B, a.T, a.H) ||
        !make_token_map(&mdv, a.dv, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    if (a.grad_f32) {                                 // dq, dk fp32: written directly, maps unused
        mdq = mq;
        mdk = mk;
    } else if (!make_token_map(&mdq, a.dq, a.B, a.T, a.H) || !make_token_map(&mdk, a.dk, a.B, a.T, a.H)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(qdelta_bwd_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int nchunks = (a.T + kC - 1) / kC;
    GradTcParams p{a.alpha, a.beta, a.lam, reinterpret_cast<const uint8_t *>(a.S_chk),
                   reinterpret_cast<const uint8_t *>(a.dS_chk), a.dq, a.dk, a.dv, a.dalpha, a.dbeta, a.dlam,
                   a.B, a.T, a.H, a.grad_f32, a.gates_f32};
    qdelta_bwd_grad_tc_kernel<<<(unsigned)(a.B * a.H * nchunks), kNT, kSmemBytes, s>>>(p, mq, mk, mv, md, mdq, mdk, mdv);
    return cudaGetLastError();
}

bool grad_tc_read_and_clear_timeout() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_grad_tc_timeout, sizeof v) != cudaSuccess) return false;
    if (v) cudaMemcpyToSymbol(g_grad_tc_timeout, &zero, sizeof zero);
    return v != 0;
}

}  // namespace qd

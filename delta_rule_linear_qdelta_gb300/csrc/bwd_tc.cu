// Reverse state-gradient sweep of the Q-Delta backward on the sm_103a tensor cores
// (tcgen05 + TMEM + TMA): bf16 inputs, dk = dv = 128, chunk C = 64.  One CTA of 12
// warps per (b, h) carries the gradient of the state, dS ([dv][dk] fp32), on chip
// from the last chunk to the first.
//
// Per chunk, in reverse ("Q-Delta: Beyond Key-Value Associative State Evolution",
// Sec. 3.3.2; the adjoint of the WY form the forward runs, the single solve
// T = (I + A)^{-1}), with l_i = sum_{j<=i} log alpha_j, gamma_i = e^{l_i},
// kappa_i = e^{l_C - l_i}, X = K + diag(lambda) Q:
//   A  = strictly_lower(beta_t e^{l_t - l_i} (X K^T)_ti),  P = incl_lower(e^{l_t - l_i} (Q K^T)_ti)
//   dZ^T  = dS (kappa K)^T + dO^T P                    (d_v x 64)
//   dRs^T = dZ^T T diag(beta gamma)                    (= (diag(gamma beta) T^T dZ)^T)
//   dS   <- gamma_C dS + dO^T (gamma Q) - dRs^T X
// and dS as it enters each chunk (the gradient reaching the state that leaves it) is
// written to the backward's checkpoint array, as an fp16 tile in the layout of a
// 128-byte-swizzled MMA operand (chk_tile_off, the format of the forward's state
// checkpoints); after the first chunk it is dS0 (fp32).
//
// The layout follows the forward kernel (chunk_tc.cu): every product has M = 128 with
// the TMEM lanes indexing d_v; a prep group (warps 0-7) does each chunk's
// state-independent work -- X, the Gram [X; Q] K^T, the masks, the inverse (with the
// column scaling beta gamma folded in), kappa K and gamma Q in place -- one chunk ahead
// of a chain group (warps 8-11) that carries dS: its bf16 copy (the A operand of
// dS (kappa K)^T) and the packed bf16 dZ^T and -dRs^T live in TMEM, the fp32 master
// accumulates the two update products after the epilogue has scaled it by the next
// chunk's gamma_C.
//   ready       prep -> chain: P(c), T2(c) and the scaled tiles of chunk c are in place
//   taken       chain -> prep: the chain has passed `ready` of index i, so `ready` may
//               complete its next phase
//   cdone[i&1]  chain -> prep: the products of chunk i have run, so its stage, P and T2
//               buffers are free (the chain then loads chunk i+2 into the stage)
//
// Shared memory (offsets from a 1024-aligned base):
//   stage s in {0,1}: XQ 32 KB (per 64-column panel: X rows 0-63 | Q rows 64-127),
//                     K 16 KB (scaled to kappa K), dO 16 KB
//   R1 17 KB (A fp32 [64][68], the solve's intermediate blocks), Y 4.5 KB (solve scratch),
//   P 2x8 KB (bf16 [64][64] by chunk parity), T2 2x8 KB (bf16 T diag(beta gamma) by parity;
//   zero above the 8x8 diagonal blocks)
// TMEM (512 columns allocated): G 0-63, dZ^T 64-127 (packed bf16 in its first 32),
// dRs^T 128-191 (packed -dRs^T in its first 32), bf16 dS 192-255, fp32 dS 256-383.
//
// Every wait is bounded; on a timeout the kernel sets its error word, waits (bounded)
// for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "qd_internal.cuh"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace qd {

__device__ unsigned int g_bwd_tc_timeout = 0;

namespace {

using namespace ptx;
using namespace tc;

constexpr int kPrepThreads = kThreads;              // warps 0-7
constexpr int kChainThreads = 128;                  // warps 8-11
constexpr int kAllThreads = kPrepThreads + kChainThreads;
constexpr int kBarPrep = 1, kBarChain = 2;
constexpr uint32_t kStageBytes = 65536;
constexpr uint32_t OFF_XQ = 0, OFF_K = 32768, OFF_DO = 49152;   // within a stage
constexpr uint32_t OFF_R1 = 2 * kStageBytes;         // 131072
constexpr uint32_t OFF_Y = OFF_R1 + 17408;           // 148480
constexpr uint32_t OFF_P = 153600;                   // two 8 KB tiles
constexpr uint32_t OFF_T = OFF_P + 16384;            // 169984: two 8 KB tiles
constexpr uint32_t kSmemUsed = OFF_T + 16384;        // 186368
static_assert(OFF_P >= OFF_Y + 32 * LY * 4 && OFF_P % 1024 == 0 && OFF_T % 1024 == 0, "tile placement");
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
constexpr uint32_t kTmaBytes = 3 * kC * kD * 2;      // Q, K, dO tiles per chunk
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t TM_G = 0, TM_DZ = 64, TM_DR = 128, TM_SB = 192, TM_S = 256;

struct BwdTcParams {
    const void *alpha, *beta, *lam;
    const float *dS_final;
    uint8_t *dS_chk;                                  // fp16 checkpoint tiles (chk_tile_off)
    float *dS0;
    int B, T, H;
    int gates_f32;
};

__global__ void __launch_bounds__(kAllThreads, 1)
qdelta_bwd_dstate_tc_kernel(const BwdTcParams p, const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmD) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_full[2], bar_g, bar_z, bar_r, bar_s, bar_ready, bar_taken, bar_cdone[2], bar_drain[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    // per-chunk gate arrays by loop index mod 4 (the chain reads the next chunk's
    // gamma_C in its epilogue while the prep builds the one after)
    __shared__ __align__(16) float g_ell[4][kC], g_beta[4][kC], g_lam[4][kC], g_gam[4][kC], g_kap[4][kC],
        g_igam[4][kC], g_bg[4][kC];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool prep = tid < kPrepThreads;
    const int q4 = warp & 3, hf = (warp >> 2) & 1;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int T = p.T, H = p.H;
    const int nchunks = (T + kC - 1) / kC;
    const bool p_issuer = (tid == 32), c_issuer = (tid == kPrepThreads);
    const int d_row = 32 * q4 + lane;
    auto chunk_of = [&](int i) { return nchunks - 1 - i; };   // loop index -> chunk, last first

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_z, 1);
        mbar_init(&bar_r, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_ready, 1);
        mbar_init(&bar_taken, 1);
        mbar_init(&bar_cdone[0], 1);
        mbar_init(&bar_cdone[1], 1);
        mbar_init(&bar_drain[0], 1);
        mbar_init(&bar_drain[1], 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    for (int i = tid; i < 16384 / 16; i += kAllThreads)   // T2 tiles: zeros above the diagonal blocks
        reinterpret_cast<uint4 *>(sm + OFF_T)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();

    auto issue_loads = [&](int i) {
        const int s = i & 1, t0 = chunk_of(i) * kC;
        uint8_t *st = sm + s * kStageBytes;
        mbar_arrive_expect_tx(&bar_full[s], kTmaBytes);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
            tma_load_4d(st + OFF_XQ + pnl * 16384 + 8192, &tmQ, &bar_full[s], 64 * pnl, h, t0, b);
            tma_load_4d(st + OFF_K + pnl * 8192, &tmK, &bar_full[s], 64 * pnl, h, t0, b);
            tma_load_4d(st + OFF_DO + pnl * 8192, &tmD, &bar_full[s], 64 * pnl, h, t0, b);
        }
    };
    // gates of loop index i's chunk: lane l of warp 4 takes tokens 2l and 2l+1
    float ra[2], rb[2], rl[2];
    auto load_gates = [&](int i) {
        const int c = chunk_of(i);
        const void *pa = opaque(p.alpha), *pl = opaque(p.lam);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = min(c * kC + 2 * lane + u, T - 1);
            const size_t tok = ((size_t)b * T + t) * H + h;
            ra[u] = pa ? gate_val<__nv_bfloat16>(pa, tok, p.gates_f32) : 1.f;
            rb[u] = gate_val<__nv_bfloat16>(p.beta, tok, p.gates_f32);
            rl[u] = pl ? gate_val<__nv_bfloat16>(pl, tok, p.gates_f32) : 0.f;
        }
    };
    auto compute_gates = [&](int i) {
        const int buf = i & 3, c = chunk_of(i);
        float la[2], gb[2], gl[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {                  // tokens past T: alpha 1, beta 0, lambda 0
            const bool ok = c * kC + 2 * lane + u < T;
            la[u] = ok ? __logf(ra[u]) : 0.f;
            gb[u] = ok ? rb[u] : 0.f;
            gl[u] = ok ? rl[u] : 0.f;
        }
        float sum = la[0] + la[1];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, sum, off);
            if (lane >= off) sum += n;
        }
        const float e1 = sum, e0 = sum - la[1];
        const float eC = __shfl_sync(0xffffffffu, sum, 31);
        const float g0 = __expf(e0), g1 = __expf(e1);
        g_ell[buf][2 * lane] = e0;
        g_ell[buf][2 * lane + 1] = e1;
        g_beta[buf][2 * lane] = gb[0];
        g_beta[buf][2 * lane + 1] = gb[1];
        g_lam[buf][2 * lane] = gl[0];
        g_lam[buf][2 * lane + 1] = gl[1];
        g_gam[buf][2 * lane] = g0;
        g_gam[buf][2 * lane + 1] = g1;
        g_kap[buf][2 * lane] = __expf(eC - e0);
        g_kap[buf][2 * lane + 1] = __expf(eC - e1);
        g_igam[buf][2 * lane] = eC > -80.f ? __expf(-e0) : 0.f;
        g_igam[buf][2 * lane + 1] = eC > -80.f ? __expf(-e1) : 0.f;
        g_bg[buf][2 * lane] = gb[0] * g0;
        g_bg[buf][2 * lane + 1] = gb[1] * g1;
    };

    if (tid == 0) {
        issue_loads(0);
        if (nchunks > 1) issue_loads(1);
    }
    if (warp == 4) {
        load_gates(0);
        compute_gates(0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);

    bool ok = true;
    auto wait_on = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_wait(bar, parity, kWaitNs)) { ok = false; abort_flag = 1; }
    };
    auto wait_mma = [&](uint64_t *bar, int i) {
        wait_on(bar, (uint32_t)(i & 1));
        tc_fence_after();
    };
    auto psync = [&]() {
        fence_proxy_async();
        tc_fence_before();
        named_sync(kBarPrep, kPrepThreads);
        tc_fence_after();
    };
    auto csync = [&]() {
        fence_proxy_async();
        tc_fence_before();
        named_sync(kBarChain, kChainThreads);
        tc_fence_after();
    };
    const uint32_t sbase = smem_u32(sm);
    auto stage_addr = [&](int i) { return sbase + (uint32_t)(i & 1) * kStageBytes; };

    // ---------------------------------------------------------------- prep group
    // X = K + lambda Q into rows 0-63 of the XQ panels (before K and Q are scaled)
    auto x_pass = [&](int i) {
        uint8_t *st = sm + (i & 1) * kStageBytes;
        const float *lam = g_lam[i & 3];
        uint4 kr[4], qr[4];
        float lm[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int u = tid + kPrepThreads * r;
            const int pnl = u >> 9;
            const uint32_t off = (uint32_t)(u & 511) << 4;
            kr[r] = *reinterpret_cast<const uint4 *>(st + OFF_K + pnl * 8192 + off);
            qr[r] = *reinterpret_cast<const uint4 *>(st + OFF_XQ + pnl * 16384 + 8192 + off);
            lm[r] = lam[off >> 7];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int u = tid + kPrepThreads * r;
            const int pnl = u >> 9;
            const uint32_t off = (uint32_t)(u & 511) << 4;
            float kf[8], qf[8], xf[8];
            unpack8(kr[r], kf);
            unpack8(qr[r], qf);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 x = ffma2(make_float2(lm[r], lm[r]), make_float2(qf[e], qf[e + 1]),
                                       make_float2(kf[e], kf[e + 1]));
                xf[e] = x.x;
                xf[e + 1] = x.y;
            }
            *reinterpret_cast<uint4 *>(st + OFF_XQ + pnl * 16384 + off) = pack8(xf);
        }
    };
    // G = [X; Q] K^T
    auto issue_gram = [&](int i) {
        if (!p_issuer) return;
        const uint32_t sXQ = stage_addr(i) + OFF_XQ, sK = stage_addr(i) + OFF_K;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_G, smem_desc(sXQ + ko, 16, 1024), smem_desc(sK + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                      idesc_bf16(128, 64, false, false), k > 0);
        }
        umma_commit(&bar_g);
    };
    // A (fp32, R1): A_ti = beta_t e^{l_t - l_i} (X K^T)_ti for i < t; P (bf16, P[i&1]):
    // P_ti = e^{l_t - l_i} (Q K^T)_ti for i <= t.  While l_C > -80 the decay factors as
    // gamma_t e^{-l_i}; otherwise each factor is its own exponential.
    auto masks = [&](int i) {
        const int gi = i & 3;
        const float *ell = g_ell[gi], *bet = g_beta[gi], *gam = g_gam[gi], *igam = g_igam[gi];
        float g[32];
        tmem_ld32(tl + TM_G + 32 * hf, g);
        tmem_ld_wait();
        const bool split = ell[kC - 1] > -80.f;
        const bool arow = q4 < 2;
        const int t = 32 * (arow ? q4 : q4 - 2) + lane;
        const int lim = arow ? t : t + 1;
        if (split) {
            const float r = arow ? bet[t] * gam[t] : gam[t];
            float fi[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(igam + 32 * hf + j);
                fi[j] = v.x; fi[j + 1] = v.y; fi[j + 2] = v.z; fi[j + 3] = v.w;
            }
#pragma unroll
            for (int cc = 0; cc < 32; cc += 2) {
                const float2 x = fmul2(fmul2(make_float2(r, r), make_float2(fi[cc], fi[cc + 1])),
                                       make_float2(g[cc], g[cc + 1]));
                g[cc] = (32 * hf + cc < lim) ? x.x : 0.f;
                g[cc + 1] = (32 * hf + cc + 1 < lim) ? x.y : 0.f;
            }
        } else {
            const float r = arow ? bet[t] : 1.f, lt = ell[t];
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
                g[cc] = (32 * hf + cc < lim) ? r * __expf(lt - ell[32 * hf + cc]) * g[cc] : 0.f;
        }
        if (arow) {
            float *Arow = reinterpret_cast<float *>(sm + OFF_R1) + t * LA + 32 * hf;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *reinterpret_cast<float4 *>(Arow + 4 * c4) = make_float4(g[4 * c4], g[4 * c4 + 1], g[4 * c4 + 2], g[4 * c4 + 3]);
        } else {
            uint8_t *P = sm + OFF_P + (i & 1) * 8192;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                *reinterpret_cast<uint4 *>(P + sw128_off(t, 32 * hf + 8 * ch)) = pack8p(g + 8 * ch);
        }
    };
    // K -> kappa K, Q -> gamma Q in place (the Gram and X have read them)
    auto scale_kq = [&](int i) {
        uint8_t *st = sm + (i & 1) * kStageBytes;
        const float *kap = g_kap[i & 3], *gam = g_gam[i & 3];
        uint4 kr[4], qr[4];
        float fk[4], fq[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {                     // all loads first
            const int u = tid + kPrepThreads * r;
            const int pnl = u >> 9;
            const uint32_t off = (uint32_t)(u & 511) << 4;
            kr[r] = *reinterpret_cast<const uint4 *>(st + OFF_K + pnl * 8192 + off);
            qr[r] = *reinterpret_cast<const uint4 *>(st + OFF_XQ + pnl * 16384 + 8192 + off);
            fk[r] = kap[off >> 7];
            fq[r] = gam[off >> 7];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int u = tid + kPrepThreads * r;
            const int pnl = u >> 9;
            const uint32_t off = (uint32_t)(u & 511) << 4;
            float kf[8], qf[8];
            unpack8(kr[r], kf);
            unpack8(qr[r], qf);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 a = fmul2(make_float2(kf[e], kf[e + 1]), make_float2(fk[r], fk[r]));
                const float2 c2 = fmul2(make_float2(qf[e], qf[e + 1]), make_float2(fq[r], fq[r]));
                kf[e] = a.x; kf[e + 1] = a.y;
                qf[e] = c2.x; qf[e + 1] = c2.y;
            }
            *reinterpret_cast<uint4 *>(st + OFF_K + pnl * 8192 + off) = pack8(kf);
            *reinterpret_cast<uint4 *>(st + OFF_XQ + pnl * 16384 + 8192 + off) = pack8(qf);
        }
    };
    // T2 = (I + A)^{-1} diag(beta gamma) into T2[i&1]; warp 4 meanwhile builds the next
    // chunk's gate arrays
    auto solve = [&](int i) {
        const int gi = i & 3;
        unit_lower_inverse<false>(reinterpret_cast<float *>(sm + OFF_R1), reinterpret_cast<float *>(sm + OFF_Y),
                                  sm + OFF_T + (i & 1) * 8192, nullptr, g_bg[gi], nullptr,
                                  [&]() { if (warp == 4 && i + 1 < nchunks) compute_gates(i + 1); },
                                  []() { named_sync(kBarPrep, kPrepThreads); });
    };

    // --------------------------------------------------------------- chain group
    // dZ^T = dS (kappa K)^T + dO^T P  into TM_DZ
    auto issue_dz = [&](int i) {
        if (!c_issuer) return;
        const uint32_t sK = stage_addr(i) + OFF_K, sD = stage_addr(i) + OFF_DO;
        const uint32_t sP = sbase + OFF_P + (uint32_t)(i & 1) * 8192;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            umma_bf16_ta(tm + TM_DZ, tm + TM_SB + 8 * k, smem_desc(sK + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                         idesc_bf16(128, 64, false, false), k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16(tm + TM_DZ, smem_desc(sD + k * 2048, 8192, 1024), smem_desc(sP + k * 2048, 8192, 1024),
                      idesc_bf16(128, 64, true, true), 1);
        umma_commit(&bar_z);
    };
    // 64 fp32 columns at `col` of this thread's lane -> 32 packed bf16 pairs at `col`
    // (negated when neg)
    auto pack64 = [&](uint32_t col, bool neg) {
        float z[64];
        tmem_ld32(tl + col, *reinterpret_cast<float(*)[32]>(z));
        tmem_ld32(tl + col + 32, *reinterpret_cast<float(*)[32]>(z + 32));
        tmem_ld_wait();
        uint32_t zp[32];
        const uint32_t flip = neg ? 0x80008000u : 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) zp[j] = pack_bf16x2(z[2 * j], z[2 * j + 1]) ^ flip;
        tmem_st32(tl + col, zp);
        tmem_st_wait();
    };
    // dRs^T = dZ^T T2  into TM_DR; A = the packed dZ^T
    auto issue_dr = [&](int i) {
        if (!c_issuer) return;
        const uint32_t sT = sbase + OFF_T + (uint32_t)(i & 1) * 8192;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16_ta(tm + TM_DR, tm + TM_DZ + 8 * k, smem_desc(sT + k * 2048, 8192, 1024),
                         idesc_bf16(128, 64, false, true), k > 0);
        umma_commit(&bar_r);
    };
    // dS += dO^T (gamma Q) + (-dRs^T) X   (dS in TMEM already scaled by gamma_C)
    auto issue_ds = [&](int i) {
        if (!c_issuer) return;
        const uint32_t sXQ = stage_addr(i) + OFF_XQ, sD = stage_addr(i) + OFF_DO;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16(tm + TM_S, smem_desc(sD + k * 2048, 8192, 1024), smem_desc(sXQ + 8192 + k * 2048, 16384, 1024),
                      idesc_bf16(128, 128, true, true), 1);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16_ta(tm + TM_S, tm + TM_DR + 8 * k, smem_desc(sXQ + k * 2048, 16384, 1024),
                         idesc_bf16(128, 128, false, true), 1);
        umma_commit(&bar_s);
    };
    // dS of this thread's row -> dst32 (an fp32 row) or dst16 (a checkpoint tile, fp16), its
    // bf16 copy into TM_SB, and (unless last) the master scaled by g
    auto state_out = [&](float *dst32, uint8_t *dst16, float g, bool last, bool from_tmem, const float *src) {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            float sv[64];
            if (from_tmem) {
                tmem_ld32(tl + TM_S + 64 * half, *reinterpret_cast<float(*)[32]>(sv));
                tmem_ld32(tl + TM_S + 64 * half + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 v = src ? *reinterpret_cast<const float4 *>(src + 64 * half + j)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    sv[j] = v.x; sv[j + 1] = v.y; sv[j + 2] = v.z; sv[j + 3] = v.w;
                }
            }
            if (dst32 && !abort_flag)
#pragma unroll
                for (int j = 0; j < 64; j += 4)
                    *reinterpret_cast<float4 *>(dst32 + 64 * half + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
            if (dst16 && !abort_flag)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(dst16 + chk_tile_off(d_row, 64 * half + 8 * ch)) = pack8hp(sv + 8 * ch);
            if (!last) {
                uint32_t sp[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) sp[j] = pack_bf16x2(sv[2 * j], sv[2 * j + 1]);
                tmem_st32(tl + TM_SB + 32 * half, sp);
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 x = fmul2(make_float2(sv[e], sv[e + 1]), make_float2(g, g));
                    sv[e] = x.x;
                    sv[e + 1] = x.y;
                }
                tmem_st32(tl + TM_S + 64 * half, *reinterpret_cast<float(*)[32]>(sv));
                tmem_st32(tl + TM_S + 64 * half + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
            }
        }
        tmem_st_wait();
    };
    auto chk_tile = [&](int c) {                      // the checkpoint tile of chunk c
        return p.dS_chk + ((size_t)bh * nchunks + c) * kChkTileBytes;
    };

    int loads_issued = nchunks > 1 ? 2 : 1;
    if (prep) {
        wait_on(&bar_full[0], 0);
        x_pass(0);
        psync();
        issue_gram(0);
        for (int i = 0; i < nchunks; ++i) {
            if (warp == 4 && i + 1 < nchunks) load_gates(i + 1);   // arrays built in solve(i)
            wait_mma(&bar_g, i);
            if (i >= 2) {                                 // P, T2 and the stage of index i-2 are free
                wait_on(&bar_cdone[i & 1], (uint32_t)(((i - 2) >> 1) & 1));
                tc_fence_after();
            }
            masks(i);
            tc_fence_before();
            named_sync(kBarPrep, kPrepThreads);          // TM_G read, A in R1
            tc_fence_after();
            scale_kq(i);
            solve(i);
            psync();                                      // P, T2, kappa K, gamma Q in place
            tc_fence_before();
            const bool stop = named_sync_or(kBarPrep, kPrepThreads, abort_flag != 0);
            tc_fence_after();
            if (tid == 0) {
                if (i >= 1) wait_on(&bar_taken, (uint32_t)((i - 1) & 1));   // the chain has taken ready(i-1)
                mbar_arrive(&bar_ready);
            }
            if (stop) break;
            if (i + 1 < nchunks) {
                wait_on(&bar_full[(i + 1) & 1], (uint32_t)(((i + 1) >> 1) & 1));
                x_pass(i + 1);
                psync();
                issue_gram(i + 1);
            }
        }
    } else {
        // dS leaving the last chunk = dS_final: its checkpoint, bf16 copy, and the master
        // scaled by that chunk's gamma_C
        {
            const float *src = p.dS_final ? p.dS_final + ((size_t)bh * kD + d_row) * kD : nullptr;
            state_out(nullptr, chk_tile(nchunks - 1), g_gam[0][kC - 1], false, false, src);
        }
        csync();
        for (int i = 0; i < nchunks; ++i) {
            const bool last = (i + 1 == nchunks);
            wait_on(&bar_ready, (uint32_t)(i & 1));
            tc_fence_after();
            if (c_issuer) mbar_arrive(&bar_taken);
            issue_dz(i);
            wait_mma(&bar_z, i);
            pack64(TM_DZ, false);
            csync();
            issue_dr(i);
            wait_mma(&bar_r, i);
            pack64(TM_DR, true);
            csync();
            issue_ds(i);
            wait_mma(&bar_s, i);
            if (c_issuer) {
                mbar_arrive(&bar_cdone[i & 1]);
                if (i + 2 < nchunks) {                    // index i's stage is consumed
                    issue_loads(i + 2);
                    ++loads_issued;
                }
            }
            // dS entering chunk_of(i) = leaving chunk_of(i) - 1: its checkpoint (dS0 after
            // the first chunk) and the operands of the next index
            float *d0 = last && p.dS0 ? p.dS0 + ((size_t)bh * kD + d_row) * kD : nullptr;
            state_out(d0, last ? nullptr : chk_tile(chunk_of(i) - 1), last ? 1.f : g_gam[(i + 1) & 3][kC - 1], last,
                      true, nullptr);
            tc_fence_before();
            const bool stop = named_sync_or(kBarChain, kChainThreads, abort_flag != 0);
            tc_fence_after();
            if (stop) break;
        }
    }

    if (abort_flag) {
        if (c_issuer)
            for (int s = 0; s < 2; ++s) {
                const int n_s = (loads_issued + 1 - s) / 2;
                if (n_s > 0) mbar_wait(&bar_full[s], (uint32_t)((n_s - 1) & 1), kWaitNs);
            }
        if (p_issuer || c_issuer) {
            uint64_t *dr = &bar_drain[p_issuer ? 0 : 1];
            umma_commit(dr);
            mbar_wait(dr, 0, kWaitNs);
        }
        if (lane == 0) atomicExch(&g_bwd_tc_timeout, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

bool qdelta_bwd_tc_supported(const QDeltaBwdArgs &a, int dtype) {
    // the checkpoints come from the tensor-core forward (fp16 tiles): its conditions too
    return dtype == kBF16 && a.nk == kD && a.nv == kD && a.T > 0 && (long long)a.T * a.H * kD * 2 < (1ll << 40);
}

cudaError_t launch_qdelta_bwd_dstate_tc(const QDeltaBwdArgs &a, cudaStream_t s) {
    CUtensorMap mq, mk, md;
    if (!make_token_map(&mq, a.q, a.B, a.T, a.H) || !make_token_map(&mk, a.k, a.B, a.T, a.H) ||
        !make_token_map(&md, a.dO, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(qdelta_bwd_dstate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    BwdTcParams p{a.alpha, a.beta, a.lam, a.dS_final, reinterpret_cast<uint8_t *>(a.dS_chk), a.dS0, a.B, a.T, a.H, a.gates_f32};
    qdelta_bwd_dstate_tc_kernel<<<a.B * a.H, kAllThreads, kSmemBytes, s>>>(p, mq, mk, md);
    return cudaGetLastError();
}

bool bwd_tc_read_and_clear_timeout() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_tc_timeout, sizeof v) != cudaSuccess) return false;
    if (v) cudaMemcpyToSymbol(g_bwd_tc_timeout, &zero, sizeof zero);
    return v != 0;
}

}  // namespace qd

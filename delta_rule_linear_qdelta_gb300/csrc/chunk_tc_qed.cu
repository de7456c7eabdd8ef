// Fused chunked QED forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA),
// bf16 inputs, dk = dv = 128, chunk C = 64.  One CTA of 8 warps per (b, h) carries
// the fp32 state on chip across the chunks.
//
// Recurrence ("The Query Knows What to Forget", Sec. 2.1-2.2: GDN-2 update of
// Eqs. 4/8, erase vector of Eq. 6), with the state kept as S^ = S^T ([dv][dk]):
//   S^_t = S^_{t-1} D_t (I - a_t k_t^T) + (w_t * v_t) k_t^T,   o_t = S^_t q_t,
//   D_t = Diag(e^{g_t}),  a_t = b_t*k_t + lam_h (u_t - k_t (k_t^T u_t)),  u_t = b_t*q_t
//   (the ablation arms of Table 1 take u_t = q_t, u_t = q_t without the projection,
//   or u_t = b_t*z_h; see qd_internal.cuh).
// Per chunk, with the in-chunk cumulative log-decay G_t = sum_{j<=t} g_j (a vector
// over the dk channels, anchored at the chunk start):
//   Ae = A*e^G, Qe = Q*e^G, Ke = K*e^-G, Kd = K*e^{G_C - G}   (elementwise, per channel)
//   G  = [Ae; Qe] Ke^T                 -> At = strictly_lower, P = incl_lower
//   Tinv = (I + At)^{-1}
//   U^T = (W*V)^T Tinv^T,  W^T = Ae^T Tinv^T,  Z^T = U^T - S^ W^T
//   O^T = S^ Qe^T + Z^T P^T
//   S^ <- S^ diag(e^{G_C}) + Z^T Kd
// The factored decay stays in fp32 range while every channel's log-decay summed
// over one chunk is >= -80.
//
// The structure, operand layouts (128-byte swizzle, M = 128 products with the TMEM
// lanes indexing a head dimension) and the solve are those of the Q-Delta kernel
// in chunk_tc.cu.  Tiles are single-buffered; the next chunk's tiles are fetched in
// three groups as soon as the buffers they overwrite are consumed:
//   g, b, w after the erase-vector pass; Q, V after the U/W products; K after the
//   state product.
//
// Shared memory (offsets from a 1024-aligned base):
//   XQ 32 KB (per 64-column panel: Ae rows 0-63 | Q -> Qe rows 64-127)
//   K 16 KB (K -> Ke -> Kd), V 16 KB (V -> W*V), G 16 KB, Bt 16 KB, Wt 16 KB (g, b, w tiles)
//   S_in 32 KB bf16 state, R1 17 KB (At fp32, the solve's intermediate blocks), R2 16 KB
//   (scratch, -W, Z^T, O staging), P 8 KB, T 8 KB (Tinv bf16, zero above the diagonal
//   blocks).
// TMEM (512 columns): G 0-63, O1 64-127, U/Z 128-191, W 192-255, O2 256-319, S 320-447.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "qd_internal.cuh"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace qd {

__device__ unsigned int g_qed_tc_timeout = 0;

namespace {

using namespace ptx;
using namespace tc;

constexpr uint32_t OFF_XQ = 0, OFF_K = 32768, OFF_V = 49152, OFF_G = 65536, OFF_BT = 81920, OFF_WT = 98304;
constexpr uint32_t OFF_S = 114688;
constexpr uint32_t OFF_R1 = OFF_S + 32768;           // 147456
constexpr uint32_t OFF_R2 = OFF_R1 + 17408;          // 164864
constexpr uint32_t OFF_P = OFF_R2 + 16384;           // 181248
constexpr uint32_t OFF_T = OFF_P + 8192;             // 189440 (Tinv, bf16 [64][64])
constexpr uint32_t kSmemUsed = OFF_T + 8192;         // 197632
static_assert(OFF_R2 % 1024 == 0 && OFF_P % 1024 == 0 && OFF_T % 1024 == 0 && OFF_S % 1024 == 0,
              "128-byte-swizzled MMA operands start on 1024-byte boundaries");
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t TM_G = 0, TM_O1 = 64, TM_U = 128, TM_W = 192, TM_O2 = 256, TM_S = 320;

struct QedTcParams {
    const float *lam_h, *S0;
    float *S_final;
    int B, T, H;
    int flags;      // kTcNoV | kTcS0Identity | kTcNoO (segment-scan passes)
    int variant;    // kQed* ablation arm
    const float *z; // [H][128] for kQedRand
};

struct QedMaps {
    CUtensorMap q, k, v, o, g, b, w;
};

// element (t, j) of a [64][128] bf16 tile stored as two 64-column 128B-swizzled panels
__device__ __forceinline__ uint32_t tile_off(int t, int j, uint32_t panel_stride) {
    return (uint32_t)(j >> 6) * panel_stride + sw128_off(t, j & 63);
}

__global__ void __launch_bounds__(kThreads, 1)
qed_fwd_tc_kernel(const QedTcParams p, const __grid_constant__ QedMaps mp) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_gbw, bar_qv, bar_k, bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float g_ku[kC], g_ps[2][kD];
    __shared__ __align__(16) float g_ecg[kD];      // read as float2 pairs

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int T = p.T;
    const int nchunks = (T + kC - 1) / kC;
    const bool producer = (tid == 0), issuer = (tid == 32);
    const float lam_h = p.lam_h[h];
    const int d_row = 32 * q4 + lane;
    // the erase vector's new term (ablation arm): b gate kept, projection kept, z_h in place of q
    const bool gate = p.variant == kQedFull || p.variant == kQedRand;
    const bool proj = p.variant != kQedNogateNoproj;
    const float *zrow = p.variant == kQedRand ? p.z + (size_t)h * kD : nullptr;
    // flags of the segment-scan passes, read through opaque() inside the chunk loop
    const uint32_t flags = (uint32_t)p.flags;
    const bool s0_id = flags & kTcS0Identity;
    auto no_v = [&]() { return (opaque(flags) & kTcNoV) != 0; };
    auto no_o = [&]() { return (opaque(flags) & kTcNoO) != 0; };

    if (tid == 0) {
        mbar_init(&bar_gbw, 1);
        mbar_init(&bar_qv, 1);
        mbar_init(&bar_k, 1);
        mbar_init(&bar_mma, 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mp.q);
        tma_prefetch_desc(&mp.k);
        tma_prefetch_desc(&mp.v);
        if (!(p.flags & kTcNoO)) tma_prefetch_desc(&mp.o);
        tma_prefetch_desc(&mp.g);
        tma_prefetch_desc(&mp.b);
        tma_prefetch_desc(&mp.w);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    for (int i = tid; i < 8192 / 16; i += kThreads)   // Tinv: zeros above the diagonal blocks
        reinterpret_cast<uint4 *>(sm + OFF_T)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();                              // ... as the tensor core will read them

    int n_gbw = 0, n_qv = 0, n_k = 0;                 // loads issued (producer), for a drain
    auto load_gbw = [&](int c) {
        ++n_gbw;
        mbar_arrive_expect_tx(&bar_gbw, 3 * kC * kD * 2);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
            tma_load_4d(sm + OFF_G + pnl * 8192, &mp.g, &bar_gbw, 64 * pnl, h, c * kC, b);
            tma_load_4d(sm + OFF_BT + pnl * 8192, &mp.b, &bar_gbw, 64 * pnl, h, c * kC, b);
            tma_load_4d(sm + OFF_WT + pnl * 8192, &mp.w, &bar_gbw, 64 * pnl, h, c * kC, b);
        }
    };
    auto load_qv = [&](int c) {
        ++n_qv;
        mbar_arrive_expect_tx(&bar_qv, (no_v() ? 1 : 2) * kC * kD * 2);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
            tma_load_4d(sm + OFF_XQ + pnl * 16384 + 8192, &mp.q, &bar_qv, 64 * pnl, h, c * kC, b);
            if (!no_v()) tma_load_4d(sm + OFF_V + pnl * 8192, &mp.v, &bar_qv, 64 * pnl, h, c * kC, b);
        }
    };
    auto load_k = [&](int c) {
        ++n_k;
        mbar_arrive_expect_tx(&bar_k, kC * kD * 2);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl)
            tma_load_4d(sm + OFF_K + pnl * 8192, &mp.k, &bar_k, 64 * pnl, h, c * kC, b);
    };

    if (producer) {
        load_gbw(0);
        load_qv(0);
        load_k(0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);

    // initial state: bf16 copy in S_in, fp32 in TMEM (scaled per channel at each chunk start)
    {
        const size_t base = ((size_t)bh * kD + d_row) * kD + 64 * hf;
        uint8_t *sp = sm + OFF_S + hf * 16384;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float sv[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 v = p.S0 ? *reinterpret_cast<const float4 *>(p.S0 + base + 32 * half + j)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                sv[j] = v.x; sv[j + 1] = v.y; sv[j + 2] = v.z; sv[j + 3] = v.w;
            }
            if (s0_id)
#pragma unroll
                for (int j = 0; j < 32; ++j) sv[j] = (64 * hf + 32 * half + j == d_row) ? 1.f : 0.f;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = sv[8 * ch + e];
                *reinterpret_cast<uint4 *>(sp + sw128_off(d_row, 32 * half + 8 * ch)) = pack8(f);
            }
            tmem_st32(tl + TM_S + 64 * hf + 32 * half, sv);
        }
        tmem_st_wait();
    }
    uint32_t mma_phase = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        if (!mbar_wait(&bar_mma, mma_phase, kWaitNs)) { ok = false; abort_flag = 1; }
        mma_phase ^= 1;
        tc_fence_after();
    };
    auto sync_for_mma = [&]() {
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    sync_for_mma();

    const uint32_t sbase = smem_u32(sm);
    const uint32_t sXQ = sbase + OFF_XQ, sK = sbase + OFF_K, sV = sbase + OFF_V, sS = sbase + OFF_S;
    const uint32_t sT = sbase + OFF_T, sR2 = sbase + OFF_R2, sP = sbase + OFF_P;
    // A [64 tokens][128] bf16 tile (two swizzled 64-column panels at dst) from this warp's
    // TMEM lanes (the tile's columns) and columns 32 hf.. (its tokens): the accumulator at
    // column c1, negated when c2 < 0, else plus the one at c2.  Each 16-lane half is read in
    // the 16x256b shape, so a thread holds two adjacent tokens of rows L + t/4 and
    // L + 8 + t/4, and the 8x8 blocks go out as transposed 16-byte stmatrix rows.
    auto tile_out = [&](uint32_t c1, int c2, uint32_t dst) {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            const int L = 32 * q4 + 16 * half;
            float a[16], b2[16];
            tmem_ld16x256_x4(tm + c1 + 32 * hf + ((uint32_t)L << 16), a);
            if (c2 >= 0) tmem_ld16x256_x4(tm + (uint32_t)c2 + 32 * hf + ((uint32_t)L << 16), b2);
            tmem_ld_wait();
            uint32_t pk[8];                                // pk[2j + h]: rows L + 8h + lane/4
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    float2 x = make_float2(a[4 * j + 2 * h2], a[4 * j + 2 * h2 + 1]);
                    if (c2 >= 0) x = ffma2(make_float2(1.f, 1.f), make_float2(b2[4 * j + 2 * h2], b2[4 * j + 2 * h2 + 1]), x);
                    uint32_t u = pack_bf16x2(x.x, x.y);
                    pk[2 * j + h2] = c2 < 0 ? u ^ 0x80008000u : u;
                }
            const int m = lane >> 3, col = L + 8 * (m & 1);
            const uint32_t base = dst + (uint32_t)(col >> 6) * 8192;
#pragma unroll
            for (int j = 0; j < 4; j += 2)
                stmatrix_x4_trans(base + sw128_off(32 * hf + 8 * (j + (m >> 1)) + (lane & 7), col & 63), pk[2 * j],
                                  pk[2 * j + 1], pk[2 * j + 2], pk[2 * j + 3]);
        }
    };
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kC;
        const uint32_t par = (uint32_t)(c & 1);

        // (1) this chunk's tiles
        if (!mbar_wait(&bar_gbw, par, kWaitNs) || !mbar_wait(&bar_qv, par, kWaitNs) ||
            !mbar_wait(&bar_k, par, kWaitNs)) { ok = false; abort_flag = 1; }
        __syncthreads();
        if (abort_flag) break;

        // (2) k_t . u_t per token (one warp per token; u = b*q, or the ablation arm's
        // q, b*z_h) and W*V in place of V
        if (proj)
#pragma unroll
        for (int it = 0; it < kC / (kThreads / 32); ++it) {   // unrolled: the eight reductions overlap
            const int t = warp + (kThreads / 32) * it, j = 4 * lane;
            const uint32_t o8 = tile_off(t, j, 8192), o16 = tile_off(t, j, 16384);
            const uint2 kk = *reinterpret_cast<const uint2 *>(sm + OFF_K + o8);
            const uint2 bb = *reinterpret_cast<const uint2 *>(sm + OFF_BT + o8);
            const uint2 qq = *reinterpret_cast<const uint2 *>(sm + OFF_XQ + 8192 + o16);
            const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kk);
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&bb);
            const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qq);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float2 kf = __bfloat1622float2(k2[e]), bf2 = __bfloat1622float2(b2[e]);
                float2 xf = __bfloat1622float2(q2[e]);
                if (zrow) xf = make_float2(zrow[j + 2 * e], zrow[j + 2 * e + 1]);
                const float u0 = gate ? bf2.x * xf.x : xf.x, u1 = gate ? bf2.y * xf.y : xf.y;
                acc = fmaf(kf.x, u0, acc);
                acc = fmaf(kf.y, u1, acc);
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) g_ku[t] = acc;
        }
        if (!no_v())
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t off = (uint32_t)(tid + kThreads * r) << 4;   // both 8 KB panels
            float vf[8], wf[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_V + off), vf);
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_WT + off), wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) vf[e] *= wf[e];
            *reinterpret_cast<uint4 *>(sm + OFF_V + off) = pack8(vf);
        }
        // partial sums of g over each half of the chunk, per channel
        {
            const int j = tid & 127, half = tid >> 7;
            float sum = 0.f;
#pragma unroll 8
            for (int t = 32 * half; t < 32 * half + 32; ++t)
                sum += bf(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_G + tile_off(t, j, 8192)));
            g_ps[half][j] = sum;
        }
        __syncthreads();

        // (3) per channel j: G_t, erase vector a_t, and the factored operands Ae, Qe, Ke
        {
            const int j = tid & 127, half = tid >> 7;
            float G = half ? g_ps[0][j] : 0.f;
            const float zj = zrow ? zrow[j] : 0.f;
#pragma unroll 8
            for (int t = 32 * half; t < 32 * half + 32; ++t) {
                const uint32_t o8 = tile_off(t, j, 8192), o16 = tile_off(t, j, 16384);
                G += bf(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_G + o8));
                const float eG = __expf(G), emG = __expf(-G);
                const float qv = bf(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_XQ + 8192 + o16));
                const float kv = bf(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_K + o8));
                const float bv = bf(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_BT + o8));
                const float xv = zrow ? zj : qv;
                const float u = gate ? bv * xv : xv;
                const float a = bv * kv + lam_h * (proj ? u - kv * g_ku[t] : u);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_XQ + o16) = __float2bfloat16_rn(a * eG);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_XQ + 8192 + o16) = __float2bfloat16_rn(qv * eG);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_K + o8) = __float2bfloat16_rn(kv * emG);
            }
            if (half) g_ecg[j] = __expf(G);                  // e^{G_C} per channel
        }
        sync_for_mma();
        if (producer && c + 1 < nchunks) load_gbw(c + 1);   // g, b, w tiles consumed

        // (4) G = [Ae; Qe] Ke^T and O1 = S^ Qe^T
        if (issuer) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                umma_bf16(tm + TM_G, smem_desc(sXQ + ko, 16, 1024),
                          smem_desc(sK + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), idesc_bf16(128, 64, false, false),
                          k > 0);
            }
            if (!no_o())
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                    umma_bf16(tm + TM_O1, smem_desc(sS + ko, 16, 1024), smem_desc(sXQ + ko + 8192, 16, 1024),
                              idesc_bf16(128, 64, false, false), k > 0);
                }
            umma_commit(&bar_mma);
        }
        wait_mma();

        // (5) masks: At (fp32, R1) and P (bf16); Ke -> Kd per channel; S in TMEM *= e^{G_C}
        {
            float g[32];
            tmem_ld32(tl + TM_G + 32 * hf, g);
            tmem_ld_wait();
            if (q4 < 2) {
                const int t = 32 * q4 + lane;
                float *Arow = reinterpret_cast<float *>(sm + OFF_R1) + t * LA + 32 * hf;
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    float a[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) a[e] = (32 * hf + 4 * c4 + e < t) ? g[4 * c4 + e] : 0.f;
                    *reinterpret_cast<float4 *>(Arow + 4 * c4) = make_float4(a[0], a[1], a[2], a[3]);
                }
            } else {
                const int t = 32 * (q4 - 2) + lane;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = (32 * hf + 8 * ch + e <= t) ? g[8 * ch + e] : 0.f;
                    *reinterpret_cast<uint4 *>(sm + OFF_P + sw128_off(t, 32 * hf + 8 * ch)) = pack8(f);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t off = (uint32_t)(tid + kThreads * r) << 4;
                const uint32_t in = off & 8191;
                const int row = in >> 7, lc = ((in >> 4) & 7) ^ (row & 7);
                const int j0 = 64 * (int)(off >> 13) + 8 * lc;
                uint4 *pk = reinterpret_cast<uint4 *>(sm + OFF_K + off);
                float kf[8];
                unpack8(*pk, kf);
#pragma unroll
                for (int e = 0; e < 8; ++e) kf[e] *= g_ecg[j0 + e];
                *pk = pack8(kf);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float sv[32];
                tmem_ld32(tl + TM_S + 64 * hf + 32 * half, sv);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 x = fmul2(make_float2(sv[e], sv[e + 1]),
                                           *reinterpret_cast<const float2 *>(g_ecg + 64 * hf + 32 * half + e));
                    sv[e] = x.x;
                    sv[e + 1] = x.y;
                }
                tmem_st32(tl + TM_S + 64 * hf + 32 * half, sv);
            }
            tmem_st_wait();
        }
        if (producer) tma_store_wait_read0();   // R2 (last chunk's O staging) is free for scratch
        tc_fence_before();
        __syncthreads();

        // (6) Tinv = (I + At)^{-1} -> T (the U and W products read the same matrix)
        unit_lower_inverse(reinterpret_cast<float *>(sm + OFF_R1), reinterpret_cast<float *>(sm + OFF_R2),
                           sm + OFF_T, nullptr, nullptr, nullptr, []() {}, []() { __syncthreads(); });
        sync_for_mma();

        // (7) U^T = (W*V)^T Tinv^T, W^T = Ae^T Tinv^T
        if (issuer) {
            if (!no_v())                               // v taken as 0: U = 0 (Z starts from -S^ W^T)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_bf16(tm + TM_U, smem_desc(sV + k * 2048, 8192, 1024), smem_desc(sT + k * 32, 16, 1024),
                              idesc_bf16(128, 64, true, false), k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_bf16(tm + TM_W, smem_desc(sXQ + k * 2048, 16384, 1024), smem_desc(sT + k * 32, 16, 1024),
                          idesc_bf16(128, 64, true, false), k > 0);
            umma_commit(&bar_mma);
        }
        wait_mma();
        if (producer && c + 1 < nchunks) load_qv(c + 1);   // Qe, W*V and Ae are consumed

        // (8) -W -> R2 as [64 tokens][dk]
        tile_out(TM_W, -1, sbase + OFF_R2);
        sync_for_mma();

        // (9) Z^T = U^T - S^ W^T
        if (issuer) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                umma_bf16(tm + TM_U, smem_desc(sS + ko, 16, 1024), smem_desc(sR2 + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                          idesc_bf16(128, 64, false, false), (no_v() && k == 0) ? 0u : 1u);
            }
            umma_commit(&bar_mma);
        }
        wait_mma();

        // (10) Z^T (bf16) -> R2 as [dv][64 tokens]
        {
            float z[32];
            tmem_ld32(tl + TM_U + 32 * hf, z);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = z[8 * ch + e];
                *reinterpret_cast<uint4 *>(sm + OFF_R2 + sw128_off(d_row, 32 * hf + 8 * ch)) = pack8(f);
            }
        }
        sync_for_mma();

        // (11) O2 = Z^T P^T ; S^ += Z^T Kd
        if (issuer) {
            if (!no_o())
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_bf16(tm + TM_O2, smem_desc(sR2 + k * 32, 16, 1024), smem_desc(sP + k * 32, 16, 1024),
                              idesc_bf16(128, 64, false, false), k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_bf16(tm + TM_S, smem_desc(sR2 + k * 32, 16, 1024), smem_desc(sK + k * 2048, 8192, 1024),
                          idesc_bf16(128, 128, false, true), 1);
            umma_commit(&bar_mma);
        }
        wait_mma();
        if (producer && c + 1 < nchunks) load_k(c + 1);    // Kd is consumed

        // (12) o = O1 + O2 -> staging (R2); state -> bf16 S_in (and S_final after the last chunk)
        {
            if (!no_o()) tile_out(TM_O1, TM_O2, sbase + OFF_R2);
            const bool last = (c + 1 == nchunks);
            uint8_t *sp = sm + OFF_S + hf * 16384;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float sv[32];
                tmem_ld32(tl + TM_S + 64 * hf + 32 * half, sv);
                tmem_ld_wait();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = sv[8 * ch + e];
                    *reinterpret_cast<uint4 *>(sp + sw128_off(d_row, 32 * half + 8 * ch)) = pack8(f);
                }
                if (last && p.S_final && !abort_flag) {
                    float *fs = p.S_final + ((size_t)bh * kD + d_row) * kD + 64 * hf + 32 * half;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4 *>(fs + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
                }
            }
        }
        sync_for_mma();
        if (producer && !no_o()) {
            tma_store_4d(&mp.o, sm + OFF_R2, 0, h, t0, b);
            tma_store_4d(&mp.o, sm + OFF_R2 + 8192, 64, h, t0, b);
            tma_store_commit();
        }
    }

    if (producer) {
        tma_store_wait_all();
        if (abort_flag) {   // drain loads that may still be landing in shared memory
            if (n_gbw) mbar_wait(&bar_gbw, (uint32_t)((n_gbw - 1) & 1), kWaitNs);
            if (n_qv) mbar_wait(&bar_qv, (uint32_t)((n_qv - 1) & 1), kWaitNs);
            if (n_k) mbar_wait(&bar_k, (uint32_t)((n_k - 1) & 1), kWaitNs);
        }
    }
    if (issuer && abort_flag) {
        umma_commit(&bar_mma);
        mbar_wait(&bar_mma, mma_phase, kWaitNs);
    }
    if ((!ok || abort_flag) && lane == 0) atomicExch(&g_qed_tc_timeout, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

bool qed_tc_supported(const QedArgs &a, int dtype) {
    return dtype == kBF16 && a.dk == kD && a.dv == kD && (long long)a.T * a.H * kD * 2 < (1ll << 40);
}

cudaError_t launch_qed_chunk_tc(const QedArgs &a, cudaStream_t s, int *nlaunch, int flags) {
    QedMaps m;
    if (!make_token_map(&m.q, a.q, a.B, a.T, a.H) || !make_token_map(&m.k, a.k, a.B, a.T, a.H) ||
        !make_token_map(&m.v, a.v, a.B, a.T, a.H) || !make_token_map(&m.g, a.g, a.B, a.T, a.H) ||
        !make_token_map(&m.b, a.b, a.B, a.T, a.H) || !make_token_map(&m.w, a.w, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    if (flags & kTcNoO) m.o = m.q;                    // not used
    else if (!make_token_map(&m.o, a.o, a.B, a.T, a.H)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(qed_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    QedTcParams p{a.lam_h, a.S0, a.S_final, a.B, a.T, a.H, flags, a.variant, a.z};
    qed_fwd_tc_kernel<<<a.B * a.H, kThreads, kSmemBytes, s>>>(p, m);
    e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

bool qed_tc_read_and_clear_timeout() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_qed_tc_timeout, sizeof v) != cudaSuccess) return false;
    if (v) cudaMemcpyToSymbol(g_qed_tc_timeout, &zero, sizeof zero);
    return v != 0;
}

}  // namespace qd

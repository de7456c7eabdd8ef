// Fused chunked Q-Delta forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA),
// bf16 inputs, dk = dv = 128, chunk C = 64, fp32 state held on chip for the whole
// sequence.  One CTA of 12 warps per (b, h).
//
// Algorithm ("Q-Delta: Beyond Key-Value Associative State Evolution", Sec. 3.3.2,
// Eqs. 20-27, with the corrected transposes and gamma_r/gamma_i decay; the two UT
// solves folded into one).  Per chunk, rows stacked, l_i = sum_{j<=i} log alpha_j,
// gamma_i = e^{l_i}, kappa_i = e^{l_C - l_i}, X = K + diag(lambda) Q:
//   G      = [X; Q] K^T                                   (one M=128 MMA)
//   A      = strictly_lower(beta_t e^{l_t - l_i} (X K^T)_ti);  P = incl_lower(e^{l_t-l_i} (Q K^T)_ti)
//   Tinv   = (I + A)^{-1}                                  (fp32, tc_common.cuh)
//   U^T    = V^T T1^T,  T1 = Tinv diag(beta);   T2 = Tinv diag(beta gamma)
//   Z^T    = U^T - (S X^T) T2^T                            (S = state entering the chunk;
//                                                            (S X^T) T2^T = S W^T, W = T2 X)
//   o_t    = gamma_t (S Q^T)_t + (Z^T P^T)_t
//   S     <- gamma_C S + Z^T diag(kappa) K
// Every product is written "transposed" so that the 128 TMEM lanes index d_v (or
// d_k) and every MMA has M = 128.  S [X; Q]^T is one N = 128 product whose halves are
// S X^T and S Q^T, the first output term.  The two output terms share one accumulator
// O = S Q^T + Zt^T Pt^T and the epilogue multiplies token t by gamma_t, with Zt, Pt
// chosen by the chunk's log-decay l_C:
//   l_C > -30 (fold):  Zt = Z diag(kappa), Pt_ti = e^{-l_C} (Q K^T)_ti   (K used as loaded)
//   l_C > -80 (split): Zt = Z, Pt_ti = e^{-l_i} (Q K^T)_ti, K scaled in place to kappa K
//   otherwise:         Zt = Z, Pt = P, kappa K in place, S Q^T scaled by gamma in TMEM
//                      before Zt^T Pt^T accumulates onto it, and no gamma_t in the
//                      epilogue (no factor can overflow)
// since (Z^T diag(kappa)) (P diag(1/kappa))^T = Z^T P^T and P_ti / gamma_t = e^{-l_i} (Q K^T)_ti.
// The master state stays in TMEM in fp32 (the MMA accumulates Zt^T (kappa) K onto it
// after the epilogue has scaled it by the chunk's gamma_C).  Its bf16 copy, the bf16
// -(S X^T) and the bf16 Zt^T also live in TMEM and are the A operands of the
// state-dependent products, so those MMAs read only their B operand from shared memory.
//
// Warp specialisation: a prep group (warps 0-7) does the state-independent work of
// each chunk -- the decay masks, the solve, U, and X and the Gram of the next chunk --
// and hands the chunk to a chain group (warps 8-11) that carries the state: S [X; Q]^T,
// Z, the coupling, Zt^T, the output and state products, the epilogue.  The two groups
// run concurrently, so the chunk period is the longer of the two instead of their sum.
// Each group synchronises on its own named barrier; hand-offs are mbarriers:
//   ready       prep -> chain: P(c), T2(c), the gates of chunk c+1 and X(c+1) in place
//   taken       chain -> prep: the chain has passed `ready` and `uw` of chunk c, so U(c+1)
//               may be issued and `ready` completed for chunk c+1 (the prep may run up to
//               two chunks ahead and must not complete a phase twice before the chain
//               has waited on the first)
//   cdone[c&1]  chain -> prep: the products of chunk c have run, so P, U, T2 and M21
//               of parity c&1 are free
// Inside the prep group three threads issue at once after the solve: the hand-off, U(c)
// and the Gram of chunk c+1; warps 4-7, idle in the solve's first phases, form X of
// chunk c+1 meanwhile.  The chain issues S [X; Q]^T of chunk c as soon as the state of
// chunk c-1 is final, before the chunk is handed over.
// Loads: K sits in a three-slot ring, X/Q and V in two stages by chunk parity, so the
// tiles of chunk c+2 go out while chunk c is still running -- K while the chain waits for
// `ready` (its slot held chunk c-1's K and then that chunk's o tile, once the o store has
// read it), Q and V as soon as S [X; Q]^T and U of chunk c have run -- and arrive in time
// for X of chunk c+2 to be formed during the solve of chunk c+1.
//
// Instruction economy on both groups (they share each SM sub-partition's issue slots):
// the output accumulator leaves TMEM in the 16x256b shape, so a thread holds two
// adjacent tokens of a d_v row and the o tile is written as transposed 16-byte
// stmatrix rows; elementwise scalings (state rescale, Zt packing, masks, X = K + lambda Q)
// use packed f32x2 arithmetic; -(S X^T) is packed first and its bf16 sign bits flipped.
//
// Shared memory (offsets from a 1024-aligned base):
//   stage s in {0,1}: XQ 32 KB (per 64-column panel: X rows 0-63 | Q rows 64-127), V 16 KB
//   K ring 3x16 KB   K of chunk c in slot c%3 (scaled in place to kappa*K under strong
//                    decay), then o(c) [64][dv] bf16 for the TMA store
//   R1   17 KB   A fp32 [64][68], overwritten by the solve's intermediate blocks
//   P    2x8 KB  bf16 Pt [64][64], by chunk parity
//   T1   8 KB    Tinv*beta (bf16 [64][64]); T2 2x8 KB Tinv*beta*gamma by chunk parity;
//                written block by block by the solve, zero above the 8x8 diagonal blocks
//   Y    4.5 KB  fp32 scratch of the solve (prep group only)
//   M21  2x2 KB  -M21 (diag(1/kappa)) bf16 [32][32] without swizzle, by chunk parity
//   ECG  512 B   QED: the chunk's e^{G_C}
// All shared-memory MMA operands use the 128-byte swizzle (TMA layout): 128-byte
// rows, 8-row groups 1024 bytes apart, 64-column panels.
// TMEM (512 columns): G 0-63, U[0] 64-127, U[1] 128-191 (Z^T accumulates there; its
// first 32 columns then hold the packed bf16 Zt^T), SK 192-255 and O 256-319 (the two
// halves of S [X; Q]^T; SK's first 32 columns then hold -(S X^T) packed), packed bf16
// state 320-383, fp32 state 384-511.
//
// Every wait is bounded; on a timeout the kernel sets the library's error word,
// waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "qd_internal.cuh"
#include "qed_derive.cuh"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace qd {

__device__ unsigned int g_tc_timeout = 0;

namespace {

using namespace ptx;
using namespace tc;

constexpr int kPrepThreads = kThreads;              // warps 0-7
constexpr int kChainThreads = 128;                  // warps 8-11
constexpr int kAllThreads = kPrepThreads + kChainThreads;
constexpr int kBarPrep = 1, kBarChain = 2, kBarX = 3;   // named barrier ids (8-13: inside the solve)
constexpr uint32_t kStageBytes = 49152;              // XQ 32 KB + V 16 KB, by chunk parity
constexpr uint32_t OFF_XQ = 0, OFF_V = 32768;
constexpr uint32_t OFF_KR = 2 * kStageBytes;         // 98304: K ring, three 16 KB slots
constexpr uint32_t OFF_R1 = OFF_KR + 3 * 16384;      // 147456
constexpr uint32_t OFF_P = OFF_R1 + 17408;           // 164864 (two 8 KB buffers)
constexpr uint32_t OFF_T = OFF_P + 16384;            // 181248 (T1, then T2 by parity; bf16)
constexpr uint32_t OFF_Y = OFF_T + 24576;            // 205824 (solve scratch, 32 x LY fp32)
constexpr uint32_t OFF_M21 = 210944;                 // two 2 KB coupling tiles
constexpr uint32_t OFF_ECG = OFF_M21 + 4096;         // 215040 (QED: e^{G_C} of the chunk, 128 fp32)
constexpr uint32_t kSmemUsed = OFF_ECG + 512;        // 215552
static_assert(OFF_M21 >= OFF_Y + 32 * LY * 4 && OFF_M21 % 1024 == 0, "tile placement");
static_assert(OFF_KR % 1024 == 0 && OFF_P % 1024 == 0 && OFF_T % 1024 == 0 && kSmemUsed + 1024 <= 232448,
              "128-byte-swizzled MMA operands start on 1024-byte boundaries");
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;    // + alignment slack
constexpr uint32_t kTmaBytes = 3 * kC * kD * 2;      // Q, K, V tiles per chunk
constexpr uint64_t kWaitNs = 2000000000ull;          // 2 s per wait

// fold kappa into Z^T (and 1/kappa into P) when the chunk's log-decay l_C exceeds this:
// then kappa >= e^-30 and Pt <= e^30 |Q K^T|, far from bf16 under/overflow
constexpr float kFoldLog = -30.f;
// below this log-decay e^{-l_i} leaves the fp32 range: the exponentials are taken
// one by one and Q carries gamma instead
constexpr float kSplitLog = -80.f;

constexpr uint32_t TM_G = 0, TM_U = 64, TM_SK = 192, TM_O = 256, TM_SB = 320, TM_S = 384;

struct TcParams {
    const __nv_bfloat16 *alpha, *beta, *lam;
    const float *S0;
    __nv_bfloat16 *o;
    float *S_final;
    int B, T, H;
    int flags;   // kTcNoV | kTcS0Identity | kTcNoO (segment-scan passes)
    const float *ecg;   // QED: e^{G_C} per chunk and channel, [B*H][nchunks][128]
    // fused QED (n_chain > 0): CTAs n_chain.. derive the operands that CTAs 0..n_chain-1
    // consume; done[bh * nchunks + chunk] counts the derived halves of each chunk (zero at
    // the launch)
    int n_chain;
    unsigned int *done;
    QedDeriveParams dp;
};

// PRO: q, k, alpha, beta, lambda arrive as projections and logits (the prologue of
// qdelta_fwd_prologue); a template parameter, so the plain kernel carries none of it.
// CHK: the state entering every chunk is written to the backward's checkpoint array,
// from the registers that already hold it on its way into TMEM: per (b*H + h, chunk) a
// 32 KB fp16 [dv][dk] tile in the layout of a 128-byte-swizzled MMA operand (two
// 64-column panels of 128 rows, chk_tile_off), which the gradient kernel copies in one
// piece.  That instance runs without output (kTcNoO) and takes the array in p.o.
// F16: q, k, v and o are fp16 instead of bf16, and so are every operand the kernel forms
// (X, Pt, the inverse, -(S X^T), Zt, the state copy); alpha must be null (the decay
// factors of the other regimes do not fit fp16's range).  The EDA forward (eda_tc.cu)
// runs its 2T'+1 sub-tokens through this instance: k holds every sub-token, while q, v
// and o are compact [B][T'][H][128] arrays read through pair maps (tc_common.cuh), so
// that sub-token 2j + p is row j of q and o (p = 0; zero / not stored for p = 1) and row
// j - 1 of v (p = 0; zero for p = 1 and j = 0).
// QED: the chain of the QED forward (chunk_tc_qed.cu) over its derived operands: tmA,
// tmQ, tmK, tmV map Ae, Qe, Ke, W*V, the X rows are loaded (Ae) instead of formed, every
// gate is a unit (alpha = 1, beta = 1, lambda = 0: the products above then are QED's
// Gram, masks, solve, U, S [A; Q]^T, Z, O and S + Z^T Ke), and the epilogue multiplies the state
// by the chunk's e^{G_C} per channel (column of the [dv][dk] state).
template <bool PRO, bool CHK = false, bool QED = false, bool F16 = false>
__global__ void __launch_bounds__(kAllThreads, 1)
qdelta_fwd_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmA) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_full[2], bar_g, bar_uw, bar_z, bar_zz, bar_cp, bar_o2, bar_ready, bar_taken, bar_cdone[2],
        bar_drain[3];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    // per-chunk gate arrays, by chunk index mod 4: while the prep group builds chunk
    // c+1's arrays (during the solve of chunk c) the chain group may still read those
    // of chunks c-2 (its epilogue), c-1 and c
    // (Loops below read what they need of these into registers before they store to
    // shared memory: the compiler cannot tell the two apart and would otherwise
    // serialise every load behind the previous store.)
    __shared__ __align__(16) float g_ell[4][kC], g_beta[4][kC], g_lam[4][kC], g_gam[4][kC], g_kap[4][kC],
        g_igam[4][kC];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if constexpr (QED) {
        // fused QED: the CTAs past the chains derive the operands, one 32-token half of one
        // chunk at a time in chunk order over all streams, on 256 threads, and count each
        // finished half in `done` (every writer fences its stores before the count)
        if (p.n_chain > 0 && (int)blockIdx.x >= p.n_chain) {
            if (tid >= kDeriveThreads) return;
            const int nd = (int)gridDim.x - p.n_chain, bhn = p.B * p.H, nch = (p.T + kC - 1) / kC;
            float (*s_part)[kGroups][kD] = reinterpret_cast<float (*)[kGroups][kD]>(sm);
            for (long long i = (long long)blockIdx.x - p.n_chain; i < 2LL * nch * bhn; i += nd) {
                const int chunk = (int)(i / (2 * bhn)), rem = (int)(i % (2 * bhn));
                qed_derive_half(p.dp, chunk, rem & 1, rem >> 1, s_part,
                                []() { named_sync(4, kDeriveThreads); });
                __threadfence();
                named_sync(4, kDeriveThreads);        // the half's stores are out; s_part is free
                if (tid == 0) atomicAdd(p.done + (size_t)(rem >> 1) * nch + chunk, 1u);
            }
            return;
        }
    }
    const bool prep = tid < kPrepThreads;
    const int q4 = warp & 3, hf = (warp >> 2) & 1;    // TMEM lane quarter; column half (prep)
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int T = p.T, H = p.H;
    const int nchunks = (T + kC - 1) / kC;
    // MMA issuers: U and the prep's hand-off (p), the next chunk's Gram (g, in parallel with
    // U), the chain's products (c)
    const bool p_issuer = (tid == 32), g_issuer = (tid == 64), c_issuer = (tid == kPrepThreads);
    const int d_row = 32 * q4 + lane;                  // this thread's TMEM lane / state row
    // flags of the segment-scan passes; read through opaque() where they are tested
    // inside the chunk loops (see tc_common.cuh)
    const uint32_t flags = (uint32_t)p.flags;
    const bool s0_id = flags & kTcS0Identity;
    auto no_v = [&]() { return (opaque(flags) & kTcNoV) != 0; };
    auto no_o = [&]() { return (opaque(flags) & kTcNoO) != 0; };
    constexpr bool prologue = PRO;

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_uw, 1);
        mbar_init(&bar_z, 1);
        mbar_init(&bar_cp, 1);
        mbar_init(&bar_o2, 1);
        mbar_init(&bar_ready, 1);
        mbar_init(&bar_taken, 1);
        mbar_init(&bar_zz, 1);
        mbar_init(&bar_cdone[0], 1);
        mbar_init(&bar_cdone[1], 1);
        mbar_init(&bar_drain[0], 1);
        mbar_init(&bar_drain[1], 1);
        mbar_init(&bar_drain[2], 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (!(p.flags & kTcNoO)) tma_prefetch_desc(&tmO);
        if (QED) tma_prefetch_desc(&tmA);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    for (int i = tid; i < 24576 / 16; i += kAllThreads)   // T1, T2: zeros above the diagonal blocks
        reinterpret_cast<uint4 *>(sm + OFF_T)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();                                  // ... as the tensor core will read them

    // fused QED: both halves of chunk c derived (bounded acquire), and the derived tiles,
    // written by generic stores, ordered before this thread's TMA reads of them
    auto derived_wait = [&](int c) {
        if (!(QED && p.n_chain > 0)) return;
        const unsigned int *d = p.done + (size_t)bh * nchunks + c;
        uint64_t t0 = 0;
        while (ld_acquire_u32(d) < 2u) {
            if (t0 == 0) t0 = globaltimer_ns();
            else if (globaltimer_ns() - t0 > kWaitNs) { abort_flag = 1; break; }
        }
        fence_proxy_async_global();
    };
    // the tiles of chunk c on bar_full[c&1], in two parts: K into its slot (arming the
    // barrier with the whole chunk's bytes), then Q (QED: and A) and V into the stage
    auto issue_k = [&](int c) {
        const int s = c & 1;
        uint8_t *kb = sm + OFF_KR + (uint32_t)(c % 3) * 16384;
        derived_wait(c);                              // fused QED: chunk c derived
        mbar_arrive_expect_tx(&bar_full[s], (no_v() ? kTmaBytes / 3 * 2 : kTmaBytes) + (QED ? kTmaBytes / 3 : 0));
#pragma unroll
        if (QED) {                                    // QED's maps take whole tiles
            tma_load_5d(kb, &tmK, &bar_full[s], 0, c * kC, 0, h, b);
        } else {
#pragma unroll
            for (int pnl = 0; pnl < 2; ++pnl) tma_load_4d(kb + pnl * 8192, &tmK, &bar_full[s], 64 * pnl, h, c * kC, b);
        }
    };
    auto issue_xqv = [&](int c) {
        const int s = c & 1;
        uint8_t *st = sm + s * kStageBytes;
        const int t0 = c * kC;
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
            if (QED) tma_load_4d(st + OFF_XQ + pnl * 16384, &tmA, &bar_full[s], 64 * pnl, h, t0, b);
            if (F16) {                                // pair maps: sub-token 2j + p is compact row j (p = 0)
                tma_load_5d(st + OFF_XQ + pnl * 16384 + 8192, &tmQ, &bar_full[s], 64 * pnl, 0, h, t0 / 2, b);
                tma_load_5d(st + OFF_V + pnl * 8192, &tmV, &bar_full[s], 64 * pnl, 0, h, t0 / 2 - 1, b);
                continue;
            }
            tma_load_4d(st + OFF_XQ + pnl * 16384 + 8192, &tmQ, &bar_full[s], 64 * pnl, h, t0, b);
            if (!QED && !no_v()) tma_load_4d(st + OFF_V + pnl * 8192, &tmV, &bar_full[s], 64 * pnl, h, t0, b);
        }
        if (QED && !no_v()) tma_load_5d(st + OFF_V, &tmV, &bar_full[s], 0, t0, 0, h, b);
    };
    auto issue_loads = [&](int c) {
        issue_k(c);
        issue_xqv(c);
    };
    // gates of a chunk: lane l of warp 4 holds tokens 2l and 2l+1.  The loads land in raw
    // bf16 registers that nothing reads until compute_gates, so they do not stall the warp.
    __nv_bfloat16 ra[2], rb[2], rl[2];
    auto load_gates = [&](int c) {
        if (QED) return;                                  // unit gates
        const __nv_bfloat16 *pa = opaque(p.alpha), *pl = opaque(p.lam);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = min(c * kC + 2 * lane + u, T - 1);
            const size_t tok = ((size_t)b * T + t) * H + h;
            if (pa) ra[u] = pa[tok];
            rb[u] = p.beta[tok];
            if (pl) rl[u] = pl[tok];
        }
    };
    // warp-wide: log-prefix l, gamma = e^l, kappa = e^{l_C - l}, e^{-l} of chunk c
    auto compute_gates = [&](int c) {
        const int buf = c & 3;
        const bool has_a = opaque(p.alpha) != nullptr, has_l = opaque(p.lam) != nullptr;
        const bool pro = prologue;
        float la[2], gb[2], gl[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {                  // tokens past T: alpha 1, beta 0, lambda 0
            const bool ok = c * kC + 2 * lane + u < T;
            if (QED) {                                 // alpha 1, beta 1, lambda 0
                la[u] = 0.f;
                gb[u] = ok ? 1.f : 0.f;
                gl[u] = 0.f;
            } else if (pro) {                          // gates from their logits
                const float x = bf(ra[u]);
                la[u] = (ok && has_a) ? -(fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)))) : 0.f;
                gb[u] = ok ? sigmoid_fast(bf(rb[u])) : 0.f;
                gl[u] = (ok && has_l) ? sigmoid_fast(bf(rl[u])) : 0.f;
            } else {
                la[u] = (ok && has_a) ? __logf(bf(ra[u])) : 0.f;
                gb[u] = ok ? bf(rb[u]) : 0.f;
                gl[u] = (ok && has_l) ? bf(rl[u]) : 0.f;
            }
        }
        const float l0 = la[0], l1 = la[1];
        float sum = l0 + l1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, sum, off);
            if (lane >= off) sum += n;
        }
        const float e1 = sum, e0 = sum - l1;
        const float eC = __shfl_sync(0xffffffffu, sum, 31);
        g_ell[buf][2 * lane] = e0;
        g_ell[buf][2 * lane + 1] = e1;
        g_beta[buf][2 * lane] = gb[0];
        g_beta[buf][2 * lane + 1] = gb[1];
        g_lam[buf][2 * lane] = gl[0];
        g_lam[buf][2 * lane + 1] = gl[1];
        g_gam[buf][2 * lane] = __expf(e0);
        g_gam[buf][2 * lane + 1] = __expf(e1);
        g_kap[buf][2 * lane] = __expf(eC - e0);
        g_kap[buf][2 * lane + 1] = __expf(eC - e1);
        // exp(l_t - l_i) = gamma_t * exp(-l_i) while exp(-l_C) stays in fp32 range
        g_igam[buf][2 * lane] = eC > -80.f ? __expf(-e0) : 0.f;
        g_igam[buf][2 * lane + 1] = eC > -80.f ? __expf(-e1) : 0.f;
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
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);   // this warp's TMEM lane quarter

    bool ok = true;
    auto wait_on = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_wait(bar, parity, kWaitNs)) { ok = false; abort_flag = 1; }
    };
    auto wait_mma = [&](uint64_t *bar, int chunk) {
        wait_on(bar, (uint32_t)(chunk & 1));
        tc_fence_after();
    };
    // a group's generic smem and TMEM work made visible to its next MMA / to the other group
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
    const uint32_t sT = sbase + OFF_T;
    auto stage_addr = [&](int c) { return sbase + (uint32_t)(c & 1) * kStageBytes; };
    auto kring = [&](int c) { return OFF_KR + (uint32_t)(c % 3) * 16384; };   // chunk c's K slot

    // ---------------------------------------------------------------- prep group
    // X = K + lambda Q into rows 0-63 of the XQ panels of chunk c's stage: by warps 4-7
    // during the solve of the chunk before, or, from projections (prologue), where K and Q
    // first become SiLU(x)/|SiLU(x)| in place, by the whole prep group after it.  Thread x
    // (of n = 128 or 256) takes, in each of 256/n rounds h2, the 16-byte chunks i = 0..3:
    // panel i / 2 and token row x/8 + 16 (2 h2 + i % 2) (n = 128) or x/8 + 32 (i % 2)
    // (n = 256); the eight threads of a row sum its squares by shuffles.
    auto x_pass = [&](int c) {
        uint8_t *st = sm + (c & 1) * kStageBytes;
        uint8_t *kb = sm + kring(c);
        const float *lam = g_lam[c & 3];
        constexpr int nx = prologue ? kPrepThreads : 128;
        const int xt = prologue ? tid : tid - 128;
#pragma unroll 1
        for (int h2 = 0; h2 < 256 / nx; ++h2) {
            auto chunk_of_i = [&](int i) {
                return prologue ? xt + 256 * i : xt + 128 * (2 * h2 + (i & 1) + 4 * (i >> 1));
            };
            uint4 kr[4], qr[4];
            float lm[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {                 // all loads first
                const int u = chunk_of_i(r);              // 16-byte chunk index, 0..1023
                const int pnl = u >> 9;
                const uint32_t off = (uint32_t)(u & 511) << 4;
                kr[r] = *reinterpret_cast<const uint4 *>(kb + pnl * 8192 + off);
                qr[r] = *reinterpret_cast<const uint4 *>(st + OFF_XQ + pnl * 16384 + 8192 + off);
                lm[r] = lam[off >> 7];
            }
            if (prologue) {
                float kf[4][8], qf[4][8], sk[2] = {0.f, 0.f}, sq[2] = {0.f, 0.f};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    unpack8(kr[r], kf[r]);
                    unpack8(qr[r], qf[r]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        kf[r][e] = silu_fast(kf[r][e]);
                        qf[r][e] = silu_fast(qf[r][e]);
                        sk[r & 1] = fmaf(kf[r][e], kf[r][e], sk[r & 1]);
                        sq[r & 1] = fmaf(qf[r][e], qf[r][e], sq[r & 1]);
                    }
                }
#pragma unroll
                for (int off = 1; off < 8; off <<= 1)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        sk[i] += __shfl_xor_sync(0xffffffffu, sk[i], off);
                        sq[i] += __shfl_xor_sync(0xffffffffu, sq[i], off);
                    }
                float ik[2], iq[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {             // zero rows (past T) stay zero
                    ik[i] = sk[i] > 0.f ? rsqrtf(sk[i]) : 1.f;
                    iq[i] = sq[i] > 0.f ? rsqrtf(sq[i]) : 1.f;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int u = chunk_of_i(r);
                    const int pnl = u >> 9;
                    const uint32_t off = (uint32_t)(u & 511) << 4;
                    float xf[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        kf[r][e] *= ik[r & 1];
                        qf[r][e] *= iq[r & 1];
                        xf[e] = fmaf(lm[r], qf[r][e], kf[r][e]);
                    }
                    *reinterpret_cast<uint4 *>(kb + pnl * 8192 + off) = pack8(kf[r]);
                    *reinterpret_cast<uint4 *>(st + OFF_XQ + pnl * 16384 + 8192 + off) = pack8(qf[r]);
                    *reinterpret_cast<uint4 *>(st + OFF_XQ + pnl * 16384 + off) = pack8(xf);
                }
                continue;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int u = chunk_of_i(r);
                const int pnl = u >> 9;
                const uint32_t off = (uint32_t)(u & 511) << 4;
                float kf[8], qf[8], xf[8];
                unpack8t<F16>(kr[r], kf);
                unpack8t<F16>(qr[r], qf);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 x = ffma2(make_float2(lm[r], lm[r]), make_float2(qf[e], qf[e + 1]),
                                           make_float2(kf[e], kf[e + 1]));
                    xf[e] = x.x;
                    xf[e + 1] = x.y;
                }
                *reinterpret_cast<uint4 *>(st + OFF_XQ + pnl * 16384 + off) = pack8t<F16>(xf);
            }
        }
    };
    // G = [X; Q] K^T
    auto issue_gram = [&](int c) {
        const uint32_t sXQ = stage_addr(c) + OFF_XQ, sK = sbase + kring(c);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(tm + TM_G, smem_desc(sXQ + ko, 16, 1024), smem_desc(sK + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024),
                      idesc_16<F16>(128, 64, false, false), k > 0);
        }
        umma_commit(&bar_g);
    };
    // decay masks: A (fp32, R1) from the X K^T rows, Pt (bf16) from the Q K^T rows.
    // Row t, column i of this thread's half: A_ti = beta_t e^{l_t - l_i} (X K^T)_ti for
    // i < t; for i <= t, Pt_ti = e^{-l_C} (Q K^T)_ti (fold), e^{-l_i} (Q K^T)_ti (split)
    // or e^{l_t - l_i} (Q K^T)_ti.  While l_C > -80 the decay factors as r_t * f_i with
    // f_i = e^{-l_i} (or 1 for fold-mode Pt); otherwise each factor is its own exponential.
    auto masks = [&](int c) {
        const int gi = c & 3;
        const float *ell = g_ell[gi], *bet = g_beta[gi], *gam = g_gam[gi], *igam = g_igam[gi];
        float g[32];
        tmem_ld32(tl + TM_G + 32 * hf, g);
        tmem_ld_wait();
        const bool split = ell[kC - 1] > kSplitLog;   // uniform: gamma_t * exp(-l_i) is safe
        const bool fold = ell[kC - 1] > kFoldLog;
        const bool arow = q4 < 2;                      // warp-uniform: A rows or P rows
        const int t = 32 * (arow ? q4 : q4 - 2) + lane;
        const int lim = arow ? t : t + 1;              // columns cc with 32 hf + cc < lim are kept
        const bool ones = !arow && fold;
        float r;
        if (arow) r = split ? bet[t] * gam[t] : bet[t];
        else r = fold ? igam[kC - 1] : 1.f;
        float fi[32];
        const float *src = (split ? igam : ell) + 32 * hf;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 v = ones ? make_float4(1.f, 1.f, 1.f, 1.f) : *reinterpret_cast<const float4 *>(src + j);
            fi[j] = v.x; fi[j + 1] = v.y; fi[j + 2] = v.z; fi[j + 3] = v.w;
        }
        if (split) {                                  // uniform branches: no exp when not needed
#pragma unroll
            for (int cc = 0; cc < 32; cc += 2) {
                const float2 x = fmul2(fmul2(make_float2(r, r), make_float2(fi[cc], fi[cc + 1])),
                                       make_float2(g[cc], g[cc + 1]));
                g[cc] = (32 * hf + cc < lim) ? x.x : 0.f;
                g[cc + 1] = (32 * hf + cc + 1 < lim) ? x.y : 0.f;
            }
        }
        else {
            const float lt = ell[t];
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) g[cc] = (32 * hf + cc < lim) ? r * __expf(lt - fi[cc]) * g[cc] : 0.f;
        }
        if (arow) {
            float *Arow = reinterpret_cast<float *>(sm + OFF_R1) + t * LA + 32 * hf;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *reinterpret_cast<float4 *>(Arow + 4 * c4) = make_float4(g[4 * c4], g[4 * c4 + 1], g[4 * c4 + 2], g[4 * c4 + 3]);
        } else {
            uint8_t *P = sm + OFF_P + (c & 1) * 8192;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                *reinterpret_cast<uint4 *>(P + sw128_off(t, 32 * hf + 8 * ch)) = pack8t<F16>(g + 8 * ch);
        }
    };
    // the two 32-token halves' inverses diag(T11, T22) -> Tinv*beta into T1, Tinv*beta*gamma
    // into T2[c&1], and the coupling -M21 (times 1/kappa in fold mode) into M21[c&1] (R1 and Y
    // as scratch); warps 4-7, idle in the solve's first phases, meanwhile turn the next
    // chunk's raw gates into arrays (warp 4) and (not from projections) form its X
    auto next_x = [&](int c) {
        if (c + 1 >= nchunks) return;
        if (warp == 4) compute_gates(c + 1);
        if (QED || prologue) return;                      // QED: the X rows (Ae) are loaded
        named_sync(kBarX, 128);                           // lambda of chunk c+1 in place
        wait_on(&bar_full[(c + 1) & 1], (uint32_t)(((c + 1) >> 1) & 1));
        x_pass(c + 1);
        fence_proxy_async();                              // X before the Gram reads it
    };
    auto solve = [&](int c) {
        const int gi = c & 3;
        const bool fold = g_ell[gi][kC - 1] > kFoldLog;
        unit_lower_inverse<true, F16>(reinterpret_cast<float *>(sm + OFF_R1), reinterpret_cast<float *>(sm + OFF_Y),
                                 sm + OFF_T, sm + OFF_T + 8192 + (c & 1) * 8192, g_beta[gi], g_gam[gi],
                                 [&]() { next_x(c); },
                                 []() { named_sync(kBarPrep, kPrepThreads); },
                                 sm + OFF_M21 + (c & 1) * 2048, fold ? g_gam[gi] : nullptr, g_igam[gi][kC - 1]);
    };
    // U^T = V^T T1^T into U[c&1] (bar_uw completes even without V)
    auto issue_u = [&](int c) {
        if (!p_issuer) return;
        const uint32_t sV = stage_addr(c) + OFF_V;
        const uint32_t tu = tm + TM_U + 64 * (uint32_t)(c & 1);
        if (!no_v())
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_bf16(tu, smem_desc(sV + k * 2048, 8192, 1024), smem_desc(sT + k * 32, 16, 1024),
                          idesc_16<F16>(128, 64, true, false), k > 0);
        umma_commit(&bar_uw);
    };

    // --------------------------------------------------------------- chain group
    // each chain thread owns TMEM lane d_row (a d_v row) and all of its columns
    // [S X^T | S Q^T] = S [X; Q]^T into SK | O (A = the bf16 state in TMEM, B = the XQ panels)
    auto issue_skq = [&](int c) {
        if (!c_issuer) return;
        wait_on(&bar_full[c & 1], (uint32_t)((c >> 1) & 1));
        const uint32_t sXQ = stage_addr(c) + OFF_XQ;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16_ta(tm + TM_SK, tm + TM_SB + 8 * k, smem_desc(sXQ + ko, 16, 1024),
                         idesc_16<F16>(128, 128, false, false), k > 0);
        }
        umma_commit(&bar_z);
    };
    // -(S X^T) as packed bf16 pairs into SK's first 32 columns (the A operand of Z)
    auto sx_pack = [&]() {
        float x[64];
        tmem_ld32(tl + TM_SK, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(tl + TM_SK + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_ld_wait();
        uint32_t xp[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) xp[j] = pack2<F16>(x[2 * j], x[2 * j + 1]) ^ 0x80008000u;
        tmem_st32(tl + TM_SK, xp);
        tmem_st_wait();
    };
    // strong decay: S Q^T <- (S Q^T) diag(gamma) in TMEM (gamma_t may underflow, the output
    // then takes no gamma), before Zt^T Pt^T accumulates onto it
    auto o_gamma = [&](int c) {
        const float *gam = g_gam[c & 3];
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
            float y[32];
            tmem_ld32(tl + TM_O + 32 * h2, y);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 v = fmul2(make_float2(y[j], y[j + 1]), *reinterpret_cast<const float2 *>(gam + 32 * h2 + j));
                y[j] = v.x;
                y[j + 1] = v.y;
            }
            tmem_st32(tl + TM_O + 32 * h2, y);
        }
        tmem_st_wait();
    };
    // K -> kappa K in place in chunk c's K slot (the operand of the state product)
    auto kappa_k = [&](int c) {
        uint8_t *st = sm + kring(c);
        const float *kap = g_kap[c & 3];
        const int ct = tid - kPrepThreads;
        uint4 kr[8];
        float ka[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {                     // all loads first
            const uint32_t off = (uint32_t)(ct + kChainThreads * r) << 4;   // both K panels
            kr[r] = *reinterpret_cast<const uint4 *>(st + off);
            ka[r] = kap[(off & 8191) >> 7];
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint32_t off = (uint32_t)(ct + kChainThreads * r) << 4;
            float kf[8];
            unpack8t<F16>(kr[r], kf);
#pragma unroll
            for (int e = 0; e < 8; ++e) kf[e] *= ka[r];
            *reinterpret_cast<uint4 *>(st + off) = pack8t<F16>(kf);
        }
    };
    // Z^T = U^T - (S X^T) T2^T = U^T - S W^T, accumulated into U[c&1] (A = -(S X^T) packed in TMEM)
    auto issue_z = [&](int c) {
        if (!c_issuer) return;
        const uint32_t tu = tm + TM_U + 64 * (uint32_t)(c & 1);
        const uint32_t sT2 = sT + 8192 + (uint32_t)(c & 1) * 8192;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16_ta(tu, tm + TM_SK + 8 * k, smem_desc(sT2 + k * 32, 16, 1024), idesc_16<F16>(128, 64, false, false),
                         (no_v() && k == 0) ? 0u : 1u);
        umma_commit(&bar_zz);
    };
    // 32 tokens of Z^T (fp32, columns 32 hf.. of U[c&1]) -> Zt^T as packed bf16 pairs into
    // columns 16 hf.. of U[c&1]; in fold mode Zt^T = Z^T diag(kappa)
    auto zt_pack = [&](int c, int hf2, bool fold) {
        const uint32_t tu = tl + TM_U + 64 * (uint32_t)(c & 1);
        const float *kap = g_kap[c & 3] + 32 * hf2;
        float z[32];
        tmem_ld32(tu + 32 * hf2, z);
        tmem_ld_wait();
        uint32_t zp[16];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {              // no shared-memory stores here: kappa read as needed
            const float4 kv = fold ? *reinterpret_cast<const float4 *>(kap + 2 * j) : make_float4(1.f, 1.f, 1.f, 1.f);
            const float2 a = fmul2(make_float2(z[2 * j], z[2 * j + 1]), make_float2(kv.x, kv.y));
            const float2 b = fmul2(make_float2(z[2 * j + 2], z[2 * j + 3]), make_float2(kv.z, kv.w));
            zp[j] = pack2<F16>(a.x, a.y);
            zp[j + 1] = pack2<F16>(b.x, b.y);
        }
        tmem_st16(tu + 16 * hf2, zp);
        tmem_st_wait();
    };
    // the solve's coupling: Z^T of tokens 32-63 -= Zt^T(tokens 0-31) (M21 diag(1/kappa))^T
    auto issue_couple = [&](int c) {
        if (!c_issuer) return;
        const uint32_t tu = tm + TM_U + 64 * (uint32_t)(c & 1);
        const uint32_t sM = sbase + OFF_M21 + (uint32_t)(c & 1) * 2048;
#pragma unroll
        for (int k = 0; k < 2; ++k)                       // K = 16 tokens = two core matrices along K
            umma_bf16_ta(tu + 32, tu + 8 * k, smem_desc_noswz(sM + k * 256, 128, 512),
                         idesc_16<F16>(128, 32, false, false), 1);
        umma_commit(&bar_cp);
    };
    // O += Zt^T Pt^T ; S += Zt^T (kappa K)  (S in TMEM already scaled by gamma_C); A = Zt^T in TMEM
    auto issue_mma2 = [&](int c) {
        if (!c_issuer) return;
        const uint32_t sK = sbase + kring(c), sP = sbase + OFF_P + (uint32_t)(c & 1) * 8192;
        const uint32_t tz = tm + TM_U + 64 * (uint32_t)(c & 1);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            umma_bf16_ta(tm + TM_S, tz + 8 * k, smem_desc(sK + k * 2048, 8192, 1024),
                         idesc_16<F16>(128, 128, false, true), 1);
        if (!no_o())
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_bf16_ta(tm + TM_O, tz + 8 * k, smem_desc(sP + k * 32, 16, 1024),
                             idesc_16<F16>(128, 64, false, false), 1);
        umma_commit(&bar_o2);
    };
    // the state of this thread's row, 64 columns from column 64 h: packed bf16 copy into
    // the state A operand, fp32 scaled by g back into the master state
    auto state_half = [&](int half, float (&sv)[64], float g, bool store_back) {
        uint32_t sp[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) sp[j] = pack2<F16>(sv[2 * j], sv[2 * j + 1]);
        tmem_st32(tl + TM_SB + 32 * half, sp);
        if (store_back) {
            if (!QED)                                 // QED: unit gates, gamma_C = 1
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 x = fmul2(make_float2(sv[e], sv[e + 1]), make_float2(g, g));
                    sv[e] = x.x;
                    sv[e + 1] = x.y;
                }
            tmem_st32(tl + TM_S + 64 * half, *reinterpret_cast<float(*)[32]>(sv));
            tmem_st32(tl + TM_S + 64 * half + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
        }
    };
    // state -> packed bf16 state for the next chunk, rescaled in TMEM by the next chunk's
    // gamma_C (or written out after the last); o_t = gamma_t O_t (or O_t) through a
    // shared-memory tile and two TMA stores
    auto epilogue = [&](int c) {
        const int t0 = c * kC;
        const bool last = (c + 1 == nchunks);
        const float gN = last ? 1.f : g_gam[(c + 1) & 3][kC - 1];
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            float sv[64];
            tmem_ld32(tl + TM_S + 64 * half, *reinterpret_cast<float(*)[32]>(sv));
            tmem_ld32(tl + TM_S + 64 * half + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
            tmem_ld_wait();
            if (QED) {                                // S <- (S + Z^T Ke) diag(e^{G_C}), staged in ECG
                const float *ecg = reinterpret_cast<const float *>(sm + OFF_ECG) + 64 * half;
#pragma unroll
                for (int e = 0; e < 64; e += 4) {
                    const float4 f = *reinterpret_cast<const float4 *>(ecg + e);
                    const float2 x = fmul2(make_float2(sv[e], sv[e + 1]), make_float2(f.x, f.y));
                    const float2 y = fmul2(make_float2(sv[e + 2], sv[e + 3]), make_float2(f.z, f.w));
                    sv[e] = x.x; sv[e + 1] = x.y; sv[e + 2] = y.x; sv[e + 3] = y.y;
                }
            }
            if (CHK && !last) {
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + ((size_t)bh * nchunks + c + 1) * kChkTileBytes;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(dst + chk_tile_off(d_row, 64 * half + 8 * ch)) = pack8hp(sv + 8 * ch);
            }
            if (last && opaque(p.S_final) && !abort_flag) {
                float *dst = p.S_final + ((size_t)bh * kD + d_row) * kD + 64 * half;
#pragma unroll
                for (int j = 0; j < 64; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
            }
            state_half(half, sv, gN, !last);
        }
        if (!no_o()) {
            const bool gscale = g_ell[c & 3][kC - 1] > kSplitLog;
            const float *gam = g_gam[c & 3];
            // [64 tokens][dv] tile, two 64-column panels (the previous tile's store has read it).
            // Each 16-lane half of this warp's TMEM quarter is read in the 16x256b shape, so a
            // thread holds two adjacent tokens of d_v rows L + t/4 and L + 8 + t/4; the 8x8
            // blocks (tokens x d_v) then go out as transposed stmatrix rows of 16 bytes.
            const int t4 = lane & 3;
            float2 gv[8];                                 // gamma of tokens 8j + 2 t4, + 1
#pragma unroll
            for (int j = 0; j < 8; ++j)
                gv[j] = gscale ? *reinterpret_cast<const float2 *>(gam + 8 * j + 2 * t4) : make_float2(1.f, 1.f);
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const int L = 32 * q4 + 16 * half;        // first d_v row of these 16 lanes
                float ov[32];
                tmem_ld16x256_x8(tm + TM_O + ((uint32_t)L << 16), ov);
                tmem_ld_wait();
                uint32_t pk[16];                          // pk[2j + h]: rows L + 8h + r8, tokens 8j + 2 t4, + 1
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 lo = fmul2(make_float2(ov[4 * j], ov[4 * j + 1]), gv[j]);
                    const float2 hi = fmul2(make_float2(ov[4 * j + 2], ov[4 * j + 3]), gv[j]);
                    pk[2 * j] = pack2<F16>(lo.x, lo.y);
                    pk[2 * j + 1] = pack2<F16>(hi.x, hi.y);
                }
                // matrix m = lane / 8 of each store: tokens 8 (j + m/2) + lane%8, d_v L + 8 (m%2) ..
                const int m = lane >> 3, col = L + 8 * (m & 1);
                const uint32_t obase = sbase + kring(c) + (uint32_t)(col >> 6) * 8192;
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    const int tok = 8 * (j + (m >> 1)) + (lane & 7);
                    stmatrix_x4_trans(obase + sw128_off(tok, col & 63), pk[2 * j], pk[2 * j + 1], pk[2 * j + 2],
                                      pk[2 * j + 3]);
                }
            }
            fence_proxy_async();
            named_sync(kBarChain, kChainThreads);
            if (c_issuer) {                               // rows past T are clipped by the copy
                if (QED) {
                    tma_store_5d(&tmO, sm + kring(c), 0, t0, 0, h, b);
                } else if (F16) {                         // odd sub-tokens fall outside the pair map;
                    if (t0 / 2 < (T - 1) / 2) {           // a chunk holding only sub-token 2T' stores nothing
                        tma_store_5d(&tmO, sm + kring(c), 0, 0, h, t0 / 2, b);
                        tma_store_5d(&tmO, sm + kring(c) + 8192, 64, 0, h, t0 / 2, b);
                    }
                } else {
                    tma_store_4d(&tmO, sm + kring(c), 0, h, t0, b);
                    tma_store_4d(&tmO, sm + kring(c) + 8192, 64, h, t0, b);
                }
                tma_store_commit();
            }
        }
        tmem_st_wait();
    };

    int loads_issued = nchunks > 1 ? 2 : 1;             // the chain issuer's bookkeeping for a drain
    if (prep) {
        // chunk 0's X and Gram; afterwards chunk c+1's X is formed during solve(c) and its
        // Gram issued beside U(c)
        wait_on(&bar_full[0], 0);
        if (!QED && (prologue || warp >= 4)) x_pass(0);   // QED: the X rows (Ae) are loaded
        psync();
        if (g_issuer) issue_gram(0);
        for (int c = 0; c < nchunks; ++c) {
            if (warp == 4 && c + 1 < nchunks) load_gates(c + 1);   // arrays built in solve(c)
            wait_mma(&bar_g, c);
            if (c >= 2) {                                 // P[c&1] and U[c&1] free
                wait_on(&bar_cdone[c & 1], (uint32_t)(((c - 2) >> 1) & 1));
                tc_fence_after();
            }
            masks(c);
            tc_fence_before();
            named_sync(kBarPrep, kPrepThreads);
            tc_fence_after();
            if (c >= 1) wait_mma(&bar_uw, c - 1);         // T1 free: U of chunk c-1 has run
            solve(c);
            psync();
            if (prologue && c + 1 < nchunks) {            // from projections: X(c+1) after the solve
                wait_on(&bar_full[(c + 1) & 1], (uint32_t)(((c + 1) >> 1) & 1));
                x_pass(c + 1);
                psync();
            }
            // three threads at once: the hand-off, U(c), the Gram of chunk c+1
            if ((tid == 0 || p_issuer) && c >= 1) wait_on(&bar_taken, (uint32_t)((c - 1) & 1));   // see `taken`
            if (tid == 0) mbar_arrive(&bar_ready);        // P(c), T2(c), gates(c+1), X(c+1) in place
            if (g_issuer && c + 1 < nchunks) {            // TM_G was read by masks(c), X(c+1) formed
                wait_on(&bar_full[(c + 1) & 1], (uint32_t)(((c + 1) >> 1) & 1));
                issue_gram(c + 1);
            }
            issue_u(c);
            tc_fence_before();
            const bool stop = named_sync_or(kBarPrep, kPrepThreads, abort_flag != 0);
            tc_fence_after();
            if (stop) break;
        }
    } else {
        // initial state: packed bf16 copy and fp32 state (scaled by chunk 0's gamma_C) in TMEM
        {
            const size_t base = ((size_t)bh * kD + d_row) * kD;
            const float g0 = g_gam[0][kC - 1];
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float sv[64];
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    float4 v = p.S0 ? *reinterpret_cast<const float4 *>(p.S0 + base + 64 * half + j)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                    sv[j] = v.x; sv[j + 1] = v.y; sv[j + 2] = v.z; sv[j + 3] = v.w;
                }
                if (s0_id)
#pragma unroll
                    for (int j = 0; j < 64; ++j) sv[j] = (64 * half + j == d_row) ? 1.f : 0.f;
                if (CHK) {
                    uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + (size_t)bh * nchunks * kChkTileBytes;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        *reinterpret_cast<uint4 *>(dst + chk_tile_off(d_row, 64 * half + 8 * ch)) = pack8hp(sv + 8 * ch);
                }
                state_half(half, sv, g0, true);
            }
            tmem_st_wait();
        }
        csync();
        for (int c = 0; c < nchunks; ++c) {
            // QED: this chunk's e^{G_C}, element d_row
            const float ecg = QED ? p.ecg[((size_t)bh * nchunks + c) * kD + d_row] : 0.f;
            // S [X; Q]^T as soon as the state of chunk c-1 is final (X of chunk c was formed
            // before `ready` of chunk c-1; that of chunk 0 before `ready` of chunk 0)
            // K of chunk c + 2 goes into the slot of chunk c - 1, whose o tile the store has read
            if (c > 0) issue_skq(c);
            if (c > 0 && c_issuer && c + 2 < nchunks) {
                tma_store_wait_read0();
                issue_k(c + 2);
            }
            wait_on(&bar_ready, (uint32_t)(c & 1));
            if (c == 0) {
                issue_skq(0);
                if (c_issuer && nchunks > 2) issue_k(2);
            }
            wait_mma(&bar_uw, c);
            if (c_issuer) mbar_arrive(&bar_taken);
            const float lC = g_ell[c & 3][kC - 1];
            const bool fold = lC > kFoldLog, split = lC > kSplitLog;
            wait_mma(&bar_z, c);
            if (!QED && c_issuer && c + 2 < nchunks) {    // S [X; Q]^T and U of chunk c have run
                issue_xqv(c + 2);
                ++loads_issued;
            }
            sx_pack();
            if (!split) o_gamma(c);
            if (!fold) kappa_k(c);
            if (QED) reinterpret_cast<float *>(sm + OFF_ECG)[d_row] = ecg;   // read after the csyncs below
            csync();
            issue_z(c);
            wait_mma(&bar_zz, c);
            zt_pack(c, 0, fold);
            csync();
            issue_couple(c);
            wait_mma(&bar_cp, c);
            zt_pack(c, 1, fold);
            csync();
            issue_mma2(c);
            if (QED && c_issuer && c + 2 < nchunks) {     // QED forms no X: the next tiles can wait
                issue_xqv(c + 2);                         // until the issuer waits anyway
                ++loads_issued;
            }
            wait_mma(&bar_o2, c);
            if (c_issuer) mbar_arrive(&bar_cdone[c & 1]);
            epilogue(c);
            tc_fence_before();
            const bool stop = named_sync_or(kBarChain, kChainThreads, abort_flag != 0);
            tc_fence_after();
            if (stop) break;
        }
    }

    if (c_issuer) tma_store_wait_all();
    if (abort_flag) {
        // wind down: let this CTA's copies and MMAs finish (bounded) before freeing TMEM
        if (c_issuer)
            for (int s = 0; s < 2; ++s) {
                const int n_s = (loads_issued + 1 - s) / 2;   // loads issued into stage s
                if (n_s > 0) mbar_wait(&bar_full[s], (uint32_t)((n_s - 1) & 1), kWaitNs);
            }
        if (p_issuer || g_issuer || c_issuer) {
            uint64_t *dr = &bar_drain[p_issuer ? 0 : g_issuer ? 2 : 1];
            umma_commit(dr);
            mbar_wait(dr, 0, kWaitNs);
        }
        if (lane == 0) atomicExch(&g_tc_timeout, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

bool qdelta_tc_supported(const QDeltaArgs &a, int dtype) {
    if (a.T <= 0) return false;
    return dtype == kBF16 && a.dk == kD && a.dv == kD && (long long)a.T * a.H * kD * 2 < (1ll << 40);
}

cudaError_t launch_qdelta_chunk_tc(const QDeltaArgs &a, cudaStream_t s, int *nlaunch, int flags) {
    CUtensorMap mq, mk, mv, mo;
    const bool f16 = (flags & kTcF16) != 0;
    if (f16) {                                        // q, v, o compact over (a.T - 1) / 2 pair rows
        if (a.S_chk || a.prologue || a.alpha || (flags & (kTcNoO | kTcNoV)) || a.T % 2 == 0)
            return cudaErrorInvalidValue;             // no decay in fp16; the EDA sub-token layout
        const int Tc = (a.T - 1) / 2;
        if (!make_pair_map(&mq, a.q, a.B, Tc, a.H) || !make_token_map(&mk, a.k, a.B, a.T, a.H) ||
            !make_pair_map(&mv, a.v, a.B, Tc, a.H) || !make_pair_map(&mo, a.o, a.B, Tc, a.H))
            return cudaErrorInvalidValue;
    } else {
        if (!make_token_map(&mq, a.q, a.B, a.T, a.H) || !make_token_map(&mk, a.k, a.B, a.T, a.H) ||
            !make_token_map(&mv, a.v, a.B, a.T, a.H))
            return cudaErrorInvalidValue;
        if (flags & kTcNoO) mo = mq;                  // not used
        else if (!make_token_map(&mo, a.o, a.B, a.T, a.H)) return cudaErrorInvalidValue;
    }
    auto kern = f16 ? qdelta_fwd_tc_kernel<false, false, false, true>
              : a.S_chk ? (a.prologue ? qdelta_fwd_tc_kernel<true, true> : qdelta_fwd_tc_kernel<false, true>)
              : a.prologue ? qdelta_fwd_tc_kernel<true> : qdelta_fwd_tc_kernel<false>;
    if (a.S_chk && !(flags & kTcNoO)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    TcParams p{(const __nv_bfloat16 *)a.alpha, (const __nv_bfloat16 *)a.beta, (const __nv_bfloat16 *)a.lam,
               a.S0, a.S_chk ? (__nv_bfloat16 *)a.S_chk : (__nv_bfloat16 *)a.o, a.S_final, a.B, a.T, a.H, flags,
               nullptr};
    kern<<<a.B * a.H, kAllThreads, kSmemBytes, s>>>(p, mq, mk, mv, mo, mq);
    e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

cudaError_t launch_qed_chain_tc(const QedArgs &a, const QedDerived &d, cudaStream_t s, int *nlaunch, int flags) {
    CUtensorMap ma, mq, mk, mv, mo;
    if (!make_token_map(&ma, d.Ae, a.B, a.T, a.H) || !make_token_map(&mq, d.Qe, a.B, a.T, a.H) ||
        !make_token_map_tile(&mk, d.Ke, a.B, a.T, a.H) || !make_token_map_tile(&mv, d.WV, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    if (flags & kTcNoO) mo = mq;                      // not used
    else if (!make_token_map_tile(&mo, a.o, a.B, a.T, a.H)) return cudaErrorInvalidValue;
    auto kern = qdelta_fwd_tc_kernel<false, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    TcParams p{nullptr, nullptr, nullptr, a.S0, (__nv_bfloat16 *)a.o, a.S_final, a.B, a.T, a.H, flags, d.ecg};
    kern<<<a.B * a.H, kAllThreads, kSmemBytes, s>>>(p, mq, mk, mv, mo, ma);
    e = cudaGetLastError();
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

// One cooperative launch (all CTAs resident at once): the chains of the B*H streams and,
// on the remaining SMs, the derive step feeding them chunk by chunk through `done`.
cudaError_t launch_qed_fused_tc(const QedArgs &a, const QedDerived &d, unsigned int *done, cudaStream_t s,
                                int *nlaunch) {
    CUtensorMap ma, mq, mk, mv, mo;
    if (!make_token_map(&ma, d.Ae, a.B, a.T, a.H) || !make_token_map(&mq, d.Qe, a.B, a.T, a.H) ||
        !make_token_map_tile(&mk, d.Ke, a.B, a.T, a.H) || !make_token_map_tile(&mv, d.WV, a.B, a.T, a.H) ||
        !make_token_map_tile(&mo, a.o, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    auto kern = qdelta_fwd_tc_kernel<false, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    int per_sm = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kAllThreads, (size_t)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int bhn = a.B * a.H, grid = sm_count() * per_sm, nchunks = (a.T + kC - 1) / kC;
    if (grid <= bhn) return cudaErrorInvalidValue;    // qed_fused_supported
    e = cudaMemsetAsync(done, 0, (size_t)bhn * nchunks * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const QedDeriveParams dp{(const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v,
                             (const __nv_bfloat16 *)a.g, (const __nv_bfloat16 *)a.b, (const __nv_bfloat16 *)a.w,
                             a.lam_h, a.z, (__nv_bfloat16 *)d.Ae, (__nv_bfloat16 *)d.Qe, (__nv_bfloat16 *)d.Ke,
                             (__nv_bfloat16 *)d.WV, d.ecg, a.B, a.T, a.H, a.variant, 0};
    const TcParams p{nullptr, nullptr, nullptr, a.S0, (__nv_bfloat16 *)a.o, a.S_final, a.B, a.T, a.H, 0, d.ecg,
                     bhn, done, dp};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kAllThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv, mo, ma);
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

bool tc_read_and_clear_timeout() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_timeout, sizeof v) != cudaSuccess) return false;
    if (v) cudaMemcpyToSymbol(g_tc_timeout, &zero, sizeof zero);
    return v != 0;
}

}  // namespace qd

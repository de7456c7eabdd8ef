// EDA, erase-then-delta ("Erase-then-Delta Attention", core method): per token,
//   M <- M - e (e^T M)                 targeted erase along e
//   M <- M - beta k (k^T M - v^T)      Delta write along the key (beta = 1 on the page)
//   o = M^T q
// held as S = M^T ([dv][dk], fp32):  S <- S - (S e) e^T,  S <- S - beta (S k - v) k^T,
// o = S q.
//
// A recurrent kernel in fp32, one CTA per (b, h): the state stays in registers for
// the whole sequence, and each token costs three row-dot products (S e, S k, S q), each
// reduced over the threads of a row by shuffles, and two rank-one updates: 5 dv dk
// multiply-adds.  The kernel is issue bound, so the thread layout is chosen to spend the
// fewest instructions beside those multiply-adds: for d_k >= 64 a thread holds four state
// rows over 8 columns, so each token slice it unpacks from bf16 and each shared-memory
// read serve four rows (at d_k = 128: 7 % faster than one row over 32 columns, and 0.5 %
// faster than two rows over 16); one row over 8 threads measured slower (one more
// shuffle level, no fewer unpacks).  The token
// vectors are staged in shared memory a tile of 16 tokens at a time by asynchronous
// copies (cp.async), the next tile's in flight while the current one is consumed, and
// converted to fp32 as they are read (a separate fp32 tile measured slower: twice the
// shared-memory reads).  Folding the two updates of a token into one (three row-dot
// products in one pass against the token scalars e.k, e.q, k.q, computed once per tile)
// shortens the dependency chain but measured 13 % slower: as many instructions plus a
// barrier per tile.
//
// Why not the chunked tensor-core forward: EDA is the Delta rule over the 2T
// sub-tokens (e_t, 0, beta 1), (k_t, v_t, beta_t), and that runs through the chunked
// kernels, but with the page's e = q/|q| the erase sub-token's residual is the whole
// S q, which the read-out then cancels to a small o; the bf16 operands of the
// tensor-core path leave an error of 2^-9 |S| on a result often ten times smaller
// than |S|.  The recurrence in fp32 has no such cancellation error.
#include "qd_internal.cuh"
#include "sm103_ptx.cuh"

namespace qd {
namespace {

using ptx::ffma2;

constexpr int kTile = 16;   // tokens per staged tile

__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// W = 4 or 8 consecutive elements at p as fp32 (fp32: 16-byte aligned; bf16: 2W-byte aligned)
template <int W>
__device__ __forceinline__ void loadw(const float *p, float (&x)[W]) {
#pragma unroll
    for (int i = 0; i < W; i += 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p + i);
        x[i] = a.x; x[i + 1] = a.y; x[i + 2] = a.z; x[i + 3] = a.w;
    }
}
template <int W>
__device__ __forceinline__ void loadw(const __nv_bfloat16 *p, float (&x)[W]) {
    uint32_t w[W / 2];
    if constexpr (W == 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        w[0] = u.x; w[1] = u.y;
    }
#pragma unroll
    for (int i = 0; i < W / 2; ++i) {                 // bf16 -> fp32 is exact: the 16 bits on top
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Shared-memory layout of one staged token (elements of TIn): e, k, q as TPR slices
// of NS elements each, every slice padded so that the slices of a vector start in
// different banks; then v (dv elements), and 16 bytes.
template <typename TIn, int DK, int TPR>
struct TokenLayout {
    static constexpr int E = (int)sizeof(TIn);
    static constexpr int NS = DK / TPR;
    // padded slice: an odd number of 16-byte groups (so the slices of a vector start in
    // different bank groups) that keeps every read of W elements aligned
    static constexpr int SL = NS + ((NS * E) % 32 == 16 ? 32 : 16) / E;
    static constexpr int VS = TPR * SL;               // one padded vector
    __host__ __device__ static int stride(int dv) { return 3 * VS + dv + 16 / E; }
    __host__ __device__ static size_t bytes(int dv) {
        return (size_t)2 * kTile * stride(dv) * E + sizeof(float) * (2 * kTile + (size_t)kTile * dv);
    }
};

// R state rows per thread (1, 2 or 4) over TPR threads per row.  A thread holds rows
// rg + rho dv/R, rho < R (rg = tid / TPR), over the same d_k/TPR columns, so one
// unpacked token slice serves R rows.  Its own row rho* = s / (TPR/R) (s = tid % TPR) is
// the one whose reduction it completes; its registers hold row rho* ^ m in slot m, so
// the partner at lane offset TPR/2, TPR/4, ... (own row rho* ^ R/2, rho* ^ R/4, ...) holds
// this thread's slot m in its slot m ^ R/2, m ^ R/4, ...: each of the first log2 R shuffle
// levels keeps the lower half of the slots and adds the partner's upper half, with no
// selects.
template <typename TIn, int DK, int TPR, int R>
__global__ void __launch_bounds__(TPR * 128 / R, 1) eda_recurrent_kernel(EdaArgs a) {
    static_assert((R == 1 || R == 2 || R == 4) && TPR % R == 0, "1, 2 or 4 rows per thread");
    using L = TokenLayout<TIn, DK, TPR>;
    constexpr int NS = L::NS, SL = L::SL, VS = L::VS, E = L::E;
    constexpr int P8 = 8 / E;                         // elements per 8-byte copy
    constexpr int W = NS >= 8 ? 8 : 4;                // elements per shared-memory read
    extern __shared__ __align__(16) uint8_t smraw[];
    const int dv = a.dv, T = a.T, H = a.H;
    const int TS = L::stride(dv);
    TIn *stage_base = reinterpret_cast<TIn *>(smraw);
    float *bet = reinterpret_cast<float *>(smraw + (size_t)2 * kTile * TS * E);   // [2][kTile]
    float *obuf = bet + 2 * kTile;                                                // [kTile][dv]

    const int tid = threadIdx.x, rg = tid / TPR, s = tid % TPR;
    const int own = s / (TPR / R);                    // rho*
    auto row_of = [&](int m) { return rg + (m ^ own) * (dv / R); };
    const int row = row_of(0);                        // own row
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v, *e = (const TIn *)a.e;
    const TIn *beta = (const TIn *)a.beta;
    const int nthreads = TPR * dv / R;
    const int per_tok = (3 * DK + dv) / P8;           // 8-byte copies per token

    float S[R][NS];                                   // slot m: row rho* ^ m
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const size_t base = ((size_t)bh * dv + row_of(r)) * DK + s * NS;
#pragma unroll
        for (int j = 0; j < NS; ++j) S[r][j] = a.S0 ? a.S0[base + j] : 0.f;
    }
    // issue the asynchronous copies of tile `tile` into buffer `buf` (tokens past T are
    // not copied: their staged values are never read); beta of token tid of the tile is
    // returned to threads tid < kTile
    auto stage = [&](int tile, int buf) {
        const int t0 = tile * kTile, nt = min(kTile, T - t0);
        TIn *dst = stage_base + (size_t)buf * kTile * TS;
        for (int u = tid; u < nt * per_tok; u += nthreads) {
            const int t = u / per_tok, c = (u % per_tok) * P8;
            const size_t tok = ((size_t)b * T + t0 + t) * H + h;
            const TIn *src;
            TIn *slot;
            if (c < 3 * DK) {
                const int which = c / DK, j = c % DK;
                src = (which == 0 ? e : which == 1 ? k : q) + tok * DK + j;
                slot = dst + t * TS + which * VS + (j / NS) * SL + j % NS;
            } else {
                src = v + tok * dv + (c - 3 * DK);
                slot = dst + t * TS + 3 * VS + (c - 3 * DK);
            }
            cp_async8(slot, src);
        }
        cp_async_commit();
        float bv = 0.f;
        if (tid < nt) bv = beta ? to_f(beta[((size_t)b * T + t0 + tid) * H + h]) : 1.f;
        return bv;
    };
    // the own row's dot product with x, reduced over the row's TPR threads (the first
    // log2 R levels trade slots, as above)
    auto rowdot = [&](const TIn *x) {                 // packed pairs: one instruction per two products
        float2 acc[R == 1 ? 2 : R];
#pragma unroll
        for (int m = 0; m < (R == 1 ? 2 : R); ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NS; j += W) {
            float w[W];
            loadw<W>(x + j, w);
#pragma unroll
            for (int i = 0; i < W; i += 2) {
                const float2 wi = make_float2(w[i], w[i + 1]);
                if constexpr (R == 1) {               // two chains over one row
                    acc[(i >> 1) & 1] = ffma2(make_float2(S[0][j + i], S[0][j + i + 1]), wi, acc[(i >> 1) & 1]);
                } else {
#pragma unroll
                    for (int m = 0; m < R; ++m)
                        acc[m] = ffma2(make_float2(S[m][j + i], S[m][j + i + 1]), wi, acc[m]);
                }
            }
        }
        float p[R == 1 ? 2 : R];
#pragma unroll
        for (int m = 0; m < (R == 1 ? 2 : R); ++m) p[m] = acc[m].x + acc[m].y;
        if constexpr (R == 1) p[0] += p[1];
        int off = TPR / 2;
#pragma unroll
        for (int half = R / 2; half; half >>= 1, off >>= 1) {
#pragma unroll
            for (int m = 0; m < half; ++m) p[m] += __shfl_xor_sync(0xffffffffu, p[m + half], off);
        }
        for (; off; off >>= 1) p[0] += __shfl_xor_sync(0xffffffffu, p[0], off);
        return p[0];
    };
    // a per-row scalar for every slot: slot m's row is the own row of lane s ^ m (TPR/R)
    auto spread = [&](float c, float (&cs)[R]) {
        cs[0] = c;
#pragma unroll
        for (int m = 1; m < R; ++m) cs[m] = __shfl_xor_sync(0xffffffffu, c, m * (TPR / R));
    };
    auto axpy = [&](const float (&cs)[R], const TIn *x) {   // slot m -= cs[m] x
#pragma unroll
        for (int j = 0; j < NS; j += W) {
            float w[W];
            loadw<W>(x + j, w);
#pragma unroll
            for (int i = 0; i < W; i += 2) {
                const float2 wi = make_float2(w[i], w[i + 1]);
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    const float2 r = ffma2(make_float2(-cs[m], -cs[m]), wi, make_float2(S[m][j + i], S[m][j + i + 1]));
                    S[m][j + i] = r.x;
                    S[m][j + i + 1] = r.y;
                }
            }
        }
    };

    const int ntiles = (T + kTile - 1) / kTile;
    if (ntiles > 0) {
        const float bv = stage(0, 0);
        if (tid < kTile) bet[tid] = bv;
    }
    for (int tile = 0; tile < ntiles; ++tile) {
        cp_async_wait_all();
        __syncthreads();                              // tile's copies and beta visible; obuf free
        float bnext = 0.f;
        if (tile + 1 < ntiles) bnext = stage(tile + 1, (tile + 1) & 1);   // buffer last read two tiles ago
        const TIn *cur = stage_base + (size_t)(tile & 1) * kTile * TS;
        const float *bcur = bet + (tile & 1) * kTile;
        const int nt = min(kTile, T - tile * kTile);
        for (int t = 0; t < nt; ++t) {
            const TIn *tk = cur + t * TS;
            const TIn *ev = tk + s * SL, *kv = tk + VS + s * SL, *qv = tk + 2 * VS + s * SL;
            const float vi = to_f(tk[3 * VS + row]), bt = bcur[t];
            float cs[R];
            spread(rowdot(ev), cs);                   // erase: S <- S - (S e) e^T
            axpy(cs, ev);
            spread(bt * (rowdot(kv) - vi), cs);       // write: S <- S - beta (S k - v) k^T
            axpy(cs, kv);
            const float o = rowdot(qv);               // o = S q
            if ((s & (TPR / R - 1)) == 0) obuf[t * dv + row] = o;
        }
        if (tile + 1 < ntiles && tid < kTile) bet[((tile + 1) & 1) * kTile + tid] = bnext;
        __syncthreads();                              // outputs of the tile complete
        const int t0 = tile * kTile;
        for (int idx = tid; idx < nt * dv; idx += nthreads) {
            const int t = idx / dv, i = idx % dv;
            ((TIn *)a.o)[(((size_t)b * T + t0 + t) * H + h) * dv + i] = from_f<TIn>(obuf[idx]);
        }
    }
    if (a.S_final) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const size_t base = ((size_t)bh * dv + row_of(r)) * DK + s * NS;
#pragma unroll
            for (int j = 0; j < NS; ++j) a.S_final[base + j] = S[r][j];
        }
    }
}

template <typename TIn, int DK, int TPR, int R>
cudaError_t run_eda(const EdaArgs &a, cudaStream_t s) {
    const size_t smem = TokenLayout<TIn, DK, TPR>::bytes(a.dv);
    auto kern = eda_recurrent_kernel<TIn, DK, TPR, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<a.B * a.H, TPR * a.dv / R, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_eda(const EdaArgs &a, cudaStream_t s) {
    switch (a.dk) {
        case 16: return run_eda<TIn, 16, 4, 1>(a, s);
        case 32: return run_eda<TIn, 32, 4, 1>(a, s);
        case 64: return run_eda<TIn, 64, 8, 4>(a, s);       // 8 columns x 4 rows a thread
        case 128: return run_eda<TIn, 128, 16, 4>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_eda(const EdaArgs &a, int dtype, cudaStream_t s, int *nlaunch) {
    cudaError_t e = dtype == kBF16 ? dispatch_eda<__nv_bfloat16>(a, s) : dispatch_eda<float>(a, s);
    if (e == cudaSuccess) *nlaunch += 1;
    return e;
}

}  // namespace qd

// Pieces shared by the tensor-core chunk kernels (Q-Delta and QED): tile sizes,
// bf16 packing, the fp32 unit-lower-triangular inverse of one 64x64 chunk matrix,
// and the TMA tensor maps of the [B][T][H][128] token tensors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace qd {
namespace tc {

using namespace ptx;

constexpr int kC = 64, kD = 128, kThreads = 256;
constexpr int LA = 68;                 // fp32 row stride of the 64x64 chunk matrix (16-byte rows)
constexpr int LY = 36;                 // fp32 row stride of the 32x32 scratch

// Named barrier `id` over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns the OR of `pred` over the participating threads,
// so that every thread of the group takes the same decision.
__device__ __forceinline__ bool named_sync_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float bf(__nv_bfloat16 x) { return __bfloat162float(x); }

// Returns v unchanged but hides it from the optimiser.  A loop-invariant flag or
// nullable pointer tested inside a long loop would otherwise let the compiler copy
// the whole loop once per value (loop unswitching), multiplying the kernel's code
// size; instruction fetch is then a measurable share of the stall cycles.
__device__ __forceinline__ uint32_t opaque(uint32_t v) {
    asm volatile("" : "+r"(v));
    return v;
}
template <typename T> __device__ __forceinline__ T *opaque(T *v) {
    asm volatile("" : "+l"(v));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
// eight consecutive floats (from f[0]) -> eight bf16
__device__ __forceinline__ uint4 pack8p(const float *f) {
    uint4 u;
    u.x = pack_bf16x2(f[0], f[1]);
    u.y = pack_bf16x2(f[2], f[3]);
    u.z = pack_bf16x2(f[4], f[5]);
    u.w = pack_bf16x2(f[6], f[7]);
    return u;
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) { return pack8p(f); }

// The same for fp16 (the operands of a kind::f16 product taken as f16)
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void unpack8h(const uint4 &u, float (&f)[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 pack8hp(const float *f) {
    uint4 u;
    u.x = pack_half2(f[0], f[1]);
    u.y = pack_half2(f[2], f[3]);
    u.z = pack_half2(f[4], f[5]);
    u.w = pack_half2(f[6], f[7]);
    return u;
}
// two 16-bit values of the chosen type
template <bool kHalf> __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kHalf ? pack_half2(lo, hi) : pack_bf16x2(lo, hi);
}
// eight 16-bit values of the chosen type to / from fp32
template <bool kHalf> __device__ __forceinline__ void unpack8t(const uint4 &u, float (&f)[8]) {
    if (kHalf) unpack8h(u, f);
    else unpack8(u, f);
}
template <bool kHalf> __device__ __forceinline__ uint4 pack8t(const float *f) {
    return kHalf ? pack8hp(f) : pack8p(f);
}
template <bool kHalf> __device__ __forceinline__ uint16_t cvt16(float x) {
    if (kHalf) {
        __half v = __float2half_rn(x);
        return *reinterpret_cast<uint16_t *>(&v);
    }
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&v);
}


// ---------------------------------------------------------- warp-level TF32 MMA
// The merge steps of the inverse are 16x8 output tiles with K = 16 or 32: too small
// and too latency-bound for tcgen05 (its TMEM round trip alone exceeds the work),
// so they run on the warp-synchronous m16n8k8 TF32 MMA with operands read straight
// from shared memory.  One TF32 product per step: its rounding (unit roundoff
// 2^-11) stays well below the bf16 rounding (2^-8) that every entry of the inverse
// receives before it is used, so a split hi/lo product would buy no accuracy.
// Fragment layout of m16n8k8 (lane = 4 g + t): A (16x8) a0 (g, t), a1 (g+8, t),
// a2 (g, t+4), a3 (g+8, t+4); B (8x8) b0 (t, g), b1 (t+4, g); C/D (16x8) c0 (g, 2t),
// c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d = C + A B for one 16x8 tile: A 16 x K (row stride lda), B K x 8 (row stride ldb),
// C 16 x 8 (row stride ldc), all fp32 in shared memory.  Every load comes before the
// caller's stores.
template <int K>
__device__ __forceinline__ void tile_cab(float (&d)[4], const float *C, int ldc, const float *A, int lda,
                                         const float *B, int ldb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint32_t a[K / 8][4], b[K / 8][2];
#pragma unroll
    for (int s = 0; s < K / 8; ++s) {                  // every operand load first
        const int k0 = 8 * s;
        a[s][0] = to_tf32(A[g * lda + k0 + t]);
        a[s][1] = to_tf32(A[(g + 8) * lda + k0 + t]);
        a[s][2] = to_tf32(A[g * lda + k0 + t + 4]);
        a[s][3] = to_tf32(A[(g + 8) * lda + k0 + t + 4]);
        b[s][0] = to_tf32(B[(k0 + t) * ldb + g]);
        b[s][1] = to_tf32(B[(k0 + t + 4) * ldb + g]);
    }
    float x[2][4] = {{C[g * ldc + 2 * t], C[g * ldc + 2 * t + 1], C[(g + 8) * ldc + 2 * t],
                      C[(g + 8) * ldc + 2 * t + 1]},
                     {0.f, 0.f, 0.f, 0.f}};             // two accumulators: short chains
#pragma unroll
    for (int s = 0; s < K / 8; ++s) mma_tf32(x[s & 1], a[s], b[s][0], b[s][1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = x[0][i] + x[1][i];
}
// stores s * d into the 16x8 tile at D (row stride ldd)
__device__ __forceinline__ void tile_store(float *D, int ldd, const float (&d)[4], float s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(D + g * ldd + 2 * t) = make_float2(s * d[0], s * d[1]);
    *reinterpret_cast<float2 *>(D + (g + 8) * ldd + 2 * t) = make_float2(s * d[2], s * d[3]);
}

// one 8x8 product on the m16n8k8 MMA (rows 8-15 of its A operand zero):
// d = C + A B, A, B, C 8x8 fp32 in shared memory; this lane receives row g, columns
// 2t and 2t+1 of d in d[0], d[1]
__device__ __forceinline__ void tile8_cab(float (&d)[4], const float *C, int ldc, const float *A, int lda,
                                          const float *B, int ldb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const uint32_t a[4] = {to_tf32(A[g * lda + t]), 0u, to_tf32(A[g * lda + t + 4]), 0u};
    const uint32_t b0 = to_tf32(B[t * ldb + g]), b1 = to_tf32(B[(t + 4) * ldb + g]);
    d[0] = C[g * ldc + 2 * t];
    d[1] = C[g * ldc + 2 * t + 1];
    d[2] = 0.f;
    d[3] = 0.f;
    mma_tf32(d, a, b0, b1);
}

// Byte offset of bf16 element (row, col) of a [32][32] K-major MMA operand without
// swizzle: 8x8 core matrices of 128 contiguous bytes (8 rows of 16 bytes), 128 bytes
// apart along K (leading offset) and 512 bytes apart along the rows (stride offset).
__device__ __forceinline__ uint32_t core_off(int row, int col) {
    return (uint32_t)((row >> 3) * 512 + (col >> 3) * 128 + (row & 7) * 16 + (col & 7) * 2);
}

// 16-bit outputs of the inverse (bf16, or fp16 with kHalf): s * Tinv(row, col) * s1[col]
// into out1 and, unless out2 is null, times s2[col] into out2 (null scales mean 1); col is
// even and (v0, v1) are columns col and col + 1 of the row.
template <bool kHalf = false>
__device__ __forceinline__ void put_pair(uint8_t *out1, uint8_t *out2, const float *s1, const float *s2, int row,
                                         int col, float v0, float v1) {
    const float a0 = s1 ? v0 * s1[col] : v0, a1 = s1 ? v1 * s1[col + 1] : v1;
    const uint32_t off = sw128_off(row, col);
    *reinterpret_cast<uint32_t *>(out1 + off) = pack2<kHalf>(a0, a1);
    if (out2)
        *reinterpret_cast<uint32_t *>(out2 + off) =
            pack2<kHalf>(s2 ? a0 * s2[col] : a0, s2 ? a1 * s2[col + 1] : a1);
}

// Tinv = (I + A)^{-1} for the 64x64 strictly lower fp32 matrix A held in M (row
// stride LA, zero on and above the diagonal).  Writes Tinv diag(s1) to out1 and
// Tinv diag(s1 s2) to out2 as bf16 (fp16 with kHalf) [64][64] tiles in the 128-byte swizzle, each
// block as soon as it is final (null scales mean 1, null out2 skips it).  out1 and
// out2 must not overlap M and must hold zeros above the 8x8 diagonal blocks (that
// part of the inverse is zero and is never written).  Y is >= 32*LY floats of
// scratch; M is overwritten with intermediate blocks.
//   a) the eight 8x8 diagonal blocks by forward substitution, one column per lane,
//      the block held in registers (warp w < 4: blocks 2w and 2w+1, lanes 0-15)
//   b) 8 -> 16:  T10 = -T11 (A10 T00), warp w merges its own two blocks
//   c) 16 -> 32: the same on 16x16 blocks, one warp per (pair, 8-column tile)
//   d) 32 -> 64: the same on the two 32x32 halves, one warp per 16x8 tile
// Every inverted block keeps only the strict lower part of its inverse (the unit
// diagonal is implied, zeros above), so each merge is two products,
// Y = A21 + A21 T11s and T21 = -(Y + T22s Y), run on the warp MMA.  Between the two
// products only the warps that read the A21 being overwritten synchronise: the
// warp itself (8 -> 16), the warp pair on named barrier 8 + pair (16 -> 32); in
// 32 -> 64 nothing is overwritten and warps w, w + 4 share their Y tiles on named
// barrier 10 + w (w < 4).  Between the phases, too, only the producers of what a
// warp reads next synchronise: a warp with itself (a -> b), a warp pair (b -> c).
// The caller orders the bf16 writes before their use (proxy fence and barrier).
// Called by kThreads threads (thread indices 0..kThreads-1) that synchronise with
// sync(); phases a-c run on warps 0-3 alone while warps 4-7 run idle().
//
// With kCouple the last merge is left to the caller: phase d then computes only
// M21 = T22 A21 (the 32x32 block coupling the two halves) and writes
// -M21 diag(s3 * s3_mul) (null s3: -M21) as a bf16 (fp16 with kHalf) [32][32] tile without swizzle
// (core_off below) to out3; out1/out2 then hold the block-diagonal inverse
// diag(T11, T22) with the same scalings.  Since T21 = -M21 T11, a solve (I + A) z = r is finished from the
// block-diagonal one, zl = diag(T11, T22) r, by z_bot = zl_bot - M21 z_top.
template <bool kCouple = false, bool kHalf = false, typename Idle, typename Sync>
__device__ __forceinline__ void unit_lower_inverse(float *M, float *Y, uint8_t *out1, uint8_t *out2,
                                                   const float *s1, const float *s2, Idle idle, Sync sync,
                                                   uint8_t *out3 = nullptr, const float *s3 = nullptr,
                                                   float s3_mul = 1.f) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp >= 4) {
        idle();
    } else {
        const int g = lane >> 2, t4 = lane & 3;
        if (lane < 16) {
            const int base = 8 * (2 * warp + (lane >> 3)), j = lane & 7;
            float a[8][8];
#pragma unroll
            for (int i = 1; i < 8; ++i) {                  // the block's rows 1-7, all loads first
                const float4 lo = *reinterpret_cast<const float4 *>(M + (base + i) * LA + base);
                const float4 hi = *reinterpret_cast<const float4 *>(M + (base + i) * LA + base + 4);
                a[i][0] = lo.x; a[i][1] = lo.y; a[i][2] = lo.z; a[i][3] = lo.w;
                a[i][4] = hi.x; a[i][5] = hi.y; a[i][6] = hi.z; a[i][7] = hi.w;
            }
            const float c1 = s1 ? s1[base + j] : 1.f;
            const float c2 = s2 ? c1 * s2[base + j] : c1;
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float acc0 = (i == j) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
                for (int m = 0; m < i; ++m) {
                    if (m & 1) acc1 = fmaf(-a[i][m], t[m], acc1);
                    else acc0 = fmaf(-a[i][m], t[m], acc0);
                }
                t[i] = (i < j) ? 0.f : acc0 + acc1;
            }
#pragma unroll
            for (int i = 1; i < 8; ++i)
                if (i > j) M[(base + i) * LA + base + j] = t[i];
#pragma unroll
            for (int i = 0; i < 8; ++i) {                  // the whole block, zeros above the diagonal
                const uint32_t off = sw128_off(base + i, base + j);
                *reinterpret_cast<uint16_t *>(out1 + off) = cvt16<kHalf>(t[i] * c1);
                if (out2) *reinterpret_cast<uint16_t *>(out2 + off) = cvt16<kHalf>(t[i] * c2);
            }
        }
        __syncwarp();
        // 8 -> 16: warp w < 4 merges the 8x8 blocks at 16 w (its own)
        {
            const int base = 16 * warp;
            float *Yw = Y + 8 * warp * LY;
            float d[4];
            tile8_cab(d, M + (base + 8) * LA + base, LA, M + (base + 8) * LA + base, LA, M + base * LA + base, LA);
            *reinterpret_cast<float2 *>(Yw + g * LY + 2 * t4) = make_float2(d[0], d[1]);
            __syncwarp();
            tile8_cab(d, Yw, LY, M + (base + 8) * LA + base + 8, LA, Yw, LY);
            *reinterpret_cast<float2 *>(M + (base + 8 + g) * LA + base + 2 * t4) = make_float2(-d[0], -d[1]);
            put_pair<kHalf>(out1, out2, s1, s2, base + 8 + g, base + 2 * t4, -d[0], -d[1]);
        }
        named_sync(8 + (warp >> 1), 64);  // the pair's two 16x16 blocks are final
        // 16 -> 32: warp w < 4 takes pair p = w / 2 (blocks at 32 p) and 8-column tile w % 2
        {
            const int p = warp >> 1, n0 = 8 * (warp & 1), base = 32 * p;
            float *Yp = Y + 16 * p * LY;
            float d[4];
            tile_cab<16>(d, M + (base + 16) * LA + base + n0, LA, M + (base + 16) * LA + base, LA,
                         M + base * LA + base + n0, LA);                // A10 + A10 T00s
            tile_store(Yp + n0, LY, d, 1.f);
            named_sync(8 + p, 64);        // the pair's A10 has been read before T10 overwrites it
            tile_cab<16>(d, Yp + n0, LY, M + (base + 16) * LA + base + 16, LA, Yp + n0, LY);   // Y + T11s Y
            tile_store(M + (base + 16) * LA + base + n0, LA, d, -1.f);
            put_pair<kHalf>(out1, out2, s1, s2, base + 16 + g, base + n0 + 2 * t4, -d[0], -d[1]);
            put_pair<kHalf>(out1, out2, s1, s2, base + 24 + g, base + n0 + 2 * t4, -d[2], -d[3]);
        }
    }
    sync();
    if (kCouple) {                    // M21 = A21 + T22s A21, warp w: rows 16 (w / 4), columns 8 (w % 4)
        const int g = lane >> 2, t4 = lane & 3;
        const int m0 = 16 * (warp >> 2), n0 = 8 * (warp & 3);
        float d[4];
        tile_cab<32>(d, M + (32 + m0) * LA + n0, LA, M + (32 + m0) * LA + 32, LA, M + 32 * LA + n0, LA);
        const int c0 = n0 + 2 * t4;
        const float f0 = s3 ? -s3[c0] * s3_mul : -1.f, f1 = s3 ? -s3[c0 + 1] * s3_mul : -1.f;
        *reinterpret_cast<uint32_t *>(out3 + core_off(m0 + g, c0)) = pack2<kHalf>(f0 * d[0], f1 * d[1]);
        *reinterpret_cast<uint32_t *>(out3 + core_off(m0 + 8 + g, c0)) = pack2<kHalf>(f0 * d[2], f1 * d[3]);
        return;
    }
    // 32 -> 64: warp w takes rows 16 (w / 4) and columns 8 (w % 4) of the 32x32 block
    {
        const int g = lane >> 2, t4 = lane & 3;
        const int m0 = 16 * (warp >> 2), n0 = 8 * (warp & 3);
        float d[4];
        tile_cab<32>(d, M + (32 + m0) * LA + n0, LA, M + (32 + m0) * LA, LA, M + n0, LA);   // A21 + A21 T11s
        tile_store(Y + m0 * LY + n0, LY, d, 1.f);
        named_sync(10 + (warp & 3), 64);   // warps w and w ^ 4: Y columns n0..n0+7, all 32 rows
        tile_cab<32>(d, Y + m0 * LY + n0, LY, M + (32 + m0) * LA + 32, LA, Y + n0, LY);    // Y + T22s Y
        put_pair<kHalf>(out1, out2, s1, s2, 32 + m0 + g, n0 + 2 * t4, -d[0], -d[1]);
        put_pair<kHalf>(out1, out2, s1, s2, 40 + m0 + g, n0 + 2 * t4, -d[2], -d[3]);
    }
}

// The backward's checkpoints on the tensor-core path: per (b*H + h, chunk) one fp16
// [128][128] state (or state gradient) tile laid out as a 128-byte-swizzled MMA operand,
// two 64-column panels of 128 rows, so that it is copied to shared memory in one piece.
constexpr uint32_t kChkTileBytes = 2 * kD * 128;
// byte offset of element (row, col) (col a multiple of 8 for a 16-byte group)
__device__ __forceinline__ uint32_t chk_tile_off(int row, int col) {
    return (uint32_t)(col >> 6) * (kD * 128) + sw128_off(row, col & 63);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// The same tensor viewed as [B][H][2 panels][T][64]: one box is a whole 64-token tile
// of one head, landing as its two 64-column panels one after the other (the layout of
// the two 4-D boxes at panel offsets 0 and 8 KB), so one TMA instruction moves it.
inline bool make_token_map_tile(CUtensorMap *m, const void *ptr, int B, int T, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5] = {64, (cuuint64_t)T, 2, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[4] = {(cuuint64_t)H * kD * 2, 64 * 2, (cuuint64_t)kD * 2, (cuuint64_t)T * H * kD * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)kC, 2, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A compact [B][Tc][H][128] 16-bit tensor seen as a sequence of 2 Tc sub-token rows, row j
// of the tensor at sub-token 2j and nothing at 2j + 1: dims {128, 1, H, Tc, B} with boxes
// {64, 2, 1, 32, 1}, so a box is 64 sub-token rows (32 pairs) of one head whose odd rows
// fall outside the size-1 dimension (zero-filled on load, not written on store).
inline bool make_pair_map(CUtensorMap *m, const void *ptr, int B, int Tc, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5] = {(cuuint64_t)kD, 1, (cuuint64_t)H, (cuuint64_t)Tc, (cuuint64_t)B};
    cuuint64_t strides[4] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                             (cuuint64_t)Tc * H * kD * 2};
    cuuint32_t box[5] = {64, 2, 1, (cuuint32_t)kC / 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B][T][H][128] bf16 tensor, boxes of 64 columns x 64 tokens of one head.
inline bool make_token_map(CUtensorMap *m, const void *ptr, int B, int T, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, (cuuint64_t)T * H * kD * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kC, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace tc
}  // namespace qd

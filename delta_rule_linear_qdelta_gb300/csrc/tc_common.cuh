// Pieces shared by the tensor-core chunk kernels (Q-Delta and QED): tile sizes,
// bf16 packing, the fp32 unit-lower-triangular inverse of one 64x64 chunk matrix,
// and the TMA tensor maps of the [B][T][H][128] token tensors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
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


// ---------------------------------------------------------- warp-level TF32 MMA
// The merge steps of the inverse are 16x8 output tiles with K = 16 or 32: too small
// and too latency-bound for tcgen05 (its TMEM round trip alone exceeds the work),
// so they run on the warp-synchronous m16n8k8 TF32 MMA with operands read straight
// from shared memory.  Each fp32 operand is split into two TF32 parts, x = hi + lo,
// and a b = a_hi b_hi + a_hi b_lo + a_lo b_hi (the a_lo b_lo term is below fp32
// rounding), which keeps the products at about fp32 accuracy.
// Fragment layout of m16n8k8 (lane = 4 g + t): A (16x8) a0 (g, t), a1 (g+8, t),
// a2 (g, t+4), a3 (g+8, t+4); B (8x8) b0 (t, g), b1 (t+4, g); C/D (16x8) c0 (g, 2t),
// c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = to_tf32(x);
    lo = to_tf32(x - __uint_as_float(hi));
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
    d[0] = C[g * ldc + 2 * t];
    d[1] = C[g * ldc + 2 * t + 1];
    d[2] = C[(g + 8) * ldc + 2 * t];
    d[3] = C[(g + 8) * ldc + 2 * t + 1];
    float x[K / 8][4];                                 // one accumulator per k-step: short chains
#pragma unroll
    for (int s = 0; s < K / 8; ++s) {
        const int k0 = 8 * s;
        uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
        split_tf32(A[g * lda + k0 + t], ah[0], al[0]);
        split_tf32(A[(g + 8) * lda + k0 + t], ah[1], al[1]);
        split_tf32(A[g * lda + k0 + t + 4], ah[2], al[2]);
        split_tf32(A[(g + 8) * lda + k0 + t + 4], ah[3], al[3]);
        split_tf32(B[(k0 + t) * ldb + g], bh0, bl0);
        split_tf32(B[(k0 + t + 4) * ldb + g], bh1, bl1);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[s][i] = 0.f;
        mma_tf32(x[s], ah, bl0, bl1);
        mma_tf32(x[s], al, bh0, bh1);
        mma_tf32(x[s], ah, bh0, bh1);
    }
#pragma unroll
    for (int s = 0; s < K / 8; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += x[s][i];
}
// stores s * d into the 16x8 tile at D (row stride ldd)
__device__ __forceinline__ void tile_store(float *D, int ldd, const float (&d)[4], float s) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(D + g * ldd + 2 * t) = make_float2(s * d[0], s * d[1]);
    *reinterpret_cast<float2 *>(D + (g + 8) * ldd + 2 * t) = make_float2(s * d[2], s * d[3]);
}

// Tinv = (I + A)^{-1} for the 64x64 strictly lower fp32 matrix A held in M (row
// stride LA, zero on and above the diagonal), then Tinv diag(s1) -> out1 and
// Tinv diag(s1 s2) -> out2 as bf16 [64][64] tiles in the 128-byte swizzle (out1
// and out2 may overlay M; null scales mean 1).  Y is >= 32*LY floats of scratch.
//   a) the four 16x16 diagonal blocks by forward substitution, one column per lane
//   b) 16 -> 32: T10 = -T11 (A10 T00) for the block pairs (0,1) and (2,3)
//   c) 32 -> 64: T21 = -T22 (A21 T11) on the two 32x32 halves
// Every inverted block keeps only the strict lower part of its inverse (the unit
// diagonal is implied, zeros above), so each merge is two products,
// Y = A21 + A21 T11s and T21 = -(Y + T22s Y), run as 16x8 tiles on the warp MMA.
// Called by kThreads threads (thread indices 0..kThreads-1) that synchronise with
// sync(); idle() runs on every one of them while warps 0-3 invert the diagonal blocks.
template <typename Idle, typename Sync>
__device__ __forceinline__ void unit_lower_inverse(float *M, float *Y, uint8_t *out1, uint8_t *out2,
                                                   const float *s1, const float *s2, Idle idle, Sync sync) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp < 4 && lane < 16) {
        const int base = 16 * warp, j = lane;
        float t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float *Ai = M + (base + i) * LA + base;
            float acc[4] = {(i == j) ? 1.f : 0.f, 0.f, 0.f, 0.f};   // four partial sums
#pragma unroll
            for (int m4 = 0; m4 < (i + 3) / 4; ++m4) {
                const float4 a = *reinterpret_cast<const float4 *>(Ai + 4 * m4);
                if (4 * m4 + 0 < i) acc[0] = fmaf(-a.x, t[4 * m4 + 0], acc[0]);
                if (4 * m4 + 1 < i) acc[1] = fmaf(-a.y, t[4 * m4 + 1], acc[1]);
                if (4 * m4 + 2 < i) acc[2] = fmaf(-a.z, t[4 * m4 + 2], acc[2]);
                if (4 * m4 + 3 < i) acc[3] = fmaf(-a.w, t[4 * m4 + 3], acc[3]);
            }
            t[i] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        __syncwarp(0x0000ffffu);
#pragma unroll
        for (int i = 1; i < 16; ++i)
            if (i > j) M[(base + i) * LA + base + j] = t[i];
    }
    idle();
    sync();
    // 16 -> 32: warp w < 4 takes pair p = w / 2 (blocks at 32 p) and 8-column tile w % 2
    {
        const int p = (warp >> 1) & 1, n0 = 8 * (warp & 1), base = 32 * p;
        float *Yp = Y + 16 * p * LY;
        float d[4];
        if (warp < 4) {
            tile_cab<16>(d, M + (base + 16) * LA + base + n0, LA, M + (base + 16) * LA + base, LA,
                         M + base * LA + base + n0, LA);                // A10 + A10 T00s
            tile_store(Yp + n0, LY, d, 1.f);
        }
        sync();
        if (warp < 4) {
            tile_cab<16>(d, Yp + n0, LY, M + (base + 16) * LA + base + 16, LA, Yp + n0, LY);   // Y + T11s Y
            tile_store(M + (base + 16) * LA + base + n0, LA, d, -1.f);
        }
    }
    sync();
    // 32 -> 64: warp w takes rows 16 (w / 4) and columns 8 (w % 4) of the 32x32 block
    {
        const int m0 = 16 * (warp >> 2), n0 = 8 * (warp & 3);
        float d[4];
        tile_cab<32>(d, M + (32 + m0) * LA + n0, LA, M + (32 + m0) * LA, LA, M + n0, LA);   // A21 + A21 T11s
        tile_store(Y + m0 * LY + n0, LY, d, 1.f);
        sync();
        tile_cab<32>(d, Y + m0 * LY + n0, LY, M + (32 + m0) * LA + 32, LA, Y + n0, LY);    // Y + T22s Y
        tile_store(M + (32 + m0) * LA + n0, LA, d, -1.f);
    }
    sync();
    // Tinv*beta and Tinv*beta*gamma as bf16 [64][64] (128B swizzle) over R1
    float tv[2][8];
    int rows[2], chs[2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        const int u = tid + kThreads * n;          // 512 chunks of 8
        rows[n] = u >> 3;
        chs[n] = u & 7;
        const float4 lo = *reinterpret_cast<const float4 *>(M + rows[n] * LA + 8 * chs[n]);
        const float4 hi = *reinterpret_cast<const float4 *>(M + rows[n] * LA + 8 * chs[n] + 4);
        const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 8 * chs[n] + e;
            tv[n][e] = (j < rows[n]) ? v[e] : (j == rows[n] ? 1.f : 0.f);
        }
    }
    // the column scales, read before any store (the compiler cannot tell them apart)
    float f1[2][8], f2[2][8];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 8 * chs[n] + e;
            f1[n][e] = s1 ? tv[n][e] * s1[j] : tv[n][e];
            f2[n][e] = s2 ? f1[n][e] * s2[j] : f1[n][e];
        }
    sync();
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        *reinterpret_cast<uint4 *>(out1 + sw128_off(rows[n], 8 * chs[n])) = pack8(f1[n]);
        *reinterpret_cast<uint4 *>(out2 + sw128_off(rows[n], 8 * chs[n])) = pack8(f2[n]);
    }
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

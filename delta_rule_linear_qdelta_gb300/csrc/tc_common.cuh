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


// Tinv = (I + A)^{-1} for the 64x64 strictly lower fp32 matrix A held in M (row
// stride LA, zero on and above the diagonal), then Tinv diag(s1) -> out1 and
// Tinv diag(s1 s2) -> out2 as bf16 [64][64] tiles in the 128-byte swizzle (out1
// and out2 may overlay M; null scales mean 1).  Y is >= 32*LY floats of scratch.
//   a) the four 16x16 diagonal blocks by forward substitution, one column per lane
//   b) 16 -> 32: T10 = -T11 (A10 T00) for the block pairs (0,1) and (2,3)
//   c) 32 -> 64: T21 = -T22 (A21 T11) on the two 32x32 halves
// Every inverted block keeps only the strict lower part of its inverse (the unit
// diagonal is implied, zeros above), so each product is a dense loop:
// Y = A21 + A21 T11s and T21 = -(Y + T22s Y).  Called by kThreads threads (thread
// indices 0..kThreads-1) that synchronise with sync(); idle() runs on every one of
// them while warps 0-3 invert the diagonal blocks.
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
            float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m4 = 0; m4 < (i + 3) / 4; ++m4) {
                const float4 a = *reinterpret_cast<const float4 *>(Ai + 4 * m4);
                if (4 * m4 + 0 < i) acc = fmaf(-a.x, t[4 * m4 + 0], acc);
                if (4 * m4 + 1 < i) acc = fmaf(-a.y, t[4 * m4 + 1], acc);
                if (4 * m4 + 2 < i) acc = fmaf(-a.z, t[4 * m4 + 2], acc);
                if (4 * m4 + 3 < i) acc = fmaf(-a.w, t[4 * m4 + 3], acc);
            }
            t[i] = acc;
        }
        __syncwarp(0x0000ffffu);
#pragma unroll
        for (int i = 1; i < 16; ++i)
            if (i > j) M[(base + i) * LA + base + j] = t[i];
    }
    idle();
    sync();
    // Y = L + L Rs (+= into out) for n x n blocks: thread owns rows r, r+n/2 and 4 columns.
    // 16 -> 32: both pairs at once (threads 0..63 pair 0, 64..127 pair 1), 2x4 outputs each
    if (tid < 128) {
        const int pr = tid >> 6, u = tid & 63, r = u >> 2, c = 4 * (u & 3), base = 32 * pr;
        const float *L0 = M + (base + 16 + r) * LA + base;        // A10 row r
        float y[4];
        {
            const float4 l0 = *reinterpret_cast<const float4 *>(L0 + c);
            y[0] = l0.x; y[1] = l0.y; y[2] = l0.z; y[3] = l0.w;
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const float4 a = *reinterpret_cast<const float4 *>(L0 + 4 * k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 tr = *reinterpret_cast<const float4 *>(M + (base + 4 * k4 + e) * LA + base + c);
                y[0] = fmaf(av[e], tr.x, y[0]); y[1] = fmaf(av[e], tr.y, y[1]);
                y[2] = fmaf(av[e], tr.z, y[2]); y[3] = fmaf(av[e], tr.w, y[3]);
            }
        }
        *reinterpret_cast<float4 *>(Y + (16 * pr + r) * LY + c) = make_float4(y[0], y[1], y[2], y[3]);
    }
    sync();
    if (tid < 128) {                                     // T10 = -(Y + T11s Y)
        const int pr = tid >> 6, u = tid & 63, r = u >> 2, c = 4 * (u & 3), base = 32 * pr;
        const float *T0 = M + (base + 16 + r) * LA + base + 16;
        const float *Yp = Y + 16 * pr * LY;
        float y[4];
        {
            const float4 y0 = *reinterpret_cast<const float4 *>(Yp + r * LY + c);
            y[0] = y0.x; y[1] = y0.y; y[2] = y0.z; y[3] = y0.w;
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const float4 a = *reinterpret_cast<const float4 *>(T0 + 4 * k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 yr = *reinterpret_cast<const float4 *>(Yp + (4 * k4 + e) * LY + c);
                y[0] = fmaf(av[e], yr.x, y[0]); y[1] = fmaf(av[e], yr.y, y[1]);
                y[2] = fmaf(av[e], yr.z, y[2]); y[3] = fmaf(av[e], yr.w, y[3]);
            }
        }
        *reinterpret_cast<float4 *>(M + (base + 16 + r) * LA + base + c) = make_float4(-y[0], -y[1], -y[2], -y[3]);
    }
    sync();
    // 32 -> 64: row r of the 32x32 blocks, columns c..c+3 (256 threads)
    {
        const int r = tid >> 3, c = 4 * (tid & 7);
        const float *L0 = M + (32 + r) * LA;                     // A21 row r
        float y0[4];
        {
            const float4 a0 = *reinterpret_cast<const float4 *>(L0 + c);
            y0[0] = a0.x; y0[1] = a0.y; y0[2] = a0.z; y0[3] = a0.w;
        }
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {                 // Y = A21 + A21 T11s
            const float4 a0 = *reinterpret_cast<const float4 *>(L0 + 4 * k4);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 tr = *reinterpret_cast<const float4 *>(M + (4 * k4 + e) * LA + c);
                y0[0] = fmaf(av0[e], tr.x, y0[0]); y0[1] = fmaf(av0[e], tr.y, y0[1]);
                y0[2] = fmaf(av0[e], tr.z, y0[2]); y0[3] = fmaf(av0[e], tr.w, y0[3]);
            }
        }
        *reinterpret_cast<float4 *>(Y + r * LY + c) = make_float4(y0[0], y0[1], y0[2], y0[3]);
        sync();
        const float *T0 = L0 + 32;                                // T22s row r
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {                 // T21 = -(Y + T22s Y)
            const float4 a0 = *reinterpret_cast<const float4 *>(T0 + 4 * k4);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 yr = *reinterpret_cast<const float4 *>(Y + (4 * k4 + e) * LY + c);
                y0[0] = fmaf(av0[e], yr.x, y0[0]); y0[1] = fmaf(av0[e], yr.y, y0[1]);
                y0[2] = fmaf(av0[e], yr.z, y0[2]); y0[3] = fmaf(av0[e], yr.w, y0[3]);
            }
        }
        *reinterpret_cast<float4 *>(M + (32 + r) * LA + c) = make_float4(-y0[0], -y0[1], -y0[2], -y0[3]);
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
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 8 * chs[n] + e;
            tv[n][e] = (j < rows[n]) ? M[rows[n] * LA + j] : (j == rows[n] ? 1.f : 0.f);
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

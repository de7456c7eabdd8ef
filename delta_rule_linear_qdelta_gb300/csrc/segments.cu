// Segment scan for long sequences over few (b, h) streams (Q-Delta and QED).
//
// A chunk of the Q-Delta recurrence maps its entering state linearly
// ("Q-Delta: Beyond Key-Value Associative State Evolution", Sec. 3.3.2: with the
// chunk's WY factors, S_out = gamma_C S_in + (U - W S_in^T)^T K_out), so
//     S_out = S_in Phi + Psi,   Phi = gamma_C I - W^T K_out  (d_k x d_k),  Psi = U^T K_out,
// and so does any run of chunks: a segment's map is the product of its chunks' maps.
// When B*H streams leave most SMs idle, each sequence is cut into G segments
// that run side by side as a [B*G][T/G] batch of the same tensor-core kernel:
//   pass 1  S0 = 0, v as given        ->  final state = Psi_g
//   pass 2  S0 = I, v taken as 0      ->  final state = Phi_g
//   combine (fp32, per (b, h) and 16 state rows, in segment order): S_start(g) = S,
//           S <- S Phi_g + Psi_g
//   pass 3  S0 = S_start(g)           ->  o, exactly as one pass over the whole sequence
// The [B][T][H][d] layout makes the segment view free: [B][G*L][H][d] is [B*G][L][H][d].
// QED ("The Query Knows What to Forget", Eqs. 4/6/8) keeps its state transposed,
// S^ = S^T in [dv][dk], and S^_t = S^_{t-1} Diag(e^{g_t}) (I - a_t k_t^T) + (w_t*v_t) k_t^T
// is the same kind of map, so the same passes and combine serve it.
// The three per-segment state arrays live in caller-provided workspace.
#include <cuda_runtime.h>

#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kD = 128;
constexpr int kLS = 132;          // smem row stride (16-byte aligned rows; 8 rows hit 8 distinct 16-byte banks)
constexpr int kCombineThreads = 256;
constexpr int kRows = 16;         // state rows per combine CTA

__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fma4(float (&acc)[4], float a, const float4 &p) {
    acc[0] = fmaf(a, p.x, acc[0]);
    acc[1] = fmaf(a, p.y, acc[1]);
    acc[2] = fmaf(a, p.z, acc[2]);
    acc[3] = fmaf(a, p.w, acc[3]);
}

// One CTA per (b, h, 16 state rows): rows of S evolve independently under
// S <- S Phi_g + Psi_g, so a head's 128 rows are spread over 8 CTAs.  Each holds its
// rows of S (two buffers, read and written in alternation) and Phi_g (fp32, two buffers:
// Phi_{g+1} is copied in by cp.async while Phi_g is used) in shared memory, so one
// barrier per segment orders everything.  Warp w computes columns 16 w .. 16 w + 15 of
// all 16 rows; lane l rows l/4 and l/4 + 8, columns 16 w + 4 (l%4) .. + 3, reading four
// k at a time (a warp's Phi reads are 64 contiguous bytes, its S reads 8 rows in 8
// distinct banks).  Psi_g is loaded into registers before the products and added after.
// Each result goes from registers to the next segment's S_start (or to S_final).
__global__ void __launch_bounds__(kCombineThreads)
segment_combine_kernel(const float *S0, const float *Phi, const float *Psi, float *S_start, float *S_final,
                       int B, int H, int G) {
    extern __shared__ float4 sm4[];
    float *sm = reinterpret_cast<float *>(sm4);
    auto Ss = [&](int i) { return sm + i * kRows * kLS; };             // S buffers 0, 1
    auto Ps = [&](int i) { return sm + 2 * kRows * kLS + i * kD * kLS; };  // Phi buffers 0, 1
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int row0 = blockIdx.y * kRows;
    const int r0 = lane >> 2, n0 = 16 * warp + 4 * (lane & 3);
    const size_t mat = (size_t)kD * kD;
    auto seg = [&](int g) { return ((size_t)(b * G + g) * H + h) * mat; };   // (b*G + g, h) in the segment batch
    auto load_phi = [&](int g) {
        const float *src = Phi + seg(g);
        float *dst = Ps(g & 1);
        for (int i = tid; i < kD * kD / 4; i += kCombineThreads)
            cp_async16(dst + (i >> 5) * kLS + 4 * (i & 31), src + 4 * i);
        cp_async_commit();
    };
    load_phi(0);
    for (int i = tid; i < kRows * kD / 4; i += kCombineThreads) {   // S_start(0) = S0 (or 0)
        const int rr = i >> 5, c = 4 * (i & 31);
        const size_t o = (size_t)(row0 + rr) * kD + c;
        const float4 v = S0 ? *reinterpret_cast<const float4 *>(S0 + (size_t)bh * mat + o)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Ss(0) + rr * kLS + c) = v;
        *reinterpret_cast<float4 *>(S_start + seg(0) + o) = v;
    }
    for (int g = 0; g < G; ++g) {
        cp_async_wait_all();
        __syncthreads();    // Phi_g and S_start(g) in place; iteration g-1 no longer reads its buffers
        if (g + 1 < G) load_phi(g + 1);
        const size_t o0 = (size_t)(row0 + r0) * kD + n0, o1 = o0 + 8 * kD;
        const float4 psi0 = *reinterpret_cast<const float4 *>(Psi + seg(g) + o0);
        const float4 psi1 = *reinterpret_cast<const float4 *>(Psi + seg(g) + o1);
        const float *S = Ss(g & 1), *P = Ps(g & 1);
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int k = 0; k < kD; k += 4) {
            const float4 s0 = *reinterpret_cast<const float4 *>(S + r0 * kLS + k);
            const float4 s1 = *reinterpret_cast<const float4 *>(S + (r0 + 8) * kLS + k);
            const float4 p0 = *reinterpret_cast<const float4 *>(P + k * kLS + n0);
            const float4 p1 = *reinterpret_cast<const float4 *>(P + (k + 1) * kLS + n0);
            const float4 p2 = *reinterpret_cast<const float4 *>(P + (k + 2) * kLS + n0);
            const float4 p3 = *reinterpret_cast<const float4 *>(P + (k + 3) * kLS + n0);
            fma4(a0, s0.x, p0); fma4(a1, s1.x, p0);
            fma4(a0, s0.y, p1); fma4(a1, s1.y, p1);
            fma4(a0, s0.z, p2); fma4(a1, s1.z, p2);
            fma4(a0, s0.w, p3); fma4(a1, s1.w, p3);
        }
        const float4 x0 = make_float4(a0[0] + psi0.x, a0[1] + psi0.y, a0[2] + psi0.z, a0[3] + psi0.w);
        const float4 x1 = make_float4(a1[0] + psi1.x, a1[1] + psi1.y, a1[2] + psi1.z, a1[3] + psi1.w);
        if (g + 1 < G) {
            float *Sn = Ss((g + 1) & 1);
            *reinterpret_cast<float4 *>(Sn + r0 * kLS + n0) = x0;
            *reinterpret_cast<float4 *>(Sn + (r0 + 8) * kLS + n0) = x1;
            *reinterpret_cast<float4 *>(S_start + seg(g + 1) + o0) = x0;
            *reinterpret_cast<float4 *>(S_start + seg(g + 1) + o1) = x1;
        } else if (S_final) {
            *reinterpret_cast<float4 *>(S_final + (size_t)bh * mat + o0) = x0;
            *reinterpret_cast<float4 *>(S_final + (size_t)bh * mat + o1) = x1;
        }
    }
}


}  // namespace

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

int qdelta_segments(int B, int T, int H, int dk, int dv, int dtype) {
    if (dtype != kBF16 || dk != kD || dv != kD) return 1;
    const long long streams = (long long)B * H;
    const int nsm = sm_count();
    int G = 1;
    while (streams * 2 * G <= nsm && T % (2 * G) == 0 && T / (2 * G) >= 1024) G *= 2;
    return G;
}

int qed_segments(int B, int T, int H, int dk, int dv, int dtype) {
    // The Q-Delta policy, for at most 16 streams.  QED derives its operands once for all
    // three passes, but each pass still repeats the chain; on the 32-stream QED workload
    // (B=4, H=8, T=4096) one pass takes 0.325 ms against 0.372 ms for four segments.
    if ((long long)B * H > 16) return 1;
    return qdelta_segments(B, T, H, dk, dv, dtype);
}

size_t qdelta_segment_workspace(int B, int H, int G) {
    return G > 1 ? 3 * (size_t)B * G * H * kD * kD * sizeof(float) : 0;
}

namespace {

// The four launches of a segment scan; Args is QDeltaArgs or QedArgs and launch(args,
// flags) runs one pass of the matching tensor-core kernel.
template <typename Args, typename Launch>
cudaError_t run_segmented(const Args &a, int G, cudaStream_t s, int *nlaunch, Launch launch) {
    const size_t n = (size_t)a.B * G * a.H * kD * kD;
    float *S_start = static_cast<float *>(a.ws), *Psi = S_start + n, *Phi = Psi + n;
    Args seg = a;
    seg.B = a.B * G;
    seg.T = a.T / G;
    seg.S0 = nullptr;
    seg.S_final = Psi;
    cudaError_t e = launch(seg, kTcNoO);
    if (e != cudaSuccess) return e;
    seg.S_final = Phi;
    e = launch(seg, kTcNoO | kTcNoV | kTcS0Identity);
    if (e != cudaSuccess) return e;
    const size_t smem = 2 * (kRows + kD) * kLS * sizeof(float);
    e = cudaFuncSetAttribute(segment_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    segment_combine_kernel<<<dim3(a.B * a.H, kD / kRows), kCombineThreads, smem, s>>>(a.S0, Phi, Psi, S_start,
                                                                                     a.S_final, a.B, a.H, G);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *nlaunch += 1;
    seg.S0 = S_start;
    seg.S_final = nullptr;
    return launch(seg, 0);
}

}  // namespace

cudaError_t launch_qdelta_segmented(const QDeltaArgs &a, int G, cudaStream_t s, int *nlaunch) {
    return run_segmented(a, G, s, nlaunch,
                         [&](const QDeltaArgs &x, int f) { return launch_qdelta_chunk_tc(x, s, nlaunch, f); });
}

cudaError_t launch_qed_segmented(const QedArgs &a, int G, const QedDerived &d, cudaStream_t s, int *nlaunch) {
    return run_segmented(a, G, s, nlaunch,
                         [&](const QedArgs &x, int f) { return launch_qed_chain_tc(x, d, s, nlaunch, f); });
}

}  // namespace qd

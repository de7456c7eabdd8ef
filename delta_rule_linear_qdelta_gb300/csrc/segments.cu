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
constexpr int kLS = 132;          // smem row stride (16-byte aligned rows)
constexpr int kCombineThreads = 256;
constexpr int kRows = 16;         // state rows per combine CTA

// One CTA per (b, h, 16 state rows): rows of S evolve independently under
// S <- S Phi_g + Psi_g, so a head's 128 rows are spread over 8 CTAs.  Each holds its
// rows of S and the whole Phi_g (fp32) in shared memory; thread t computes row t/16,
// columns 8 (t%16) .. 8 (t%16) + 7 of the product.
__global__ void __launch_bounds__(kCombineThreads)
segment_combine_kernel(const float *S0, const float *Phi, const float *Psi, float *S_start, float *S_final,
                       int B, int H, int G) {
    extern __shared__ float sm[];
    float *Ss = sm, *Ps = sm + kRows * kLS;
    const int tid = threadIdx.x;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int row0 = blockIdx.y * kRows;
    const int r = tid >> 4, c0 = 8 * (tid & 15);
    const size_t mat = (size_t)kD * kD;
    for (int i = tid; i < kRows * kD / 4; i += kCombineThreads) {
        const int rr = (4 * i) / kD, c = (4 * i) % kD;
        const float4 v = S0 ? *reinterpret_cast<const float4 *>(S0 + (size_t)bh * mat + (size_t)(row0 + rr) * kD + c)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Ss + rr * kLS + c) = v;
    }
    __syncthreads();
    for (int g = 0; g < G; ++g) {
        const size_t seg = ((size_t)(b * G + g) * H + h) * mat;   // (b*G + g, h) in the segment batch
        for (int i = tid; i < kRows * kD / 4; i += kCombineThreads) {
            const int rr = (4 * i) / kD, c = (4 * i) % kD;
            *reinterpret_cast<float4 *>(S_start + seg + (size_t)(row0 + rr) * kD + c) =
                *reinterpret_cast<const float4 *>(Ss + rr * kLS + c);
        }
        for (int i = tid; i < kD * kD / 4; i += kCombineThreads) {
            const int rr = (4 * i) / kD, c = (4 * i) % kD;
            *reinterpret_cast<float4 *>(Ps + rr * kLS + c) = reinterpret_cast<const float4 *>(Phi + seg)[i];
        }
        float acc[8];
        {
            const float *src = Psi + seg + (size_t)(row0 + r) * kD + c0;
            const float4 u = *reinterpret_cast<const float4 *>(src), w = *reinterpret_cast<const float4 *>(src + 4);
            acc[0] = u.x; acc[1] = u.y; acc[2] = u.z; acc[3] = u.w;
            acc[4] = w.x; acc[5] = w.y; acc[6] = w.z; acc[7] = w.w;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kD; ++k) {
            const float a = Ss[r * kLS + k];
            const float4 p0 = *reinterpret_cast<const float4 *>(Ps + k * kLS + c0);
            const float4 p1 = *reinterpret_cast<const float4 *>(Ps + k * kLS + c0 + 4);
            acc[0] = fmaf(a, p0.x, acc[0]); acc[1] = fmaf(a, p0.y, acc[1]);
            acc[2] = fmaf(a, p0.z, acc[2]); acc[3] = fmaf(a, p0.w, acc[3]);
            acc[4] = fmaf(a, p1.x, acc[4]); acc[5] = fmaf(a, p1.y, acc[5]);
            acc[6] = fmaf(a, p1.z, acc[6]); acc[7] = fmaf(a, p1.w, acc[7]);
        }
        __syncthreads();
        *reinterpret_cast<float4 *>(Ss + r * kLS + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(Ss + r * kLS + c0 + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        __syncthreads();
    }
    if (S_final)
        for (int i = tid; i < kRows * kD / 4; i += kCombineThreads) {
            const int rr = (4 * i) / kD, c = (4 * i) % kD;
            *reinterpret_cast<float4 *>(S_final + (size_t)bh * mat + (size_t)(row0 + rr) * kD + c) =
                *reinterpret_cast<const float4 *>(Ss + rr * kLS + c);
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
    const size_t smem = (kRows + kD) * kLS * sizeof(float);
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

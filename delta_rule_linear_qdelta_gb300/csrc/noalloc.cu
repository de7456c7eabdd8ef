// qdelta_fwd_static_scratch: the chunked Q-Delta forward for callers that cannot
// allocate device memory at call time.
//
// Some callers cannot hand this library a workspace: plain C code that holds only
// the input and output pointers and no device allocator, or a serving loop whose
// device memory is reserved up front and that must not call cudaMalloc (which can
// synchronise the device and can fail under memory pressure) in the middle of a
// step.  For them this entry point takes no workspace and allocates nothing: when
// the long-sequence segment scan needs scratch, it uses a fixed array that lives
// in this library's device image (g_static_scratch below), held by every GPU that
// loads the library until the process exits.
//
// The array is kStaticScratchBytes = 24 MiB: room for 128 segment-heads (B * G * H,
// G segments per sequence) of three 128 x 128 fp32 states.  Larger problems are
// rejected with QD_ERR_WORKSPACE; problems that need no scratch run as usual.
// Arguments are checked first, exactly as qdelta_fwd checks them, so a bad argument
// returns QD_ERR_ARG (or QD_ERR_UNSUPPORTED) before any CUDA call is made.
//
// Host code may not use the array's name as a device address: here it stands for a
// host-side shadow.  The device address is taken with cudaGetSymbolAddress with the
// device current, on the first call made on that device, and kept together with the
// id of the context it belongs to; a call that finds another context current (after
// cudaDeviceReset, say) looks the address up again.  That first call on a device or
// context should therefore come before any stream capture.  All calls share the one
// array: calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on it.  Nothing in it needs to start at zero: every call writes
// all the scratch it later reads.
#include <cuda.h>

#include <mutex>

#include "../../include/qdelta.h"
#include "qd_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)24 << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
    void *ptr;
    unsigned long long ctx_id;   // the context the address belongs to
};
ScratchAddr g_scratch_dev[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current context (0 when there is none yet or the
// driver cannot say).  Context ids are never reused within a process.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device (set up on first use
// in each context).
qd_status static_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qd::report_error(QD_ERR_CUDA, "qdelta_fwd_static_scratch: cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return qd::report_error(QD_ERR_UNSUPPORTED, "qdelta_fwd_static_scratch: device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &slot = g_scratch_dev[dev];
    const unsigned long long id = current_context_id();
    if (!slot.ptr || id == 0 || id != slot.ctx_id) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);   // makes the device's context current if needed
        if (e != cudaSuccess || !p)
            return qd::report_error(QD_ERR_CUDA, "qdelta_fwd_static_scratch: cudaGetSymbolAddress failed");
        slot.ptr = p;
        slot.ctx_id = current_context_id();
    }
    *out = slot.ptr;
    return QD_OK;
}

}  // namespace

extern "C" qd_status qdelta_fwd_static_scratch(const void *q, const void *k, const void *v, const void *alpha,
                                               const void *beta, const void *lam, const float *S0, void *o,
                                               float *S_final, int B, int T, int H, int dk, int dv, int chunk,
                                               qd_dtype dtype, cudaStream_t stream) {
    const qd_status arg = qd::check_qdelta_fwd_args("qdelta_fwd_static_scratch", q, k, v, alpha, beta, lam, S0, o,
                                                    S_final, B, T, H, dk, dv, chunk, dtype);
    if (arg != QD_OK) return arg;
    const size_t need = qdelta_workspace_bytes(B, T, H, dk, dv, chunk, dtype);
    if (need == 0)
        return qdelta_fwd(q, k, v, alpha, beta, lam, S0, o, S_final, B, T, H, dk, dv, chunk, dtype, nullptr, 0,
                          stream);
    if (need > kStaticScratchBytes)
        return qd::report_error(QD_ERR_WORKSPACE,
                                "qdelta_fwd_static_scratch: these sizes need more scratch than the library's "
                                "fixed 24 MiB (at most 128 segment-heads); use qdelta_fwd with a workspace");
    void *ws = nullptr;
    const qd_status st = static_scratch(&ws);
    if (st != QD_OK) return st;
    return qdelta_fwd(q, k, v, alpha, beta, lam, S0, o, S_final, B, T, H, dk, dv, chunk, dtype, ws,
                      kStaticScratchBytes, stream);
}

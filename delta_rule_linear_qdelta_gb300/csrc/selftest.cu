// The failure path of a bounded wait, on its own (qd_selftest_bounded_wait): one CTA
// waits, with the library's bounded mbarrier wait, on a barrier that nothing ever
// arrives on; when the limit runs out it records the timeout in a device word that
// qd_device_status reads like the tensor-core kernels' own, and exits.  No trap, no
// fault, no unbounded spin.
#include "qd_internal.cuh"
#include "sm103_ptx.cuh"

namespace qd {
namespace {

__device__ unsigned int g_selftest_timeout = 0;

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, limit_ns)) atomicExch(&g_selftest_timeout, 1u);
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

bool selftest_read_and_clear_timeout() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_selftest_timeout, sizeof v) != cudaSuccess) return false;
    if (v) cudaMemcpyToSymbol(g_selftest_timeout, &zero, sizeof zero);
    return v != 0;
}

}  // namespace qd

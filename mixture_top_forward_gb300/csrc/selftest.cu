// Self-test of the bounded device-side wait that every tensor-core kernel of
// the library uses for its mbarrier handshakes (umma.cuh). One thread arms a
// shared-memory mbarrier that nothing ever completes and waits on it with a
// short limit; the wait gives up, records MITA_ERR_TIMEOUT in the status word
// and the kernel returns. Nothing spins without a bound, traps or faults.
// The pages describe no such part: it exists so that the timeout path the
// forward kernels rely on can be exercised on a GPU.
#include "umma.cuh"

namespace mita {

namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        umma::mbar_init(&bar, 1);  // one arrival expected; none comes
        umma::fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) umma::mbar_wait(&bar, 0, status, limit_ns);
    __syncwarp();
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mita

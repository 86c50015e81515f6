// Self-test of the bounded waits: a kernel waits on an mbarrier that nothing
// ever signals, with a caller-given poll limit, gives up, and records the
// failure in the workspace's error word the way the library's kernels do.
#include "common.cuh"
#include "umma.cuh"

namespace csa2 {

__global__ void k_selftest_wait(uint32_t max_polls, int* __restrict__ err) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x == 0) {
        umma::mbar_init(umma::smem_u32(&bar), 1);     // one arrival expected; none will come
        umma::fence_mbar_init();
    }
    __syncthreads();
    const bool ok = umma::mbar_wait(umma::smem_u32(&bar), 0, max_polls);
    if (!ok && threadIdx.x == 0) atomicExch(err, 1);
}

cudaError_t launch_selftest_wait(uint32_t max_polls, int* err, cudaStream_t st) {
    k_selftest_wait<<<1, 32, 0, st>>>(max_polls, err);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa2

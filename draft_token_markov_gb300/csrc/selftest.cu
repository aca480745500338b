// selftest.cu -- failure detection without a GPU fault: the kernels' bounded
// waits, run on a wait that nothing can complete, must give up after their
// limit, record MARKOV_ETIMEOUT and return.
#include <cstdint>

#include "../../include/markov.h"
#include "common.cuh"
#include "tc.cuh"

namespace dtm {
namespace {

// [0] barrier counter, [1] unused, [2] status code, [3] where
__device__ uint32_t g_selftest[4];

// One CTA.  which 0: the chain's grid barrier with a target one arrival
// beyond the grid (the counter can never reach it); which 1: an mbarrier
// phase that nothing arrives on, awaited as the tcgen05 chain awaits its
// MMA and TMA barriers.  Either wait gives up after timeout_ns.
__global__ void selftest_wait_kernel(int which, uint64_t timeout_ns) {
    __shared__ uint32_t flag;
    __shared__ __align__(8) uint64_t bar;
    if (which == 0) {
        grid_barrier(&g_selftest[0], 2u, &g_selftest[2], timeout_ns, 0xE000u, &flag);
    } else {
        if (threadIdx.x == 0) {
            tc::mbar_init(tc::smem_u32(&bar), 1);
            tc::mbar_init_fence();
        }
        __syncthreads();
        if (threadIdx.x == 0 &&
            !tc::mbar_wait(tc::smem_u32(&bar), 0u, tc::now_ns() + timeout_ns))
            set_status(&g_selftest[2], 4u /* MARKOV_ETIMEOUT */, 0xE001u);
        __syncthreads();
    }
}

}  // namespace
}  // namespace dtm

using namespace dtm;

extern "C" markov_status markov_selftest_wait(int32_t which, int32_t timeout_us, void *stream) {
    if ((which != 0 && which != 1) || timeout_us < 1 || timeout_us > 1000000) return MARKOV_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t zero[4] = {0u, 0u, 0u, 0u};
    if (cudaMemcpyToSymbolAsync(g_selftest, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return MARKOV_ECUDA;
    selftest_wait_kernel<<<1, 32, 0, s>>>(which, (uint64_t)timeout_us * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return MARKOV_ECUDA;
    uint32_t out[4];
    if (cudaMemcpyFromSymbolAsync(out, g_selftest, sizeof(out), 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MARKOV_ECUDA;
    return (markov_status)out[2];
}

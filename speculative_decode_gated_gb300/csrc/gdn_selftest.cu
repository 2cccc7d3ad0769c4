// Self-check of the bounded pipeline wait.  The chunked kernel waits on
// shared-memory mbarriers for its TMA copies and tensor-core products; if one
// of them never completed, the wait gives up after about two seconds and the
// block reports GDN_DEVERR_TIMEOUT instead of hanging the GPU.  Nothing in a
// correct run makes a copy that never lands, so this kernel runs the same wait
// on a barrier that no one arrives on: the expiry path, exercised without
// provoking any fault.
#include <cstdint>

#include "gdn_device.cuh"
#include "gdn_launch.h"
#include "gdn_wait.cuh"

namespace gdn {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(int32_t *dev_err) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) mbar_init(b, 1);  // one expected arrival, which never comes
    __syncthreads();
    if (threadIdx.x == 0 && !wait_parity(b, 0)) atomicOr(dev_err, GDN_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t *dev_err, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(dev_err);
    return cudaGetLastError();
}

}  // namespace gdn

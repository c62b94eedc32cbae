// wait_selftest.cu -- a check of the bounded mbarrier waits that guard every
// tensor-core kernel of the library: one thread waits for phase 0 of a barrier
// that nothing arrives on, with the polling wait (mbar_wait_bounded) or the
// sleeping one (mbar_wait_sleep), and writes FP4_ERR_TIMEOUT to the status word
// when the wait gives up. Mode 2 arrives first (the phase completes) and leaves
// the status alone. Nothing faults, traps or hangs: the kernel ends when its
// wait's limit runs out (a fraction of a second), and the context stays usable.
#include "fp4mx.h"
#include "launch.h"
#include "tc_sm103.cuh"

namespace fp4mx {
namespace {

__global__ void wait_selftest_kernel(int32_t mode, int32_t *__restrict__ status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (mode == 2) mbar_arrive(b);  // the control case: phase 0 completes
    const bool ok = mode == 1 ? mbar_wait_sleep(b, 0) : mbar_wait_bounded(b, 0);
    if (!ok) atomicExch(status, FP4_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t mode, int32_t *status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(mode, status);
    return cudaGetLastError();
}

}  // namespace fp4mx

// The bounded wait every pipelined kernel here uses on its shared-memory
// mbarriers (ring stages, accumulator hand-offs), run on its own so its
// time-out path can be checked: a wait whose phase never completes gives up
// after a fixed number of polls, records ERRF_WAIT_TIMEOUT in the error word
// the host reads, and returns, leaving the device usable.  No step of the
// forward pass runs it.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tma.cuh"

namespace llm {

namespace {

__global__ void wait_check_kernel(int arrive, uint32_t polls, uint32_t *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (arrive) mbar_arrive(b);
    for (uint32_t i = 0; i < polls; ++i)
        if (mbar_try_wait(b, 0)) return;
    raise_error(err, ERRF_WAIT_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_check(int arrive, uint32_t polls, uint32_t *err, cudaStream_t st) {
    wait_check_kernel<<<1, 32, 0, st>>>(arrive, polls, err);
    return cudaGetLastError();
}

}  // namespace llm

// diag.cu -- a self-test of the bounded device-side waits.
//
// Every wait in the tcgen05 kernels gives up after a limit, records
// MOE_ERR_TIMEOUT in the forward's status word and lets the CTA exit, so a
// lost arrival becomes an error status instead of a hung GPU.  This entry
// point exercises that machinery on its own: one thread waits, with a short
// limit, on an mbarrier that nothing ever arrives on, and records the timeout
// in a caller-provided status word.  No counterpart on the pages.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

__global__ void wait_timeout_kernel(uint64_t timeout_ns, int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_s;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_s = 0;
        ptx::fence_mbar_init();
        // nothing arrives on `bar`: the bounded wait has to give up
        if (!ptx::mbar_wait_bounded(&bar, 0u, &abort_s, timeout_ns))
            atomicExch(status, MOE_ERR_TIMEOUT);
    }
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_dbg_wait_timeout(long long timeout_ns, int32_t* status, void* stream) {
    if (timeout_ns < 1 || timeout_ns > 1000000000LL || !status) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(status) & 3u) return MOE_ERR_ALIGNMENT;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)timeout_ns, status);
    count_launches(1);
    return cuda_status(cudaGetLastError());
}

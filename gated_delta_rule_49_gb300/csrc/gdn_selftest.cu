// Self-test of the bounded-wait path used by the tensor-core prefill: a wait
// on an mbarrier that never completes must give up, record the timeout in the
// device status word and return (no trap, no hang).
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

__global__ void wait_timeout_kernel(long long limit, int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_mbar_init();
        // nothing ever arrives: the phase with parity 0 never completes
        if (!sm100::mbar_wait(&bar, 0, limit) && status) atomicOr(status, kStatusTimeout);
    }
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_selftest_wait_timeout(long long limit_cycles, void *stream) {
    if (limit_cycles < 1 || limit_cycles > (1LL << 31)) return GDN_ERR_INVALID_ARG;
    gdn::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        limit_cycles, gdn::device_status_ptr());
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// gdn_selftest.cu -- exercises the bounded-wait path of the tensor-core kernels without
// faulting or hanging anything: one thread waits on an mbarrier phase that nothing
// completes, with the same wait helper and a caller-given limit, and records the
// outcome in a status word.
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"

namespace {

__global__ void wait_timeout_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    gdn::sm100::mbar_init(&bar, 1);
    gdn::sm100::fence_mbar_init();
    // phase 0 needs one arrival that never comes: the wait must give up after limit_ns
    const uint64_t t0 = gdn::sm100::globaltimer_ns();
    const bool done = gdn::sm100::mbar_wait(&bar, 0, limit_ns);
    const uint64_t waited = gdn::sm100::globaltimer_ns() - t0;
    status[0] = done ? GDN_OK : GDN_ERR_TIMEOUT;
    const uint64_t us = waited / 1000u;
    status[1] = us > 0x7fffffffull ? 0x7fffffff : (int32_t)us;   // microseconds waited
}

}  // namespace

extern "C" int gdn_selftest_wait_timeout(int32_t *status, uint64_t limit_ns, void *cuda_stream) {
    if (!status) return GDN_ERR_INVALID_ARG;
    if ((uintptr_t)status & 3u) return GDN_ERR_MISALIGNED;
    if (limit_ns == 0 || limit_ns > 2000000000ull) return GDN_ERR_INVALID_ARG;   // at most 2 s
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)cuda_stream>>>(status, limit_ns);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

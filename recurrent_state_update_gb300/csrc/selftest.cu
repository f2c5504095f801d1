// selftest.cu -- a diagnostic entry point that makes one bounded wait run out on purpose.
//
// Every kernel in this library waits on its asynchronous copies and tensor-core operations for at
// most umma::kWaitPolls mbarrier polls (about one second); a wait that runs out ORs
// MAMBA_ERR_TIMEOUT into the caller's error word and the kernel winds down instead of hanging.  This kernel waits, with the
// same helper and the same poll bound as the kernels, on a barrier phase that nothing completes,
// so a caller (a test, or an operator checking a new driver) can see that path end, read the
// flag, time the wait, and find the context still usable afterwards.  It touches no other memory.
#include "common.cuh"
#include "umma.cuh"

namespace ms {

__global__ void __launch_bounds__(32) k_wait_timeout(int32_t *err, uint64_t *elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    umma::mbar_init(&bar, 1);  // one arrival expected, and none is ever made
    umma::fence_mbar_init();
    uint64_t t0, t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    const bool done = umma::mbar_wait(&bar, 0, umma::kWaitPolls);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (!done) flag_error(err, MAMBA_ERR_TIMEOUT);
    if (elapsed_ns) *elapsed_ns = t1 - t0;
}

}  // namespace ms

using namespace ms;

extern "C" int mamba_selftest_wait_timeout(int32_t *err_word, uint64_t *elapsed_ns, void *stream) {
    MS_TRACE("mamba_selftest_wait_timeout");
    if (!err_word) return MAMBA_EINVAL;
    k_wait_timeout<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err_word, elapsed_ns);
    return launch_status();
}

// diag.cu -- kda_selftest_bounded_wait: the bounded-wait path of the kernels,
// exercised on purpose.
//
// Every wait of the tensor-core kernels (for a TMA copy or an MMA batch) is a
// bounded poll of an mbarrier that gives up, reports KDA_DEV_TIMEOUT and lets
// the kernel drain and return instead of spinning forever.  This entry point
// runs that same helper on an mbarrier nothing ever arrives on, so a test can
// watch the wait run out, read the status on the host and go on using the
// context; no copy or MMA is in flight, so nothing needs draining.
#include "kda_common.cuh"
#include "kda_host.h"
#include "umma.cuh"

namespace kda {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(uint32_t polls, int32_t* __restrict__ dev_status,
                                                          unsigned long long* __restrict__ cycles) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = umma::smem_u32(&bar);
    umma::mbar_init(b, 1);  // one arrival expected; none comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const long long t0 = clock64();
    const bool done = umma::mbar_wait(b, 0, polls);
    const long long t1 = clock64();
    if (!done) report(dev_status, KDA_DEV_TIMEOUT);
    if (cycles) *cycles = (unsigned long long)(t1 - t0);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_selftest_bounded_wait(uint32_t polls, int32_t* dev_status,
                                                unsigned long long* cycles, void* stream) {
    KDA_REQUIRE(dev_status != nullptr && aligned16(dev_status), KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(cycles == nullptr || aligned16(cycles), KDA_ERR_INVALID_ARG);
    bounded_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(polls, dev_status, cycles);
    return launch_status();
}

// selftest.cu - gdn_selftest_wait_timeout: exercises the bounded mbarrier
// wait that every wait of the chunked kernel goes through.
//
// One warp initialises an mbarrier that nothing ever arrives on and waits for
// its first phase with the library's bounded wait (mbar_wait).  The wait must
// give up after the limit and the kernel must record GDN_ERR_TIMEOUT and
// return, leaving the context usable.  This is how the library's failure path
// is tested without faulting or hanging the GPU.
#include "../../include/gdn.h"
#include "internal.h"
#include "sm100.cuh"

namespace gdn {
namespace {

__global__ void wait_timeout_probe_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_mbar_init();
    }
    __syncwarp();
    // phase 0 needs one arrival and none comes
    const bool done = sm100::mbar_wait(&bar, 0, limit_ns);
    if (threadIdx.x == 0) atomicExch(status, done ? GDN_OK : GDN_ERR_TIMEOUT);
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_selftest_wait_timeout(int32_t *status, int limit_us, void *stream) {
    if (!status) return gdn::set_error(GDN_ERR_NULL, "status is required");
    if (limit_us < 1 || limit_us > 1000000)
        return gdn::set_error(GDN_ERR_SHAPE, "limit_us=%d outside [1, 1000000]", limit_us);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gdn::wait_timeout_probe_kernel<<<1, 32, 0, s>>>(status, (uint64_t)limit_us * 1000u);
    gdn::note_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return gdn::set_error(GDN_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return GDN_OK;
}

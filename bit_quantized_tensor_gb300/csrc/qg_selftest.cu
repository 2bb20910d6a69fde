// qg_selftest_wait_timeout: exercises the failure path of the bounded waits
// on the device without faulting or hanging it.  One CTA waits on an
// mbarrier that nothing ever arrives on, under a caller-given limit; the wait
// runs out, the kernel records QG_ERR_TIMEOUT in the device status word (as
// any kernel of the library does when a copy or an MMA never completes) and
// returns, so the context stays usable and qg_device_status reports it.
#include "qg_internal.h"
#include "qg_ptx.cuh"

namespace qg {

constexpr int kSiteSelftest = 900;

__global__ void k_selftest_wait(Ctl ctl) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // one arrival expected; none is made
        fence_mbar_init();
    }
    __syncwarp();
    const bool done = bounded_wait(smem_u32(&bar), 0u, nullptr, ctl, kSiteSelftest);
    (void)done;  // false: the status word now holds QG_ERR_TIMEOUT
}

}  // namespace qg

extern "C" int qg_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
    if (limit_ns < 1 || limit_ns > 1000000000ull) return QG_ERR_INVALID_ARG;
    const int dev = qg::current_device();
    if (dev < 0) return QG_ERR_CUDA;
    qg::Ctl ctl = qg::host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    ctl.timeout_ns = limit_ns;
    qg::k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctl);
    return qg::map_cuda(cudaGetLastError());
}

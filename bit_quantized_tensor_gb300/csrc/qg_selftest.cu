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

// The three ways a hand-built pipeline deadlocks ("Warp-Specialized Kernel
// Implementation for W4A4 MatMul ...", section 3), each staged on purpose
// with bounded waits so that it ends in a recorded timeout instead of a hang:
//   kMissingArrival  a barrier expects two producer arrivals; the second
//                    producer skips its arrive, so the consumer's phase
//                    never completes.
//   kPhaseMismatch   the producer fills the slot once (phase 0 completes);
//                    the consumer starts with the wrong parity and waits for
//                    phase 1, which nobody will complete.
//   kCycle           a drain warp waits for the MMA warp's "full" barrier
//                    before arriving on "empty", and the MMA warp waits on
//                    "empty" before arriving on "full".
// The first role to give up raises a shared abort flag, which the other role
// polls and leaves on; each role records a site tag of its own.
constexpr int kMissingArrival = 1, kPhaseMismatch = 2, kCycle = 3;
constexpr int kSiteMissingArrival = 901, kSitePhaseMismatch = 902, kSiteCycleDrain = 903,
              kSiteCycleMma = 904;

__global__ void k_selftest_deadlock(Ctl ctl, int pattern) {
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    const bool leader = (threadIdx.x & 31) == 0;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar[0]), pattern == kMissingArrival ? 2 : 1);
        mbar_init(smem_u32(&bar[1]), 1);
        abort_flag = 0;
        fence_mbar_init();
        // phase 0 completes before anyone waits, so the consumer's wrong
        // parity always names the open phase 1 (had it waited first, parity 1
        // would have named the already-closed preceding phase and passed)
        if (pattern == kPhaseMismatch) mbar_arrive(smem_u32(&bar[0]));
    }
    __syncthreads();
    volatile int* abort_ptr = &abort_flag;
    if (pattern == kMissingArrival) {
        if (warp == 0 && leader) mbar_arrive(smem_u32(&bar[0]));  // producer 0 arrives
        // producer 1 (warp 1) skips its arrival
        if (warp == 2) bounded_wait(smem_u32(&bar[0]), 0u, abort_ptr, ctl, kSiteMissingArrival);
    } else if (pattern == kPhaseMismatch) {
        if (warp == 1) {
            const uint32_t wrong_parity = 1u;  // a consumer that starts on the wrong phase
            bounded_wait(smem_u32(&bar[0]), wrong_parity, abort_ptr, ctl, kSitePhaseMismatch);
        }
    } else {  // kCycle: bar[0] = full (MMA -> drain), bar[1] = empty (drain -> MMA)
        if (warp == 0) {  // drain
            if (bounded_wait(smem_u32(&bar[0]), 0u, abort_ptr, ctl, kSiteCycleDrain) && leader)
                mbar_arrive(smem_u32(&bar[1]));
        } else if (warp == 1) {  // MMA
            if (bounded_wait(smem_u32(&bar[1]), 0u, abort_ptr, ctl, kSiteCycleMma) && leader)
                mbar_arrive(smem_u32(&bar[0]));
        }
    }
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

extern "C" int qg_selftest_deadlock(int pattern, uint64_t limit_ns, void* stream) {
    if (pattern < qg::kMissingArrival || pattern > qg::kCycle) return QG_ERR_INVALID_ARG;
    if (limit_ns < 1 || limit_ns > 1000000000ull) return QG_ERR_INVALID_ARG;
    const int dev = qg::current_device();
    if (dev < 0) return QG_ERR_CUDA;
    qg::Ctl ctl = qg::host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    ctl.timeout_ns = limit_ns;
    qg::k_selftest_deadlock<<<1, 96, 0, static_cast<cudaStream_t>(stream)>>>(ctl, pattern);
    return qg::map_cuda(cudaGetLastError());
}

// Internal definitions shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qgemm.h"

#include <nvtx3/nvToolsExt.h>

namespace qg {

// An NVTX range named after a C-ABI call for the object's lifetime, so each
// call shows on a profiler's timeline (no effect unless a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Device status word layout (one per device, in qg_api.cu):
//   [0] first error code recorded (0 = none)
//   [1] call-site tag of that error (which role of which kernel)
//   [2] number of errors recorded
//   [3] block index that recorded the first error
//   [4] phase parity the timed-out wait was waiting for
//   [5] shared-memory address of the barrier it waited on (the ring slot)
constexpr int kStatusWords = 6;

// Backstop on bounded_wait when %globaltimer does not advance.
constexpr uint32_t kMaxWaitIterations = 1u << 30;

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

struct Ctl {
    int* status;          // device status word (kStatusWords ints)
    uint64_t timeout_ns;  // limit of every bounded wait
};

__device__ __forceinline__ void report_error(const Ctl& ctl, int code, int site, uint32_t bar = 0,
                                             uint32_t parity = 0) {
    if (atomicCAS(ctl.status, 0, code) == 0) {
        ctl.status[1] = site;
        ctl.status[3] = static_cast<int>(blockIdx.x);
        ctl.status[4] = static_cast<int>(parity);
        ctl.status[5] = static_cast<int>(bar);
    }
    atomicAdd(ctl.status + 2, 1);
}

// Resource budget of one kernel instance: what a CTA of it asks of an SM and
// how many CTAs of it the design counts on finding resident on one SM.  Each
// translation unit registers the instances it launches (QG_KERNEL_BUDGET) at
// load time; the C ABI lists them (qg_kernel_budget_*), so that tests can
// check the accounting on the host and the real residency (registers
// included) on a device.
struct KernelBudget {
    const char* name;     // kernel with its template arguments
    const void* func;     // host stub, for occupancy queries
    int threads;          // threads per CTA
    int smem_bytes;       // largest dynamic shared memory a launch requests
    int tmem_cols;        // tensor-memory columns each CTA allocates (0 = none)
    int cluster;          // CTAs per cluster
    int min_ctas_per_sm;  // CTAs of this kernel the design needs resident per SM
};
int register_kernel_budget(const KernelBudget& b);

#define QG_BUDGET_CAT2(a, b) a##b
#define QG_BUDGET_CAT(a, b) QG_BUDGET_CAT2(a, b)
#define QG_KERNEL_BUDGET(...)                                       \
    static const int QG_BUDGET_CAT(qg_kernel_budget_, __COUNTER__) = \
        ::qg::register_kernel_budget(::qg::KernelBudget{__VA_ARGS__})

// Workspace bytes of qgemm_s8_host (qg_hostio.cu).
size_t s8_host_workspace(int64_t M, int64_t N, int64_t K);

// Host helpers (qg_api.cu).
Ctl host_ctl(int device);  // status pointer of `device` + current timeout
int num_sms(int device);
int current_device();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Records the code of a failed runtime call (positive) or driver call
// (negative) for qg_last_cuda_error(); returns QG_ERR_CUDA.
int record_cuda_error(int code);

inline int map_cuda(cudaError_t e) {
    return e == cudaSuccess ? QG_OK : record_cuda_error(static_cast<int>(e));
}

}  // namespace qg

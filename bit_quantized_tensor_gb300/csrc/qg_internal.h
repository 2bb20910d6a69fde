// Internal definitions shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qgemm.h"

namespace qg {

// Device status word layout (one per device, in qg_api.cu):
//   [0] first error code recorded (0 = none)
//   [1] call-site tag of that error
//   [2] number of errors recorded
//   [3] block index that recorded the first error
constexpr int kStatusWords = 4;

// Backstop on bounded_wait when %globaltimer does not advance.
constexpr uint32_t kMaxWaitIterations = 1u << 30;

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

struct Ctl {
    int* status;          // device status word (kStatusWords ints)
    uint64_t timeout_ns;  // limit of every bounded wait
};

__device__ __forceinline__ void report_error(const Ctl& ctl, int code, int site) {
    if (atomicCAS(ctl.status, 0, code) == 0) {
        ctl.status[1] = site;
        ctl.status[3] = static_cast<int>(blockIdx.x);
    }
    atomicAdd(ctl.status + 2, 1);
}

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

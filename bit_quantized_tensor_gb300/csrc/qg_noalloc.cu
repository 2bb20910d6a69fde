// qgemm_s8_noalloc: the exact INT8 GEMM for callers that cannot allocate.
//
// qgemm_s8 needs a scratch workspace (fp16 copies of both operands) that the
// caller allocates.  Some callers have no way to do that: plugin hosts that
// hand a kernel only its inputs and outputs and own every allocation,
// inference engines whose memory plan is frozen after start-up, and code
// that must not call cudaMalloc because it would synchronize the device or
// is not allowed at that point.  For them this entry point uses a fixed
// scratch array that lives in the library's device image instead:
//
//  - the array is a file-scope static __device__ array of kScratchBytes
//    (16 MiB); every GPU that loads this library holds it until the process
//    exits;
//  - problems whose scratch need, 2*K*(M+N) bytes rounded up to 256-byte
//    boundaries per operand, exceeds it are rejected with QG_ERR_WORKSPACE
//    before anything is enqueued;
//  - the first call on each device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture on the device;
//  - the stream must belong to the current device (checked: the cached
//    address is that device's); the cache lives as long as the library and
//    is not refreshed if a device is reset (cudaDeviceReset), so the library
//    must not be used on a device after that device was reset;
//  - every call shares the one array and it keeps the last call's contents.
//    Nothing in it has to start at zero (each call overwrites the part it
//    reads first), but calls that overlap on the GPU (different streams, or
//    different host threads without ordering) race on it and must be
//    serialized by the caller.
// Apart from where the scratch comes from, the work is exactly qgemm_s8's.
#include <mutex>

#include "qg_internal.h"

namespace {

constexpr size_t kScratchBytes = QG_S8_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_s8_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_s8_scratch on the current device (set up once per
// device; a failed lookup is retried on the next call).
int scratch_address(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_s8_scratch);
        if (e != cudaSuccess || p == nullptr) return qg::map_cuda(e == cudaSuccess ? cudaErrorUnknown : e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QG_OK;
}

}  // namespace

extern "C" int qgemm_s8_noalloc(int64_t M, int64_t N, int64_t K, const int8_t* A, int64_t lda,
                                int layout_a, const int8_t* B, int64_t ldb, int layout_b,
                                int32_t* C, int64_t ldc, void* stream) {
    const qg::NvtxRange nvtx_range("qgemm_s8_noalloc");
    if (M < 1 || N < 1 || K < 1) return QG_ERR_INVALID_ARG;
    const size_t need = qg_workspace_size(QG_OP_S8, M, N, K);
    if (need == 0 || need > kScratchBytes) return QG_ERR_WORKSPACE;
    const int dev = qg::current_device();
    if (dev < 0 || dev >= kMaxDevices) return QG_ERR_CUDA;
    if (stream) {
        // the scratch address is per device: a stream of another device would
        // run the kernels against the wrong device's array
        int sdev = -1;
        if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
            cudaGetLastError();
            return QG_ERR_INVALID_ARG;
        }
        if (sdev != dev) return QG_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    const int rc = scratch_address(dev, &scratch);
    if (rc != QG_OK) return rc;
    return qgemm_s8(M, N, K, A, lda, layout_a, B, ldb, layout_b, C, ldc, scratch, kScratchBytes,
                    stream);
}

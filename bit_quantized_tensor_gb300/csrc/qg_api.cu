// Library-wide C ABI pieces: status strings, workspace sizes, the device
// status word written by bounded waits, and the wait time limit.
#include <atomic>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "qg_internal.h"

namespace {

// One status word per device (see qg::kStatusWords).  A device variable is
// instantiated, zero-filled, on every device that loads the module.
__device__ int g_status[qg::kStatusWords];

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::once_flag g_status_once[kMaxDevices];
int g_sms[kMaxDevices] = {};
std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<int> g_last_cuda_error{0};

uint64_t timeout_from_env() {
    const char* e = std::getenv("QG_TIMEOUT_NS");
    if (e && *e) {
        unsigned long long v = std::strtoull(e, nullptr, 10);
        if (v > 0) return v;
    }
    return qg::kDefaultTimeoutNs;
}

std::vector<qg::KernelBudget>& budgets() {
    static std::vector<qg::KernelBudget> v;
    return v;
}

std::mutex& budgets_mutex() {
    static std::mutex m;
    return m;
}

}  // namespace

namespace qg {

int register_kernel_budget(const KernelBudget& b) {
    std::lock_guard<std::mutex> g(budgets_mutex());
    budgets().push_back(b);
    return static_cast<int>(budgets().size()) - 1;
}

int record_cuda_error(int code) {
    g_last_cuda_error.store(code);
    return QG_ERR_CUDA;
}

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

Ctl host_ctl(int device) {
    Ctl c{nullptr, 0};
    if (device < 0 || device >= kMaxDevices) return c;
    std::call_once(g_status_once[device], [device] {
        void* p = nullptr;
        int prev = 0;
        cudaGetDevice(&prev);
        cudaSetDevice(device);
        if (cudaGetSymbolAddress(&p, g_status) == cudaSuccess) g_status_ptr[device] = static_cast<int*>(p);
        cudaSetDevice(prev);
    });
    uint64_t t = g_timeout_ns.load();
    if (t == 0) {
        t = timeout_from_env();
        g_timeout_ns.store(t);
    }
    c.status = g_status_ptr[device];
    c.timeout_ns = t;
    return c;
}

int num_sms(int device) {
    if (device < 0 || device >= kMaxDevices) return 1;
    if (g_sms[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
            n = 1;
        g_sms[device] = n;
    }
    return g_sms[device];
}

}  // namespace qg

static size_t round_up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

extern "C" {

const char* qg_status_string(int status) {
    switch (status) {
        case QG_OK: return "QG_OK";
        case QG_ERR_INVALID_ARG: return "QG_ERR_INVALID_ARG";
        case QG_ERR_UNSUPPORTED: return "QG_ERR_UNSUPPORTED";
        case QG_ERR_MISALIGNED: return "QG_ERR_MISALIGNED";
        case QG_ERR_WORKSPACE: return "QG_ERR_WORKSPACE";
        case QG_ERR_CUDA: return "QG_ERR_CUDA";
        case QG_ERR_TIMEOUT: return "QG_ERR_TIMEOUT";
        default: return "QG_ERR_UNKNOWN";
    }
}

int qg_version(void) { return 100; }

size_t qg_workspace_size(int op, int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const size_t m = static_cast<size_t>(M), n = static_cast<size_t>(N), k = static_cast<size_t>(K);
    switch (op) {
        case QG_OP_S8:  // fp16 copies of both operands (exact for int8 values)
            return round_up256(2 * m * k) + round_up256(2 * n * k);
        case QG_OP_S4:  // e4m3 copies of both operands (exact for int4 values)
            return round_up256(m * k) + round_up256(n * k);
        case QG_OP_S8_HOST:  // device copies of A, B, C and fp16 forms of A, B
            return qg::s8_host_workspace(M, N, K);
        case QG_OP_W4A4: {  // e4m3 operands, transposed fp32 scale tables
            const size_t nblk = k / 64 + 1;
            const size_t mp = (m + 3) & ~static_cast<size_t>(3), np = (n + 3) & ~static_cast<size_t>(3);
            return round_up256(m * k) + round_up256(n * k) + round_up256(4 * nblk * mp) +
                   round_up256(4 * nblk * np);
        }
        case QG_OP_W4A4_PREPACKED: {  // the X side only
            const size_t nblk = k / 64 + 1;
            const size_t mp = (m + 3) & ~static_cast<size_t>(3);
            return round_up256(m * k) + round_up256(4 * nblk * mp);
        }
        case QG_OP_W4A4_WEIGHTS: {  // packed weights: e4m3 codes, transposed scale table (M unused)
            const size_t nblk = k / 64 + 1;
            const size_t np = (n + 3) & ~static_cast<size_t>(3);
            return round_up256(n * k) + round_up256(4 * nblk * np);
        }
        default:
            return 0;
    }
}

int qg_last_cuda_error(void) { return g_last_cuda_error.exchange(0); }

int qg_set_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns == 0 ? timeout_from_env() : ns);
    return QG_OK;
}

int qg_device_status_detail(int* words, void* stream) {
    const int dev = qg::current_device();
    if (dev < 0) return QG_ERR_CUDA;
    qg::Ctl c = qg::host_ctl(dev);
    if (!c.status) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return QG_ERR_CUDA;
    int h[qg::kStatusWords] = {};
    if (cudaMemcpy(h, c.status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return QG_ERR_CUDA;
    if (words) {
        for (int i = 0; i < qg::kStatusWords; ++i) words[i] = h[i];
    }
    if (h[0] != 0) {
        const int z[qg::kStatusWords] = {};
        if (cudaMemcpy(c.status, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return QG_ERR_CUDA;
        return h[0];
    }
    return QG_OK;
}

int qg_device_status(void* stream) { return qg_device_status_detail(nullptr, stream); }

int qg_kernel_budget_count(void) {
    std::lock_guard<std::mutex> g(budgets_mutex());
    return static_cast<int>(budgets().size());
}

int qg_kernel_budget_get(int index, qg_kernel_budget* out) {
    if (!out) return QG_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(budgets_mutex());
    if (index < 0 || index >= static_cast<int>(budgets().size())) return QG_ERR_INVALID_ARG;
    const qg::KernelBudget& b = budgets()[static_cast<size_t>(index)];
    out->kernel = b.name;
    out->threads = b.threads;
    out->smem_bytes = b.smem_bytes;
    out->tmem_cols = b.tmem_cols;
    out->cluster = b.cluster;
    out->min_ctas_per_sm = b.min_ctas_per_sm;
    return QG_OK;
}

int qg_kernel_budget_measure(int index, int* regs_per_thread, int* static_smem_bytes,
                             int* ctas_per_sm) {
    if (!regs_per_thread || !static_smem_bytes || !ctas_per_sm) return QG_ERR_INVALID_ARG;
    qg::KernelBudget b;
    {
        std::lock_guard<std::mutex> g(budgets_mutex());
        if (index < 0 || index >= static_cast<int>(budgets().size())) return QG_ERR_INVALID_ARG;
        b = budgets()[static_cast<size_t>(index)];
    }
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, b.func);
    if (e != cudaSuccess) return qg::map_cuda(e);
    *regs_per_thread = fa.numRegs;
    *static_smem_bytes = static_cast<int>(fa.sharedSizeBytes);
    if (b.smem_bytes > 0) {
        e = cudaFuncSetAttribute(b.func, cudaFuncAttributeMaxDynamicSharedMemorySize, b.smem_bytes);
        if (e != cudaSuccess) return qg::map_cuda(e);
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, b.func, b.threads,
                                                      static_cast<size_t>(b.smem_bytes));
    if (e != cudaSuccess) return qg::map_cuda(e);
    *ctas_per_sm = n;
    return QG_OK;
}

}  // extern "C"

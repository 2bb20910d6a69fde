// qgemm_s8_host: the exact INT8 GEMM with its operands and result in host
// memory.
//
// A host-resident problem crosses the host link three times (A and B in, C
// out; for a square int8 problem C alone is twice the size of both inputs),
// and on this machine the link, not the tensor cores, sets the time.  The
// call therefore cuts the problem into pieces (row slices of A times row
// slices of B) and overlaps three queues, each an internal stream of the
// current device:
//   copy-in    A slices and B slices, host -> device, each exactly once, in
//              the order the pieces need them (A0, B0, B1, ..., A1, A2, ...);
//   compute    each slice converted to fp16 once (exact for int8), then one
//              tensor-core GEMM per piece into a device copy of C;
//   copy-out   each piece of C, device -> host, as soon as its GEMM is done.
// The first piece needs one A slice and one B slice only, so results flow
// back while the rest of the inputs are still arriving, and the copy-out
// queue (the longest) runs from then on without gaps.
//
// Ordering: the queues start after the work already enqueued on the caller's
// stream, and the caller's stream waits for the last copy-out, so the call
// behaves as one operation on that stream.  The queues and their events are
// created once per device and shared by every call on that device (calls are
// enqueued under a per-device lock).
#include <mutex>

#include <cuda_fp16.h>

#include "qg_gemm_host.h"
#include "qg_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxASlices = 8;
constexpr int kMaxBSlices = 2;
constexpr int64_t kMinASliceRows = 1024;
constexpr int64_t kSplitBFrom = 4096;  // N from which B is cut in two slices
constexpr int kEvents = 4 + kMaxASlices + kMaxBSlices + kMaxASlices * kMaxBSlices;

struct Queues {
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t ev[kEvents] = {};
    bool ready = false;
};

std::mutex g_mu[kMaxDevices];
Queues g_queues[kMaxDevices];

void destroy(Queues& q) {
    for (cudaEvent_t& e : q.ev)
        if (e) {
            cudaEventDestroy(e);
            e = nullptr;
        }
    for (cudaStream_t* s : {&q.in, &q.comp, &q.out})
        if (*s) {
            cudaStreamDestroy(*s);
            *s = nullptr;
        }
}

// The device's queues, created on first use (caller holds g_mu[dev]).
int get_queues(int dev, Queues** out) {
    Queues& q = g_queues[dev];
    if (!q.ready) {
        cudaError_t e = cudaSuccess;
        for (cudaStream_t* s : {&q.in, &q.comp, &q.out})
            if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
        for (cudaEvent_t& ev : q.ev)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            destroy(q);
            return qg::map_cuda(e);
        }
        q.ready = true;
    }
    *out = &q;
    return QG_OK;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// How the problem is cut: A in `a` slices of `ra` rows (the last one
// shorter), B in `b` slices of `cb` rows.  Slices are multiples of 256 rows
// (whole 256 x 256 tiles of the paired GEMM kernel) except the last.
struct Plan {
    int64_t ra, cb;
    int a, b;
};

Plan make_plan(int64_t M, int64_t N) {
    Plan p;
    p.ra = round_up((M + kMaxASlices - 1) / kMaxASlices, 256);
    if (p.ra < kMinASliceRows) p.ra = kMinASliceRows;
    if (p.ra > M) p.ra = M;
    p.a = static_cast<int>((M + p.ra - 1) / p.ra);
    p.cb = N >= kSplitBFrom ? round_up((N + kMaxBSlices - 1) / kMaxBSlices, 256) : N;
    p.b = static_cast<int>((N + p.cb - 1) / p.cb);
    return p;
}

// Device buffers inside the workspace, each at a 256-byte boundary.
struct Buffers {
    int8_t *a8, *b8;
    __half *a16, *b16;
    int32_t* c32;
    int64_t ldc32;  // row stride of the device copy of C, in elements
    size_t bytes;
};

Buffers carve(void* ws, int64_t M, int64_t N, int64_t K) {
    Buffers b;
    const size_t m = static_cast<size_t>(M), n = static_cast<size_t>(N), k = static_cast<size_t>(K);
    b.ldc32 = round_up(N, 4);
    auto r = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    const size_t o_b8 = r(m * k), o_a16 = o_b8 + r(n * k), o_b16 = o_a16 + r(2 * m * k),
                 o_c32 = o_b16 + r(2 * n * k);
    b.bytes = o_c32 + r(4 * m * static_cast<size_t>(b.ldc32));
    uint8_t* base = static_cast<uint8_t*>(ws);
    b.a8 = reinterpret_cast<int8_t*>(base);
    b.b8 = reinterpret_cast<int8_t*>(base + o_b8);
    b.a16 = reinterpret_cast<__half*>(base + o_a16);
    b.b16 = reinterpret_cast<__half*>(base + o_b16);
    b.c32 = reinterpret_cast<int32_t*>(base + o_c32);
    return b;
}

}  // namespace

namespace qg {

size_t s8_host_workspace(int64_t M, int64_t N, int64_t K) { return carve(nullptr, M, N, K).bytes; }

}  // namespace qg

extern "C" int qgemm_s8_host(int64_t M, int64_t N, int64_t K, const int8_t* A, int64_t lda, const int8_t* B,
                             int64_t ldb, int32_t* C, int64_t ldc, void* ws, size_t ws_bytes, void* stream) {
    const qg::NvtxRange nvtx_range("qgemm_s8_host");
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX) return QG_ERR_INVALID_ARG;
    if (!A || !B || !C) return QG_ERR_INVALID_ARG;
    if (K % 16 || K >= 131072) return QG_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldc < N) return QG_ERR_INVALID_ARG;
    if (!ws || ws_bytes < qg::s8_host_workspace(M, N, K)) return QG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QG_ERR_MISALIGNED;
    const int dev = qg::current_device();
    if (dev < 0 || dev >= kMaxDevices) return QG_ERR_CUDA;
    qg::Ctl ctl = qg::host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;

    std::lock_guard<std::mutex> lock(g_mu[dev]);
    Queues* q = nullptr;
    int rc = get_queues(dev, &q);
    if (rc) return rc;
    const Plan p = make_plan(M, N);
    const Buffers d = carve(ws, M, N, K);
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    cudaEvent_t ev_start = q->ev[0], ev_end = q->ev[1], ev_in_end = q->ev[2], ev_comp_end = q->ev[3];
    cudaEvent_t* ev_a = q->ev + 4;
    cudaEvent_t* ev_b = ev_a + kMaxASlices;
    cudaEvent_t* ev_piece = ev_b + kMaxBSlices;
    auto rows_a = [&](int i) { return i + 1 < p.a ? p.ra : M - static_cast<int64_t>(i) * p.ra; };
    auto rows_b = [&](int j) { return j + 1 < p.b ? p.cb : N - static_cast<int64_t>(j) * p.cb; };

    cudaError_t e = cudaEventRecord(ev_start, user);
    for (cudaStream_t s : {q->in, q->comp, q->out})
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_start, 0);

    // copy-in, in the order the pieces use the slices
    auto copy_a = [&](int i) {
        const int64_t r0 = static_cast<int64_t>(i) * p.ra;
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(d.a8 + r0 * K, static_cast<size_t>(K), A + r0 * lda, static_cast<size_t>(lda),
                                  static_cast<size_t>(K), static_cast<size_t>(rows_a(i)), cudaMemcpyHostToDevice,
                                  q->in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_a[i], q->in);
    };
    auto copy_b = [&](int j) {
        const int64_t r0 = static_cast<int64_t>(j) * p.cb;
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(d.b8 + r0 * K, static_cast<size_t>(K), B + r0 * ldb, static_cast<size_t>(ldb),
                                  static_cast<size_t>(K), static_cast<size_t>(rows_b(j)), cudaMemcpyHostToDevice,
                                  q->in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_b[j], q->in);
    };
    // Copy-in order A0, B0, A1, B1, A2, ...: the first pieces need only the
    // first slices, and the first rows of C start back across the link early
    // (with all of B first, the second row of pieces waited behind it).
    const int nin = p.a > p.b ? p.a : p.b;
    for (int k = 0; k < nin; ++k) {
        if (k < p.a) copy_a(k);
        if (k < p.b) copy_b(k);
    }

    // One piece: convert its slices on first use, GEMM, copy the piece of C out.
    bool a_conv[kMaxASlices] = {}, b_conv[kMaxBSlices] = {};
    auto piece = [&](int i, int j) {
        const int64_t r0 = static_cast<int64_t>(i) * p.ra;
        const int64_t c0 = static_cast<int64_t>(j) * p.cb;
        if (!a_conv[i]) {
            if (e == cudaSuccess) e = cudaStreamWaitEvent(q->comp, ev_a[i], 0);
            if (e == cudaSuccess && rc == QG_OK)
                rc = qg::s8_to_f16_rows(d.a8 + r0 * K, rows_a(i), K, d.a16 + r0 * K, K, dev, q->comp);
            a_conv[i] = true;
        }
        if (!b_conv[j]) {
            if (e == cudaSuccess) e = cudaStreamWaitEvent(q->comp, ev_b[j], 0);
            if (e == cudaSuccess && rc == QG_OK)
                rc = qg::s8_to_f16_rows(d.b8 + c0 * K, rows_b(j), K, d.b16 + c0 * K, K, dev, q->comp);
            b_conv[j] = true;
        }
        if (e != cudaSuccess || rc != QG_OK) return;
        rc = qg::run_gemm_s8_converted(d.a16 + r0 * K, d.b16 + c0 * K, rows_a(i), rows_b(j), K,
                                       d.c32 + r0 * d.ldc32 + c0, d.ldc32, ctl, q->comp);
        if (rc != QG_OK) return;
        cudaEvent_t ev = ev_piece[i * kMaxBSlices + j];
        e = cudaEventRecord(ev, q->comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(q->out, ev, 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(C + r0 * ldc + c0, static_cast<size_t>(ldc) * 4, d.c32 + r0 * d.ldc32 + c0,
                                  static_cast<size_t>(d.ldc32) * 4, static_cast<size_t>(rows_b(j)) * 4,
                                  static_cast<size_t>(rows_a(i)), cudaMemcpyDeviceToHost, q->out);
    };
    // Pieces in the order their slices arrive: each slice, once copied in,
    // completes the pieces whose other slice is already there.
    for (int k = 0; k < nin && e == cudaSuccess && rc == QG_OK; ++k) {
        if (k < p.a)
            for (int j = 0; j < p.b && j < k && e == cudaSuccess && rc == QG_OK; ++j) piece(k, j);
        if (k < p.b)
            for (int i = 0; i < p.a && i <= k && e == cudaSuccess && rc == QG_OK; ++i) piece(i, k);
    }
    if (e == cudaSuccess && rc == QG_OK) {
        // join all three queues back into the caller's stream (the copy-out
        // queue ends last; the other two are joined explicitly so that a
        // stream capture sees every fork closed)
        e = cudaEventRecord(ev_end, q->out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in_end, q->in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_comp_end, q->comp);
        for (cudaEvent_t ev : {ev_in_end, ev_comp_end, ev_end})
            if (e == cudaSuccess) e = cudaStreamWaitEvent(user, ev, 0);
        if (e == cudaSuccess) return QG_OK;
    }
    // Something failed part-way: let what was enqueued finish before the
    // buffers go back to the caller.
    for (cudaStream_t s : {q->in, q->comp, q->out}) cudaStreamSynchronize(s);
    return rc != QG_OK ? rc : qg::map_cuda(e);
}

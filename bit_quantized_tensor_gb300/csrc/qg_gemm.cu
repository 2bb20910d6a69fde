// Dense GEMM entry points on the tcgen05 kernel: gemm_f16, qgemm_s8, qgemm_s4.
//
// sm_103a has no integer tcgen05 MMA kind, so the exact integer GEMMs carry
// their integer operands in floating-point types that hold them exactly:
//   int8 -> fp16 (every integer of magnitude <= 2048 is exact), kind::f16,
//           fp32 accumulation cut into K-chunks of at most 1024 so every
//           partial sum is an integer of magnitude <= 128*128*1024 = 2^24;
//   int4 -> e4m3 (every integer in [-8, 8] is exact), kind::f8f6f4, partial
//           sums of magnitude <= 64*K, exact in fp32 for K < 2^18.
// Source of the operations: "Hand-Written PTX Tensor-Core GEMM Kernels: A
// Multi-Precision Study on NVIDIA L4" (abstract): exact INT8 / INT4 GEMM with
// 32-bit results, and FP16 GEMM as the comparison point.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>
#include <mutex>

#include "qg_gemm_host.h"
#include "tc_gemm2.cuh"

namespace qg {

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int64_t inner,
                 int64_t outer, int64_t row_stride_bytes, int box_inner, int box_outer,
                 CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return QG_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QG_OK : record_cuda_error(-static_cast<int>(r));
}

int make_tmap_kmajor(CUtensorMap* map, bool fp16, const void* base, int64_t k_elems, int64_t rows,
                     int64_t row_stride_bytes, int box_k, int box_rows) {
    return make_tmap_2d(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        base, k_elems, rows, row_stride_bytes, box_k, box_rows,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

// ------------------------------------------------------------ tc GEMM launch

// Caller-owned CUDA events recorded around every tcgen05 GEMM launch while
// set (measurement of the main kernel alone); null = off.
static std::atomic<void*> g_prof_before{nullptr}, g_prof_after{nullptr};

void profile_events(void** before, void** after) {
    *before = g_prof_before.load();
    *after = g_prof_after.load();
}

template <class Cfg>
static int launch_tc(const void* A, int64_t lda_bytes, const void* B, int64_t ldb_bytes, int64_t M,
                     int64_t N, int64_t K, void* C, int64_t ldc, int chunk_kb, const __half* bias,
                     const Ctl& ctl, cudaStream_t stream) {
    constexpr bool f16 = Cfg::KIND == MmaKind::F16;
    CUtensorMap ta, tb;
    int rc = make_tmap_kmajor(&ta, f16, A, K, M, lda_bytes, Cfg::BK, Cfg::BM);
    if (rc) return rc;
    rc = make_tmap_kmajor(&tb, f16, B, K, N, ldb_bytes, Cfg::BK, Cfg::BN);
    if (rc) return rc;

    const int dev = current_device();
    if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
    static std::mutex mu;
    static bool attr_set[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<Cfg>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }

    TcGemmParams p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>((K + Cfg::BK - 1) / Cfg::BK);
    p.chunk_kb = chunk_kb > 0 ? chunk_kb : p.num_kb;
    p.C = C;
    p.ldc = ldc;
    p.bias = bias;
    p.ctl = ctl;
    const int64_t tiles = ((M + Cfg::BM - 1) / Cfg::BM) * ((N + Cfg::BN - 1) / Cfg::BN);
    const int grid = static_cast<int>(tiles < num_sms(dev) ? tiles : num_sms(dev));
    cudaEvent_t ev0 = static_cast<cudaEvent_t>(g_prof_before.load());
    cudaEvent_t ev1 = static_cast<cudaEvent_t>(g_prof_after.load());
    if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return QG_ERR_CUDA;
    tc_gemm_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, p);
    rc = map_cuda(cudaGetLastError());
    if (!rc && ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return QG_ERR_CUDA;
    return rc;
}

// Paired-CTA version (cta_group::2, 256 x 256 tiles per SM pair).
template <class Cfg>
static int launch_tc2(const void* A, int64_t lda_bytes, const void* B, int64_t ldb_bytes, int64_t M,
                      int64_t N, int64_t K, void* C, int64_t ldc, int chunk_kb, const __half* bias,
                      const Ctl& ctl, cudaStream_t stream) {
    constexpr bool f16 = Cfg::KIND == MmaKind::F16;
    CUtensorMap ta, tb;
    int rc = make_tmap_kmajor(&ta, f16, A, K, M, lda_bytes, Cfg::BK, Cfg::BM);
    if (rc) return rc;
    rc = make_tmap_kmajor(&tb, f16, B, K, N, ldb_bytes, Cfg::BK, Cfg::B_ROWS);
    if (rc) return rc;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
    static std::mutex mu;
    static bool attr_set[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(tc_gemm2_kernel<Cfg>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }
    TcGemmParams p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>((K + Cfg::BK - 1) / Cfg::BK);
    p.chunk_kb = chunk_kb > 0 ? chunk_kb : p.num_kb;
    p.C = C;
    p.ldc = ldc;
    p.bias = bias;
    p.ctl = ctl;
    const int64_t tiles = ((M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * ((N + Cfg::BN - 1) / Cfg::BN);
    const int64_t max_pairs = num_sms(dev) / 2;
    const int grid = 2 * static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
    void *pb = nullptr, *pa = nullptr;
    profile_events(&pb, &pa);
    if (pb && cudaEventRecord(static_cast<cudaEvent_t>(pb), stream) != cudaSuccess) return QG_ERR_CUDA;
    tc_gemm2_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, p);
    rc = map_cuda(cudaGetLastError());
    if (!rc && pa && cudaEventRecord(static_cast<cudaEvent_t>(pa), stream) != cudaSuccess)
        return QG_ERR_CUDA;
    return rc;
}

// GEMM kernel choice: 0 = by shape (pairs when M >= 256 and N >= 256),
// 1 = always one CTA per tile, 2 = always CTA pairs.  Testing hook.
static std::atomic<int> g_gemm_path{0};

int gemm_path() { return g_gemm_path.load(); }

static bool use_pairs(int64_t M, int64_t N) {
    const int path = g_gemm_path.load();
    if (path == 1) return false;
    if (path == 2) return true;
    return M >= 256 && N >= 256;
}

template <MmaKind KIND, Epi EPI>
static int launch_gemm(const void* A, int64_t lda_bytes, const void* B, int64_t ldb_bytes, int64_t M,
                       int64_t N, int64_t K, void* C, int64_t ldc, int chunk_kb, const __half* bias,
                       const Ctl& ctl, cudaStream_t stream) {
    if (use_pairs(M, N))
        return launch_tc2<Tc2Cfg<KIND, EPI>>(A, lda_bytes, B, ldb_bytes, M, N, K, C, ldc, chunk_kb,
                                            bias, ctl, stream);
    return launch_tc<TcGemmCfg<KIND, EPI>>(A, lda_bytes, B, ldb_bytes, M, N, K, C, ldc, chunk_kb,
                                          bias, ctl, stream);
}

int run_gemm_f16_tc(const __half* A, int64_t lda, const __half* B, int64_t ldb, int64_t M, int64_t N,
                    int64_t K, __half* C, int64_t ldc, const __half* bias, const Ctl& ctl,
                    cudaStream_t stream) {
    return launch_gemm<MmaKind::F16, Epi::F16>(A, lda * 2, B, ldb * 2, M, N, K, C, ldc, 0, bias, ctl,
                                               stream);
}

// -------------------------------------------------------- operand converters

// int8 -> fp16, 16 elements per thread; cols is a multiple of 16.
__global__ void k_s8_to_f16(const int8_t* __restrict__ src, int64_t rows, int64_t cols, int64_t lds,
                            __half* __restrict__ dst, int64_t ldd) {
    const int64_t per_row = cols / 16;
    const int64_t total = rows * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / per_row;
        const int64_t c = (i - r * per_row) * 16;
        const int4 v = __ldg(reinterpret_cast<const int4*>(src + r * lds + c));
        const int8_t* b = reinterpret_cast<const int8_t*>(&v);
        uint4 o[2];
        __half2* h = reinterpret_cast<__half2*>(o);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            h[j] = __halves2half2(__short2half_rn(b[2 * j]), __short2half_rn(b[2 * j + 1]));
        uint4* d = reinterpret_cast<uint4*>(dst + r * ldd + c);
        d[0] = o[0];
        d[1] = o[1];
    }
}

// Packed signed 4-bit (low nibble = even k) -> one e4m3 byte per value.
// 16 packed bytes (32 values) per thread; bytes_per_row is a multiple of 16.
__global__ void k_s4_to_e4m3(const uint8_t* __restrict__ src, int64_t rows, int64_t bytes_per_row,
                             int64_t lds, uint8_t* __restrict__ dst, int64_t ldd) {
    // e4m3 code of each nibble value, built with the hardware conversion.
    uint64_t lut_lo = 0, lut_hi = 0;  // nibbles 0..7 and 8..15
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const float v = static_cast<float>(n < 8 ? n : n - 16);
        const uint64_t code =
            static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
        if (n < 8)
            lut_lo |= code << (8 * n);
        else
            lut_hi |= code << (8 * (n - 8));
    }
    const int64_t per_row = bytes_per_row / 16;
    const int64_t total = rows * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / per_row;
        const int64_t c = (i - r * per_row) * 16;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * lds + c));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t nib = (w[q] >> (4 * (4 * h + j))) & 0xFu;
                    const uint64_t tab = nib < 8 ? lut_lo : lut_hi;
                    const uint32_t code = static_cast<uint32_t>(tab >> (8 * (nib & 7u))) & 0xFFu;
                    o |= code << (8 * j);
                }
                out[2 * q + h] = o;
            }
        }
        uint4* d = reinterpret_cast<uint4*>(dst + r * ldd + 2 * c);
        d[0] = make_uint4(out[0], out[1], out[2], out[3]);
        d[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
}

int s4_to_e4m3(const uint8_t* src, int64_t rows, int64_t K, int64_t lds_bytes, uint8_t* dst,
               int64_t ldd, int dev, cudaStream_t s) {
    k_s4_to_e4m3<<<conv_grid(dev, rows * K / 32), 256, 0, s>>>(src, rows, K / 2, lds_bytes, dst, ldd);
    return map_cuda(cudaGetLastError());
}

int conv_grid(int dev, int64_t work_items) {
    const int64_t per_block = 256;
    int64_t g = (work_items + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(num_sms(dev)) * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

// Chunk length (in k-blocks of 64) of the exact int8 path; <= 16 keeps
// every fp32 partial sum within 2^24.  Adjustable for tests.
static int g_s8_chunk_kb = 16;

}  // namespace qg

using namespace qg;

static bool bad_layouts(int la, int lb) { return la != QG_ROW_MAJOR || lb != QG_COL_MAJOR; }

extern "C" {

int qg_set_profile_events(void* before, void* after) {
    if ((before == nullptr) != (after == nullptr)) return QG_ERR_INVALID_ARG;
    g_prof_before.store(before);
    g_prof_after.store(after);
    return QG_OK;
}

int qg_set_gemm_path(int path) {
    if (path < 0 || path > 2) return QG_ERR_INVALID_ARG;
    g_gemm_path.store(path);
    return QG_OK;
}

int qg_set_s8_chunk(int kblocks) {
    if (kblocks < 1 || kblocks > 16) return QG_ERR_INVALID_ARG;
    g_s8_chunk_kb = kblocks;
    return QG_OK;
}

int gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int layout_a,
             const uint16_t* B, int64_t ldb, int layout_b, uint16_t* C, int64_t ldc, void* stream) {
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return QG_ERR_INVALID_ARG;
    if (!A || !B || !C) return QG_ERR_INVALID_ARG;
    if (bad_layouts(layout_a, layout_b)) return QG_ERR_UNSUPPORTED;
    if (K % 8) return QG_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldc < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 8 || ldb % 8)
        return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0) return QG_ERR_CUDA;
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    return run_gemm_f16_tc(reinterpret_cast<const __half*>(A), lda, reinterpret_cast<const __half*>(B),
                           ldb, M, N, K, reinterpret_cast<__half*>(C), ldc, nullptr, ctl,
                           static_cast<cudaStream_t>(stream));
}

int qgemm_s8(int64_t M, int64_t N, int64_t K, const int8_t* A, int64_t lda, int layout_a,
             const int8_t* B, int64_t ldb, int layout_b, int32_t* C, int64_t ldc, void* ws,
             size_t ws_bytes, void* stream) {
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX) return QG_ERR_INVALID_ARG;
    if (!A || !B || !C) return QG_ERR_INVALID_ARG;
    if (bad_layouts(layout_a, layout_b)) return QG_ERR_UNSUPPORTED;
    if (K % 16 || K >= 131072) return QG_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldc < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 16 || ldb % 16)
        return QG_ERR_MISALIGNED;
    const size_t need = qg_workspace_size(QG_OP_S8, M, N, K);
    if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0) return QG_ERR_CUDA;
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    __half* A16 = static_cast<__half*>(ws);
    __half* B16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) +
                                            ((static_cast<size_t>(M) * K * 2 + 255) & ~size_t(255)));
    k_s8_to_f16<<<conv_grid(dev, M * K / 16), 256, 0, s>>>(A, M, K, lda, A16, K);
    k_s8_to_f16<<<conv_grid(dev, N * K / 16), 256, 0, s>>>(B, N, K, ldb, B16, K);
    int rc = map_cuda(cudaGetLastError());
    if (rc) return rc;
    return launch_gemm<MmaKind::F16, Epi::S32>(A16, K * 2, B16, K * 2, M, N, K, C, ldc,
                                               g_s8_chunk_kb, nullptr, ctl, s);
}

int qgemm_s4(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda_bytes, int layout_a,
             const uint8_t* B, int64_t ldb_bytes, int layout_b, int32_t* C, int64_t ldc, void* ws,
             size_t ws_bytes, void* stream) {
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX) return QG_ERR_INVALID_ARG;
    if (!A || !B || !C) return QG_ERR_INVALID_ARG;
    if (bad_layouts(layout_a, layout_b)) return QG_ERR_UNSUPPORTED;
    if (K % 32 || K >= 262144) return QG_ERR_INVALID_ARG;
    if (lda_bytes < K / 2 || ldb_bytes < K / 2 || ldc < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda_bytes % 16 || ldb_bytes % 16)
        return QG_ERR_MISALIGNED;
    const size_t need = qg_workspace_size(QG_OP_S4, M, N, K);
    if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0) return QG_ERR_CUDA;
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    uint8_t* A8 = static_cast<uint8_t*>(ws);
    uint8_t* B8 = static_cast<uint8_t*>(ws) + ((static_cast<size_t>(M) * K + 255) & ~size_t(255));
    k_s4_to_e4m3<<<conv_grid(dev, M * K / 32), 256, 0, s>>>(A, M, K / 2, lda_bytes, A8, K);
    k_s4_to_e4m3<<<conv_grid(dev, N * K / 32), 256, 0, s>>>(B, N, K / 2, ldb_bytes, B8, K);
    int rc = map_cuda(cudaGetLastError());
    if (rc) return rc;
    // Partial sums are bounded by 64*K < 2^24: one accumulation unit per tile.
    return launch_gemm<MmaKind::F8F6F4, Epi::S32>(A8, K, B8, K, M, N, K, C, ldc, 0, nullptr, ctl, s);
}

}  // extern "C"

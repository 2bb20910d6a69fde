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
#include "tc_gemm2_s4raw.cuh"

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

// L2 policy mode of the tensor-core GEMM kernels (qg_set_l2_policy): 0 =
// evict-normal loads, 1 = A evict-last / B evict-first, 2 = as 1 plus
// streaming output stores.
static std::atomic<int> g_l2_mode{0};

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
    p.l2_mode = g_l2_mode.load();
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
    p.l2_mode = g_l2_mode.load();
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

// qgemm_s4 route (qg_set_s4_path): 0 = the in-kernel nibble conversion where
// it applies (CTA pairs, K <= 65536), 1 = always the conversion pre-pass.
static std::atomic<int> g_s4_path{0};

// INT4 GEMM straight from the packed operands (tc_gemm2_s4raw_kernel).
static int launch_s4raw(const uint8_t* A, int64_t lda_bytes, const uint8_t* B, int64_t ldb_bytes, int64_t M,
                        int64_t N, int64_t K, int32_t* C, int64_t ldc, const Ctl& ctl, cudaStream_t stream) {
    using Cfg = S4RawCfg;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
    static std::mutex mu;
    static bool attr_set[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(tc_gemm2_s4raw_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }
    // the packed operands, 64 bytes (one 128-wide K stage) x the CTA's 128 rows per box
    CUtensorMap ta, tb;
    int rc0 = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K / 2, M, lda_bytes, Cfg::RAW_ROW, Cfg::BM,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!rc0)
        rc0 = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K / 2, N, ldb_bytes, Cfg::RAW_ROW, Cfg::B_ROWS,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc0) return rc0;
    S4RawParams p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = static_cast<int>((K + Cfg::BK - 1) / Cfg::BK);
    p.C = C;
    p.ldc = ldc;
    p.ctl = ctl;
    const int64_t tiles = ((M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * ((N + Cfg::BN - 1) / Cfg::BN);
    const int64_t max_pairs = num_sms(dev) / 2;
    const int grid = 2 * static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
    void *pb = nullptr, *pa = nullptr;
    profile_events(&pb, &pa);
    if (pb && cudaEventRecord(static_cast<cudaEvent_t>(pb), stream) != cudaSuccess) return QG_ERR_CUDA;
    tc_gemm2_s4raw_kernel<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, p);
    int rc = map_cuda(cudaGetLastError());
    if (!rc && pa && cudaEventRecord(static_cast<cudaEvent_t>(pa), stream) != cudaSuccess) return QG_ERR_CUDA;
    return rc;
}

int run_gemm_f16_tc(const __half* A, int64_t lda, const __half* B, int64_t ldb, int64_t M, int64_t N,
                    int64_t K, __half* C, int64_t ldc, const __half* bias, const Ctl& ctl,
                    cudaStream_t stream) {
    return launch_gemm<MmaKind::F16, Epi::F16>(A, lda * 2, B, ldb * 2, M, N, K, C, ldc, 0, bias, ctl,
                                               stream);
}

// -------------------------------------------------------- operand converters
//
// Both converters expand 8 source bytes into 16 destination bytes (int8 ->
// fp16; two packed nibbles -> two e4m3 bytes), so one kernel shape serves
// both: a warp takes a 512-byte segment of a source row, lane l the 8-byte
// pieces at 8 l and 256 + 8 l, and writes their 16-byte results at 16 l and
// 512 + 16 l of the 1024-byte output segment, so every store instruction of
// the warp fills 512 contiguous bytes (a thread converting 16 contiguous
// source bytes would store two 16-byte halves 32 bytes apart, half-filling
// the sectors of each store: 86 us against 70 us for two 8192 x 8192 int8
// operands).  CTAs are strided over rows, blockIdx.z selects the operand (A
// and B in one launch).  Both are HBM-bound: 3 bytes of traffic per int8
// value, 1.5 per int4 value.

struct ExpandJob {
    const uint8_t* src;
    int64_t rows, lds;  // source row stride in bytes
    uint8_t* dst;
    int64_t ldd;        // destination row stride in bytes
};
struct ExpandJobs {
    ExpandJob job[2];
    int64_t chunks;     // 16-byte source chunks per row (same for every job)
};

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// int8 -> fp16, exact: the byte XOR 0x80 (offset binary, 0..255) placed under
// the fp16 exponent of 1024 is 1024 + b + 128; subtracting 1152 leaves b.
struct S8ToF16 {
    __device__ __forceinline__ uint4 operator()(const uint2& in) const {
        const __half2 c1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        const uint32_t w[2] = {in.x ^ 0x80808080u, in.y ^ 0x80808080u};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t lo = __byte_perm(w[q], 0x64646464u, 0x4140);  // bytes 0, 1
            const uint32_t hi = __byte_perm(w[q], 0x64646464u, 0x4342);  // bytes 2, 3
            __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), c1152);
            __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), c1152);
            o[2 * q] = *reinterpret_cast<uint32_t*>(&a);
            o[2 * q + 1] = *reinterpret_cast<uint32_t*>(&b);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

// Signed nibble (low nibble = even k) -> e4m3 byte, exact for -8..7.  Four
// nibbles (16 bits) are a prmt selector: with table P = e4m3(0..7) a
// selector n < 8 picks P[n], and n >= 8 (bit 3 = sign-replicate mode) gives
// 0x00 because every P entry is positive; with the selector's bit 3 flipped
// and table Q[i] = e4m3(8 - i), the magnitude of n - 16 = -(8 - (n & 7)),
// n >= 8 picks Q[n & 7] and n < 8 gives 0x00.  The sign bit is set on the
// nonzero bytes of the second lookup (all Q entries are nonzero and below
// 0x80, so the per-byte add cannot carry).  The tables come from the
// hardware float -> e4m3 conversion.
struct S4ToE4M3 {
    uint32_t p_lo, p_hi, q_lo, q_hi;
    __device__ __forceinline__ S4ToE4M3() {
        p_lo = p_hi = q_lo = q_hi = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t pc = static_cast<uint8_t>(__nv_cvt_float_to_fp8(static_cast<float>(i), __NV_SATFINITE, __NV_E4M3));
            const uint32_t qc = static_cast<uint8_t>(__nv_cvt_float_to_fp8(static_cast<float>(8 - i), __NV_SATFINITE, __NV_E4M3));
            if (i < 4) {
                p_lo |= pc << (8 * i);
                q_lo |= qc << (8 * i);
            } else {
                p_hi |= pc << (8 * (i - 4));
                q_hi |= qc << (8 * (i - 4));
            }
        }
    }
    // prmt in its default mode: bit 3 of a selector nibble replicates the
    // selected byte's sign (the __byte_perm intrinsic ignores that bit).
    __device__ __forceinline__ static uint32_t prmt_sign(uint32_t a, uint32_t b, uint32_t sel) {
        uint32_t d;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
        return d;
    }
    __device__ __forceinline__ uint32_t four(uint32_t sel) const {
        const uint32_t pos = prmt_sign(p_lo, p_hi, sel);
        const uint32_t mag = prmt_sign(q_lo, q_hi, sel ^ 0x8888u);
        const uint32_t sign = (mag + 0x7F7F7F7Fu) & 0x80808080u;
        return pos | mag | sign;
    }
    __device__ __forceinline__ uint4 operator()(const uint2& in) const {
        return make_uint4(four(in.x & 0xFFFFu), four(in.x >> 16), four(in.y & 0xFFFFu), four(in.y >> 16));
    }
};

template <class Conv>
__global__ void __launch_bounds__(256) k_expand(const ExpandJobs jobs) {
    const ExpandJob jb = blockIdx.z == 0 ? jobs.job[0] : jobs.job[1];  // no dynamic index into parameters
    const Conv conv;
    const int lane = threadIdx.x & 31;
    const int64_t row_bytes = 16 * jobs.chunks;
    const int64_t soff = (blockIdx.x * 8 + (threadIdx.x >> 5)) * 512 + 8 * lane;
    if (soff >= row_bytes) return;
    // the last segment of a row may be partial: each 8-byte piece is whole
    // (row_bytes is a multiple of 16) and either inside the row or not
    const bool second = soff + 256 < row_bytes;
    const int64_t doff = 2 * soff;
    // four rows per pass, loads first: 64 bytes in flight per thread
    constexpr int U = 4;
    const int64_t step = gridDim.y;
    int64_t r = blockIdx.y;
    for (; r + (U - 1) * step < jb.rows; r += U * step) {
        uint2 v[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint8_t* p = jb.src + (r + u * step) * jb.lds + soff;
            v[u][0] = ld_stream8(p);
            v[u][1] = second ? ld_stream8(p + 256) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint8_t* d = jb.dst + (r + u * step) * jb.ldd + doff;
            *reinterpret_cast<uint4*>(d) = conv(v[u][0]);
            if (second) *reinterpret_cast<uint4*>(d + 512) = conv(v[u][1]);
        }
    }
    for (; r < jb.rows; r += step) {
        const uint8_t* p = jb.src + r * jb.lds + soff;
        uint8_t* d = jb.dst + r * jb.ldd + doff;
        *reinterpret_cast<uint4*>(d) = conv(ld_stream8(p));
        if (second) *reinterpret_cast<uint4*>(d + 512) = conv(ld_stream8(p + 256));
    }
}

// Launches k_expand over one or two operands with the same chunk count: 8
// warps (eight 512-byte source segments) per CTA along a row, up to 16 CTAs
// per SM in all (two waves of 8; measured 3% faster than one wave at two
// 8192 x 8192 int8 operands).
template <class Conv>
static int launch_expand(const ExpandJob* jobs, int njobs, int64_t chunks, int dev, cudaStream_t s) {
    ExpandJobs js;
    js.job[0] = jobs[0];
    js.job[1] = njobs > 1 ? jobs[1] : jobs[0];
    js.chunks = chunks;
    int64_t rows = jobs[0].rows;
    if (njobs > 1 && jobs[1].rows > rows) rows = jobs[1].rows;
    const int64_t segs = (chunks + 31) / 32;  // 512-byte source segments per row
    const int64_t gx = (segs + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms(dev)) * 16 / njobs;
    int64_t gy = cap / gx;
    if (gy > rows) gy = rows;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    if (gx > 2147483647) return QG_ERR_INVALID_ARG;
    k_expand<Conv><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(njobs)), 256,
                     0, s>>>(js);
    return map_cuda(cudaGetLastError());
}

int s8_to_f16_rows(const int8_t* src, int64_t rows, int64_t lds, __half* dst, int64_t K, int dev,
                   cudaStream_t s) {
    const ExpandJob job = {reinterpret_cast<const uint8_t*>(src), rows, lds, reinterpret_cast<uint8_t*>(dst),
                           K * 2};
    return launch_expand<S8ToF16>(&job, 1, K / 16, dev, s);
}

int s4_to_e4m3_pair(const uint8_t* a, int64_t a_rows, int64_t a_lds, uint8_t* a_dst, const uint8_t* b,
                    int64_t b_rows, int64_t b_lds, uint8_t* b_dst, int64_t K, int dev, cudaStream_t s) {
    const ExpandJob jobs[2] = {{a, a_rows, a_lds, a_dst, K}, {b, b_rows, b_lds, b_dst, K}};
    return launch_expand<S4ToE4M3>(jobs, 2, K / 32, dev, s);
}

int s4_to_e4m3_rows(const uint8_t* src, int64_t rows, int64_t lds, uint8_t* dst, int64_t K, int dev,
                    cudaStream_t s) {
    const ExpandJob job = {src, rows, lds, dst, K};
    return launch_expand<S4ToE4M3>(&job, 1, K / 32, dev, s);
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
static std::atomic<int> g_s8_chunk_kb{16};  // qg_set_s8_chunk; read once per call

int run_gemm_s8_converted(const __half* A16, const __half* B16, int64_t M, int64_t N, int64_t K, int32_t* C,
                          int64_t ldc, const Ctl& ctl, cudaStream_t stream) {
    return launch_gemm<MmaKind::F16, Epi::S32>(A16, K * 2, B16, K * 2, M, N, K, C, ldc, g_s8_chunk_kb.load(), nullptr,
                                               ctl, stream);
}

// Resource budgets of the instances launched above.
#define QG_TC_BUDGET(CFG, NAME, CLUSTER)                                                      \
    QG_KERNEL_BUDGET(NAME, reinterpret_cast<const void*>(CFG), CFG##_Cfg::THREADS,              \
                     CFG##_Cfg::SMEM_BYTES, CFG##_Cfg::TMEM_COLS, CLUSTER, 1)
using TcS8_Cfg = TcGemmCfg<MmaKind::F16, Epi::S32>;
using TcS4_Cfg = TcGemmCfg<MmaKind::F8F6F4, Epi::S32>;
using TcF16_Cfg = TcGemmCfg<MmaKind::F16, Epi::F16>;
using Tc2S8_Cfg = Tc2Cfg<MmaKind::F16, Epi::S32>;
using Tc2S4_Cfg = Tc2Cfg<MmaKind::F8F6F4, Epi::S32>;
using Tc2F16_Cfg = Tc2Cfg<MmaKind::F16, Epi::F16>;
static constexpr auto TcS8 = tc_gemm_kernel<TcS8_Cfg>;
static constexpr auto TcS4 = tc_gemm_kernel<TcS4_Cfg>;
static constexpr auto TcF16 = tc_gemm_kernel<TcF16_Cfg>;
static constexpr auto Tc2S8 = tc_gemm2_kernel<Tc2S8_Cfg>;
static constexpr auto Tc2S4 = tc_gemm2_kernel<Tc2S4_Cfg>;
static constexpr auto Tc2F16 = tc_gemm2_kernel<Tc2F16_Cfg>;
QG_TC_BUDGET(TcS8, "tc_gemm_kernel<F16,S32>", 1);
QG_TC_BUDGET(TcS4, "tc_gemm_kernel<F8F6F4,S32>", 1);
QG_TC_BUDGET(TcF16, "tc_gemm_kernel<F16,F16>", 1);
QG_TC_BUDGET(Tc2S8, "tc_gemm2_kernel<F16,S32>", 2);
QG_TC_BUDGET(Tc2S4, "tc_gemm2_kernel<F8F6F4,S32>", 2);
QG_TC_BUDGET(Tc2F16, "tc_gemm2_kernel<F16,F16>", 2);
#undef QG_TC_BUDGET
QG_KERNEL_BUDGET("tc_gemm2_s4raw_kernel", reinterpret_cast<const void*>(tc_gemm2_s4raw_kernel), S4RawCfg::THREADS,
                 S4RawCfg::SMEM_BYTES, S4RawCfg::TMEM_COLS, 2, 1);
QG_KERNEL_BUDGET("k_expand<S8ToF16>", reinterpret_cast<const void*>(k_expand<S8ToF16>), 256, 0, 0, 1, 1);
QG_KERNEL_BUDGET("k_expand<S4ToE4M3>", reinterpret_cast<const void*>(k_expand<S4ToE4M3>), 256, 0, 0, 1, 1);

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

int qg_set_s4_path(int path) {
    if (path < 0 || path > 1) return QG_ERR_INVALID_ARG;
    g_s4_path.store(path);
    return QG_OK;
}

int qg_set_l2_policy(int mode) {
    if (mode < 0 || mode > 2) return QG_ERR_INVALID_ARG;
    g_l2_mode.store(mode);
    return QG_OK;
}

int qg_set_s8_chunk(int kblocks) {
    if (kblocks < 1 || kblocks > 16) return QG_ERR_INVALID_ARG;
    g_s8_chunk_kb.store(kblocks);
    return QG_OK;
}

int gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int layout_a,
             const uint16_t* B, int64_t ldb, int layout_b, uint16_t* C, int64_t ldc, void* stream) {
    const qg::NvtxRange nvtx_range("gemm_f16");
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
    const qg::NvtxRange nvtx_range("qgemm_s8");
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
    const ExpandJob jobs[2] = {{reinterpret_cast<const uint8_t*>(A), M, lda, reinterpret_cast<uint8_t*>(A16), K * 2},
                               {reinterpret_cast<const uint8_t*>(B), N, ldb, reinterpret_cast<uint8_t*>(B16), K * 2}};
    int rc = launch_expand<S8ToF16>(jobs, 2, K / 16, dev, s);
    if (rc) return rc;
    return launch_gemm<MmaKind::F16, Epi::S32>(A16, K * 2, B16, K * 2, M, N, K, C, ldc,
                                               g_s8_chunk_kb.load(), nullptr, ctl, s);
}

int qgemm_s4(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda_bytes, int layout_a,
             const uint8_t* B, int64_t ldb_bytes, int layout_b, int32_t* C, int64_t ldc, void* ws,
             size_t ws_bytes, void* stream) {
    const qg::NvtxRange nvtx_range("qgemm_s4");
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

    // the in-kernel conversion saves a launch and a pass over the operands,
    // but its transform warps (shared-memory reads, conversion, generic
    // stores, the stage hand-off) pace its K loop at about 1.7x the MMA time
    // of a stage: 2.13 against 3.67 POPS at 8192^3, so large problems keep
    // the TMA-fed kernel behind the pre-pass
    if (g_s4_path.load() == 0 && use_pairs(M, N) && K <= S4RawCfg::MAX_K && M * N * K <= (int64_t(1) << 34))
        return launch_s4raw(A, lda_bytes, B, ldb_bytes, M, N, K, C, ldc, ctl, s);
    uint8_t* A8 = static_cast<uint8_t*>(ws);
    uint8_t* B8 = static_cast<uint8_t*>(ws) + ((static_cast<size_t>(M) * K + 255) & ~size_t(255));
    const ExpandJob jobs[2] = {{A, M, lda_bytes, A8, K}, {B, N, ldb_bytes, B8, K}};
    int rc = launch_expand<S4ToE4M3>(jobs, 2, K / 32, dev, s);
    if (rc) return rc;
    // Partial sums are bounded by 64*K < 2^24: one accumulation unit per tile.
    return launch_gemm<MmaKind::F8F6F4, Epi::S32>(A8, K, B8, K, M, N, K, C, ldc, 0, nullptr, ctl, s);
}

}  // extern "C"

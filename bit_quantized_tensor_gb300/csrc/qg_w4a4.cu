// W4A4 with a low-rank residual:  Y = (Q(X) . Q(W)^T) (.) scale + L(X) + b
// ("Warp-Specialized Kernel Implementation for W4A4 MatMul on Latest GPU
// Architectures", section 1).
//
// w4a4_quantize  one pass over X (fp32): per row and 64-element K block the
//                symmetric absmax quantizer (bit-exact IEEE binary32 steps),
//                fused with the low-rank down-projection XU = X . U.
// w4a4_gemm      the block-scaled GEMM of w4a4_gemm.cuh: exact integer block
//                partials on the tensor cores, both block scales applied in
//                fp32 by the epilogue, the low-rank term as one extra MMA
//                unit, the bias before the fp16 store.  A short pre-pass
//                turns the packed operands into e4m3 bytes and the scales
//                into transposed fp32 tables (one row per K block plus a
//                constant-1 row for the low-rank unit).
#include <cuda_fp16.h>

#include <mutex>

#include "qg_gemm_host.h"
#include "w4a4_gemm.cuh"

namespace qg {

constexpr int kW4A4Block = 64;
constexpr int kW4A4MaxRank = 32;

// ------------------------------------------------ quantizer (+ X . U)
//
// CTA: 128 threads, 16 rows.  Thread (row r = tid/8, segment j = tid%8)
// owns K positions [64*b + 8j, 64*b + 8j + 8) of every block b of its row:
// it quantizes them (absmax shared by the 8 segment lanes of the row through
// shuffles) and accumulates their contribution to all `rank` columns of XU;
// the 8 segment partial sums are added at the end.  U is staged per block in
// shared memory as fp32, double buffered, with its 16-byte chunks rotated by
// the segment index so the 8 lanes of a row read distinct banks.
constexpr int kQRows = 16;
constexpr int kQThreads = 128;

__device__ __forceinline__ int u_swz(int k, int r) {  // rank r of K row k, rotated
    return k * kW4A4MaxRank + ((r + 4 * (k >> 3)) & (kW4A4MaxRank - 1));
}

__global__ void __launch_bounds__(kQThreads)
    k_w4a4_quantize(int M, int K, const float* __restrict__ X, int64_t ldx,
                    const __half* __restrict__ U, int rank, uint8_t* __restrict__ Xq,
                    __half* __restrict__ Xs, __half* __restrict__ XU) {
    __shared__ __align__(16) float us[2][kW4A4Block * kW4A4MaxRank];
    const int tid = threadIdx.x;
    const int r = tid >> 3;                 // row within the CTA
    const int seg = tid & 7;                // 8-element segment within a block
    const int row = blockIdx.x * kQRows + r;
    const bool live = row < M;
    const int nblk = K / kW4A4Block;
    const bool lowrank = rank > 0;

    float acc[kW4A4MaxRank];
#pragma unroll
    for (int i = 0; i < kW4A4MaxRank; ++i) acc[i] = 0.f;

    auto stage_u = [&](int b, int buf) {
        // 64 x 32 fp16 = 256 chunks of 8 halves; 2 chunks per thread.
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int chunk = tid * 2 + c;
            const int k = chunk >> 2;
            const int r0 = (chunk & 3) * 8;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                U + static_cast<int64_t>(b * kW4A4Block + k) * kW4A4MaxRank + r0));
            const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(h[q]);
                us[buf][u_swz(k, r0 + 2 * q)] = f.x;
                us[buf][u_swz(k, r0 + 2 * q + 1)] = f.y;
            }
        }
    };

    if (lowrank) stage_u(0, 0);
    for (int b = 0; b < nblk; ++b) {
        const int buf = b & 1;
        float x[8];
        if (live) {
            const float4* src =
                reinterpret_cast<const float4*>(X + static_cast<int64_t>(row) * ldx + b * kW4A4Block +
                                                seg * 8);
            const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
            x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
            x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = 0.f;
        }
        // Absmax over the 64-element block (8 lanes x 8 values).
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        const __half sh = __float2half_rn(__fdiv_rn(a, 7.0f));
        const float s = __half2float(sh);
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = 0;
            if (s != 0.f) {
                float t = rintf(__fdiv_rn(x[i], s));
                t = fminf(fmaxf(t, -8.f), 7.f);
                q = static_cast<int>(t);
            }
            packed |= (static_cast<uint32_t>(q) & 0xFu) << (4 * i);
        }
        if (live) {
            *reinterpret_cast<uint32_t*>(Xq + static_cast<int64_t>(row) * (K / 2) + b * 32 + seg * 4) =
                packed;
            if (seg == 0) Xs[static_cast<int64_t>(row) * nblk + b] = sh;
        }
        if (lowrank) {
            __syncthreads();                              // us[buf] complete
            if (b + 1 < nblk) stage_u(b + 1, buf ^ 1);    // overlaps the FMAs below
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = seg * 8 + i;
                const float* urow = &us[buf][k * kW4A4MaxRank];
                const int rot = 4 * (k >> 3);
#pragma unroll
                for (int c = 0; c < kW4A4MaxRank; c += 4) {
                    const float4 u = *reinterpret_cast<const float4*>(urow + ((c + rot) & 31));
                    acc[c] = fmaf(x[i], u.x, acc[c]);
                    acc[c + 1] = fmaf(x[i], u.y, acc[c + 1]);
                    acc[c + 2] = fmaf(x[i], u.z, acc[c + 2]);
                    acc[c + 3] = fmaf(x[i], u.w, acc[c + 3]);
                }
            }
            __syncthreads();                              // us[buf] may be overwritten
        }
    }
    if (lowrank) {
#pragma unroll
        for (int i = 0; i < kW4A4MaxRank; ++i) {
            acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
            acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 2);
            acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 4);
        }
        if (live) {
            // Lane `seg` writes ranks 4*seg .. 4*seg+3.
            float o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float v = 0.f;
#pragma unroll
                for (int c = 0; c < kW4A4MaxRank; ++c)
                    if (c == 4 * seg + q) v = acc[c];
                o[q] = v;
            }
            __half2 h0 = __floats2half2_rn(o[0], o[1]);
            __half2 h1 = __floats2half2_rn(o[2], o[3]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&h0);
            pk.y = *reinterpret_cast<uint32_t*>(&h1);
            *reinterpret_cast<uint2*>(XU + static_cast<int64_t>(row) * kW4A4MaxRank + 4 * seg) = pk;
        }
    }
}

// ------------------------------------------------ GEMM pre-pass

// St[j][r] = S[r][j] (fp16 -> fp32) for j < nblk; St[nblk][r] = 1; columns
// r in [rows, rows_p) are 0.  S: rows x nblk, St: (nblk + 1) x rows_p.
__global__ void k_scales_transposed(int64_t rows, int64_t rows_p, int nblk,
                                    const __half* __restrict__ S, float* __restrict__ St) {
    const int64_t total = static_cast<int64_t>(nblk + 1) * rows_p;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = i / rows_p;
        const int64_t r = i - j * rows_p;
        float v = 0.f;
        if (r < rows) v = (j == nblk) ? 1.f : __half2float(S[r * nblk + j]);
        St[i] = v;
    }
}

// Vt[n][j] = V[j][n];  V: rank x N, Vt: N x rank.
__global__ void k_transpose_v(int N, int rank, const __half* __restrict__ V, __half* __restrict__ Vt) {
    const int64_t total = static_cast<int64_t>(N) * rank;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / rank;
        const int j = static_cast<int>(i - n * rank);
        Vt[i] = V[static_cast<int64_t>(j) * N + n];
    }
}

}  // namespace qg

using namespace qg;

extern "C" {

int w4a4_quantize(int64_t M, int64_t K, const float* X, int64_t ldx, const uint16_t* U, int64_t rank,
                  uint8_t* Xq, uint16_t* Xscale, uint16_t* XU, int64_t block, void* stream) {
    if (M < 1 || K < 1 || M > INT32_MAX || K > INT32_MAX) return QG_ERR_INVALID_ARG;
    if (block != kW4A4Block) return QG_ERR_UNSUPPORTED;
    if (K % kW4A4Block) return QG_ERR_INVALID_ARG;
    if (rank != 0 && rank != kW4A4MaxRank) return QG_ERR_UNSUPPORTED;
    if (!X || !Xq || !Xscale || (rank && (!U || !XU))) return QG_ERR_INVALID_ARG;
    if (ldx < K) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || ldx % 4 || !aligned16(Xq) || !aligned16(Xscale) ||
        (rank && (!aligned16(U) || !aligned16(XU))))
        return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0) return QG_ERR_CUDA;
    const int grid = static_cast<int>((M + kQRows - 1) / kQRows);
    k_w4a4_quantize<<<grid, kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<int>(M), static_cast<int>(K), X, ldx, reinterpret_cast<const __half*>(U),
        static_cast<int>(rank), Xq, reinterpret_cast<__half*>(Xscale), reinterpret_cast<__half*>(XU));
    return map_cuda(cudaGetLastError());
}

int w4a4_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* Xq, const uint16_t* Xscale,
              const uint8_t* Wq, const uint16_t* Wscale, int64_t block, const uint16_t* XU,
              const uint16_t* V, int64_t rank, const uint16_t* bias, uint16_t* Y, int64_t ldy,
              void* ws, size_t ws_bytes, void* stream) {
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return QG_ERR_INVALID_ARG;
    if (block != kW4A4Block) return QG_ERR_UNSUPPORTED;
    if (K % kW4A4Block) return QG_ERR_INVALID_ARG;
    if (rank != 0 && rank != kW4A4MaxRank) return QG_ERR_UNSUPPORTED;
    if (!Xq || !Xscale || !Wq || !Wscale || !Y || (rank && (!XU || !V))) return QG_ERR_INVALID_ARG;
    if (ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(Y) || (rank && !aligned16(XU)))
        return QG_ERR_MISALIGNED;
    const size_t need = qg_workspace_size(QG_OP_W4A4, M, N, K);
    if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    const int nblk = static_cast<int>(K / kW4A4Block);
    const int64_t Mp = (M + 3) & ~int64_t(3), Np = (N + 3) & ~int64_t(3);
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t* A8 = base;
    uint8_t* B8 = A8 + up(static_cast<size_t>(M) * K);
    float* SXt = reinterpret_cast<float*>(B8 + up(static_cast<size_t>(N) * K));
    float* SWt = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(SXt) +
                                          up(4ull * (nblk + 1) * Mp));
    __half* Vt = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(SWt) +
                                           up(4ull * (nblk + 1) * Np));

    int rc = s4_to_e4m3(Xq, M, K, K / 2, A8, K, dev, s);
    if (!rc) rc = s4_to_e4m3(Wq, N, K, K / 2, B8, K, dev, s);
    if (rc) return rc;
    k_scales_transposed<<<conv_grid(dev, (nblk + 1) * Mp), 256, 0, s>>>(
        M, Mp, nblk, reinterpret_cast<const __half*>(Xscale), SXt);
    k_scales_transposed<<<conv_grid(dev, (nblk + 1) * Np), 256, 0, s>>>(
        N, Np, nblk, reinterpret_cast<const __half*>(Wscale), SWt);
    if (rank)
        k_transpose_v<<<conv_grid(dev, N * rank), 256, 0, s>>>(
            static_cast<int>(N), static_cast<int>(rank), reinterpret_cast<const __half*>(V), Vt);
    rc = map_cuda(cudaGetLastError());
    if (rc) return rc;

    using Cfg = W4A4Cfg;
    CUtensorMap tA, tB, tXU, tVt, tSX, tSW;
    rc = make_tmap_kmajor(&tA, false, A8, K, M, K, Cfg::BK, Cfg::BM);
    if (!rc) rc = make_tmap_kmajor(&tB, false, B8, K, N, K, Cfg::BK, Cfg::BN);
    if (!rc) rc = make_tmap_2d(&tSX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SXt, Mp, nblk + 1, Mp * 4,
                               Cfg::BM, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!rc) rc = make_tmap_2d(&tSW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SWt, Np, nblk + 1, Np * 4,
                               Cfg::BN, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rank) {
        // 32 low-rank columns in a 64-wide (128-byte) box: TMA zero-fills the rest
        if (!rc) rc = make_tmap_kmajor(&tXU, true, XU, rank, M, rank * 2, 64, Cfg::BM);
        if (!rc) rc = make_tmap_kmajor(&tVt, true, Vt, rank, N, rank * 2, 64, Cfg::BN);
    } else {
        tXU = tA;  // never read without the low-rank unit
        tVt = tB;
    }
    if (rc) return rc;

    static std::mutex mu;
    static bool attr_set[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(
                w4a4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }
    W4A4Params p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_ks = static_cast<int>((K + Cfg::BK - 1) / Cfg::BK);
    p.nblk = nblk;
    p.lowrank = rank ? 1 : 0;
    p.Y = reinterpret_cast<__half*>(Y);
    p.ldy = ldy;
    p.bias = reinterpret_cast<const __half*>(bias);
    p.ctl = ctl;
    const int64_t tiles = ((M + Cfg::BM - 1) / Cfg::BM) * ((N + Cfg::BN - 1) / Cfg::BN);
    const int grid = static_cast<int>(tiles < num_sms(dev) ? tiles : num_sms(dev));
    void *pb = nullptr, *pa = nullptr;
    profile_events(&pb, &pa);
    if (pb && cudaEventRecord(static_cast<cudaEvent_t>(pb), s) != cudaSuccess) return QG_ERR_CUDA;
    w4a4_gemm_kernel<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, s>>>(tA, tB, tXU, tVt, tSX, tSW, p);
    rc = map_cuda(cudaGetLastError());
    if (!rc && pa && cudaEventRecord(static_cast<cudaEvent_t>(pa), s) != cudaSuccess)
        return QG_ERR_CUDA;
    return rc;
}

}  // extern "C"

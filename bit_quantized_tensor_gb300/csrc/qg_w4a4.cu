// W4A4 with a low-rank residual:  Y = (Q(X) . Q(W)^T) (.) scale + L(X) + b
// ("Warp-Specialized Kernel Implementation for W4A4 MatMul on Latest GPU
// Architectures", section 1).
//
// w4a4_quantize  one pass over X (fp32): per row and 64-element K block the
//                symmetric absmax quantizer (bit-exact IEEE binary32 steps),
//                fused with the low-rank down-projection XU = X . U.
// w4a4_gemm      folds each block scale into its 4-bit values (fp16 q*s, one
//                rounding), appends the low-rank factors as `rank` extra K
//                columns ([q*sX | XU] against [q*sW | V^T]), and runs the
//                tcgen05 fp16 GEMM whose epilogue adds the bias per column.
//                The block-wise scale therefore acts inside the K sum, block
//                by block, as the scaled product requires.
#include <cuda_fp16.h>

#include "qg_gemm_host.h"

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

// ------------------------------------------------ scale folding
//
// Dst[row][k] = fp16(q[row][k] * s[row][k / 64]) for k < K: the integer
// times the fp16 scale is exact in fp32 and rounds once to fp16.  16 values
// per thread (8 packed bytes, inside one block).
__global__ void k_w4a4_fold(int64_t rows, int K, const uint8_t* __restrict__ Q,
                            const __half* __restrict__ S, __half* __restrict__ Dst, int64_t ldd) {
    const int per_row = K / 16;
    const int64_t total = rows * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / per_row;
        const int c = static_cast<int>(i - r * per_row) * 16;
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(Q + r * (K / 2) + c / 2));
        const float s = __half2float(S[r * (K / kW4A4Block) + c / kW4A4Block]);
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t word = j < 4 ? w.x : w.y;
            const int sh = 8 * (j & 3);
            const int lo = static_cast<int>((word >> sh) & 0xFu);
            const int hi = static_cast<int>((word >> (sh + 4)) & 0xFu);
            const float vlo = static_cast<float>(lo < 8 ? lo : lo - 16) * s;
            const float vhi = static_cast<float>(hi < 8 ? hi : hi - 16) * s;
            __half2 h = __floats2half2_rn(vlo, vhi);
            out[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        uint4* d = reinterpret_cast<uint4*>(Dst + r * ldd + c);
        d[0] = make_uint4(out[0], out[1], out[2], out[3]);
        d[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
}

// Low-rank columns: A'[m][K + j] = XU[m][j] and B'[n][K + j] = V[j][n].
__global__ void k_w4a4_lowrank_cols(int M, int N, int K, int rank, const __half* __restrict__ XU,
                                    const __half* __restrict__ V, __half* __restrict__ A,
                                    __half* __restrict__ B, int64_t ld) {
    const int64_t totalA = static_cast<int64_t>(M) * rank;
    const int64_t total = totalA + static_cast<int64_t>(N) * rank;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (i < totalA) {
            const int64_t m = i / rank;
            const int j = static_cast<int>(i - m * rank);
            A[m * ld + K + j] = XU[m * rank + j];
        } else {
            const int64_t e = i - totalA;
            const int64_t n = e / rank;
            const int j = static_cast<int>(e - n * rank);
            B[n * ld + K + j] = V[static_cast<int64_t>(j) * N + n];
        }
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
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX - 64)
        return QG_ERR_INVALID_ARG;
    if (block != kW4A4Block) return QG_ERR_UNSUPPORTED;
    if (K % kW4A4Block) return QG_ERR_INVALID_ARG;
    if (rank != 0 && rank != kW4A4MaxRank) return QG_ERR_UNSUPPORTED;
    if (!Xq || !Xscale || !Wq || !Wscale || !Y || (rank && (!XU || !V))) return QG_ERR_INVALID_ARG;
    if (ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(Y)) return QG_ERR_MISALIGNED;
    const size_t need = qg_workspace_size(QG_OP_W4A4, M, N, K);
    if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0) return QG_ERR_CUDA;
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int64_t ke = K + rank;  // multiple of 32 halves: 16-byte aligned rows
    __half* A16 = static_cast<__half*>(ws);
    __half* B16 = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) +
                                            ((static_cast<size_t>(M) * ke * 2 + 255) & ~size_t(255)));
    k_w4a4_fold<<<conv_grid(dev, M * K / 16), 256, 0, s>>>(M, static_cast<int>(K), Xq,
                                                           reinterpret_cast<const __half*>(Xscale),
                                                           A16, ke);
    k_w4a4_fold<<<conv_grid(dev, N * K / 16), 256, 0, s>>>(N, static_cast<int>(K), Wq,
                                                           reinterpret_cast<const __half*>(Wscale),
                                                           B16, ke);
    if (rank)
        k_w4a4_lowrank_cols<<<conv_grid(dev, (M + N) * rank), 256, 0, s>>>(
            static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), static_cast<int>(rank),
            reinterpret_cast<const __half*>(XU), reinterpret_cast<const __half*>(V), A16, B16, ke);
    int rc = map_cuda(cudaGetLastError());
    if (rc) return rc;
    return run_gemm_f16_tc(A16, ke, B16, ke, M, N, ke, reinterpret_cast<__half*>(Y), ldy,
                           reinterpret_cast<const __half*>(bias), ctl, s);
}

}  // extern "C"

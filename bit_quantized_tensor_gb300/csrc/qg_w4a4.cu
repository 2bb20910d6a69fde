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

#include <atomic>
#include <mutex>

#include "qg_gemm_host.h"
#include "tc_gemm2.cuh"
#include "w4a4_gemm.cuh"
#include "w4a4_gemm2.cuh"

namespace qg {

// Which paired W4A4 kernel runs (qg_set_w4a4_pair_form): 0 the default
// (256 x 256 tiles), 1 256 x 192 tiles.
static std::atomic<int> g_w4a4_pair_form{0};
static int w4a4_pair_form() { return g_w4a4_pair_form.load(); }

constexpr int kW4A4Block = 64;
constexpr int kW4A4MaxRank = 32;

// ------------------------------------------------ quantizer (+ X . U)
//
// CTA: 8 warps on one 16-row tile of X, warp w on K slice w (a contiguous
// range of 64-element blocks).  Each warp streams its blocks through a
// private kQStages-deep ring in shared memory: lane 0 loads a block as two
// TMA boxes of 16 rows x 32 floats (128-byte rows, 128-byte swizzle) and the
// warp waits on the stage's mbarrier.  Lane (g, t) owns rows g and g + 8 at
// the 16 positions [16t, 16t + 16) of every block, read as four 16-byte
// chunks; lanes t = 2, 3 take their chunks in the order 2, 3, 0, 1, which
// together with the swizzle puts the eight lanes of every shared-memory
// phase on distinct banks.  x[4i + j] is position 16t + 4 (i ^ 2 (t / 2)) + j.
// Per row and block: absmax through two shuffles, s = fp16(max / 7), codes
// q = clamp(rint(fl(x / s)), -8, 7) (codes_fast, codes_exact), the lane's 8
// code bytes stored at once.
// X . U on mma.sync m16n8k16 (X rounded to fp16, fp32 accumulation): in step
// i the lane's chunk i is its A fragment (k slots 2t, 2t+1 <- its first two
// values, 2t+8, 2t+9 <- the other two) and the B fragment holds U at the same
// four positions, read from U stored rank x K (row 8n + g) with two 16-byte
// loads per n-tile.  The eight slices' partial X . U tiles are added through
// shared memory at the end.
constexpr int kQWarps = 8;
constexpr int kQThreads = 32 * kQWarps;
constexpr int kQStages = 3;
constexpr int kQStageBytes = 16 * kW4A4Block * 4;                        // 4 KiB: 16 rows x 64 fp32
constexpr int kQSmemBytes = kQWarps * kQStages * kQStageBytes + 1024;    // + alignment slack

__device__ __forceinline__ void mma_16816_q(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Codes of one lane-row: four 16-bit groups, group i holding the codes of the
// lane's chunk i (x[4i + j] in nibble j).  The definition is
// q = s == 0 ? 0 : clamp(rint(fl(x / s)), -8, 7) with s = fp16(max / 7).
//
// Exact slow form: the IEEE division itself.
__device__ __forceinline__ void codes_exact(const float (&x)[16], float s, uint32_t (&grp)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int q = 0;
            if (s != 0.f)
                q = static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(x[4 * c + j], s)), -8.f), 7.f));
            w |= (static_cast<uint32_t>(q) & 0xFu) << (4 * j);
        }
        grp[c] = w;
    }
}

// Fast form, y = fl(x * fl(1 / s)) instead of fl(x / s).  It is kept for a
// row only when s is a normal fp16 value and no y is within 2^-17 of a
// half-integer; then it gives the same codes:
//  - a normal s is within a factor (1 +- 2^-11) of max / 7, so |x / s| and
//    |y| stay below 7.004: rint never leaves [-7, 7] and the clamp is idle;
//  - |y - x / s| <= |x / s| (2^-24 + 2^-24 + 2^-48) < 2^-20 and
//    |fl(x / s) - x / s| <= 2^-22 below 8, so a y more than 2^-17 from every
//    half-integer has fl(x / s) on the same side of each of them;
//  - y + 1.5 * 2^23 rounds y to an integer with ties to even (the sum's ulp
//    is 1 and 1.5 * 2^23 is even), and the sum's four low mantissa bits are
//    that integer's two's-complement nibble;
//  - d = y - rint(y) is exact and |d| <= 1/2; "near a tie" is
//    |d| > 1/2 - 2^-17.
// Returns true when the row needs the exact form.
__device__ __forceinline__ bool codes_fast(const float (&x)[16], float r, uint32_t (&grp)[4]) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    constexpr float kNearTie = 0.5f - 0x1p-17f;
    // the same IEEE operations on pairs of values (f32x2), and the largest
    // |d| of the row compared once
    const uint64_t r2 = pack_f32x2(r, r), magic2 = pack_f32x2(kMagic, kMagic);
    float dmax = 0.f;
    uint32_t pair[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const uint64_t y = mul2(pack_f32x2(x[2 * p], x[2 * p + 1]), r2);
        const uint64_t tq = add2(y, magic2);
        const float2 d = unpack_f32x2(sub2(y, sub2(tq, magic2)));
        dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
        const float2 tf = unpack_f32x2(tq);
        // low nibble <- the pair's first value, high nibble <- its second
        pair[p] = (__float_as_uint(tf.x) & 0x0Fu) | ((__float_as_uint(tf.y) << 4) & 0xF0u);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) grp[c] = __byte_perm(pair[2 * c], pair[2 * c + 1], 0x0040);
    return dmax > kNearTie;
}

__device__ __forceinline__ float absmax16(const float (&x)[16]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(x[i]), fabsf(x[i + 8]));
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], m[i + 4]);
    return fmaxf(fmaxf(m[0], m[2]), fmaxf(m[1], m[3]));
}

// The lane's 8 code bytes in position order from its chunk groups (chunk
// order 0..3, or 2, 3, 0, 1 when `swapped`).
__device__ __forceinline__ uint2 code_bytes(const uint32_t (&grp)[4], bool swapped) {
    const uint32_t lo = __byte_perm(grp[0], grp[1], 0x5410);
    const uint32_t hi = __byte_perm(grp[2], grp[3], 0x5410);
    return swapped ? make_uint2(hi, lo) : make_uint2(lo, hi);
}

template <bool LOWRANK>
__global__ void __launch_bounds__(kQThreads, 2)
    k_w4a4_quantize(const __grid_constant__ CUtensorMap tmX, int M, int K,
                    const __half* __restrict__ Ut, uint8_t* __restrict__ Xq, __half* __restrict__ Xs,
                    __half* __restrict__ XU, const Ctl ctl) {
    extern __shared__ uint8_t qsmem_raw[];
    __shared__ __align__(8) uint64_t full[kQWarps][kQStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nblk = K / kW4A4Block;
    const int bpw = (nblk + kQWarps - 1) / kQWarps;
    const int bbeg = min(nblk, warp * bpw), bend = min(nblk, bbeg + bpw);
    const int tile_row = blockIdx.x * 16;
    const int row0 = tile_row + g, row1 = row0 + 8;
    const bool live0 = row0 < M, live1 = row1 < M;
    const bool swapped = t >= 2;  // chunk order 2, 3, 0, 1

    // 1024-byte aligned ring (the 128-byte swizzle repeats every 1024 bytes)
    const uint32_t ring_base =
        ((smem_u32(qsmem_raw) + 1023u) & ~1023u) + warp * (kQStages * kQStageBytes);
    uint8_t* const ring_gen = qsmem_raw + (ring_base - smem_u32(qsmem_raw));
    const uint32_t bar0 = smem_u32(&full[warp][0]);
    if (lane == 0) {
        for (int s = 0; s < kQStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int b, int st) {  // lane 0 only
        const uint32_t bar = bar0 + 8 * st;
        const uint32_t dst = ring_base + st * kQStageBytes;
        mbar_arrive_expect_tx(bar, kQStageBytes);
        tma_load_2d(dst, &tmX, b * kW4A4Block, tile_row, bar, pol);
        tma_load_2d(dst + kQStageBytes / 2, &tmX, b * kW4A4Block + 32, tile_row, bar, pol);
    };
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kQStages; ++i)
            if (bbeg + i < bend) issue(bbeg + i, i);
    }

    // shared-memory offsets of the lane's chunk i in rows g and g + 8
    uint32_t off[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ch = 4 * (t & 1) + (i ^ (swapped ? 2 : 0));  // chunk within the 128-byte half-row
        off[i] = (t >> 1) * (kQStageBytes / 2) + g * 128 + ((ch ^ g) << 4);
    }

    float acc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;

    int fail_b = -1;
    int stage = 0;
    uint32_t phase = 0;
    for (int b = bbeg; b < bend; ++b) {
        uint4 u[4][2];
        if constexpr (LOWRANK) {
            // piece h ^ swapped of the lane's 32 bytes of U row 8n + g
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    u[n][h] = __ldg(reinterpret_cast<const uint4*>(
                        Ut + static_cast<int64_t>(8 * n + g) * K + b * kW4A4Block + 16 * t +
                        8 * (h ^ (swapped ? 1 : 0))));
        }
        if (!__all_sync(0xffffffffu, bounded_wait(bar0 + 8 * stage, phase, nullptr, ctl, 20))) {
            fail_b = b;
            break;
        }
        float x0[16], x1[16];
        {
            const uint8_t* st = ring_gen + stage * kQStageBytes;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v0 = *reinterpret_cast<const float4*>(st + off[i]);
                const float4 v1 = *reinterpret_cast<const float4*>(st + off[i] + 8 * 128);
                x0[4 * i] = v0.x; x0[4 * i + 1] = v0.y; x0[4 * i + 2] = v0.z; x0[4 * i + 3] = v0.w;
                x1[4 * i] = v1.x; x1[4 * i + 1] = v1.y; x1[4 * i + 2] = v1.z; x1[4 * i + 3] = v1.w;
            }
        }
        // Per-row block absmax over the 4 lanes t of the row.
        float m0 = absmax16(x0), m1 = absmax16(x1);
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
        // Every lane has used its values of the stage (the absmax reads all of
        // them): only now may the TMA overwrite it.  Refilling right after the
        // loads, before their registers were used, raced in a ring built the
        // same way (a slot refilled before all of its loads had read it).
        __syncwarp();
        if (lane == 0 && b + kQStages < bend) issue(b + kQStages, stage);
        if (++stage == kQStages) {
            stage = 0;
            phase ^= 1u;
        }
        const __half h0 = __float2half_rn(__fdiv_rn(m0, 7.0f));
        const __half h1 = __float2half_rn(__fdiv_rn(m1, 7.0f));
        const float s0 = __half2float(h0), s1 = __half2float(h1);
        uint32_t q0[4], q1[4];
        const bool slow0 = codes_fast(x0, __frcp_rn(s0), q0) || !(s0 >= 0x1p-14f);
        const bool slow1 = codes_fast(x1, __frcp_rn(s1), q1) || !(s1 >= 0x1p-14f);
        if (__any_sync(0xffffffffu, slow0 || slow1)) {  // rare: near a tie, or a tiny block
            if (slow0) codes_exact(x0, s0, q0);
            if (slow1) codes_exact(x1, s1, q1);
        }
        if (live0) {
            *reinterpret_cast<uint2*>(Xq + static_cast<int64_t>(row0) * (K / 2) + b * 32 + 8 * t) =
                code_bytes(q0, swapped);
            if (t == 0) Xs[static_cast<int64_t>(row0) * nblk + b] = h0;
        }
        if (live1) {
            *reinterpret_cast<uint2*>(Xq + static_cast<int64_t>(row1) * (K / 2) + b * 32 + 8 * t) =
                code_bytes(q1, swapped);
            if (t == 0) Xs[static_cast<int64_t>(row1) * nblk + b] = h1;
        }
        if constexpr (LOWRANK) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t a0 = pack_f16x2(x0[4 * i], x0[4 * i + 1]);
                const uint32_t a1 = pack_f16x2(x1[4 * i], x1[4 * i + 1]);
                const uint32_t a2 = pack_f16x2(x0[4 * i + 2], x0[4 * i + 3]);
                const uint32_t a3 = pack_f16x2(x1[4 * i + 2], x1[4 * i + 3]);
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    const uint4& p = u[n][i >> 1];
                    mma_16816_q(acc[n], a0, a1, a2, a3, (i & 1) ? p.z : p.x, (i & 1) ? p.w : p.y);
                }
            }
        }
    }
    if (fail_b >= 0) {
        // A load did not arrive in time (recorded): wait, bounded, for the
        // loads still in flight, blocks [fail_b, fail_b + kQStages), before
        // the ring is reused or the CTA's shared memory is released.
        if (lane == 0)
            for (int bb = fail_b; bb < min(bend, fail_b + kQStages); ++bb)
                bounded_wait(bar0 + 8 * ((bb - bbeg) % kQStages), ((bb - bbeg) / kQStages) & 1, nullptr,
                             ctl, 21);
        __syncwarp();
    }
    if constexpr (LOWRANK) {
        // warp w's 16 x 32 partial into its own (drained) ring, then warp 0 sums
        float* red = reinterpret_cast<float*>(ring_gen);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[(4 * n + i) * 32 + lane] = acc[n][i];
        __syncthreads();
        if (warp == 0) {
            const float* red0 = reinterpret_cast<const float*>(ring_gen);
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kQWarps; ++w)
                        sum += red0[w * (kQStages * kQStageBytes / 4) + (4 * n + i) * 32 + lane];
                    v[i] = sum;
                }
                // C fragment: (row g, cols 2t, 2t+1) and (row g+8, same cols) of n-tile n
                const int col = 8 * n + 2 * t;
                if (live0)
                    *reinterpret_cast<uint32_t*>(XU + static_cast<int64_t>(row0) * kW4A4MaxRank + col) =
                        pack_f16x2(v[0], v[1]);
                if (live1)
                    *reinterpret_cast<uint32_t*>(XU + static_cast<int64_t>(row1) * kW4A4MaxRank + col) =
                        pack_f16x2(v[2], v[3]);
            }
        }
    }
}

// ------------------------------------------------ GEMM pre-pass

// St[j][r] = S[r][j] (fp16 -> fp32) for j < nblk; St[nblk][r] = 1; columns
// r in [rows, rows_p) are 0.  S: rows x nblk, St: (nblk + 1) x rows_p.
// With `alpha` (one fp16 multiplier per row of S, i.e. per output column of
// the GEMM) every entry of row r, the constant one included, is multiplied by
// alpha[r]: that applies the column-wise affine calibration's multiplier to
// both the block-scaled product and the low-rank unit.  An fp16 scale times
// an fp16 multiplier has at most 22 significant bits, so the fp32 product is
// exact.
__global__ void __launch_bounds__(256) k_scales_transposed(int64_t rows, int64_t rows_p, int nblk,
                                                          const __half* __restrict__ S,
                                                          const __half* __restrict__ alpha,
                                                          float* __restrict__ St) {
    // 32 x 32 tiles through shared memory: a warp reads 32 consecutive
    // blocks of one row and writes 32 consecutive rows of one block
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
    const int64_t rtiles = (rows_p + 31) / 32, jtiles = (nblk + 1 + 31) / 32;
    for (int64_t t = blockIdx.x; t < rtiles * jtiles; t += gridDim.x) {
        const int64_t r0 = (t % rtiles) * 32;
        const int64_t j0 = (t / rtiles) * 32;
        const int64_t j = j0 + tx;
        for (int rr = ty; rr < 32; rr += 8) {
            const int64_t r = r0 + rr;
            float v = 0.f;
            if (r < rows && j <= nblk) {
                v = (j == nblk) ? 1.f : __half2float(S[r * nblk + j]);
                if (alpha) v *= __half2float(alpha[r]);
            }
            tile[rr][tx] = v;
        }
        __syncthreads();
        const int64_t r = r0 + tx;
        for (int jj = ty; jj < 32; jj += 8)
            if (j0 + jj <= nblk && r < rows_p) St[(j0 + jj) * rows_p + r] = tile[tx][jj];
        __syncthreads();
    }
}

}  // namespace qg

namespace qg {

// Tensor maps and launch of one of the two W4A4 GEMM kernels (one CTA per
// 128 x 192 tile, or CTA pairs per 256 x 192 tile).
template <class Cfg, bool PAIR, auto KERNEL>
static int launch_w4a4(const uint8_t* A8, const uint8_t* B8, const float* SXt, const float* SWt,
                       const uint16_t* XU, const uint16_t* V, int64_t M, int64_t N, int64_t K,
                       int64_t Mp, int64_t Np, int64_t rank, const W4A4Params& p, int dev,
                       cudaStream_t s) {
    constexpr int B_ROWS = PAIR ? Cfg::BN / 2 : Cfg::BN;
    const int nblk = p.nblk;
    CUtensorMap tA, tB, tXU, tV, tSX, tSW;
    int rc = make_tmap_kmajor(&tA, false, A8, K, M, K, Cfg::BK, Cfg::BM);
    if (!rc) rc = make_tmap_kmajor(&tB, false, B8, K, N, K, Cfg::BK, B_ROWS);
    if (!rc) rc = make_tmap_2d(&tSX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SXt, Mp, nblk + 1, Mp * 4,
                               Cfg::BM, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!rc) rc = make_tmap_2d(&tSW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SWt, Np, nblk + 1, Np * 4,
                               Cfg::BN, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rank) {
        // 32 low-rank columns in a 64-wide (128-byte) box: TMA zero-fills the rest
        if (!rc) rc = make_tmap_kmajor(&tXU, true, XU, rank, M, rank * 2, 64, Cfg::BM);
        if (!rc) rc = make_tmap_kmajor(&tV, true, V, rank, N, rank * 2, 64, B_ROWS);
    } else {
        tXU = tA;  // never read without the low-rank unit
        tV = tB;
    }
    if (rc) return rc;

    auto kernel = KERNEL;
    static std::mutex mu;
    static bool attr_set[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(
                kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }
    int grid;
    if (PAIR) {
        const int64_t tiles = ((M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * ((N + Cfg::BN - 1) / Cfg::BN);
        const int64_t max_pairs = num_sms(dev) / 2;
        grid = 2 * static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
    } else {
        const int64_t tiles = ((M + Cfg::BM - 1) / Cfg::BM) * ((N + Cfg::BN - 1) / Cfg::BN);
        grid = static_cast<int>(tiles < num_sms(dev) ? tiles : num_sms(dev));
    }
    void *pb = nullptr, *pa = nullptr;
    profile_events(&pb, &pa);
    if (pb && cudaEventRecord(static_cast<cudaEvent_t>(pb), s) != cudaSuccess) return QG_ERR_CUDA;
    kernel<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, s>>>(tA, tB, tXU, tV, tSX, tSW, p);
    rc = map_cuda(cudaGetLastError());
    if (!rc && pa && cudaEventRecord(static_cast<cudaEvent_t>(pa), s) != cudaSuccess)
        return QG_ERR_CUDA;
    return rc;
}

// Resource budgets of the instances launched above.  The quantizer counts on
// two CTAs per SM.
QG_KERNEL_BUDGET("k_w4a4_quantize<true>", reinterpret_cast<const void*>(k_w4a4_quantize<true>), kQThreads,
                 kQSmemBytes, 0, 1, 2);
QG_KERNEL_BUDGET("k_w4a4_quantize<false>", reinterpret_cast<const void*>(k_w4a4_quantize<false>), kQThreads,
                 kQSmemBytes, 0, 1, 2);
QG_KERNEL_BUDGET("k_scales_transposed", reinterpret_cast<const void*>(k_scales_transposed), 256, 0, 0, 1, 1);
QG_KERNEL_BUDGET("w4a4_gemm_kernel", reinterpret_cast<const void*>(w4a4_gemm_kernel), W4A4Cfg::THREADS,
                 W4A4Cfg::SMEM_BYTES, W4A4Cfg::TMEM_COLS, 1, 1);
QG_KERNEL_BUDGET("w4a4_gemm2_kernel<W4A4PairCfgT<256,4>>",
                 reinterpret_cast<const void*>(w4a4_gemm2_kernel<W4A4PairCfgT<256, 4>>),
                 W4A4PairCfgT<256, 4>::THREADS, W4A4PairCfgT<256, 4>::SMEM_BYTES, W4A4PairCfgT<256, 4>::TMEM_COLS,
                 2, 1);
QG_KERNEL_BUDGET("w4a4_gemm2_kernel", reinterpret_cast<const void*>(w4a4_gemm2_kernel<W4A4PairCfg>), W4A4PairCfg::THREADS,
                 W4A4PairCfg::SMEM_BYTES, W4A4PairCfg::TMEM_COLS, 2, 1);

}  // namespace qg

using namespace qg;

extern "C" {

int w4a4_quantize(int64_t M, int64_t K, const float* X, int64_t ldx, const uint16_t* U, int64_t rank,
                  uint8_t* Xq, uint16_t* Xscale, uint16_t* XU, int64_t block, void* stream) {
    const qg::NvtxRange nvtx_range("w4a4_quantize");
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
    if (dev >= 64) return QG_ERR_CUDA;
    {
        static std::mutex mu;
        static bool attr_set[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(k_w4a4_quantize<true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(k_w4a4_quantize<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    CUtensorMap tX;
    // two boxes of 16 rows x 32 floats (128-byte rows) per 64-element block
    int rc = make_tmap_2d(&tX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, X, K, M, ldx * 4, 32, 16,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    const int grid = static_cast<int>((M + 15) / 16);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rank)
        k_w4a4_quantize<true><<<grid, kQThreads, kQSmemBytes, s>>>(
            tX, static_cast<int>(M), static_cast<int>(K), reinterpret_cast<const __half*>(U), Xq,
            reinterpret_cast<__half*>(Xscale), reinterpret_cast<__half*>(XU), ctl);
    else
        k_w4a4_quantize<false><<<grid, kQThreads, kQSmemBytes, s>>>(
            tX, static_cast<int>(M), static_cast<int>(K), nullptr, Xq,
            reinterpret_cast<__half*>(Xscale), nullptr, ctl);
    return map_cuda(cudaGetLastError());
}

}  // extern "C"

namespace qg {

// The GEMM on converted operands: A8 / B8 e4m3 codes (M x K, N x K), SXt /
// SWt the transposed fp32 scale tables (K/64 + 1 rows of Mp / Np floats).
static int w4a4_run(int64_t M, int64_t N, int64_t K, const uint8_t* A8, const float* SXt, const uint8_t* B8,
                    const float* SWt, const uint16_t* XU, const uint16_t* V, int64_t rank, const uint16_t* bias,
                    uint16_t* Y, int64_t ldy, const Ctl& ctl, int dev, cudaStream_t s) {
    const int nblk = static_cast<int>(K / kW4A4Block);
    const int64_t Mp = (M + 3) & ~int64_t(3), Np = (N + 3) & ~int64_t(3);
    W4A4Params p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_ks = static_cast<int>((K + W4A4Cfg::BK - 1) / W4A4Cfg::BK);
    p.nblk = nblk;
    p.lowrank = rank ? 1 : 0;
    p.Y = reinterpret_cast<__half*>(Y);
    p.ldy = ldy;
    p.bias = reinterpret_cast<const __half*>(bias);
    p.ctl = ctl;
    const int path = gemm_path();
    const bool pairs = path == 2 || (path == 0 && M > W4A4Cfg::BM);
    if (!pairs)
        return launch_w4a4<W4A4Cfg, false, w4a4_gemm_kernel>(A8, B8, SXt, SWt, XU, V, M, N, K, Mp, Np, rank,
                                                             p, dev, s);
    // 256 x 256 tiles (four epilogue warps per TMEM lane quadrant) by
    // default; 256 x 192 tiles (three per quadrant) as the ablation form
    using P256 = W4A4PairCfgT<256, 4>;
    if (w4a4_pair_form() == 1)
        return launch_w4a4<W4A4PairCfg, true, w4a4_gemm2_kernel<W4A4PairCfg>>(A8, B8, SXt, SWt, XU, V, M, N, K,
                                                                               Mp, Np, rank, p, dev, s);
    return launch_w4a4<P256, true, w4a4_gemm2_kernel<P256>>(A8, B8, SXt, SWt, XU, V, M, N, K, Mp, Np, rank, p,
                                                             dev, s);
}

// w4a4_gemm and w4a4_gemm_affine: alpha == nullptr is the formula as printed.
static int w4a4_gemm_impl(int64_t M, int64_t N, int64_t K, const uint8_t* Xq, const uint16_t* Xscale,
                          const uint8_t* Wq, const uint16_t* Wscale, int64_t block, const uint16_t* XU,
                          const uint16_t* V, int64_t rank, const uint16_t* alpha, const uint16_t* bias,
                          uint16_t* Y, int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return QG_ERR_INVALID_ARG;
    if (block != kW4A4Block) return QG_ERR_UNSUPPORTED;
    if (K % kW4A4Block) return QG_ERR_INVALID_ARG;
    if (rank != 0 && rank != kW4A4MaxRank) return QG_ERR_UNSUPPORTED;
    if (!Xq || !Xscale || !Wq || !Wscale || !Y || (rank && (!XU || !V))) return QG_ERR_INVALID_ARG;
    if (ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(Y) || (rank && (!aligned16(XU) || !aligned16(V))))
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

    int rc = s4_to_e4m3_pair(Xq, M, K / 2, A8, Wq, N, K / 2, B8, K, dev, s);
    if (rc) return rc;
    k_scales_transposed<<<conv_grid(dev, 256 * ((nblk + 32) / 32) * ((Mp + 31) / 32)), 256, 0, s>>>(
        M, Mp, nblk, reinterpret_cast<const __half*>(Xscale), nullptr, SXt);
    k_scales_transposed<<<conv_grid(dev, 256 * ((nblk + 32) / 32) * ((Np + 31) / 32)), 256, 0, s>>>(
        N, Np, nblk, reinterpret_cast<const __half*>(Wscale), reinterpret_cast<const __half*>(alpha),
        SWt);
    rc = map_cuda(cudaGetLastError());
    if (rc) return rc;
    return w4a4_run(M, N, K, A8, SXt, B8, SWt, XU, V, rank, bias, Y, ldy, ctl, dev, s);
}

// Offset of the scale table inside a buffer of packed weights (after the
// e4m3 codes, N x K bytes).
static size_t w4a4_packed_scales_offset(int64_t N, int64_t K) {
    return (static_cast<size_t>(N) * static_cast<size_t>(K) + 255) & ~static_cast<size_t>(255);
}

}  // namespace qg

extern "C" {

int w4a4_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* Xq, const uint16_t* Xscale,
              const uint8_t* Wq, const uint16_t* Wscale, int64_t block, const uint16_t* XU,
              const uint16_t* V, int64_t rank, const uint16_t* bias, uint16_t* Y, int64_t ldy,
              void* ws, size_t ws_bytes, void* stream) {
    const qg::NvtxRange nvtx_range("w4a4_gemm");
    return w4a4_gemm_impl(M, N, K, Xq, Xscale, Wq, Wscale, block, XU, V, rank, nullptr, bias, Y, ldy,
                          ws, ws_bytes, stream);
}

int w4a4_gemm_affine(int64_t M, int64_t N, int64_t K, const uint8_t* Xq, const uint16_t* Xscale,
                     const uint8_t* Wq, const uint16_t* Wscale, int64_t block, const uint16_t* XU,
                     const uint16_t* V, int64_t rank, const uint16_t* alpha, const uint16_t* bias,
                     uint16_t* Y, int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
    const qg::NvtxRange nvtx_range("w4a4_gemm_affine");
    if (!alpha) return QG_ERR_INVALID_ARG;
    return w4a4_gemm_impl(M, N, K, Xq, Xscale, Wq, Wscale, block, XU, V, rank, alpha, bias, Y, ldy,
                          ws, ws_bytes, stream);
}

int w4a4_prepack_weights(int64_t N, int64_t K, const uint8_t* Wq, const uint16_t* Wscale, int64_t block,
                         const uint16_t* alpha, void* packed, size_t packed_bytes, void* stream) {
    const qg::NvtxRange nvtx_range("w4a4_prepack_weights");
    if (N < 1 || K < 1 || N > INT32_MAX || K > INT32_MAX) return QG_ERR_INVALID_ARG;
    if (block != kW4A4Block) return QG_ERR_UNSUPPORTED;
    if (K % kW4A4Block) return QG_ERR_INVALID_ARG;
    if (!Wq || !Wscale || !packed) return QG_ERR_INVALID_ARG;
    if (!aligned16(Wq) || (reinterpret_cast<uintptr_t>(packed) & 255u)) return QG_ERR_MISALIGNED;
    if (packed_bytes < qg_workspace_size(QG_OP_W4A4_WEIGHTS, 1, N, K)) return QG_ERR_WORKSPACE;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int nblk = static_cast<int>(K / kW4A4Block);
    const int64_t Np = (N + 3) & ~int64_t(3);
    uint8_t* B8 = static_cast<uint8_t*>(packed);
    float* SWt = reinterpret_cast<float*>(B8 + w4a4_packed_scales_offset(N, K));
    int rc = s4_to_e4m3_rows(Wq, N, K / 2, B8, K, dev, s);
    if (rc) return rc;
    k_scales_transposed<<<conv_grid(dev, 256 * ((nblk + 32) / 32) * ((Np + 31) / 32)), 256, 0, s>>>(
        N, Np, nblk, reinterpret_cast<const __half*>(Wscale), reinterpret_cast<const __half*>(alpha), SWt);
    return map_cuda(cudaGetLastError());
}

int w4a4_gemm_prepacked(int64_t M, int64_t N, int64_t K, const uint8_t* Xq, const uint16_t* Xscale,
                        const void* packed, size_t packed_bytes, int64_t block, const uint16_t* XU,
                        const uint16_t* V, int64_t rank, const uint16_t* bias, uint16_t* Y, int64_t ldy,
                        void* ws, size_t ws_bytes, void* stream) {
    const qg::NvtxRange nvtx_range("w4a4_gemm_prepacked");
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return QG_ERR_INVALID_ARG;
    if (block != kW4A4Block) return QG_ERR_UNSUPPORTED;
    if (K % kW4A4Block) return QG_ERR_INVALID_ARG;
    if (rank != 0 && rank != kW4A4MaxRank) return QG_ERR_UNSUPPORTED;
    if (!Xq || !Xscale || !packed || !Y || (rank && (!XU || !V))) return QG_ERR_INVALID_ARG;
    if (ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(Xq) || !aligned16(Y) || (rank && (!aligned16(XU) || !aligned16(V))) ||
        (reinterpret_cast<uintptr_t>(packed) & 255u))
        return QG_ERR_MISALIGNED;
    if (packed_bytes < qg_workspace_size(QG_OP_W4A4_WEIGHTS, 1, N, K)) return QG_ERR_INVALID_ARG;
    if (!ws || ws_bytes < qg_workspace_size(QG_OP_W4A4_PREPACKED, M, N, K)) return QG_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QG_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
    Ctl ctl = host_ctl(dev);
    if (!ctl.status) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int nblk = static_cast<int>(K / kW4A4Block);
    const int64_t Mp = (M + 3) & ~int64_t(3);
    uint8_t* A8 = static_cast<uint8_t*>(ws);
    float* SXt = reinterpret_cast<float*>(A8 + ((static_cast<size_t>(M) * K + 255) & ~static_cast<size_t>(255)));
    int rc = s4_to_e4m3_rows(Xq, M, K / 2, A8, K, dev, s);
    if (rc) return rc;
    k_scales_transposed<<<conv_grid(dev, 256 * ((nblk + 32) / 32) * ((Mp + 31) / 32)), 256, 0, s>>>(
        M, Mp, nblk, reinterpret_cast<const __half*>(Xscale), nullptr, SXt);
    rc = map_cuda(cudaGetLastError());
    if (rc) return rc;
    const uint8_t* B8 = static_cast<const uint8_t*>(packed);
    const float* SWt = reinterpret_cast<const float*>(B8 + w4a4_packed_scales_offset(N, K));
    return w4a4_run(M, N, K, A8, SXt, B8, SWt, XU, V, rank, bias, Y, ldy, ctl, dev, s);
}

int qg_set_w4a4_pair_form(int form) {
    if (form < 0 || form > 1) return QG_ERR_INVALID_ARG;
    g_w4a4_pair_form.store(form);
    return QG_OK;
}

}  // extern "C"

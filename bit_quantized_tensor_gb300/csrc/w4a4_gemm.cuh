// W4A4 block-scaled GEMM with low-rank residual and bias, for sm_103a:
//
//   Y[m][n] = sum_j sX[m][j] * sW[n][j] * P_j[m][n]  +  (XU . V)[m][n]  +  b[n]
//   P_j[m][n] = sum_{k in block j} qX[m][k] * qW[n][k]      (64-wide K blocks)
//
// ("Warp-Specialized Kernel Implementation for W4A4 MatMul on Latest GPU
// Architectures", sections 1 and 5.)  The 4-bit values travel as e4m3 bytes
// (every integer in [-8, 8] is exact in e4m3), so each block partial P_j is
// an exact integer computed by tcgen05 kind::f8f6f4 into its own TMEM
// buffer.  The epilogue warps apply the two block scales in fp32 and add the
// result to a register-resident fp32 tile:
//     c = sW[n][j] * sX[m][j]   (packed f32x2, two columns per instruction)
//     acc = fma(P_j, c, acc)    (one rounding per block)  The low-rank
// term XU . V is one more accumulation unit per tile: a kind::f16 MMA over
// the 32 low-rank columns (TMA zero-fills them to a 64-wide tile), scaled by
// the constant 1 row appended to the scale tables.  The bias is added before
// the fp16 store.
//
// Three rings advance independently ("three independent pipelines: main
// operands, low-rank branch, drain"):
//   operand ring   STAGES x (A 128x128 B, B 192x128 B), TMA -> MMA
//   scale ring     SC_STAGES x (sX 2x128, sW 2x192 fp32), TMA -> epilogue
//   accumulators   2 TMEM buffers of 128 x 192 fp32, MMA -> epilogue
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "tc_gemm.cuh"

namespace qg {

// Packed pairs of fp32 values in one 64-bit register (low half = first).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ uint64_t pack_u32x2(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

struct W4A4Cfg {
    // N = 192 lets 16 epilogue warps (4 per TMEM lane quadrant, 48 columns
    // each) hold their fp32 accumulators in registers within an 18-warp block.
    static constexpr int BM = 128, BN = 192;
    static constexpr int ROW_BYTES = 128;                 // 128 e4m3 per stage row = 2 blocks
    static constexpr int BK = 128;
    static constexpr int QBLOCK = 64;                     // scale block along K
    static constexpr int A_BYTES = BM * ROW_BYTES;        // 16 KB
    static constexpr int B_BYTES = BN * ROW_BYTES;        // 24 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 5;
    static constexpr int SC_STAGES = 6;
    static constexpr int SX_BYTES = 2 * BM * 4;           // two blocks of row scales (fp32)
    static constexpr int SW_BYTES = 2 * BN * 4;           // two blocks of column scales
    static constexpr int SC_BYTES = SX_BYTES + SW_BYTES;
    static constexpr int BARRIER_BYTES = 256;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + SC_STAGES * SC_BYTES + BARRIER_BYTES + ALIGN_SLACK;
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 16;
    static constexpr int EPI_COLS = BN / 4;               // columns per epilogue warp
    static constexpr int THREADS = 32 * (2 + EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * SC_STAGES + 2 * ACC_BUFS + 1;
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, BM, BN);  // e4m3 or f16 x2, f32 acc

    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared-memory budget exceeded");
    static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM keeps all 512 TMEM columns free");
    static_assert(NUM_BARRIERS * 8 + 8 <= BARRIER_BYTES, "barrier area too small");
    static_assert(ACC_BUFS * BN <= TMEM_COLS, "TMEM budget exceeded");
    static_assert(SC_BYTES % 128 == 0 && STAGE_BYTES % 1024 == 0, "alignment of ring slots");
    static_assert(EPI_COLS % 16 == 0 && BN % 16 == 0 && BN <= 256, "epilogue column split");
    static_assert(THREADS <= 576, "more than 18 warps would cap registers below 112");
};

struct W4A4Params {
    int M, N, K;
    int num_ks;          // ceil(K / 128) operand stages per tile
    int nblk;            // K / 64: row index of the constant-1 scale row
    int lowrank;         // 1 when the XU . V unit is present
    __half* Y;
    int64_t ldy;
    const __half* bias;  // may be null
    Ctl ctl;
};

enum W4A4Site : int {
    kSiteW4ProdEmpty = 201,
    kSiteW4ProdScale = 202,
    kSiteW4MmaAcc = 203,
    kSiteW4MmaFull = 204,
    kSiteW4EpiScale = 205,
    kSiteW4EpiAcc = 206,
    kSiteW4DrainTma = 207,
    kSiteW4DrainMma = 208,
};

__global__ void __launch_bounds__(W4A4Cfg::THREADS, 1)
    w4a4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmXU, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmSX, const __grid_constant__ CUtensorMap tmSW,
                     const W4A4Params p) {
    using Cfg = W4A4Cfg;
    constexpr int STAGES = Cfg::STAGES, SCS = Cfg::SC_STAGES, ACC = Cfg::ACC_BUFS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t* sS = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sS + SCS * Cfg::SC_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto scf_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto sce_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + SCS + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * SCS + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * SCS + ACC + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * SCS + 2 * ACC);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < SCS; ++s) {
            mbar_init(scf_bar(s), 1);
            mbar_init(sce_bar(s), Cfg::EPI_WARPS);
        }
        for (int b = 0; b < ACC; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), Cfg::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSX);
        tma_prefetch_desc(&tmSW);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int num_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int ntiles = num_m * num_n;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            Ring<STAGES> ps;
            Ring<SCS> ss;
            uint32_t armed = 0, armed_phase = 0, sarmed = 0, sarmed_phase = 0;
            const uint64_t pol = l2_policy_evict_normal();
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb);
                const int steps = p.num_ks + p.lowrank;
                for (int ks = 0; ks < steps; ++ks) {
                    const bool lr = ks == p.num_ks;
                    if (!bounded_wait(empty_bar(ps.slot()), ps.parity() ^ 1u, abort_flag, p.ctl,
                                      kSiteW4ProdEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(ps.slot()), Cfg::STAGE_BYTES);
                    const uint32_t da = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                    const uint32_t db = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
                    if (!lr) {
                        tma_load_2d(da, &tmA, ks * Cfg::BK, mb * Cfg::BM, full_bar(ps.slot()), pol);
                        tma_load_2d(db, &tmB, ks * Cfg::BK, nb * Cfg::BN, full_bar(ps.slot()), pol);
                    } else {
                        tma_load_2d(da, &tmXU, 0, mb * Cfg::BM, full_bar(ps.slot()), pol);
                        tma_load_2d(db, &tmV, 0, nb * Cfg::BN, full_bar(ps.slot()), pol);
                    }
                    armed |= 1u << ps.slot();
                    armed_phase = (armed_phase & ~(1u << ps.slot())) | (ps.parity() << ps.slot());
                    ps.next();

                    if (!bounded_wait(sce_bar(ss.slot()), ss.parity() ^ 1u, abort_flag, p.ctl,
                                      kSiteW4ProdScale)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(scf_bar(ss.slot()), Cfg::SC_BYTES);
                    const uint32_t dsx = smem_u32(sS + ss.slot() * Cfg::SC_BYTES);
                    const int row = lr ? p.nblk : 2 * ks;
                    tma_load_2d(dsx, &tmSX, mb * Cfg::BM, row, scf_bar(ss.slot()), pol);
                    tma_load_2d(dsx + Cfg::SX_BYTES, &tmSW, nb * Cfg::BN, row, scf_bar(ss.slot()), pol);
                    sarmed |= 1u << ss.slot();
                    sarmed_phase = (sarmed_phase & ~(1u << ss.slot())) | (ss.parity() << ss.slot());
                    ss.next();
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s))
                        bounded_wait(full_bar(s), (armed_phase >> s) & 1u, nullptr, p.ctl,
                                     kSiteW4DrainTma);
                for (int s = 0; s < SCS; ++s)
                    if (sarmed & (1u << s))
                        bounded_wait(scf_bar(s), (sarmed_phase >> s) & 1u, nullptr, p.ctl,
                                     kSiteW4DrainTma);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            Ring<STAGES> ps;
            Ring<ACC> as;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                const int steps = p.num_ks + p.lowrank;
                for (int ks = 0; ok && ks < steps; ++ks) {
                    const bool lr = ks == p.num_ks;
                    if (!bounded_wait(full_bar(ps.slot()), ps.parity(), abort_flag, p.ctl,
                                      kSiteW4MmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
                    const int units = lr ? 1 : 2;
                    for (int h = 0; h < units; ++h) {
                        if (!bounded_wait(acce_bar(as.slot()), as.parity() ^ 1u, abort_flag, p.ctl,
                                          kSiteW4MmaAcc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + static_cast<uint32_t>(as.slot() * Cfg::BN);
                        if (!lr) {
                            // one 64-wide block = bytes [64h, 64h + 64) of each row: 2 MMAs
#pragma unroll
                            for (int k = 0; k < 2; ++k)
                                tc_mma<MmaKind::F8F6F4>(
                                    d, smem_desc_sw128(a_addr + 64u * h + 32u * k),
                                    smem_desc_sw128(b_addr + 64u * h + 32u * k), Cfg::IDESC,
                                    k > 0 ? 1u : 0u);
                        } else {
                            // 64 fp16 columns (32 low-rank + 32 zero-filled): 4 MMAs
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma<MmaKind::F16>(d, smem_desc_sw128(a_addr + 32u * k),
                                                     smem_desc_sw128(b_addr + 32u * k), Cfg::IDESC,
                                                     k > 0 ? 1u : 0u);
                        }
                        tc_commit(accf_bar(as.slot()));
                        as.next();
                    }
                    if (!ok) break;
                    tc_commit(empty_bar(ps.slot()));
                    ps.next();
                }
            }
            tc_commit(drain_bar);
            bounded_wait(drain_bar, 0u, nullptr, p.ctl, kSiteW4DrainMma);
        }
    } else {
        // ---------------------------------------------------- epilogue
        // Warp (quad, colpart) owns TMEM lanes [32 quad, 32 quad + 32) and
        // columns [48 colpart, 48 colpart + 48) of the tile, read as two
        // 16-lane halves in the m16n8-accumulator layout: lane (g, q) holds
        // rows 32 quad + 16 hf + g (+ 8) and columns 8c + 2q (+ 1) for the
        // six column groups c, so per block it needs 4 row scales and 6
        // column-scale pairs, all from distinct shared-memory words.  The
        // three 16-column chunks are loaded one ahead of the arithmetic.
        constexpr int NCH = Cfg::EPI_COLS / 16;
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int colpart = (warp - 2) >> 2;     // which quarter of the tile's columns
        const int g = lane >> 2, q = lane & 3;
        Ring<ACC> as;
        Ring<SCS> ss;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb);
            // acc[hf][c][2e + d]: row 16 hf + g + 8e, column 8c + 2q + d
            float acc[2][2 * NCH][4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int c = 0; c < 2 * NCH; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[hf][c][i] = 0.f;
            const int steps = p.num_ks + p.lowrank;
            for (int ks = 0; ok && ks < steps; ++ks) {
                const int units = (ks == p.num_ks) ? 1 : 2;
                bool got = bounded_wait(scf_bar(ss.slot()), ss.parity(), abort_flag, p.ctl,
                                        kSiteW4EpiScale);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const float* sx_s = reinterpret_cast<const float*>(sS + ss.slot() * Cfg::SC_BYTES);
                const float* sw_s = sx_s + 2 * Cfg::BM;
                for (int h = 0; h < units; ++h) {
                    got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl,
                                       kSiteW4EpiAcc);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float* sxr = sx_s + h * Cfg::BM + quad * 32 + g;
                    const float* swc = sw_s + h * Cfg::BN + colpart * Cfg::EPI_COLS + 2 * q;
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                           static_cast<uint32_t>(as.slot() * Cfg::BN +
                                                                 colpart * Cfg::EPI_COLS);
                    uint32_t rb[2][2][8];  // [buffer][half][x2 registers]
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tmem_ld_16x256b_x2(taddr + (static_cast<uint32_t>(16 * hf) << 16), rb[0][hf]);
                    // row-scale pairs (s, s) for rows g, g + 8, 16 + g, 24 + g
                    uint64_t sxp[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) sxp[k] = pack_f32x2(sxr[8 * k], sxr[8 * k]);
                    tmem_wait_ld();
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        if (ch + 1 < NCH) {
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
                                tmem_ld_16x256b_x2(taddr + (static_cast<uint32_t>(16 * hf) << 16) +
                                                       static_cast<uint32_t>(16 * (ch + 1)),
                                                   rb[(ch + 1) & 1][hf]);
                        } else {
                            // the buffer's last TMEM reads completed at the
                            // previous tcgen05.wait::ld: hand it back before
                            // the last chunk's arithmetic
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(acce_bar(as.slot()));
                        }
                        // c = sW * sX for the chunk's 2 column pairs and 4 rows, as
                        // packed pairs (both factors already paired in registers)
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const uint64_t w = *reinterpret_cast<const uint64_t*>(swc + 16 * ch + 8 * i);
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const float2 c = unpack_f32x2(mul2(w, sxp[2 * hf + e]));
                                    const uint32_t* r = &rb[ch & 1][hf][4 * i + 2 * e];
                                    float* a = &acc[hf][2 * ch + i][2 * e];
                                    a[0] = __fmaf_rn(__uint_as_float(r[0]), c.x, a[0]);
                                    a[1] = __fmaf_rn(__uint_as_float(r[1]), c.y, a[1]);
                                }
                        }
                        if (ch + 1 < NCH) tmem_wait_ld();
                    }
                    as.next();
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(sce_bar(ss.slot()));
                ss.next();
            }
            if (!ok) break;
            // fp16 store (+ bias): per row pairs of adjacent columns
            const int colb = nb * Cfg::BN + colpart * Cfg::EPI_COLS + 2 * q;
            const bool pair_ok = (p.ldy & 1) == 0;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = mb * Cfg::BM + quad * 32 + 16 * hf + 8 * e + g;
                    if (row >= p.M) continue;
                    __half* yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
#pragma unroll
                    for (int c = 0; c < 2 * NCH; ++c) {
                        const int col = colb + 8 * c;
                        float v0 = acc[hf][c][2 * e], v1 = acc[hf][c][2 * e + 1];
                        if (p.bias) {
                            if (col < p.N) v0 += __half2float(p.bias[col]);
                            if (col + 1 < p.N) v1 += __half2float(p.bias[col + 1]);
                        }
                        if (pair_ok && col + 1 < p.N) {
                            *reinterpret_cast<__half2*>(yrow + col) = __floats2half2_rn(v0, v1);
                        } else {
                            if (col < p.N) yrow[col] = __float2half_rn(v0);
                            if (col + 1 < p.N) yrow[col + 1] = __float2half_rn(v1);
                        }
                    }
                }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace qg

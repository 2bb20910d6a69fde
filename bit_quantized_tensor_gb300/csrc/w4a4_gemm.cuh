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
//     t = P_j * sW[n][j]   (exact: 13-bit integer times an fp16 value)
//     acc = fma(t, sX[m][j], acc)   (one rounding per block)
// using packed f32x2 arithmetic, two columns per instruction.  The low-rank
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

__device__ __forceinline__ void mul_f32x2(float& d0, float& d1, float a0, float a1, float b0,
                                          float b1) {
    asm("{\n.reg .b64 a, b, d;\nmov.b64 a, {%2, %3};\nmov.b64 b, {%4, %5};\n"
        "mul.rn.f32x2 d, a, b;\nmov.b64 {%0, %1}, d;\n}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, float b0,
                                          float b1) {
    asm("{\n.reg .b64 a, b, d;\nmov.b64 a, {%2, %3};\nmov.b64 b, {%4, %5};\n"
        "mov.b64 d, {%0, %1};\nfma.rn.f32x2 d, a, b, d;\nmov.b64 {%0, %1}, d;\n}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

struct W4A4Cfg {
    // N = 192 lets 12 epilogue warps (3 per TMEM lane quadrant, 64 columns
    // each) hold their fp32 accumulators in registers within a 14-warp block.
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
    static constexpr int EPI_WARPS = 12;
    static constexpr int EPI_COLS = BN / 3;               // columns per epilogue warp
    static constexpr int THREADS = 32 * (2 + EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * SC_STAGES + 2 * ACC_BUFS + 1;
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, BM, BN);  // e4m3 or f16 x2, f32 acc

    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared-memory budget exceeded");
    static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM keeps all 512 TMEM columns free");
    static_assert(NUM_BARRIERS * 8 + 8 <= BARRIER_BYTES, "barrier area too small");
    static_assert(ACC_BUFS * BN <= TMEM_COLS, "TMEM budget exceeded");
    static_assert(SC_BYTES % 128 == 0 && STAGE_BYTES % 1024 == 0, "alignment of ring slots");
    static_assert(EPI_COLS % 16 == 0 && BN % 16 == 0 && BN <= 256, "epilogue column split");
    static_assert(THREADS <= 512, "more than 16 warps would cap registers at 96");
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
            PipeState<STAGES> ps;
            PipeState<SCS> ss;
            uint32_t armed = 0, armed_phase = 0, sarmed = 0, sarmed_phase = 0;
            const uint64_t pol = l2_policy_evict_normal();
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb);
                const int steps = p.num_ks + p.lowrank;
                for (int ks = 0; ks < steps; ++ks) {
                    const bool lr = ks == p.num_ks;
                    if (!bounded_wait(empty_bar(ps.index), ps.phase ^ 1u, abort_flag, p.ctl,
                                      kSiteW4ProdEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(ps.index), Cfg::STAGE_BYTES);
                    const uint32_t da = smem_u32(sA + ps.index * Cfg::A_BYTES);
                    const uint32_t db = smem_u32(sB + ps.index * Cfg::B_BYTES);
                    if (!lr) {
                        tma_load_2d(da, &tmA, ks * Cfg::BK, mb * Cfg::BM, full_bar(ps.index), pol);
                        tma_load_2d(db, &tmB, ks * Cfg::BK, nb * Cfg::BN, full_bar(ps.index), pol);
                    } else {
                        tma_load_2d(da, &tmXU, 0, mb * Cfg::BM, full_bar(ps.index), pol);
                        tma_load_2d(db, &tmV, 0, nb * Cfg::BN, full_bar(ps.index), pol);
                    }
                    armed |= 1u << ps.index;
                    armed_phase = (armed_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
                    ps.advance();

                    if (!bounded_wait(sce_bar(ss.index), ss.phase ^ 1u, abort_flag, p.ctl,
                                      kSiteW4ProdScale)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(scf_bar(ss.index), Cfg::SC_BYTES);
                    const uint32_t dsx = smem_u32(sS + ss.index * Cfg::SC_BYTES);
                    const int row = lr ? p.nblk : 2 * ks;
                    tma_load_2d(dsx, &tmSX, mb * Cfg::BM, row, scf_bar(ss.index), pol);
                    tma_load_2d(dsx + Cfg::SX_BYTES, &tmSW, nb * Cfg::BN, row, scf_bar(ss.index), pol);
                    sarmed |= 1u << ss.index;
                    sarmed_phase = (sarmed_phase & ~(1u << ss.index)) | (ss.phase << ss.index);
                    ss.advance();
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
            PipeState<STAGES> ps;
            PipeState<ACC> as;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                const int steps = p.num_ks + p.lowrank;
                for (int ks = 0; ok && ks < steps; ++ks) {
                    const bool lr = ks == p.num_ks;
                    if (!bounded_wait(full_bar(ps.index), ps.phase, abort_flag, p.ctl,
                                      kSiteW4MmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + ps.index * Cfg::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + ps.index * Cfg::B_BYTES);
                    const int units = lr ? 1 : 2;
                    for (int h = 0; h < units; ++h) {
                        if (!bounded_wait(acce_bar(as.index), as.phase ^ 1u, abort_flag, p.ctl,
                                          kSiteW4MmaAcc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + static_cast<uint32_t>(as.index * Cfg::BN);
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
                        tc_commit(accf_bar(as.index));
                        as.advance();
                    }
                    if (!ok) break;
                    tc_commit(empty_bar(ps.index));
                    ps.advance();
                }
            }
            tc_commit(drain_bar);
            bounded_wait(drain_bar, 0u, nullptr, p.ctl, kSiteW4DrainMma);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int colpart = (warp - 2) >> 2;     // which third of the tile's columns
        PipeState<ACC> as;
        PipeState<SCS> ss;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb);
            const int rloc = quad * 32 + lane;
            const int row = mb * Cfg::BM + rloc;
            const int col0 = nb * Cfg::BN + colpart * Cfg::EPI_COLS;
            float acc[Cfg::EPI_COLS];
#pragma unroll
            for (int i = 0; i < Cfg::EPI_COLS; ++i) acc[i] = 0.f;
            const int steps = p.num_ks + p.lowrank;
            for (int ks = 0; ok && ks < steps; ++ks) {
                const int units = (ks == p.num_ks) ? 1 : 2;
                bool got = bounded_wait(scf_bar(ss.index), ss.phase, abort_flag, p.ctl,
                                        kSiteW4EpiScale);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const float* sx_s = reinterpret_cast<const float*>(sS + ss.index * Cfg::SC_BYTES);
                const float* sw_s = sx_s + 2 * Cfg::BM;
                for (int h = 0; h < units; ++h) {
                    got = bounded_wait(accf_bar(as.index), as.phase, abort_flag, p.ctl,
                                       kSiteW4EpiAcc);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float sx = sx_s[h * Cfg::BM + rloc];
                    const float* swc = sw_s + h * Cfg::BN + colpart * Cfg::EPI_COLS;
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                           static_cast<uint32_t>(as.index * Cfg::BN +
                                                                 colpart * Cfg::EPI_COLS);
#pragma unroll
                    for (int c = 0; c < Cfg::EPI_COLS / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(taddr + 16u * c, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 w = *reinterpret_cast<const float4*>(swc + 16 * c + i);
                            float t0, t1, t2, t3;
                            mul_f32x2(t0, t1, __uint_as_float(r[i]), __uint_as_float(r[i + 1]), w.x,
                                      w.y);
                            mul_f32x2(t2, t3, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]),
                                      w.z, w.w);
                            fma_f32x2(acc[16 * c + i], acc[16 * c + i + 1], t0, t1, sx, sx);
                            fma_f32x2(acc[16 * c + i + 2], acc[16 * c + i + 3], t2, t3, sx, sx);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(as.index));
                    as.advance();
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(sce_bar(ss.index));
                ss.advance();
            }
            if (!ok) break;
            if (row < p.M)
                store_row_f16<Cfg::EPI_COLS>(p.Y + static_cast<int64_t>(row) * p.ldy + col0, col0, p.N,
                                             acc, p.bias);
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

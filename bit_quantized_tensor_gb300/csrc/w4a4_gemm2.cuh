// Paired-CTA (cta_group::2) form of the W4A4 block-scaled GEMM:
//
//   Y[m][n] = sum_j sX[m][j] * sW[n][j] * P_j[m][n]  +  (XU . V)[m][n]  +  b[n]
//
// with the same arithmetic as w4a4_gemm.cuh (exact integer block partials
// P_j from kind::f8f6f4 on e4m3 bytes, c = sW * sX in packed fp32, acc =
// fma(P_j, c, acc), the low-rank term as one kind::f16 unit scaled by the
// constant-1 scale row, bias before the fp16 store).  ("Warp-Specialized
// Kernel Implementation for W4A4 MatMul on Latest GPU Architectures",
// sections 4 and 5.)
//
// What changes is the data flow.  The two CTAs of a cluster share a 256 x BN
// output tile (BN = 256 by default, 192 as the ablation form): CTA r owns
// rows [128 r, 128 r + 128), loads its own 128 rows of A and its own BN / 2
// rows of B (half of the tile's columns), and the leader issues
// tcgen05.mma.cta_group::2 with M = 256 that writes each CTA's 128 x BN
// block partial into that CTA's TMEM (two buffers).  Per 64-wide K block an
// SM then loads 8 KB of A and BN / 2 x 64 bytes of B; at BN = 256 each
// paired fp8 MMA instruction (N = 256, K = 32) carries enough tensor work
// to cover its own issue cost, which the N = 128 instruction does not.
//
// Synchronization:
//   full[s]     leader only; armed by the leader's producer for both CTAs'
//               bytes, completed by both CTAs' TMA loads
//   empty[s]    both CTAs; one multicast commit from the leader
//   scf/sce[s]  per CTA: its own scale tables (sX of its rows, sW of the tile)
//   accf[b]     both CTAs; multicast commit after a block's MMAs
//   acce[b]     leader only; the epilogue warps of both CTAs arrive remotely
//               (relaxed: one arrive per warp per 64-wide block)
// Every wait is bounded; the CTAs leave only after a cluster barrier.
#pragma once
#include "w4a4_gemm.cuh"

namespace qg {

template <int BN_ = 192, int EPQ_ = 3>
struct W4A4PairCfgT {
    static constexpr int BM = 128;                        // rows per CTA (256 per pair)
    static constexpr int BN = BN_;                        // columns of the pair's tile
    static constexpr int B_ROWS = BN / 2;                 // B rows loaded per CTA
    static constexpr int ROW_BYTES = 128;                 // 128 e4m3 per stage row = 2 blocks
    static constexpr int BK = 128;
    static constexpr int A_BYTES = BM * ROW_BYTES;        // 16 KB
    static constexpr int B_BYTES = B_ROWS * ROW_BYTES;    // 12 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SC_STAGES = 8;
    static constexpr int SX_BYTES = 2 * BM * 4;           // two blocks of row scales (fp32)
    static constexpr int SW_BYTES = 2 * BN * 4;           // two blocks of column scales
    static constexpr int SC_BYTES = SX_BYTES + SW_BYTES;
    static constexpr int BARRIER_BYTES = 512;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int STAGES =
        (SMEM_LIMIT - SC_STAGES * SC_BYTES - BARRIER_BYTES - ALIGN_SLACK) / STAGE_BYTES;
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + SC_STAGES * SC_BYTES + BARRIER_BYTES + ALIGN_SLACK;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 4 * EPQ_;            // EPQ_ per TMEM lane quadrant
    static constexpr int EPI_COLS = BN / EPQ_;            // columns per epilogue warp
    static constexpr int THREADS = 32 * (2 + EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * SC_STAGES + 2 * ACC_BUFS + 1;
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, 2 * BM, BN);  // M = 256 across the pair

    static_assert(STAGES >= 5, "operand ring too shallow");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared-memory budget exceeded");
    static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM keeps all 512 TMEM columns free");
    static_assert(NUM_BARRIERS * 8 + 8 <= BARRIER_BYTES, "barrier area too small");
    static_assert(ACC_BUFS * BN <= TMEM_COLS, "TMEM budget exceeded");
    static_assert(SC_BYTES % 128 == 0 && B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0,
                  "alignment of ring slots");
    static_assert(EPI_COLS % 8 == 0, "epilogue reads 8-column groups");
    static_assert(THREADS <= 640, "register file split");
};
using W4A4PairCfg = W4A4PairCfgT<>;

enum W4A4PairSite : int {
    kSiteW4PProdEmpty = 221,
    kSiteW4PProdScale = 222,
    kSiteW4PMmaAcc = 223,
    kSiteW4PMmaFull = 224,
    kSiteW4PEpiScale = 225,
    kSiteW4PEpiAcc = 226,
    kSiteW4PDrainTma = 227,
    kSiteW4PDrainMma = 228,
};

template <class Cfg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::THREADS, 1)
    w4a4_gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmXU, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmSX, const __grid_constant__ CUtensorMap tmSW,
                      const W4A4Params p) {
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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

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
            mbar_init(acce_bar(b), 2 * Cfg::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSX);
        tma_prefetch_desc(&tmSW);
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialized and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int num_m = (p.M + 2 * Cfg::BM - 1) / (2 * Cfg::BM);
    const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int ntiles = num_m * num_n;
    const int steps = p.num_ks + p.lowrank;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            Ring<STAGES> ps;
            Ring<SCS> ss;
            uint32_t armed = 0, armed_phase = 0, sarmed = 0, sarmed_phase = 0;
            const uint64_t pol = l2_policy_evict_normal();
            bool ok = true;
            for (int t = pair; ok && t < ntiles; t += npairs) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb, kGroupMPairs);
                const int arow = mb * 2 * Cfg::BM + static_cast<int>(rank) * Cfg::BM;
                const int brow = nb * Cfg::BN + static_cast<int>(rank) * Cfg::B_ROWS;
                for (int ks = 0; ks < steps; ++ks) {
                    const bool lr = ks == p.num_ks;
                    if (!bounded_wait(empty_bar(ps.slot()), ps.parity() ^ 1u, abort_flag, p.ctl,
                                      kSiteW4PProdEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t lead_full = mapa_shared(full_bar(ps.slot()), 0);
                    if (leader) {
                        mbar_arrive_expect_tx(full_bar(ps.slot()), 2 * Cfg::STAGE_BYTES);
                        armed |= 1u << ps.slot();
                        armed_phase = (armed_phase & ~(1u << ps.slot())) | (ps.parity() << ps.slot());
                    }
                    const uint32_t da = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                    const uint32_t db = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
                    if (!lr) {
                        tma_load_2d_pair(da, &tmA, ks * Cfg::BK, arow, lead_full, pol);
                        tma_load_2d_pair(db, &tmB, ks * Cfg::BK, brow, lead_full, pol);
                    } else {
                        tma_load_2d_pair(da, &tmXU, 0, arow, lead_full, pol);
                        tma_load_2d_pair(db, &tmV, 0, brow, lead_full, pol);
                    }
                    ps.next();

                    if (!bounded_wait(sce_bar(ss.slot()), ss.parity() ^ 1u, abort_flag, p.ctl,
                                      kSiteW4PProdScale)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(scf_bar(ss.slot()), Cfg::SC_BYTES);
                    const uint32_t dsx = smem_u32(sS + ss.slot() * Cfg::SC_BYTES);
                    const int row = lr ? p.nblk : 2 * ks;
                    tma_load_2d(dsx, &tmSX, arow, row, scf_bar(ss.slot()), pol);
                    tma_load_2d(dsx + Cfg::SX_BYTES, &tmSW, nb * Cfg::BN, row, scf_bar(ss.slot()), pol);
                    sarmed |= 1u << ss.slot();
                    sarmed_phase = (sarmed_phase & ~(1u << ss.slot())) | (ss.parity() << ss.slot());
                    ss.next();
                }
            }
            if (!ok) {
                for (int s = 0; s < SCS; ++s)
                    if (sarmed & (1u << s))
                        bounded_wait(scf_bar(s), (sarmed_phase >> s) & 1u, nullptr, p.ctl,
                                     kSiteW4PDrainTma);
                if (leader) {
                    for (int s = 0; s < STAGES; ++s)
                        if (armed & (1u << s))
                            bounded_wait(full_bar(s), (armed_phase >> s) & 1u, nullptr, p.ctl,
                                         kSiteW4PDrainTma);
                } else {
                    // The partner's barrier cannot be polled from here: give the
                    // operand copies already issued a fixed time to land.
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < kPeerDrainNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (leader)
            Ring<STAGES> ps;
            Ring<ACC> as;
            bool ok = true;
            for (int t = pair; ok && t < ntiles; t += npairs) {
                for (int ks = 0; ok && ks < steps; ++ks) {
                    const bool lr = ks == p.num_ks;
                    if (!bounded_wait(full_bar(ps.slot()), ps.parity(), abort_flag, p.ctl,
                                      kSiteW4PMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
                    const int units = lr ? 1 : 2;
                    for (int h = 0; h < units; ++h) {
                        if (!bounded_wait(acce_bar(as.slot()), as.parity() ^ 1u, abort_flag, p.ctl,
                                          kSiteW4PMmaAcc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + static_cast<uint32_t>(as.slot() * Cfg::BN);
                        if (!lr) {
                            // one 64-wide block = bytes [64h, 64h + 64) of each row: 2 MMAs
#pragma unroll
                            for (int k = 0; k < 2; ++k)
                                tc_mma_pair<MmaKind::F8F6F4>(
                                    d, smem_desc_sw128(a_addr + 64u * h + 32u * k),
                                    smem_desc_sw128(b_addr + 64u * h + 32u * k), Cfg::IDESC,
                                    k > 0 ? 1u : 0u);
                        } else {
                            // 64 fp16 columns (32 low-rank + 32 zero-filled): 4 MMAs
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma_pair<MmaKind::F16>(d, smem_desc_sw128(a_addr + 32u * k),
                                                          smem_desc_sw128(b_addr + 32u * k),
                                                          Cfg::IDESC, k > 0 ? 1u : 0u);
                        }
                        tc_commit_pair(accf_bar(as.slot()), 0x3);
                        as.next();
                    }
                    if (!ok) break;
                    tc_commit_pair(empty_bar(ps.slot()), 0x3);
                    ps.next();
                }
            }
            tc_commit_pair(drain_bar, 0x1);
            bounded_wait(drain_bar, 0u, nullptr, p.ctl, kSiteW4PDrainMma);
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        // Warp (quad, colpart) owns TMEM lanes [32 quad, 32 quad + 32) and
        // columns [64 colpart, 64 colpart + 64) of the tile (three parts),
        // read as two 16-lane halves in the m16n8-accumulator layout: lane
        // (g, q) holds rows 32 quad + 16 hf + g (+ 8) and columns 8c + 2q (+ 1)
        // for the eight column groups c, so per block it needs 4 row scales
        // and 8 column-scale pairs, all from distinct shared-memory words.
        // Each 8-column group is loaded one ahead of the arithmetic.
        constexpr int NG = Cfg::EPI_COLS / 8;  // 8-column groups per warp
        const int quad = warp & 3;
        const int colpart = (warp - 2) >> 2;
        const int g = lane >> 2, q = lane & 3;
        const uint32_t lead_acce0 = mapa_shared(acce_bar(0), 0);
        Ring<ACC> as;
        Ring<SCS> ss;
        bool ok = true;
        for (int t = pair; ok && t < ntiles; t += npairs) {
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb, kGroupMPairs);
            // acc[hf][c][2e + d]: row 16 hf + g + 8e, column 8c + 2q + d
            float acc[2][NG][4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int c = 0; c < NG; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[hf][c][i] = 0.f;
            for (int ks = 0; ok && ks < steps; ++ks) {
                const int units = (ks == p.num_ks) ? 1 : 2;
                bool got = bounded_wait(scf_bar(ss.slot()), ss.parity(), abort_flag, p.ctl,
                                        kSiteW4PEpiScale);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const float* sx_s = reinterpret_cast<const float*>(sS + ss.slot() * Cfg::SC_BYTES);
                const float* sw_s = sx_s + 2 * Cfg::BM;
                for (int h = 0; h < units; ++h) {
                    got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl,
                                       kSiteW4PEpiAcc);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                           static_cast<uint32_t>(as.slot() * Cfg::BN +
                                                                 colpart * Cfg::EPI_COLS);
                    const float* sxr = sx_s + h * Cfg::BM + quad * 32 + g;
                    const float* swc = sw_s + h * Cfg::BN + colpart * Cfg::EPI_COLS + 2 * q;
                    // row-scale pairs (s, s) for rows g, g + 8, 16 + g, 24 + g
                    uint64_t sxp[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) sxp[k] = pack_f32x2(sxr[8 * k], sxr[8 * k]);
                    uint32_t rb[2][2][4];  // [buffer][half][x1 registers]
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tmem_ld_16x256b_x1(taddr + (static_cast<uint32_t>(16 * hf) << 16), rb[0][hf]);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < NG; ++c) {
                        if (c + 1 < NG) {
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
                                tmem_ld_16x256b_x1(taddr + (static_cast<uint32_t>(16 * hf) << 16) +
                                                       static_cast<uint32_t>(8 * (c + 1)),
                                                   rb[(c + 1) & 1][hf]);
                        } else {
                            // the buffer's last TMEM reads completed at the
                            // previous tcgen05.wait::ld: hand it back before
                            // the last group's arithmetic, with the arrival
                            // only (no cluster-scope release needed)
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster_relaxed(lead_acce0 + 8u * as.slot());
                        }
                        const uint64_t w = *reinterpret_cast<const uint64_t*>(swc + 8 * c);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float2 cs = unpack_f32x2(mul2(w, sxp[2 * hf + e]));
                                const uint32_t* rr = &rb[c & 1][hf][2 * e];
                                float* a = &acc[hf][c][2 * e];
                                a[0] = __fmaf_rn(__uint_as_float(rr[0]), cs.x, a[0]);
                                a[1] = __fmaf_rn(__uint_as_float(rr[1]), cs.y, a[1]);
                            }
                        if (c + 1 < NG) tmem_wait_ld();
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
                    const int row = mb * 2 * Cfg::BM + static_cast<int>(rank) * Cfg::BM + quad * 32 +
                                    16 * hf + 8 * e + g;
                    if (row >= p.M) continue;
                    __half* yrow = p.Y + static_cast<int64_t>(row) * p.ldy;
#pragma unroll
                    for (int c = 0; c < NG; ++c) {
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
    cluster_sync();  // neither CTA leaves while its partner may still use it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace qg

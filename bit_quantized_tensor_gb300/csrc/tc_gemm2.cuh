// Paired-CTA (cta_group::2) persistent tcgen05 GEMM for sm_103a: D = A . B^T.
//
// Two CTAs of a cluster share one 256 x 256 output tile: CTA r of the pair
// owns output rows [128 r, 128 r + 128) and loads its own 128 rows of A and
// its own 128 rows of B (half of the tile's columns) into a 7-stage ring;
// the leader CTA (rank 0) alone issues tcgen05.mma.cta_group::2 with M = 256,
// which reads both CTAs' operand halves and writes each CTA's 128 x 256 fp32
// accumulator into that CTA's TMEM.  Compared with one CTA per 128 x 256
// tile, every SM loads half as much B per MMA (less L2 traffic, more stages
// in the same shared memory) -- the "cross-CTA paired MMA" of
// "Warp-Specialized Kernel Implementation for W4A4 MatMul on Latest GPU
// Architectures", section 4, with the data flow re-divided as it describes.
//
// Synchronization (each role keeps its own position in each ring it walks):
//   full[s]      leader only; armed by the leader's producer for both CTAs'
//                bytes, completed by both CTAs' TMA loads (cta_group::2 TMA
//                signals the leader's barrier)
//   empty[s]     both CTAs; one multicast tcgen05.commit from the leader frees
//                stage s in both
//   acc_full[b]  both CTAs; multicast commit after a unit's last MMA
//   acc_empty[b] leader only; 8 epilogue warps of each CTA arrive remotely
//                (relaxed: the TMEM reads are complete at tcgen05.wait::ld)
// Every wait is bounded.  The CTAs leave only after a cluster barrier, so no
// CTA exits while its partner may still read its shared memory or signal it.
#pragma once
#include "tc_gemm.cuh"

namespace qg {

template <MmaKind KIND_, Epi EPI_>
struct Tc2Cfg {
    static constexpr MmaKind KIND = KIND_;
    static constexpr Epi EPI = EPI_;
    static constexpr int BM = 128;                      // rows per CTA (256 per pair)
    static constexpr int BN = 256;                      // columns of the pair's tile
    static constexpr int B_ROWS = BN / 2;               // B rows loaded per CTA
    static constexpr int ROW_BYTES = 128;
    static constexpr int ELEM_BYTES = (KIND == MmaKind::F16) ? 2 : 1;
    static constexpr int BK = ROW_BYTES / ELEM_BYTES;
    static constexpr int MMA_K = 32 / ELEM_BYTES;
    static constexpr int KSTEPS = BK / MMA_K;
    static constexpr int A_BYTES = BM * ROW_BYTES;      // 16 KB
    static constexpr int B_BYTES = B_ROWS * ROW_BYTES;  // 16 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int BARRIER_BYTES = 256;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int STAGES = (SMEM_LIMIT - BARRIER_BYTES - ALIGN_SLACK) / STAGE_BYTES;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BARRIER_BYTES + ALIGN_SLACK;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 32 * (2 + EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * ACC_BUFS + 1;
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, 2 * BM, BN);  // M = 256 across the pair

    static_assert(STAGES >= 2, "operand ring needs at least double buffering");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared-memory budget exceeded");
    static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM keeps all 512 TMEM columns free");
    static_assert(NUM_BARRIERS * 8 + 8 <= BARRIER_BYTES, "barrier area too small");
    static_assert(ACC_BUFS * BN <= TMEM_COLS, "TMEM budget exceeded");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

constexpr int kSitePairProdEmpty = 111;
constexpr int kSitePairMmaAcc = 112;
constexpr int kSitePairMmaFull = 113;
constexpr int kSitePairEpiAcc = 114;
constexpr int kSitePairDrainTma = 115;
constexpr int kSitePairDrainMma = 116;
constexpr uint64_t kPeerDrainNs = 1000000;  // 1 ms

template <class Cfg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::THREADS, 1)
    tc_gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const TcGemmParams p) {
    constexpr int STAGES = Cfg::STAGES;
    constexpr int ACC_BUFS = Cfg::ACC_BUFS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + ACC_BUFS + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * ACC_BUFS);
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
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * Cfg::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
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
    const int units = (p.num_kb + p.chunk_kb - 1) / p.chunk_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            Ring<STAGES> ps;
            uint32_t armed = 0, armed_phase = 0;
            const L2Policies pol = l2_policies(p.l2_mode);
            bool ok = true;
            for (int t = pair; ok && t < ntiles; t += npairs) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb, kGroupMPairs);
                const int arow = mb * 2 * Cfg::BM + static_cast<int>(rank) * Cfg::BM;
                const int brow = nb * Cfg::BN + static_cast<int>(rank) * Cfg::B_ROWS;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!bounded_wait(empty_bar(ps.slot()), ps.parity() ^ 1u, abort_flag, p.ctl,
                                      kSitePairProdEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t lead_full = mapa_shared(full_bar(ps.slot()), 0);
                    if (leader) {
                        mbar_arrive_expect_tx(full_bar(ps.slot()), 2 * Cfg::STAGE_BYTES);
                        armed |= 1u << ps.slot();
                        armed_phase = (armed_phase & ~(1u << ps.slot())) | (ps.parity() << ps.slot());
                    }
                    tma_load_2d_pair(smem_u32(sA + ps.slot() * Cfg::A_BYTES), &tmA, kb * Cfg::BK, arow,
                                     lead_full, pol.a);
                    tma_load_2d_pair(smem_u32(sB + ps.slot() * Cfg::B_BYTES), &tmB, kb * Cfg::BK, brow,
                                     lead_full, pol.b);
                    ps.next();
                }
            }
            if (!ok) {
                if (leader) {
                    // Both CTAs' copies of an armed stage complete the leader's barrier.
                    for (int s = 0; s < STAGES; ++s)
                        if (armed & (1u << s))
                            bounded_wait(full_bar(s), (armed_phase >> s) & 1u, nullptr, p.ctl,
                                         kSitePairDrainTma);
                } else {
                    // The partner's barrier cannot be polled from here: give the
                    // copies already issued a fixed time to land.
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
            Ring<ACC_BUFS> as;
            bool ok = true;
            for (int t = pair; ok && t < ntiles; t += npairs) {
                for (int u = 0; ok && u < units; ++u) {
                    const int kb0 = u * p.chunk_kb;
                    const int kb1 = min(p.num_kb, kb0 + p.chunk_kb);
                    if (!bounded_wait(acce_bar(as.slot()), as.parity() ^ 1u, abort_flag, p.ctl,
                                      kSitePairMmaAcc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as.slot() * Cfg::BN);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!bounded_wait(full_bar(ps.slot()), ps.parity(), abort_flag, p.ctl,
                                          kSitePairMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                        const uint32_t b_addr = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
#pragma unroll
                        for (int k = 0; k < Cfg::KSTEPS; ++k)
                            tc_mma_pair<Cfg::KIND>(d_tmem, smem_desc_sw128(a_addr + 32u * k),
                                                   smem_desc_sw128(b_addr + 32u * k), Cfg::IDESC,
                                                   (kb > kb0 || k > 0) ? 1u : 0u);
                        tc_commit_pair(empty_bar(ps.slot()), 0x3);
                        ps.next();
                    }
                    if (!ok) break;
                    tc_commit_pair(accf_bar(as.slot()), 0x3);
                    as.next();
                }
            }
            tc_commit_pair(drain_bar, 0x1);
            bounded_wait(drain_bar, 0u, nullptr, p.ctl, kSitePairDrainMma);
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int quad = warp & 3;
        const int colhalf = (warp - 2) >> 2;
        Ring<ACC_BUFS> as;
        bool ok = true;
        for (int t = pair; ok && t < ntiles; t += npairs) {
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb, kGroupMPairs);
            const int row = mb * 2 * Cfg::BM + static_cast<int>(rank) * Cfg::BM + quad * 32 + lane;
            const int col0 = nb * Cfg::BN + colhalf * 128;
            if constexpr (Cfg::EPI == Epi::S32) {
                int32_t sum[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) sum[i] = 0;
                for (int u = 0; u < units; ++u) {
                    bool got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl,
                                            kSitePairEpiAcc);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                           static_cast<uint32_t>(as.slot() * Cfg::BN + colhalf * 128);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(taddr + 32u * c, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            sum[32 * c + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                    // The buffer's TMEM reads completed at tcgen05.wait::ld, so the
                    // leader needs the arrival only, not a cluster-scope release.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(acce_bar(as.slot()), 0));
                    as.next();
                }
                if (!ok) break;
                if (row < p.M)
                    store_row_s32<128>(static_cast<int32_t*>(p.C) + static_cast<int64_t>(row) * p.ldc +
                                           col0,
                                       col0, p.N, sum, p.l2_mode == 2);
            } else {
                bool got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl,
                                        kSitePairEpiAcc);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                       static_cast<uint32_t>(as.slot() * Cfg::BN + colhalf * 128);
                float v[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + 32u * c, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(acce_bar(as.slot()), 0));
                as.next();
                if (row < p.M)
                    store_row_f16<128>(static_cast<__half*>(p.C) + static_cast<int64_t>(row) * p.ldc +
                                           col0,
                                       col0, p.N, v, p.bias, p.l2_mode == 2);
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

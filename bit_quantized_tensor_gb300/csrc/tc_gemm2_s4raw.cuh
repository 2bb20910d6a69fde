// Paired-CTA INT4 GEMM that reads the packed nibbles itself: C = A . B^T in
// int32, A and B in the "s4p" format (two signed 4-bit values per byte along
// K, low nibble = even k), no conversion pass before the kernel
// ("Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study on
// NVIDIA L4", abstract: exact INT4 GEMM; nibble sign extension on the way
// into shared memory).
//
// The tensor cores have no 4-bit integer MMA on sm_103a, so the nibbles are
// carried as e4m3 bytes (tcgen05 kind::f8f6f4).  Instead of sign-extending
// each nibble (a table lookup per four values), the transform warps use the
// offset-binary form: with u = n XOR 8 the value is q = u - 8, and the byte
// 0000uuuu read as e4m3 is exactly u * 2^-9 (u = 0..7 are the subnormals
// u * 2^-9, u = 8..15 the normals (8 + (u - 8)) * 2^-9).  So per 32-bit word
// of eight packed nibbles the even and odd nibbles become two words of four
// bytes with three logic operations, and the MMA accumulates
//     D[m][n] = sum_k u_a[m][k] u_b[n][k] * 2^-18        (exact in fp32 while
//                                                          225 K < 2^24)
// from which the epilogue recovers
//     C[m][n] = 2^18 D[m][n] - 8 RA[m] - 8 RB[n] + 64 K,
//     RA[m] = sum_k u_a[m][k],  RB[n] = sum_k u_b[n][k].
// The K order inside each 32-value chunk is permuted (even nibbles first) in
// the same way for A and B, which leaves every dot product unchanged.  K
// values past the end of the matrix are written as u = 0 (zero products) and
// left out of the sums.
//
// Roles (23 warps):
//   warp 0       TMEM owner; lane 0 of the leader CTA issues the paired MMAs
//   warp 1       lane 0: TMA producer of the packed bytes (this CTA's 128 rows
//                of A and of B per 128-wide K stage) into a RAW_STAGES ring
//   warps 2..17  transform: packed bytes (shared memory) -> e4m3 bytes in the
//                128-byte swizzled K-major MMA stage; row sums of the rows
//                they convert
//   warp 18      signaler: forwards each finished stage to the MMA
//   warps 19..22 epilogue: TMEM -> registers, the correction, int32 stores
//                (one warp per TMEM lane quadrant, all 256 columns; it runs
//                once per tile, under the next tile's K loop)
// The packed bytes come in by TMA rather than by per-thread global loads: a
// global load costs the load/store pipe one wavefront per 32-byte sector,
// a shared-memory read one per 128 bytes, and with global loads that pipe
// was the bottleneck (1.95 POPS at 8192^3).
// Synchronization:
//   raw_full/    per CTA: the producer's TMA completes raw_full; the transform
//   raw_empty    warps arrive on raw_empty once they have used the bytes
//   slot s       named barrier 1 + s: the transform threads arrive (bar.arrive,
//                after their stores and fence.proxy.async) and the signaler
//                waits
//   full[s]      leader only: armed by the leader's signaler (arrive with 32
//                expected bytes); each CTA's signaler then issues a 16-byte
//                shared-memory bulk copy into the leader that completes on it.
//                The async-proxy completion orders the stage's (fenced) stores
//                before the MMA as a TMA load's completion would; an arrive
//                with release at cluster scope costs about a microsecond.
//   empty[s]     both CTAs; one multicast commit from the leader
//   accf/acce    as in tc_gemm2_kernel
//   sums_full    per CTA; the transform warps of both CTAs arrive after
//                storing this tile's row sums of A (own CTA) and B (both
//                halves: each CTA writes its half into both CTAs)
//   sums_empty   per CTA; the epilogue warps of both CTAs arrive after
//                reading them
// Every wait is bounded; the CTAs leave only after a cluster barrier.
#pragma once
#include "tc_gemm2.cuh"

namespace qg {

struct S4RawCfg {
    static constexpr int BM = 128;                        // rows per CTA (256 per pair)
    static constexpr int BN = 256;                        // columns of the pair's tile
    static constexpr int B_ROWS = BN / 2;                 // B rows converted per CTA
    static constexpr int BK = 128;                        // k per stage: one 128-byte e4m3 row
    static constexpr int RAW_ROW = BK / 2;                // packed bytes per row per stage
    static constexpr int KSTEPS = 4;                      // MMAs per stage (K = 32 each)
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = B_ROWS * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int RAW_A_BYTES = BM * RAW_ROW;      // packed bytes of a stage (A, B halves)
    static constexpr int RAW_B_BYTES = B_ROWS * RAW_ROW;
    static constexpr int RAW_BYTES = RAW_A_BYTES + RAW_B_BYTES;
    static constexpr int STAGES = 5;                      // e4m3 MMA operand ring
    static constexpr int RAW_STAGES = 4;                  // packed-byte ring
    static constexpr int SUMS_BYTES = (BM + BN) * 4;      // RA of this CTA's rows, RB of the tile
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int BARRIER_BYTES = 256;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + RAW_STAGES * RAW_BYTES + SUMS_BYTES + BARRIER_BYTES + ALIGN_SLACK;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int PROD_WARP = 1;
    static constexpr int XF_WARP0 = 2, XF_WARPS = 16;
    static constexpr int SIG_WARP = XF_WARP0 + XF_WARPS;  // forwards each stage to the MMA
    static constexpr int EPI_WARP0 = SIG_WARP + 1, EPI_WARPS = 4;  // one per TMEM lane quadrant
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr int XF_THREADS = 32 * XF_WARPS;
    // each transform thread: one 16-byte quarter of a 64-byte raw row segment
    static constexpr int ROW_SLOTS = XF_THREADS / 4;      // rows covered per pass
    static constexpr int A_TASKS = BM / ROW_SLOTS;        // A rows per thread per stage
    static constexpr int B_TASKS = B_ROWS / ROW_SLOTS;
    static constexpr int TASKS = A_TASKS + B_TASKS;
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * RAW_STAGES + 2 * ACC_BUFS + 3;
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, 2 * BM, BN);  // e4m3 x e4m3, M = 256
    static constexpr int64_t MAX_K = 65536;               // 225 * K < 2^24: exact fp32 sums

    static_assert(STAGES >= 4 && RAW_STAGES >= 3, "rings too shallow");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared-memory budget exceeded");
    static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM keeps all 512 TMEM columns free");
    static_assert(NUM_BARRIERS * 8 + 8 + 16 + 32 <= BARRIER_BYTES, "barrier area too small");
    static_assert(ACC_BUFS * BN <= TMEM_COLS, "TMEM budget exceeded");
    static_assert(A_TASKS * ROW_SLOTS == BM && B_TASKS * ROW_SLOTS == B_ROWS, "row split");
    static_assert(225 * MAX_K < (1 << 24), "offset-binary partial sums stay exact in fp32");
    static_assert(STAGES + 1 <= 16, "one named barrier per ring slot (ids 1..STAGES)");
};

struct S4RawParams {
    int M, N, K;
    int num_kb;                 // ceil(K / 128)
    int32_t* C;
    int64_t ldc;
    Ctl ctl;
};

enum S4RawSite : int {
    kSiteS4Prod = 138,
    kSiteS4XfRaw = 139,
    kSiteS4Drain = 130,
    kSiteS4XfEmpty = 131,
    kSiteS4XfSums = 132,
    kSiteS4MmaAcc = 133,
    kSiteS4MmaFull = 134,
    kSiteS4EpiAcc = 135,
    kSiteS4EpiSums = 136,
    kSiteS4DrainMma = 137,
};

// Named CTA barriers: `count` threads in all (whole warps); arrive does not wait.
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Eight packed nibbles -> the even ones (k = 0, 2, 4, 6) and the odd ones
// (k = 1, 3, 5, 7) as offset-binary bytes u = n XOR 8.
__device__ __forceinline__ void split_offset(uint32_t w, uint32_t& even, uint32_t& odd) {
    even = (w ^ 0x88888888u) & 0x0F0F0F0Fu;
    odd = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(S4RawCfg::THREADS, 1)
    tc_gemm2_s4raw_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const S4RawParams p) {
    using Cfg = S4RawCfg;
    constexpr int STAGES = Cfg::STAGES, ACC = Cfg::ACC_BUFS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t* sRaw = smem + STAGES * Cfg::STAGE_BYTES;  // RAW_STAGES x (A rows, B rows) x 64 bytes
    int32_t* sRA = reinterpret_cast<int32_t*>(sRaw + Cfg::RAW_STAGES * Cfg::RAW_BYTES);
    int32_t* sRB = sRA + Cfg::BM;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRB + Cfg::BN);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + ACC + b); };
    constexpr int RS = Cfg::RAW_STAGES;
    auto rawf_bar = [&](int r) { return bar0 + 8u * (2 * STAGES + 2 * ACC + r); };
    auto rawe_bar = [&](int r) { return bar0 + 8u * (2 * STAGES + 2 * ACC + RS + r); };
    const uint32_t sumsf_bar = bar0 + 8u * (2 * STAGES + 2 * ACC + 2 * RS);
    const uint32_t sumse_bar = sumsf_bar + 8u;
    const uint32_t drain_bar = sumse_bar + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // 16-byte source and destination of the stage-ready bulk copies
    const uint32_t sig_src = (smem_u32(tmem_holder + 2) + 15u) & ~15u;
    const uint32_t sig_dst = sig_src + 16u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < ACC; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * Cfg::EPI_WARPS);
        }
        for (int r = 0; r < RS; ++r) {
            mbar_init(rawf_bar(r), 1);
            mbar_init(rawe_bar(r), Cfg::XF_WARPS);
        }
        mbar_init(sumsf_bar, 2 * Cfg::XF_WARPS);
        mbar_init(sumse_bar, 2 * Cfg::EPI_WARPS);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 0) tmem_alloc_pair(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialized and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int num_m = (p.M + 2 * Cfg::BM - 1) / (2 * Cfg::BM);
    const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int ntiles = num_m * num_n;
    const int kbytes = p.K / 2;  // packed bytes per row

    if (warp == 0) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (leader)
            Ring<STAGES> ps;
            Ring<ACC> as;
            bool ok = true;
            for (int t = pair; ok && t < ntiles; t += npairs) {
                if (!bounded_wait(acce_bar(as.slot()), as.parity() ^ 1u, abort_flag, p.ctl,
                                  kSiteS4MmaAcc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as.slot() * Cfg::BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    // completed by async-proxy transfers (the signalers' bulk
                    // copies), as a TMA-fed ring is: CTA-scope wait
                    if (!bounded_wait(full_bar(ps.slot()), ps.parity(), abort_flag, p.ctl, kSiteS4MmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
#pragma unroll
                    for (int k = 0; k < Cfg::KSTEPS; ++k)
                        tc_mma_pair<MmaKind::F8F6F4>(d_tmem, smem_desc_sw128(a_addr + 32u * k),
                                                     smem_desc_sw128(b_addr + 32u * k), Cfg::IDESC,
                                                     (kb > 0 || k > 0) ? 1u : 0u);
                    tc_commit_pair(empty_bar(ps.slot()), 0x3);
                    ps.next();
                }
                if (!ok) break;
                tc_commit_pair(accf_bar(as.slot()), 0x3);
                as.next();
            }
            tc_commit_pair(drain_bar, 0x1);
            bounded_wait(drain_bar, 0u, nullptr, p.ctl, kSiteS4DrainMma);
        }
    } else if (warp == Cfg::PROD_WARP) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            Ring<RS> rr;
            uint32_t armed = 0, armed_phase = 0;
            const uint64_t pol = l2_policy_evict_normal();
            bool ok = true;
            for (int t = pair; ok && t < ntiles; t += npairs) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb, kGroupMPairs);
                const int arow = mb * 2 * Cfg::BM + static_cast<int>(rank) * Cfg::BM;
                const int brow = nb * Cfg::BN + static_cast<int>(rank) * Cfg::B_ROWS;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!bounded_wait(rawe_bar(rr.slot()), rr.parity() ^ 1u, abort_flag, p.ctl, kSiteS4Prod)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(rawf_bar(rr.slot()), Cfg::RAW_BYTES);
                    armed |= 1u << rr.slot();
                    armed_phase = (armed_phase & ~(1u << rr.slot())) | (rr.parity() << rr.slot());
                    uint8_t* dst = sRaw + rr.slot() * Cfg::RAW_BYTES;
                    // 64 packed bytes of each row (k = 128 kb ... 128 kb + 127); rows
                    // and bytes past the matrix are filled with zeros
                    tma_load_2d(smem_u32(dst), &tmA, kb * Cfg::RAW_ROW, arow, rawf_bar(rr.slot()), pol);
                    tma_load_2d(smem_u32(dst + Cfg::RAW_A_BYTES), &tmB, kb * Cfg::RAW_ROW, brow,
                                rawf_bar(rr.slot()), pol);
                    rr.next();
                }
            }
            if (!ok)
                for (int r = 0; r < RS; ++r)
                    if (armed & (1u << r))
                        bounded_wait(rawf_bar(r), (armed_phase >> r) & 1u, nullptr, p.ctl, kSiteS4Drain);
        }
    } else if (warp < Cfg::SIG_WARP) {
        // ---------------------------------------------------- transform (both CTAs)
        // Thread x: quarter q (16 packed bytes = 32 values) of row slot rs;
        // it converts rows rs + ROW_SLOTS * i of this CTA's A and B halves.
        const int x = threadIdx.x - 32 * Cfg::XF_WARP0;
        const int rs = x >> 2, q = x & 3;
        const uint32_t peer_rb = mapa_shared(smem_u32(sRB), rank ^ 1u);
        const uint32_t peer_sumsf = mapa_shared(sumsf_bar, rank ^ 1u);
        Ring<STAGES> ps;
        Ring<RS> rr;
        uint32_t sums_lap = 0;
        int signaled = 0;  // stages this thread has arrived on (the signaler counts on all)
        int32_t rsum[Cfg::TASKS];
        bool ok = true;
        for (int t = pair; ok && t < ntiles; t += npairs) {
#pragma unroll
            for (int i = 0; i < Cfg::TASKS; ++i) rsum[i] = 0;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                bool got = bounded_wait(rawf_bar(rr.slot()), rr.parity(), abort_flag, p.ctl, kSiteS4XfRaw);
                if (got) got = bounded_wait(empty_bar(ps.slot()), ps.parity() ^ 1u, abort_flag, p.ctl,
                                            kSiteS4XfEmpty);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const bool inside = kb * Cfg::RAW_ROW + 16 * q < kbytes;
                const uint8_t* raw = sRaw + rr.slot() * Cfg::RAW_BYTES;
                uint4 w[Cfg::TASKS];
#pragma unroll
                for (int i = 0; i < Cfg::TASKS; ++i) {
                    const int r = rs + Cfg::ROW_SLOTS * (i < Cfg::A_TASKS ? i : i - Cfg::A_TASKS);
                    const uint8_t* src = raw + (i < Cfg::A_TASKS ? 0 : Cfg::RAW_A_BYTES) + r * Cfg::RAW_ROW + 16 * q;
                    w[i] = *reinterpret_cast<const uint4*>(src);
                }
#pragma unroll
                for (int i = 0; i < Cfg::TASKS; ++i) {
                    uint32_t e0, o0, e1, o1, e2, o2, e3, o3;
                    split_offset(w[i].x, e0, o0);
                    split_offset(w[i].y, e1, o1);
                    split_offset(w[i].z, e2, o2);
                    split_offset(w[i].w, e3, o3);
                    if (inside) {
                        const uint32_t bytes = (e0 + o0) + (e1 + o1) + (e2 + o2) + (e3 + o3);  // <= 120 each
                        rsum[i] = static_cast<int32_t>(__dp4a(bytes, 0x01010101u, static_cast<uint32_t>(rsum[i])));
                    } else {
                        // past the end of K: zero products, nothing in the sums
                        e0 = o0 = e1 = o1 = e2 = o2 = e3 = o3 = 0u;
                    }
                    const int r = rs + Cfg::ROW_SLOTS * (i < Cfg::A_TASKS ? i : i - Cfg::A_TASKS);
                    uint8_t* base = (i < Cfg::A_TASKS) ? sA + ps.slot() * Cfg::A_BYTES : sB + ps.slot() * Cfg::B_BYTES;
                    // 32 output bytes = 16-byte chunks 2q and 2q + 1 of the 128-byte
                    // row r, placed by the 128-byte swizzle (chunk c at c ^ (r & 7))
                    uint8_t* row = base + r * 128;
                    *reinterpret_cast<uint4*>(row + (((2 * q) ^ (r & 7)) << 4)) = make_uint4(e0, o0, e1, o1);
                    *reinterpret_cast<uint4*>(row + (((2 * q + 1) ^ (r & 7)) << 4)) = make_uint4(e2, o2, e3, o3);
                }
                // the packed bytes have been used: the producer may refill the slot
                __syncwarp();
                if (lane == 0) mbar_arrive(rawe_bar(rr.slot()));
                rr.next();
                fence_proxy_async_smem();
                named_bar_arrive(1 + ps.slot(), Cfg::XF_THREADS + 32);
                ps.next();
                ++signaled;
            }
            if (!ok) break;
            // row sums of this tile: the four quarters of a row are lanes 4j..4j+3
#pragma unroll
            for (int i = 0; i < Cfg::TASKS; ++i) {
                rsum[i] += __shfl_xor_sync(0xffffffffu, rsum[i], 1);
                rsum[i] += __shfl_xor_sync(0xffffffffu, rsum[i], 2);
            }
            bool got = bounded_wait_cluster(sumse_bar, sums_lap ^ 1u, abort_flag, p.ctl, kSiteS4XfSums);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            if (q == 0) {
#pragma unroll
                for (int i = 0; i < Cfg::TASKS; ++i) {
                    if (i < Cfg::A_TASKS) {
                        sRA[rs + Cfg::ROW_SLOTS * i] = rsum[i];
                    } else {
                        // this CTA's half of the tile's B rows, in both CTAs
                        const int c = static_cast<int>(rank) * Cfg::B_ROWS + rs + Cfg::ROW_SLOTS * (i - Cfg::A_TASKS);
                        sRB[c] = rsum[i];
                        st_shared_cluster_u32(peer_rb + 4u * c, static_cast<uint32_t>(rsum[i]));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sumsf_bar);
                mbar_arrive_cluster(peer_sumsf);  // release: orders the remote stores above
            }
            sums_lap ^= 1u;
        }
        // after an abort: the remaining arrivals, so that the signaler's
        // (unbounded) named-barrier waits all complete
        const int stages_total = p.num_kb * ((ntiles - pair + npairs - 1) / npairs);
        for (; pair < ntiles && signaled < stages_total; ++signaled) {
            named_bar_arrive(1 + ps.slot(), Cfg::XF_THREADS + 32);
            ps.next();
        }
    } else if (warp == Cfg::SIG_WARP) {
        // ---------------------------------------------------- signaler (both CTAs)
        const uint32_t lead_full0 = mapa_shared(full_bar(0), 0);
        Ring<STAGES> ps;
        const int stages_total = p.num_kb * ((ntiles - pair + npairs - 1) / npairs);
        const uint32_t lead_dst = mapa_shared(sig_dst, 0);
        bool aborted = false;
        for (int i = 0; i < (pair < ntiles ? stages_total : 0); ++i) {
            named_bar_sync(1 + ps.slot(), Cfg::XF_THREADS + 32);
            if (*abort_flag) {
                aborted = true;
                break;
            }
            if (lane == 0) {
                if (leader) mbar_arrive_expect_tx(full_bar(ps.slot()), 32);
                bulk_copy_s2s_cluster(lead_dst, sig_src, 16, lead_full0 + 8u * ps.slot());
            }
            ps.next();
        }
        if (aborted) {
            // give the 16-byte copies already issued a fixed time to land
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < kPeerDrainNs) {
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int quad = warp & 3;
        const uint32_t lead_acce0 = mapa_shared(acce_bar(0), 0);
        const uint32_t peer_sumse = mapa_shared(sumse_bar, rank ^ 1u);
        Ring<ACC> as;
        uint32_t sums_lap = 0;
        const int32_t k64 = 64 * p.K;
        bool ok = true;
        for (int t = pair; ok && t < ntiles; t += npairs) {
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb, kGroupMPairs);
            const int row = mb * 2 * Cfg::BM + static_cast<int>(rank) * Cfg::BM + quad * 32 + lane;
            const int col0 = nb * Cfg::BN;
            bool got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl, kSiteS4EpiAcc);
            if (got) got = bounded_wait_cluster(sumsf_bar, sums_lap, abort_flag, p.ctl, kSiteS4EpiSums);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int32_t base_m = k64 - 8 * sRA[quad * 32 + lane];
            const int32_t* rb = sRB;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(as.slot() * Cfg::BN);
            int32_t* crow = p.C + static_cast<int64_t>(row) * p.ldc + col0;
#pragma unroll 1
            for (int c = 0; c < Cfg::BN / 16; ++c) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(taddr + 16u * c, r);
                tmem_wait_ld();
                if (c == Cfg::BN / 16 - 1) {
                    // all of this warp's TMEM reads are complete: hand the buffer
                    // and the sums back before the stores
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(lead_acce0 + 8u * as.slot());
                }
                int32_t v[16];
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const int4 b4 = *reinterpret_cast<const int4*>(rb + 16 * c + i);  // broadcast
                    v[i] = __float2int_rn(__uint_as_float(r[i]) * 262144.f) + base_m - 8 * b4.x;
                    v[i + 1] = __float2int_rn(__uint_as_float(r[i + 1]) * 262144.f) + base_m - 8 * b4.y;
                    v[i + 2] = __float2int_rn(__uint_as_float(r[i + 2]) * 262144.f) + base_m - 8 * b4.z;
                    v[i + 3] = __float2int_rn(__uint_as_float(r[i + 3]) * 262144.f) + base_m - 8 * b4.w;
                }
                if (c == Cfg::BN / 16 - 1) {
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(sumse_bar);
                        mbar_arrive_cluster(peer_sumse);
                    }
                }
                if (row < p.M) store_row_s32<16>(crow + 16 * c, col0 + 16 * c, p.N, v);
            }
            as.next();
            sums_lap ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while its partner may still use it
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace qg

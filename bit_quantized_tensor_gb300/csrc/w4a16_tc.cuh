// W4A16 on the tensor cores for batches above the decode shapes:
//
//   Y[m][n] = sum_k X[m][k] * (s[n][k / 128] * q[n][k])
//
// ("fused-int4-gemm-sm75" README: weight-only int4 with group-128 scales.)
// A cluster of 4 CTAs owns 128 output columns (128 weight rows) for up to 128
// batch rows and splits K four ways: CTA r handles a contiguous quarter of
// the K groups.  Per K stage a CTA
//  - TMA-loads its 128-row tile of X (and, in the ring form, the packed
//    weight rows of the stage); in the resident form (a quarter of at most 8
//    groups, K <= 4096) all packed rows of the quarter (64 KB) are loaded
//    before the programmatic dependent wait and only X streams;
//  - dequantizes in registers, as the SM75 page does: each weight becomes
//    the fp16 product q * s (rounded once, at most 2^-11 of the weight); the
//    128 rows go to the 128-byte-swizzled K-major layout of the MMA's B
//    operand.  Groups of warps take alternate stages: one warp's pass over a
//    stage is latency-bound (shared-memory loads, the proxy fence, the
//    barrier arrival), so two stages in flight double the transform rate;
//  - issues tcgen05.mma kind::f16 M=128 N=128 (one thread) into a 128-column
//    TMEM accumulator.
// What paces the loop (globaltimer traces of a chain of calls, M = 128,
// N = K = 4096): one such MMA runs in about 30 ns, but each stage also costs
// the issuing thread about 200 ns of barrier waits, fences and commits, so
// the resident form takes 128-wide stages (8 MMAs and one commit each; the X
// and B rings have one depth, so one commit frees both slots): 12.2 -> 10.6
// us per call.  With MMAs skipped the transform alone takes about as long as
// the loop now does.  An exact alternative to the rounded q * s (two exact
// fp16 rows, q * s_hi and q * s_lo, with s_hi the scale with its three
// lowest mantissa bits cleared) doubles the B operand and was slower by that.
// At the end every CTA stores its 128 x 128 fp32
// partial tile in shared memory and, once every CTA of the cluster is past
// its K loop, bulk-copies rows [32 r, 32 r + 32) of it into CTA r's shared
// memory (the copy engine signals CTA r's barrier with the byte count); CTA r
// adds the four partials of its rows and stores them as fp16.  The copies
// run at about 20 bytes per clock (1.4 us for 50 KB; 16-byte copies take
// 0.26 us); sending the rows from registers with 16-byte st.async stores
// (2.7 us) or plain remote stores and a release/acquire cluster barrier
// (3.0 us) was slower.  Both cluster barriers are relaxed: the copies carry
// their own completion, and a barrier with release semantics cost about half
// a microsecond here.  Weight rows and scales are fetched before the
// programmatic dependent wait; X after it.  Every wait is bounded.  Scales
// must stay below 8188 in magnitude (8 * s must be a finite fp16).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "qg_internal.h"
#include "qg_ptx.cuh"

namespace qg {

// Execution barrier over all threads of the cluster, without memory ordering.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\nbarrier.cluster.wait.aligned;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to the
// shared memory of a CTA of the cluster; completes on that CTA's mbarrier.
__device__ __forceinline__ void bulk_copy_s2cluster(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                    uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

// WRES: the CTA's packed weights stay resident.  When a K quarter holds at
// most 8 groups (K <= 4096) all of its packed rows (64 KB) are bulk-loaded
// before the programmatic dependent wait, each ring stage's rows on a barrier
// of their own, so the transform never waits on a refill and the first B slots
// are dequantized before X (the previous kernel's output) may be read; only
// X streams through the ring.  Otherwise X and the packed rows share one
// ring, refilled as the MMA frees it.
template <bool WRES_, int STAGES_, int BSLOTS_, int MAXG_, int SUB_, int XGROUPS_>
struct W16TcCfgT {
    static constexpr bool WRES = WRES_;
    static constexpr int KSPLIT = 4;                    // CTAs per cluster, one K quarter each
    static constexpr int BM = 128;                      // batch rows per launch
    static constexpr int BN = 128;                      // weight rows (output columns) per cluster
    static constexpr int BK = 64;                       // K per sub-tile: 128 bytes of fp16
    // 64-wide sub-tiles per ring stage: a stage's MMAs (4 per sub-tile) share
    // one pair of barrier waits and one commit, which cost the issuing
    // thread more than the MMAs themselves
    static constexpr int SUB = SUB_;
    static constexpr int X_SUB = BM * BK * 2;           // 16 KB
    static constexpr int B_ROWS = BN;                   // q * s rows
    static constexpr int B_SUB = B_ROWS * BK * 2;       // 16 KB fp16 operand
    static constexpr int W_SUB = BN * BK / 2;           // 4 KB packed nibbles
    static constexpr int X_BYTES = SUB * X_SUB, B_BYTES = SUB * B_SUB, W_BYTES = SUB * W_SUB;
    static constexpr int STAGES = STAGES_;              // X (+ packed-weight) ring (memory latency)
    static constexpr int BSLOTS = BSLOTS_;              // B operand ring (transform -> MMA)
    static constexpr int MAX_SLICE_GROUPS = MAXG_;      // K groups per quarter, at most
    static constexpr int W_SLOTS = WRES ? 2 * MAX_SLICE_GROUPS / SUB : STAGES;  // packed stages held
    // X and B rings of one depth move together: one commit per stage frees
    // both slots (a tcgen05.commit costs the issuing thread about as much as
    // an MMA: 30 ns)
    static constexpr bool ONE_FREE = STAGES == BSLOTS;
    static constexpr int XFORM_WARPS = 16;
    static constexpr int XFORM_GROUPS = XGROUPS_;       // groups of warps on alternate stages
    static constexpr int GROUP_WARPS = XFORM_WARPS / XFORM_GROUPS;
    static constexpr int THREADS = 32 * (2 + XFORM_WARPS);  // producer, MMA, transform/epilogue
    static constexpr int TMEM_COLS = 128;
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * BSLOTS + 2 + (WRES ? W_SLOTS : 0);
    static constexpr int BAR_BYTES = 512;
    static constexpr int SCALE_BYTES = BN * MAX_SLICE_GROUPS * 2;
    static constexpr int RING_BYTES = STAGES * X_BYTES + W_SLOTS * W_BYTES + BSLOTS * B_BYTES;
    static constexpr int SMEM_BYTES = RING_BYTES + BAR_BYTES + SCALE_BYTES + 1024;
    static constexpr int RED_STRIDE = BN + 4;           // floats per partial-tile row (bank spread)
    static constexpr int SLICE_ROWS = BM / KSPLIT;      // output rows each CTA finishes
    static constexpr int SLICE_BYTES = SLICE_ROWS * RED_STRIDE * 4;  // one bulk copy
    static constexpr int RX_OFF = (BM * RED_STRIDE * 4 + 1023) / 1024 * 1024;  // received partials
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, BM, B_ROWS);

    static_assert(X_SUB % 1024 == 0 && B_SUB % 1024 == 0,
                  "swizzle atoms need 1 KB alignment");
    static_assert(SUB == 1 || SUB == 2, "a stage is one or two 64-wide sub-tiles (at most one K group)");
    static constexpr int TPR = 32 * GROUP_WARPS / BN;   // transform threads per weight row
    static constexpr int WPT = 8 / TPR;                 // packed 32-bit words per thread per sub-tile
    static_assert(TPR * BN == 32 * GROUP_WARPS && (WPT == 2 || WPT == 4), "transform thread mapping");
    static_assert(NUM_BARRIERS * 8 + 16 <= BAR_BYTES, "barrier area too small");
    static_assert(SMEM_BYTES <= 232448, "shared-memory budget exceeded");
    static_assert(RX_OFF + KSPLIT * SLICE_BYTES <= RING_BYTES, "partial tiles reuse the rings");
    static_assert(SLICE_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
};
using W16TcCfg = W16TcCfgT<false, 8, 3, 64, 1, 2>;    // any K up to 32768
using W16TcResCfg = W16TcCfgT<true, 2, 2, 8, 2, 2>;   // K <= 4096: 128-wide stages

struct W16TcParams {
    int M, N, K;
    int m0;           // first batch row of this launch
    __half* Y;
    int64_t ldy;
    const __half* S;  // N x K/128 group scales
    Ctl ctl;
};

enum W16TcSite : int {
    kSiteW16TcEmpty = 311,
    kSiteW16TcFull = 312,
    kSiteW16TcReady = 313,
    kSiteW16TcXform = 314,
    kSiteW16TcAcc = 315,
    kSiteW16TcRx = 316,
};

template <class Cfg>
__global__ void __cluster_dims__(Cfg::KSPLIT, 1, 1) __launch_bounds__(Cfg::THREADS, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const W16TcParams p) {
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int NB = Cfg::BSLOTS;
    uint8_t* sX = smem;                                   // S x 16 KB
    uint8_t* sB = sX + S * Cfg::X_BYTES;                  // NB x 32 KB
    uint8_t* sW = sB + NB * Cfg::B_BYTES;                 // W_SLOTS x 4 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(sW + Cfg::W_SLOTS * Cfg::W_BYTES);
    unsigned short* sS = reinterpret_cast<unsigned short*>(reinterpret_cast<uint8_t*>(bars) + Cfg::BAR_BYTES);
    float* red = reinterpret_cast<float*>(smem);          // partial tile, after the K loop
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };             // X (+ W) of stage s landed
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };      // MMA done with stage s
    auto ready_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };  // B slot b written
    auto bfree_bar = [&](int b) {  // MMA done with B slot b
        return Cfg::ONE_FREE ? empty_bar(b) : bar0 + 8u * (2 * S + NB + b);
    };
    const uint32_t accf_bar = bar0 + 8u * (2 * S + 2 * NB);
    const uint32_t rx_bar = bar0 + 8u * (2 * S + 2 * NB + 1);  // partials of this CTA's rows arrived
    auto wfull_bar = [&](int i) { return bar0 + 8u * (2 * S + 2 * NB + 2 + i); };  // WRES: packed stage i
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();              // K quarter of this CTA
    const int n0 = static_cast<int>(blockIdx.x / Cfg::KSPLIT) * Cfg::BN;
    const int G = p.K / 128;
    const int gq = (G + Cfg::KSPLIT - 1) / Cfg::KSPLIT;   // groups per quarter
    const int g_beg = min(G, static_cast<int>(rank) * gq), g_end = min(G, g_beg + gq);
    const int ng = g_end - g_beg;
    const int num_kb = 2 * ng / Cfg::SUB;                 // ring stages of this quarter
    const int kb0 = 2 * g_beg;                            // first global 64-wide sub-tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(ready_bar(b), Cfg::GROUP_WARPS);  // one group transforms a stage
            if constexpr (!Cfg::ONE_FREE) mbar_init(bfree_bar(b), 1);
        }
        mbar_init(accf_bar, 1);
        mbar_init(rx_bar, 1);
        if constexpr (Cfg::WRES)
            for (int i = 0; i < Cfg::W_SLOTS; ++i) mbar_init(wfull_bar(i), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_launch_dependents();

    bool ok = true;  // per role; a timed-out role skips its remaining work
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            const int pre = num_kb < S ? num_kb : S;
            constexpr uint32_t kStageTx = Cfg::WRES ? Cfg::X_BYTES : Cfg::X_BYTES + Cfg::W_BYTES;
            if constexpr (Cfg::WRES) {
                for (int i = 0; i < num_kb; ++i) {  // every packed stage, before the wait
                    mbar_arrive_expect_tx(wfull_bar(i), Cfg::W_BYTES);
                    for (int h = 0; h < Cfg::SUB; ++h)
                        tma_load_2d(smem_u32(sW + i * Cfg::W_BYTES + h * Cfg::W_SUB), &tmW,
                                    (kb0 + Cfg::SUB * i + h) * (Cfg::BK / 2), n0, wfull_bar(i), pol_w);
                }
            } else {
                for (int i = 0; i < pre; ++i) {  // weights of the first stages before the wait
                    mbar_arrive_expect_tx(full_bar(i), kStageTx);
                    for (int h = 0; h < Cfg::SUB; ++h)
                        tma_load_2d(smem_u32(sW + i * Cfg::W_BYTES + h * Cfg::W_SUB), &tmW,
                                    (kb0 + Cfg::SUB * i + h) * (Cfg::BK / 2), n0, full_bar(i), pol_w);
                }
            }
            pdl_wait_prior_grid();  // X may be the previous kernel's output
            // the previous kernel wrote X with ordinary stores; these loads
            // are TMA (async proxy) reads
            asm volatile("fence.proxy.async.global;" ::: "memory");
            for (int i = 0; i < pre; ++i) {
                if constexpr (Cfg::WRES) mbar_arrive_expect_tx(full_bar(i), kStageTx);
                for (int h = 0; h < Cfg::SUB; ++h)
                    tma_load_2d(smem_u32(sX + i * Cfg::X_BYTES + h * Cfg::X_SUB), &tmX,
                                (kb0 + Cfg::SUB * i + h) * Cfg::BK, p.m0, full_bar(i), pol_x);
            }
            for (int i = pre; i < num_kb; ++i) {
                const int s = i % S;
                const uint32_t ph = static_cast<uint32_t>(i / S - 1) & 1u;  // round just finished
                if (!bounded_wait(empty_bar(s), ph, abort_flag, p.ctl, kSiteW16TcEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(s), kStageTx);
                for (int h = 0; h < Cfg::SUB; ++h) {
                    const int kb = kb0 + Cfg::SUB * i + h;
                    if constexpr (!Cfg::WRES)
                        tma_load_2d(smem_u32(sW + s * Cfg::W_BYTES + h * Cfg::W_SUB), &tmW, kb * (Cfg::BK / 2),
                                    n0, full_bar(s), pol_w);
                    tma_load_2d(smem_u32(sX + s * Cfg::X_BYTES + h * Cfg::X_SUB), &tmX, kb * Cfg::BK, p.m0,
                                full_bar(s), pol_x);
                }
            }
            if (!ok) {
                // copies already issued get a fixed time to land before the
                // shared memory is reused or released
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            for (int i = 0; i < num_kb; ++i) {
                const int s = i % S, b = i % NB;
                const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
                const uint32_t bph = static_cast<uint32_t>(i / NB) & 1u;
                if (!bounded_wait(full_bar(s), ph, abort_flag, p.ctl, kSiteW16TcFull) ||
                    !bounded_wait(ready_bar(b), bph, abort_flag, p.ctl, kSiteW16TcReady))
                    break;
                tc_fence_after();
                const uint32_t xa = smem_u32(sX + s * Cfg::X_BYTES);
                const uint32_t ba = smem_u32(sB + b * Cfg::B_BYTES);
#pragma unroll
                for (int k = 0; k < 4 * Cfg::SUB; ++k) {
                    const uint32_t kk = 32u * (k & 3);  // 16 values of K inside a 64-wide sub-tile
                    tc_mma<MmaKind::F16>(tmem_base, smem_desc_sw128(xa + (k >> 2) * Cfg::X_SUB + kk),
                                         smem_desc_sw128(ba + (k >> 2) * Cfg::B_SUB + kk), Cfg::IDESC,
                                         (i > 0 || k > 0) ? 1u : 0u);
                }
                tc_commit(empty_bar(s));
                if constexpr (!Cfg::ONE_FREE) tc_commit(bfree_bar(b));
            }
            tc_commit(accf_bar);  // also when stopped early: lets the epilogue leave
        }
    } else {
        // ---------------------------------------- transform, then epilogue
        const int tid = threadIdx.x - 64;                 // 0..511
        for (int i = tid; i < Cfg::BN * ng; i += 32 * Cfg::XFORM_WARPS) {  // this quarter's scales
            const int r = i / ng, gi = i - r * ng;
            sS[r * Cfg::MAX_SLICE_GROUPS + gi] =
                (n0 + r < p.N) ? __half_as_ushort(p.S[static_cast<int64_t>(n0 + r) * G + g_beg + gi]) : 0;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::XFORM_WARPS) : "memory");
        const int grp = (warp - 2) / Cfg::GROUP_WARPS;    // stages grp, grp + 2, ...
        const int gt = tid - grp * 32 * Cfg::GROUP_WARPS;  // 0..255 within the group
        const int r = gt / Cfg::TPR, q = gt % Cfg::TPR;   // weight row, part of the row's 64 values
        const uint32_t bw = (r >> 3) * 1024 + (r & 7) * 128;  // row start in the swizzled B stage
        for (int i = grp; i < num_kb; i += Cfg::XFORM_GROUPS) {
            const int s = i % S, b = i % NB;
            const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
            // the weights of stage i have landed and the MMA is done with the
            // B slot's previous contents (stage i - NB)
            bool got = Cfg::WRES ? bounded_wait(wfull_bar(i), 0u, abort_flag, p.ctl, kSiteW16TcXform)
                                 : bounded_wait(full_bar(s), ph, abort_flag, p.ctl, kSiteW16TcXform);
            if (got && i >= NB)
                got = bounded_wait(bfree_bar(b), static_cast<uint32_t>(i / NB - 1) & 1u, abort_flag, p.ctl,
                                   kSiteW16TcXform);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const int wslot = Cfg::WRES ? i : s;
#pragma unroll
            for (int sub = 0; sub < Cfg::SUB; ++sub) {
                const uint8_t* wsrc = sW + wslot * Cfg::W_BYTES + sub * Cfg::W_SUB + r * 32 + q * 4 * Cfg::WPT;
                uint32_t words[Cfg::WPT];
                if constexpr (Cfg::WPT == 4) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(wsrc);
                    words[0] = wv.x, words[1] = wv.y, words[2] = wv.z, words[3] = wv.w;
                } else {
                    const uint2 wv = *reinterpret_cast<const uint2*>(wsrc);
                    words[0] = wv.x, words[1] = wv.y;
                }
                const __half sc = __ushort_as_half(sS[r * Cfg::MAX_SLICE_GROUPS + ((Cfg::SUB * i + sub) >> 1)]);
                const __half2 s2 = __halves2half2(sc, sc);
                uint8_t* bst = sB + b * Cfg::B_BYTES + sub * Cfg::B_SUB + bw;
#pragma unroll
                for (int h = 0; h < Cfg::WPT; ++h) {
                    uint32_t pr[4];
                    dequant_word_fast(words[h], pr);  // (k0,k4) (k1,k5) (k2,k6) (k3,k7)
                    const uint32_t nat[4] = {__byte_perm(pr[0], pr[1], 0x5410), __byte_perm(pr[2], pr[3], 0x5410),
                                             __byte_perm(pr[0], pr[1], 0x7632), __byte_perm(pr[2], pr[3], 0x7632)};
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const __half2 qv = *reinterpret_cast<const __half2*>(&nat[j]);
                        __half2 a = __hmul2(qv, s2);  // q * s, rounded to fp16
                        w[j] = *reinterpret_cast<uint32_t*>(&a);
                    }
                    const int c = Cfg::WPT * q + h;  // 16-byte chunk: k = 8c .. 8c + 7
                    const uint32_t off = static_cast<uint32_t>((c ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4*>(bst + off) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready_bar(b));
        }
        // partial tile: TMEM lanes 32 (warp % 4) .. + 32, columns [32 ch, 32 ch + 32),
        // stored to shared memory
        const bool got = bounded_wait(accf_bar, 0u, nullptr, p.ctl, kSiteW16TcAcc);
        const int quad = warp & 3, ch = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::XFORM_WARPS) : "memory");  // stages no longer read
        const bool have = ok && __all_sync(0xffffffffu, got) && !*abort_flag && num_kb > 0;
        uint32_t vh[32];
        if (have) {
            tc_fence_after();
            const uint32_t ta = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                static_cast<uint32_t>(32 * ch);
            tmem_ld_32x32b_x32(ta, vh);
            tmem_wait_ld();
        }
        float* dst = red + row * Cfg::RED_STRIDE + 32 * ch;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (have)
                v = make_float4(__uint_as_float(vh[j]), __uint_as_float(vh[j + 1]), __uint_as_float(vh[j + 2]),
                                __uint_as_float(vh[j + 3]));
            *reinterpret_cast<float4*>(dst + j) = v;
        }
        fence_proxy_async_smem();  // the bulk copies read these rows
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_arrive_expect_tx(rx_bar, static_cast<uint32_t>((Cfg::KSPLIT - 1) * Cfg::SLICE_BYTES));
    // every CTA of the cluster is past its K loop: its rings, where the
    // partials land, are free (all MMAs, hence all their operand reads, done)
    cluster_sync_relaxed();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    const uint32_t red_u32 = smem_u32(red), rx_u32 = smem_u32(smem + Cfg::RX_OFF);
    if (threadIdx.x == 0) {
        for (int d = 1; d < Cfg::KSPLIT; ++d) {  // rows of CTA `dst` into its slot `rank`
            const uint32_t dst = (rank + static_cast<uint32_t>(d)) % Cfg::KSPLIT;
            bulk_copy_s2cluster(mapa_shared(rx_u32 + rank * Cfg::SLICE_BYTES, dst),
                                red_u32 + dst * Cfg::SLICE_BYTES, Cfg::SLICE_BYTES, mapa_shared(rx_bar, dst));
        }
    }
    if (warp >= 2) {
        // rows [32 rank, 32 rank + 32): own partial plus the three received
        const int tid = threadIdx.x - 64;
        const bool got = bounded_wait(rx_bar, 0u, nullptr, p.ctl, kSiteW16TcRx);
        const float* own = red + static_cast<int>(rank) * Cfg::SLICE_ROWS * Cfg::RED_STRIDE;
        const float* rx = reinterpret_cast<const float*>(smem + Cfg::RX_OFF);
        constexpr int E = Cfg::SLICE_ROWS * (Cfg::BN / 4) / (32 * Cfg::XFORM_WARPS);  // float4s per thread
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int idx = tid + 32 * Cfg::XFORM_WARPS * e;  // 32 rows x 32 four-column chunks
            const int t = idx >> 5, c4 = idx & 31;
            const int o = t * Cfg::RED_STRIDE + 4 * c4;
            float4 sum = *reinterpret_cast<const float4*>(own + o);
#pragma unroll
            for (int c = 0; c < Cfg::KSPLIT; ++c) {
                if (c == static_cast<int>(rank)) continue;
                const float4 v = *reinterpret_cast<const float4*>(rx + c * (Cfg::SLICE_BYTES / 4) + o);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const int m = p.m0 + static_cast<int>(rank) * Cfg::SLICE_ROWS + t, col = n0 + 4 * c4;
            if (got && m < p.M && col < p.N) {
                __half* dst = p.Y + static_cast<int64_t>(m) * p.ldy + col;
                if (col + 4 <= p.N && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
                    __half2 a = __floats2half2_rn(sum.x, sum.y), b = __floats2half2_rn(sum.z, sum.w);
                    *reinterpret_cast<uint2*>(dst) =
                        make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
                } else {
                    const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
                    for (int j = 0; j < 4 && col + j < p.N; ++j) dst[j] = __float2half_rn(vv[j]);
                }
            }
        }
    }
    // a CTA's outgoing copies have been read once every destination has
    // seen its barrier complete: only then may the source CTA leave
    cluster_sync_relaxed();
}

}  // namespace qg

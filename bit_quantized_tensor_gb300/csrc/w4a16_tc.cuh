// W4A16 on the tensor cores for batches above the decode shapes:
//
//   Y[m][n] = sum_k X[m][k] * (s[n][k / 128] * q[n][k])
//
// ("fused-int4-gemm-sm75" README: weight-only int4 with group-128 scales.)
// Each CTA owns 32 output columns (32 weight rows) for up to 128 batch rows.
// Per 64-wide K stage:
//  - X, the operand every CTA needs, is loaded once per cluster of 4 CTAs:
//    CTA r fetches rows [32 r, 32 r + 32) of the 128 x 64 fp16 tile with a
//    TMA load multicast to all 4 CTAs (128-byte swizzle).  Clusters of 8
//    were measured 1.8x slower (CTAs of this size did not all fit at once);
//  - each CTA fetches its own 32 packed weight rows (32 bytes each);
//  - four transform warps turn the nibbles into two exact fp16 operand rows
//    per weight row: q * s_hi and q * s_lo, where s_hi is the group scale with
//    its three lowest mantissa bits cleared and s_lo = s - s_hi.  q has at
//    most three significant bits, so both products are exact in fp16 and
//    q * s_hi + q * s_lo = q * s; rounding q * s to fp16 instead (a plain
//    dequantize-then-GEMM) costs up to 2^-12 of every weight, which breaks
//    the per-element tolerance once outputs grow large (a chain of layers);
//    the rows go to the swizzled K-major layout of the MMA's B operand;
//  - one thread issues tcgen05.mma kind::f16 M=128 N=64 (32 "hi" and 32 "lo"
//    columns) into a 64-column TMEM accumulator; every product is exact in
//    fp32, so the only rounding is the fp32 accumulation.  It commits to the
//    stage-empty barrier of all 4 CTAs, so a stage is refilled only when every
//    CTA of the cluster has consumed it.
// The four transform warps then drain TMEM (one lane quadrant each), add the
// two halves and store fp16 rows.  Scales must stay below 8192 in magnitude
// (8 * s_hi must be a finite fp16).  Weight rows and scales are fetched before the programmatic
// dependent wait; X after it.  Every wait is bounded; the CTAs of a cluster
// leave only after a cluster barrier.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "qg_internal.h"
#include "qg_ptx.cuh"

namespace qg {

// TMA load multicast to the CTAs of `mask`: lands at the same shared-memory
// offset in each and signals the mbarrier at the same offset in each.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                               uint32_t bar, uint16_t mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::"
        "cluster.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar), "h"(mask), "l"(policy)
        : "memory");
}

// Arrives once on the mbarrier at offset `bar` of every CTA in `mask` when
// this thread's earlier tcgen05 operations have completed.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// Orders this thread's shared-memory writes before later reads by the async
// proxy (the tensor core's operand fetch).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

constexpr uint16_t kClusterMask = 0xF;  // all CTAs of a cluster of 4

struct W16TcCfg {
    static constexpr int CLUSTER = 4;
    static constexpr int BM = 128;                      // batch rows per launch
    static constexpr int BN = 32;                       // weight rows (output columns) per CTA
    static constexpr int BK = 64;                       // K per stage: 128 bytes of fp16
    static constexpr int X_BYTES = BM * BK * 2;         // 16 KB
    static constexpr int X_SLICE = X_BYTES / CLUSTER;   // 32 rows fetched by each CTA
    static constexpr int B_ROWS = 2 * BN;               // q * s_hi rows, then q * s_lo rows
    static constexpr int B_BYTES = B_ROWS * BK * 2;     // 8 KB fp16 operand
    static constexpr int W_BYTES = BN * BK / 2;         // 1 KB packed nibbles
    static constexpr int STAGES = 7;
    static constexpr int THREADS = 32 * 6;              // producer, MMA, 4 transform/epilogue warps
    static constexpr int TMEM_COLS = 64;
    static constexpr int MAX_GROUPS = 512;              // K <= 65536: scales staged whole
    static constexpr int NUM_BARRIERS = 3 * STAGES + 1;
    static constexpr int FIXED_BYTES = STAGES * (X_BYTES + B_BYTES + W_BYTES) + 256 + 1024;
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, BM, B_ROWS);

    static_assert((1 << CLUSTER) - 1 == kClusterMask, "cluster mask");
    static_assert(X_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && X_SLICE % 1024 == 0 && BN % 8 == 0,
                  "swizzle atoms need 1 KB alignment");
    static_assert(NUM_BARRIERS * 8 + 16 <= 256, "barrier area too small");
};

// Dynamic shared memory of a launch: stages, barriers, alignment slack and the
// 32 rows' group scales.
__host__ __device__ constexpr size_t w16_tc_smem_bytes(int64_t K) {
    return W16TcCfg::FIXED_BYTES + ((static_cast<size_t>(32) * (K / 128) * 2 + 15) / 16) * 16;
}

struct W16TcParams {
    int M, N, K;
    int m0;          // first batch row of this launch
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
};

__global__ void __cluster_dims__(W16TcCfg::CLUSTER, 1, 1) __launch_bounds__(W16TcCfg::THREADS, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const W16TcParams p) {
    using Cfg = W16TcCfg;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sX = smem;                                   // S x 16 KB
    uint8_t* sB = sX + S * Cfg::X_BYTES;                  // S x 8 KB
    uint8_t* sW = sB + S * Cfg::B_BYTES;                  // S x 1 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(sW + S * Cfg::W_BYTES);
    unsigned short* sS = reinterpret_cast<unsigned short*>(reinterpret_cast<uint8_t*>(bars) + 256);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto ready_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    const uint32_t accf_bar = bar0 + 8u * (3 * S);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int n0 = blockIdx.x * Cfg::BN;
    const int G = p.K / 128;
    const int num_kb = p.K / Cfg::BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(ready_bar(s), 4);
            mbar_init(empty_bar(s), Cfg::CLUSTER);
        }
        mbar_init(accf_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tc_fence_before();
    cluster_sync();  // every CTA's barriers exist before any multicast or remote commit
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            const int pre = num_kb < S ? num_kb : S;
            // weights of the first stages before the dependency wait
            for (int kb = 0; kb < pre; ++kb) {
                mbar_arrive_expect_tx(full_bar(kb), Cfg::X_BYTES + Cfg::W_BYTES);
                tma_load_2d(smem_u32(sW + kb * Cfg::W_BYTES), &tmW, kb * (Cfg::BK / 2), n0,
                            full_bar(kb), pol_w);
            }
            pdl_wait_prior_grid();  // X may be the previous kernel's output
            // the previous kernel wrote X with ordinary stores; these loads
            // are TMA (async proxy) reads
            asm volatile("fence.proxy.async.global;" ::: "memory");
            for (int kb = 0; kb < pre; ++kb)
                tma_load_2d_mc(smem_u32(sX + kb * Cfg::X_BYTES + rank * Cfg::X_SLICE), &tmX, kb * Cfg::BK,
                               p.m0 + static_cast<int>(rank) * (Cfg::BM / Cfg::CLUSTER), full_bar(kb),
                               kClusterMask, pol_x);
            bool ok = true;
            for (int kb = pre; ok && kb < num_kb; ++kb) {
                const int s = kb % S;
                const uint32_t ph = static_cast<uint32_t>(kb / S - 1) & 1u;  // round just finished
                if (!bounded_wait(empty_bar(s), ph, abort_flag, p.ctl, kSiteW16TcEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(s), Cfg::X_BYTES + Cfg::W_BYTES);
                tma_load_2d(smem_u32(sW + s * Cfg::W_BYTES), &tmW, kb * (Cfg::BK / 2), n0, full_bar(s),
                            pol_w);
                tma_load_2d_mc(smem_u32(sX + s * Cfg::X_BYTES + rank * Cfg::X_SLICE), &tmX, kb * Cfg::BK,
                               p.m0 + static_cast<int>(rank) * (Cfg::BM / Cfg::CLUSTER), full_bar(s),
                               kClusterMask, pol_x);
            }
            if (!ok) {
                // Copies already issued (by this CTA into every CTA of the
                // cluster) get a fixed time to land before anyone leaves.
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 1000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            for (int kb = 0; kb < num_kb; ++kb) {
                const int s = kb % S;
                const uint32_t ph = static_cast<uint32_t>(kb / S) & 1u;
                if (!bounded_wait(full_bar(s), ph, abort_flag, p.ctl, kSiteW16TcFull) ||
                    !bounded_wait(ready_bar(s), ph, abort_flag, p.ctl, kSiteW16TcReady))
                    break;
                tc_fence_after();
                const uint32_t xa = smem_u32(sX + s * Cfg::X_BYTES);
                const uint32_t ba = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc_mma<MmaKind::F16>(tmem_base, smem_desc_sw128(xa + 32u * k),
                                         smem_desc_sw128(ba + 32u * k), Cfg::IDESC,
                                         (kb > 0 || k > 0) ? 1u : 0u);
                tc_commit_mc(empty_bar(s), kClusterMask);
            }
            tc_commit(accf_bar);  // also when stopped early: lets the epilogue leave
        }
    } else {
        // ---------------------------------------- transform, then epilogue
        const int tid = threadIdx.x - 64;                 // 0..127
        for (int i = tid; i < Cfg::BN * G; i += 128) {    // the 32 rows' group scales
            const int r = i / G, gi = i - r * G;
            sS[i] = (n0 + r < p.N) ? __half_as_ushort(p.S[static_cast<int64_t>(n0 + r) * G + gi]) : 0;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int r = tid >> 2, q = tid & 3;              // weight row, 16-value quarter of the stage
        const uint32_t bw = (r >> 3) * 1024 + (r & 7) * 128;  // row start in the swizzled B stage
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
            const int s = kb % S;
            const uint32_t ph = static_cast<uint32_t>(kb / S) & 1u;
            const bool got = bounded_wait(full_bar(s), ph, abort_flag, p.ctl, kSiteW16TcXform);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint2 wv = *reinterpret_cast<const uint2*>(sW + s * Cfg::W_BYTES + r * 32 + q * 8);
            const unsigned short sbits = sS[r * G + (kb >> 1)];
            const __half shi = __ushort_as_half(static_cast<unsigned short>(sbits & 0xFFF8u));
            const __half slo = __float2half_rn(__half2float(__ushort_as_half(sbits)) - __half2float(shi));
            const __half2 shi2 = __halves2half2(shi, shi), slo2 = __halves2half2(slo, slo);
            uint8_t* bst = sB + s * Cfg::B_BYTES + bw;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pr[4];
                dequant_word_fast(h ? wv.y : wv.x, pr);  // (k0,k4) (k1,k5) (k2,k6) (k3,k7)
                const uint32_t nat[4] = {__byte_perm(pr[0], pr[1], 0x5410), __byte_perm(pr[2], pr[3], 0x5410),
                                         __byte_perm(pr[0], pr[1], 0x7632), __byte_perm(pr[2], pr[3], 0x7632)};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 qv = *reinterpret_cast<const __half2*>(&nat[j]);
                    __half2 a = __hmul2(qv, shi2), b = __hmul2(qv, slo2);
                    hi[j] = *reinterpret_cast<uint32_t*>(&a);
                    lo[j] = *reinterpret_cast<uint32_t*>(&b);
                }
                const int c = 2 * q + h;                   // 16-byte chunk: k = 8c .. 8c + 7
                const uint32_t off = static_cast<uint32_t>((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4*>(bst + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                // row 32 + r: four atoms further, same swizzle phase
                *reinterpret_cast<uint4*>(bst + 4 * 1024 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready_bar(s));
        }
        // epilogue: TMEM lanes 32 (warp % 4) .. + 32, 32 fp32 columns each
        const bool got = bounded_wait(accf_bar, 0u, nullptr, p.ctl, kSiteW16TcAcc);
        if (ok && __all_sync(0xffffffffu, got) && !*abort_flag) {
            tc_fence_after();
            const int quad = warp & 3;
            uint32_t v[32], vl[32];
            tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16), v);
            tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + 32u, vl);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(vl[j]));
            const int row = p.m0 + quad * 32 + lane;
            if (row < p.M) {
                __half* dst = p.Y + static_cast<int64_t>(row) * p.ldy + n0;
                const bool vec = n0 + 32 <= p.N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
                if (vec) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            __half2 h2 = __floats2half2_rn(__uint_as_float(v[8 * c + 2 * j]),
                                                           __uint_as_float(v[8 * c + 2 * j + 1]));
                            pk[j] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n0 + j < p.N) dst[j] = __float2half_rn(__uint_as_float(v[j]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still write its shared memory
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace qg

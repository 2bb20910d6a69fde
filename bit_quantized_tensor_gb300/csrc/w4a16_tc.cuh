// W4A16 on the tensor cores for batches above the decode shapes:
//
//   Y[m][n] = sum_k X[m][k] * (s[n][k / 128] * q[n][k])
//
// ("fused-int4-gemm-sm75" README: weight-only int4 with group-128 scales.)
// A cluster of 4 CTAs owns 128 output columns (128 weight rows) for up to 128
// batch rows and splits K four ways: CTA r handles a contiguous quarter of
// the K groups.  Per 64-wide K stage a CTA
//  - TMA-loads its 128 x 64 fp16 tile of X and its 128 rows x 32 bytes of
//    packed weights into a 4-deep ring (covers the memory latency);
//  - turns the nibbles (eight transform warps) into two exact fp16 operand
//    rows per weight row, q * s_hi and q * s_lo, where s_hi is the group scale
//    with its three lowest mantissa bits cleared and s_lo = s - s_hi: q has at
//    most three significant bits, so both products are exact in fp16 and
//    q * s_hi + q * s_lo = q * s (rounding q * s to fp16, a plain
//    dequantize-then-GEMM, costs up to 2^-12 of every weight); the 256 rows go
//    to the 128-byte-swizzled K-major layout of the MMA's B operand, in a
//    ring of three slots (with two, the transform of a stage waited for the
//    MMA two stages back to complete, which paced the loop);
//  - issues tcgen05.mma kind::f16 M=128 N=256 (one thread) into a 256-column
//    TMEM accumulator.  Every product is exact in fp32, so the only rounding
//    is the fp32 accumulation.  Wide MMAs matter here: an instruction costs
//    about 128 cycles whatever its width, so N=64 ran at a quarter of the rate.
// At the end every CTA adds its hi and lo halves into a 128 x 128 fp32
// partial tile in shared memory; after a cluster barrier CTA r sums rows
// [32 r, 32 r + 32) of the four partial tiles through distributed shared
// memory and stores them as fp16.  Weight rows and scales are fetched before
// the programmatic dependent wait; X after it.  Every wait is bounded; the
// CTAs of a cluster leave only after a second cluster barrier.  Scales must
// stay below 8192 in magnitude (8 * s_hi must be a finite fp16).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "qg_internal.h"
#include "qg_ptx.cuh"

namespace qg {

// Orders this thread's shared-memory writes before later reads by the async
// proxy (the tensor core's operand fetch).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte load from the shared memory of another CTA of the cluster.
__device__ __forceinline__ float4 ld_shared_cluster_f4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

struct W16TcCfg {
    static constexpr int KSPLIT = 4;                    // CTAs per cluster, one K quarter each
    static constexpr int BM = 128;                      // batch rows per launch
    static constexpr int BN = 128;                      // weight rows (output columns) per cluster
    static constexpr int BK = 64;                       // K per stage: 128 bytes of fp16
    static constexpr int X_BYTES = BM * BK * 2;         // 16 KB
    static constexpr int B_ROWS = 2 * BN;               // q * s_hi rows, then q * s_lo rows
    static constexpr int B_BYTES = B_ROWS * BK * 2;     // 32 KB fp16 operand
    static constexpr int W_BYTES = BN * BK / 2;         // 4 KB packed nibbles
    static constexpr int STAGES = 4;                    // X + packed-weight ring (memory latency)
    static constexpr int BSLOTS = 3;                    // B operand ring (transform -> MMA)
    static constexpr int XFORM_WARPS = 8;
    static constexpr int THREADS = 32 * (2 + XFORM_WARPS);  // producer, MMA, transform/epilogue
    static constexpr int TMEM_COLS = 256;
    static constexpr int MAX_SLICE_GROUPS = 64;         // K groups per quarter: K <= 32768
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * BSLOTS + 1;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SCALE_BYTES = BN * MAX_SLICE_GROUPS * 2;  // 16 KB
    static constexpr int RING_BYTES = STAGES * (X_BYTES + W_BYTES) + BSLOTS * B_BYTES;
    static constexpr int SMEM_BYTES = RING_BYTES + BAR_BYTES + SCALE_BYTES + 1024;
    static constexpr int RED_STRIDE = BN + 4;           // floats per partial-tile row (bank spread)
    static constexpr uint32_t IDESC = make_idesc(0u, 0u, BM, B_ROWS);

    static_assert(X_BYTES % 1024 == 0 && B_BYTES % 1024 == 0,
                  "swizzle atoms need 1 KB alignment");
    static_assert(NUM_BARRIERS * 8 + 16 <= BAR_BYTES, "barrier area too small");
    static_assert(SMEM_BYTES <= 232448, "shared-memory budget exceeded");
    static_assert(BM * RED_STRIDE * 4 <= RING_BYTES, "partial tile reuses the rings");
};

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
};

__global__ void __cluster_dims__(W16TcCfg::KSPLIT, 1, 1) __launch_bounds__(W16TcCfg::THREADS, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const W16TcParams p) {
    using Cfg = W16TcCfg;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int NB = Cfg::BSLOTS;
    uint8_t* sX = smem;                                   // S x 16 KB
    uint8_t* sB = sX + S * Cfg::X_BYTES;                  // NB x 32 KB
    uint8_t* sW = sB + NB * Cfg::B_BYTES;                 // S x 4 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(sW + S * Cfg::W_BYTES);
    unsigned short* sS = reinterpret_cast<unsigned short*>(reinterpret_cast<uint8_t*>(bars) + Cfg::BAR_BYTES);
    float* red = reinterpret_cast<float*>(smem);          // partial tile, after the K loop
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };             // X + W of stage s landed
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };      // MMA done with stage s
    auto ready_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };  // B slot b written
    auto bfree_bar = [&](int b) { return bar0 + 8u * (2 * S + NB + b); };  // MMA done with B slot b
    const uint32_t accf_bar = bar0 + 8u * (2 * S + 2 * NB);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();              // K quarter of this CTA
    const int n0 = static_cast<int>(blockIdx.x / Cfg::KSPLIT) * Cfg::BN;
    const int G = p.K / 128;
    const int gq = (G + Cfg::KSPLIT - 1) / Cfg::KSPLIT;   // groups per quarter
    const int g_beg = min(G, static_cast<int>(rank) * gq), g_end = min(G, g_beg + gq);
    const int ng = g_end - g_beg;
    const int num_kb = 2 * ng;                            // 64-wide stages of this quarter
    const int kb0 = 2 * g_beg;                            // first global stage

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(ready_bar(b), Cfg::XFORM_WARPS);
            mbar_init(bfree_bar(b), 1);
        }
        mbar_init(accf_bar, 1);
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
            for (int i = 0; i < pre; ++i) {  // weights of the first stages before the wait
                mbar_arrive_expect_tx(full_bar(i), Cfg::X_BYTES + Cfg::W_BYTES);
                tma_load_2d(smem_u32(sW + i * Cfg::W_BYTES), &tmW, (kb0 + i) * (Cfg::BK / 2), n0,
                            full_bar(i), pol_w);
            }
            pdl_wait_prior_grid();  // X may be the previous kernel's output
            // the previous kernel wrote X with ordinary stores; these loads
            // are TMA (async proxy) reads
            asm volatile("fence.proxy.async.global;" ::: "memory");
            for (int i = 0; i < pre; ++i)
                tma_load_2d(smem_u32(sX + i * Cfg::X_BYTES), &tmX, (kb0 + i) * Cfg::BK, p.m0, full_bar(i),
                            pol_x);
            for (int i = pre; i < num_kb; ++i) {
                const int s = i % S;
                const uint32_t ph = static_cast<uint32_t>(i / S - 1) & 1u;  // round just finished
                if (!bounded_wait(empty_bar(s), ph, abort_flag, p.ctl, kSiteW16TcEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(s), Cfg::X_BYTES + Cfg::W_BYTES);
                tma_load_2d(smem_u32(sW + s * Cfg::W_BYTES), &tmW, (kb0 + i) * (Cfg::BK / 2), n0,
                            full_bar(s), pol_w);
                tma_load_2d(smem_u32(sX + s * Cfg::X_BYTES), &tmX, (kb0 + i) * Cfg::BK, p.m0, full_bar(s),
                            pol_x);
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
                for (int k = 0; k < 4; ++k)
                    tc_mma<MmaKind::F16>(tmem_base, smem_desc_sw128(xa + 32u * k),
                                         smem_desc_sw128(ba + 32u * k), Cfg::IDESC,
                                         (i > 0 || k > 0) ? 1u : 0u);
                tc_commit(empty_bar(s));
                tc_commit(bfree_bar(b));
            }
            tc_commit(accf_bar);  // also when stopped early: lets the epilogue leave
        }
    } else {
        // ---------------------------------------- transform, then epilogue
        const int tid = threadIdx.x - 64;                 // 0..255
        for (int i = tid; i < Cfg::BN * ng; i += 32 * Cfg::XFORM_WARPS) {  // this quarter's scales
            const int r = i / ng, gi = i - r * ng;
            sS[r * Cfg::MAX_SLICE_GROUPS + gi] =
                (n0 + r < p.N) ? __half_as_ushort(p.S[static_cast<int64_t>(n0 + r) * G + g_beg + gi]) : 0;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::XFORM_WARPS) : "memory");
        const int r = tid >> 1, q = tid & 1;              // weight row, 32-value half of the stage
        const uint32_t bw = (r >> 3) * 1024 + (r & 7) * 128;  // row start in the swizzled B stage
        for (int i = 0; i < num_kb; ++i) {
            const int s = i % S, b = i % NB;
            const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
            // the weights of stage i have landed and the MMA is done with the
            // B slot's previous contents (stage i - NB)
            bool got = bounded_wait(full_bar(s), ph, abort_flag, p.ctl, kSiteW16TcXform);
            if (got && i >= NB)
                got = bounded_wait(bfree_bar(b), static_cast<uint32_t>(i / NB - 1) & 1u, abort_flag, p.ctl,
                                   kSiteW16TcXform);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint4 wv = *reinterpret_cast<const uint4*>(sW + s * Cfg::W_BYTES + r * 32 + q * 16);
            const unsigned short sbits = sS[r * Cfg::MAX_SLICE_GROUPS + (i >> 1)];
            const __half shi = __ushort_as_half(static_cast<unsigned short>(sbits & 0xFFF8u));
            const __half slo = __float2half_rn(__half2float(__ushort_as_half(sbits)) - __half2float(shi));
            const __half2 shi2 = __halves2half2(shi, shi), slo2 = __halves2half2(slo, slo);
            uint8_t* bst = sB + b * Cfg::B_BYTES + bw;
            const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t pr[4];
                dequant_word_fast(words[h], pr);  // (k0,k4) (k1,k5) (k2,k6) (k3,k7)
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
                const int c = 4 * q + h;                   // 16-byte chunk: k = 8c .. 8c + 7
                const uint32_t off = static_cast<uint32_t>((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4*>(bst + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                // row 128 + r: sixteen atoms further, same swizzle phase
                *reinterpret_cast<uint4*>(bst + 16 * 1024 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready_bar(b));
        }
        // partial tile: TMEM lanes 32 (warp % 4) .. + 32, columns [64 ch, 64 ch + 64)
        // (hi) and [128 + 64 ch, ...) (lo), added and stored to shared memory
        const bool got = bounded_wait(accf_bar, 0u, nullptr, p.ctl, kSiteW16TcAcc);
        const int quad = warp & 3, ch = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::XFORM_WARPS) : "memory");  // stages no longer read
        const bool have = ok && __all_sync(0xffffffffu, got) && !*abort_flag && num_kb > 0;
        if (have) tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t vh[32], vl[32];
            if (have) {
                const uint32_t ta = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                    static_cast<uint32_t>(64 * ch + 32 * part);
                tmem_ld_32x32b_x32(ta, vh);
                tmem_ld_32x32b_x32(ta + 128u, vl);
                tmem_wait_ld();
            }
            float* dst = red + row * Cfg::RED_STRIDE + 64 * ch + 32 * part;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (have)
                    v = make_float4(__uint_as_float(vh[j]) + __uint_as_float(vl[j]),
                                    __uint_as_float(vh[j + 1]) + __uint_as_float(vl[j + 1]),
                                    __uint_as_float(vh[j + 2]) + __uint_as_float(vl[j + 2]),
                                    __uint_as_float(vh[j + 3]) + __uint_as_float(vl[j + 3]));
                *reinterpret_cast<float4*>(dst + j) = v;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the four partial tiles are complete
    if (warp >= 2) {
        // rows [32 rank, 32 rank + 32) of the sum of the four partial tiles
        const int tid = threadIdx.x - 64;
        const uint32_t red_local = smem_u32(red);
        uint32_t peer[Cfg::KSPLIT];
#pragma unroll
        for (int c = 0; c < Cfg::KSPLIT; ++c) peer[c] = mapa_shared(red_local, static_cast<uint32_t>(c));
        float4 part[4][Cfg::KSPLIT];                      // all remote loads first, then the sums
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = tid + 256 * e;                // 32 rows x 32 four-column chunks
            const int trow = static_cast<int>(rank) * 32 + (idx >> 5);  // row of the 128-row tile
            const uint32_t off = static_cast<uint32_t>((trow * Cfg::RED_STRIDE + 4 * (idx & 31)) * 4);
#pragma unroll
            for (int c = 0; c < Cfg::KSPLIT; ++c) part[e][c] = ld_shared_cluster_f4(peer[c] + off);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = tid + 256 * e;
            const int trow = static_cast<int>(rank) * 32 + (idx >> 5);
            const int c4 = idx & 31;
            float4 sum = part[e][0];
#pragma unroll
            for (int c = 1; c < Cfg::KSPLIT; ++c) {
                sum.x += part[e][c].x;
                sum.y += part[e][c].y;
                sum.z += part[e][c].z;
                sum.w += part[e][c].w;
            }
            const int m = p.m0 + trow, col = n0 + 4 * c4;
            if (m < p.M && col < p.N) {
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
    cluster_sync();  // no CTA leaves while a peer may still read its partial tile
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace qg

// Persistent, warp-specialized tcgen05 GEMM for sm_103a:  D = A . B^T.
//
//   A : M x K tile source, K-major, loaded by TMA (128-byte swizzle).
//   B : N x K tile source, K-major, loaded by TMA (128-byte swizzle).
//   D : fp32 accumulators in tensor memory (TMEM), drained by epilogue warps.
//
// Roles (one CTA per SM, tiles claimed round-robin until none remain):
//   warp 0      TMA producer: fills a STAGES-deep shared-memory ring.
//   warp 1      MMA issuer (one thread) and TMEM owner.
//   warps 2..9  epilogue: TMEM -> registers -> global memory.
// Two rings advance independently: the operand ring (full/empty barriers
// per stage) and the accumulator ring (acc_full/acc_empty per TMEM buffer),
// so loading, MMA and draining overlap ("Warp-Specialized Kernel
// Implementation for W4A4 MatMul on Latest GPU Architectures", sections 4-5:
// warp specialization, explicit per-warp pipeline state, persistent tile
// scheduling).
//
// Epilogues:
//   Epi::F16  one accumulation unit per tile (the whole K); fp32 -> fp16 with
//             round-to-nearest-even, optional per-column fp16 bias.
//   Epi::S32  exact integer GEMM carried in floating-point operands: the K
//             loop is cut into chunks of `chunk_kb` k-blocks whose fp32 sums
//             stay within 2^24 in magnitude (so every partial sum is an exactly
//             representable integer); each chunk is converted to int32 and
//             added in registers; the int32 tile is stored at the end.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "qg_ptx.cuh"

namespace qg {

enum class Epi { F16, S32 };

// Call-site tags recorded with QG_ERR_TIMEOUT.
enum WaitSite : int {
    kSiteProducerEmpty = 101,
    kSiteMmaAccEmpty = 102,
    kSiteMmaFull = 103,
    kSiteEpiAccFull = 104,
    kSiteDrainTma = 105,
    kSiteDrainMma = 106,
};

// Tile configuration with its shared-memory budget solved at compile time:
// stages * (bytes_A + bytes_B) + barriers + alignment slack <= per-block limit,
// maximizing the number of stages ("Warp-Specialized Kernel Implementation
// for W4A4 MatMul ...", section 6).  Each CTA loads its own A and B tiles
// (1-CTA MMA), so nothing is amortized across CTAs in this budget.
template <MmaKind KIND_, Epi EPI_>
struct TcGemmCfg {
    static constexpr MmaKind KIND = KIND_;
    static constexpr Epi EPI = EPI_;
    static constexpr int BM = 128;                       // UMMA M (rows per CTA tile)
    static constexpr int BN = 256;                       // UMMA N
    static constexpr int ROW_BYTES = 128;                // one 128B-swizzle row along K
    static constexpr int ELEM_BYTES = (KIND == MmaKind::F16) ? 2 : 1;
    static constexpr int BK = ROW_BYTES / ELEM_BYTES;    // K elements per stage
    static constexpr int MMA_K = 32 / ELEM_BYTES;        // K per tcgen05.mma (32 bytes)
    static constexpr int KSTEPS = BK / MMA_K;            // MMAs per stage
    static constexpr int A_BYTES = BM * ROW_BYTES;
    static constexpr int B_BYTES = BN * ROW_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_LIMIT = 232448;            // 227 KB per block (opt-in)
    static constexpr int BARRIER_BYTES = 256;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int STAGES = (SMEM_LIMIT - BARRIER_BYTES - ALIGN_SLACK) / STAGE_BYTES;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BARRIER_BYTES + ALIGN_SLACK;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 32 * (2 + EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 * ACC_BUFS + 1;
    static constexpr uint32_t IDESC =
        make_idesc(0u, 0u, static_cast<uint32_t>(BM), static_cast<uint32_t>(BN));

    static_assert(STAGES >= 2, "operand ring needs at least double buffering");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared-memory budget exceeded");
    static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM keeps all 512 TMEM columns free");
    static_assert(NUM_BARRIERS * 8 + 8 <= BARRIER_BYTES, "barrier area too small");
    static_assert(ACC_BUFS * BN <= TMEM_COLS, "TMEM budget exceeded");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "invalid UMMA N for M = 128");
    static_assert(EPI_WARPS == 8 && BN == 256, "epilogue maps 2 warps x 128 columns per lane quadrant");
};

struct TcGemmParams {
    int M, N, K;
    int num_kb;     // ceil(K / BK)
    int chunk_kb;   // k-blocks per accumulation unit (Epi::S32); >= num_kb for Epi::F16
    void* C;        // int32 (S32) or fp16 (F16) output, row-major
    int64_t ldc;    // in elements
    const __half* bias;  // optional per-column bias (F16 epilogue), may be null
    Ctl ctl;
    int l2_mode;    // L2 policy of the operand loads and output stores (qg_set_l2_policy)
};

// L2 policies of one GEMM launch.  Mode 0: every TMA load evict-normal.
// Modes 1 and 2 follow the tile order below: a group of row-blocks is
// finished against every column block before the next group starts, so an
// A tile is read again in later rounds (evict-last) while a B tile is read by
// the row-blocks of one group at about the same time and then not for a
// whole group (evict-first).  Mode 2 also writes the output with streaming
// (evict-first) stores, which are not read again by this kernel.
struct L2Policies {
    uint64_t a, b;
};
__device__ __forceinline__ L2Policies l2_policies(int mode) {
    if (mode == 0) {
        const uint64_t n = l2_policy_evict_normal();
        return {n, n};
    }
    return {l2_policy_evict_last(), l2_policy_evict_first()};
}

// 16-byte global store, with the streaming (evict-first) hint when `cs`.
__device__ __forceinline__ void st_global_16(void* dst, uint4 v, bool cs) {
    if (cs)
        __stcs(reinterpret_cast<uint4*>(dst), v);
    else
        *reinterpret_cast<uint4*>(dst) = v;
}

// One 32-byte store (dst 32-byte aligned).  An epilogue thread owns one
// output row, so the lanes of a warp store to 32 different rows: a 32-byte
// piece per lane fills whole sectors, where 16-byte pieces would half-fill
// each sector and take twice the store instructions.
__device__ __forceinline__ void st_global_32(void* dst, uint4 a, uint4 b, bool cs) {
    if (cs)
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a.x),
                     "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
    else
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a.x),
                     "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
}

// Tiles are visited in groups of `group_m` row-blocks (column-major inside a
// group) so that the CTAs running at the same time cover a compact block of
// the output and share their A and B tiles through L2: one CTA per SM covers
// 16 row-blocks x ~10 column-blocks, CTA pairs 8 x ~10.
constexpr int kGroupM = 16;
constexpr int kGroupMPairs = 8;
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& mb, int& nb,
                                            int group_m = kGroupM) {
    const int group_size = group_m * num_n;
    const int g = t / group_size;
    const int first_m = g * group_m;
    const int gm = min(group_m, num_m - first_m);
    const int local = t - g * group_size;
    mb = first_m + local % gm;
    nb = local / gm;
}

__device__ __forceinline__ uint4 pack_f16x8(const float* f) {
    uint4 pk;
    __half2 h0 = __floats2half2_rn(f[0], f[1]);
    __half2 h1 = __floats2half2_rn(f[2], f[3]);
    __half2 h2 = __floats2half2_rn(f[4], f[5]);
    __half2 h3 = __floats2half2_rn(f[6], f[7]);
    pk.x = *reinterpret_cast<uint32_t*>(&h0);
    pk.y = *reinterpret_cast<uint32_t*>(&h1);
    pk.z = *reinterpret_cast<uint32_t*>(&h2);
    pk.w = *reinterpret_cast<uint32_t*>(&h3);
    return pk;
}

template <int N>
__device__ __forceinline__ void store_row_f16(__half* dst, int col0, int N_total, const float* v,
                                              const __half* bias, bool cs = false) {
#pragma unroll
    for (int c = 0; c < N; c += 16) {
        float f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = v[c + i];
        if (bias) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int col = col0 + c + i;
                if (col < N_total) f[i] += __half2float(bias[col]);
            }
        }
        if (col0 + c + 16 <= N_total && (reinterpret_cast<uintptr_t>(dst + c) & 31u) == 0) {
            st_global_32(dst + c, pack_f16x8(f), pack_f16x8(f + 8), cs);
            continue;
        }
#pragma unroll
        for (int h = 0; h < 16; h += 8) {
            if (col0 + c + h + 8 <= N_total && (reinterpret_cast<uintptr_t>(dst + c + h) & 15u) == 0) {
                st_global_16(dst + c + h, pack_f16x8(f + h), cs);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (col0 + c + h + i < N_total) dst[c + h + i] = __float2half_rn(f[h + i]);
            }
        }
    }
}

template <int N>  // N: a multiple of 8
__device__ __forceinline__ void store_row_s32(int32_t* dst, int col0, int N_total,
                                              const int32_t* v, bool cs = false) {
    auto pack4 = [&](int c) {
        return make_uint4(static_cast<uint32_t>(v[c]), static_cast<uint32_t>(v[c + 1]),
                          static_cast<uint32_t>(v[c + 2]), static_cast<uint32_t>(v[c + 3]));
    };
#pragma unroll
    for (int c = 0; c < N; c += 8) {
        if (col0 + c + 8 <= N_total && (reinterpret_cast<uintptr_t>(dst + c) & 31u) == 0) {
            st_global_32(dst + c, pack4(c), pack4(c + 4), cs);
            continue;
        }
#pragma unroll
        for (int h = 0; h < 8; h += 4) {
            if (col0 + c + h + 4 <= N_total && (reinterpret_cast<uintptr_t>(dst + c + h) & 15u) == 0) {
                st_global_16(dst + c + h, pack4(c + h), cs);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (col0 + c + h + i < N_total) dst[c + h + i] = v[c + h + i];
            }
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), Cfg::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int num_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int ntiles = num_m * num_n;
    const int units = (p.num_kb + p.chunk_kb - 1) / p.chunk_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            Ring<STAGES> ps;
            uint32_t armed = 0, armed_phase = 0;  // bit s: slot s armed / its phase
            const L2Policies pol = l2_policies(p.l2_mode);
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!bounded_wait(empty_bar(ps.slot()), ps.parity() ^ 1u, abort_flag, p.ctl,
                                      kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(ps.slot()), Cfg::STAGE_BYTES);
                    tma_load_2d(smem_u32(sA + ps.slot() * Cfg::A_BYTES), &tmA, kb * Cfg::BK,
                                mb * Cfg::BM, full_bar(ps.slot()), pol.a);
                    tma_load_2d(smem_u32(sB + ps.slot() * Cfg::B_BYTES), &tmB, kb * Cfg::BK,
                                nb * Cfg::BN, full_bar(ps.slot()), pol.b);
                    armed |= 1u << ps.slot();
                    armed_phase = (armed_phase & ~(1u << ps.slot())) | (ps.parity() << ps.slot());
                    ps.next();
                }
            }
            if (!ok) {
                // Leave only after the copies already issued have landed.
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s))
                        bounded_wait(full_bar(s), (armed_phase >> s) & 1u, nullptr, p.ctl,
                                     kSiteDrainTma);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            Ring<STAGES> ps;
            Ring<ACC_BUFS> as;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                for (int u = 0; ok && u < units; ++u) {
                    const int kb0 = u * p.chunk_kb;
                    const int kb1 = min(p.num_kb, kb0 + p.chunk_kb);
                    if (!bounded_wait(acce_bar(as.slot()), as.parity() ^ 1u, abort_flag, p.ctl,
                                      kSiteMmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as.slot() * Cfg::BN);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!bounded_wait(full_bar(ps.slot()), ps.parity(), abort_flag, p.ctl,
                                          kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(sA + ps.slot() * Cfg::A_BYTES);
                        const uint32_t b_addr = smem_u32(sB + ps.slot() * Cfg::B_BYTES);
#pragma unroll
                        for (int k = 0; k < Cfg::KSTEPS; ++k) {
                            const uint64_t ad = smem_desc_sw128(a_addr + 32u * k);
                            const uint64_t bd = smem_desc_sw128(b_addr + 32u * k);
                            tc_mma<Cfg::KIND>(d_tmem, ad, bd, Cfg::IDESC,
                                              (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        tc_commit(empty_bar(ps.slot()));
                        ps.next();
                    }
                    if (!ok) break;
                    tc_commit(accf_bar(as.slot()));
                    as.next();
                }
            }
            // Every MMA issued by this thread has completed before the CTA
            // can release TMEM or shared memory.
            tc_commit(drain_bar);
            bounded_wait(drain_bar, 0u, nullptr, p.ctl, kSiteDrainMma);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int colhalf = (warp - 2) >> 2;     // 0: columns [0,128), 1: [128,256)
        Ring<ACC_BUFS> as;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb);
            const int row = mb * Cfg::BM + quad * 32 + lane;
            const int col0 = nb * Cfg::BN + colhalf * 128;
            if constexpr (Cfg::EPI == Epi::S32) {
                int32_t sum[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) sum[i] = 0;
                for (int u = 0; u < units; ++u) {
                    bool got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl,
                                            kSiteEpiAccFull);
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
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(as.slot()));
                    as.next();
                }
                if (!ok) break;
                if (row < p.M)
                    store_row_s32<128>(static_cast<int32_t*>(p.C) + static_cast<int64_t>(row) * p.ldc +
                                           col0,
                                       col0, p.N, sum, p.l2_mode == 2);
            } else {
                bool got = bounded_wait(accf_bar(as.slot()), as.parity(), abort_flag, p.ctl,
                                        kSiteEpiAccFull);
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
                if (lane == 0) mbar_arrive(acce_bar(as.slot()));
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
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace qg

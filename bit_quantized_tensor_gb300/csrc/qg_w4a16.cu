// W4A16 weight-only linear ("fused-int4-gemm-sm75" README: packed INT4
// weights, sign extension and dequantization in registers, tensor-core MMA,
// per-group scales with group_size = 128):
//
//   Y[m][n] = sum_k X[m][k] * (q[n][k] * s[n][k / 128]),  fp32 accumulation.
//
// Decode shapes (small M) are bound by streaming the packed weights from
// HBM, so the kernel is organized around that stream:
//  - every thread issues all of its weight loads (16 bytes per 128-wide
//    group) at entry, before anything else, so each SM keeps tens of KB of
//    weight reads in flight;
//  - with programmatic dependent launch the weight and scale loads are issued
//    before the previous kernel on the stream has finished; X (possibly that
//    kernel's output) is read only after griddepcontrol.wait;
//  - a 32-bit word of 8 nibbles is turned into four fp16 pairs with an XOR
//    (two's complement -> offset binary), a mask-or into the fp16 pattern of
//    1024 + n, and one fp16 subtraction of 1032: exact, ~1 instruction per
//    value;
//  - the dequantized pairs feed mma.sync m16n8k16 (fp16 x fp16 -> fp32) as
//    the B operand; because a dot product does not depend on the order of k,
//    each thread's logical MMA k slots are mapped onto the physical k of the
//    word it loaded (pairs (k0,k4), (k1,k5), (k2,k6), (k3,k7)), and the same
//    mapping is applied to the X fragments, which are loaded 16 bytes at a
//    time and regrouped with byte permutes;
//  - each group's MMAs accumulate into a fresh fp32 tile that is scaled by
//    the group's fp16 scales in fp32 and added to the running sum, so the
//    weights are never rounded after dequantization;
//  - the K range is split over the CTA's warps and the partial tiles are
//    added through shared memory.
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "qg_gemm_host.h"
#include "qg_ptx.cuh"

namespace qg {

constexpr int kGroup = 128;
constexpr int kW16Threads = 256;   // 8 warps
// Groups whose weights are in flight per thread: all 8 for decode shapes,
// fewer when more m16 tiles need registers.
template <int MT>
__host__ __device__ constexpr int w16_batch() { return MT <= 1 ? 8 : (MT == 2 ? 4 : 2); }

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16 bytes of X.  X may be the output of the kernel launched just before
// (programmatic dependent launch), so it must be read only after
// griddepcontrol.wait.  A __ldg is an invariant load that the compiler may
// hoist above that wait; this load is a volatile asm statement, which keeps
// its place after the wait (also a volatile asm statement).  It is a plain
// weak load: after the wait the prior grid's writes are visible to this grid.
__device__ __forceinline__ uint4 ld_x_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned short ld_nc_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four fp16 pairs of the 8 signed nibbles of `w` (nibble j = physical k_j):
// p[0] = (k0, k4), p[1] = (k1, k5), p[2] = (k2, k6), p[3] = (k3, k7).
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t u = w ^ 0x88888888u;  // nibble n -> n ^ 8 = value + 8 in [0, 15]
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t h = ((u >> (4 * j)) & 0x000F000Fu) | 0x64006400u;  // 1024 + (value + 8)
        __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
        p[j] = *reinterpret_cast<uint32_t*>(&v);
    }
}

// X fragment words for physical k = k0 .. k0+7 of one row, regrouped as the
// pairs (x0,x4), (x1,x5), (x2,x6), (x3,x7).
__device__ __forceinline__ void x_pairs(const __half* row, uint32_t (&p)[4]) {
    const uint4 v = ld_x_u4(row);
    p[0] = __byte_perm(v.x, v.z, 0x5410);
    p[1] = __byte_perm(v.x, v.z, 0x7632);
    p[2] = __byte_perm(v.y, v.w, 0x5410);
    p[3] = __byte_perm(v.y, v.w, 0x7632);
}

// MT: m16 tiles per CTA (M <= 16*MT); NT: n8 tiles per CTA; the CTA's 8
// warps are NT n-tiles x (8/NT) K slices.
template <int MT, int NT>
__global__ void __launch_bounds__(kW16Threads)
    k_w4a16(int M, int N, int K, const __half* __restrict__ X, int64_t ldx,
            const uint8_t* __restrict__ Wq, const __half* __restrict__ S, __half* __restrict__ Y,
            int64_t ldy) {
    constexpr int KQ = 8 / NT;
    constexpr int kW16Batch = w16_batch<MT>();
    __shared__ float red[8][MT * 4][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = warp % NT, kq = warp / NT;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int gpw = (G + KQ - 1) / KQ;
    const int gbeg = min(G, kq * gpw), gend = min(G, gbeg + gpw);
    const int n0 = (blockIdx.x * NT + nt) * 8;
    const int wrow = n0 + g;          // W row whose bytes this lane loads
    const int c0 = n0 + 2 * t;        // the two output columns this lane accumulates
    const int64_t wstride = K / 2;
    const int64_t sstride = G;

    pdl_launch_dependents();

    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;

    bool waited = false;
    for (int gb = gbeg; gb < gend; gb += kW16Batch) {
        uint4 w[kW16Batch];
        float s0[kW16Batch], s1[kW16Batch];
#pragma unroll
        for (int b = 0; b < kW16Batch; ++b) {
            const int gi = gb + b;
            w[b] = make_uint4(0u, 0u, 0u, 0u);  // decodes to zeros
            s0[b] = 0.f;
            s1[b] = 0.f;
            if (gi < gend) {
                if (wrow < N) w[b] = ld_stream_u4(Wq + wrow * wstride + gi * 64 + 16 * t);
                if (c0 < N) s0[b] = __half2float(S[c0 * sstride + gi]);
                if (c0 + 1 < N) s1[b] = __half2float(S[(c0 + 1) * sstride + gi]);
            }
        }
        if (!waited) {
            pdl_wait_prior_grid();  // X may be the previous kernel's output
            waited = true;
        }
#pragma unroll
        for (int b = 0; b < kW16Batch; ++b) {
            const int gi = gb + b;
            if (gi >= gend) break;
            float tmp[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) tmp[mt][i] = 0.f;
            const uint32_t wv[4] = {w[b].x, w[b].y, w[b].z, w[b].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t p[4];
                dequant_word(wv[i], p);
                const int kx = gi * kGroup + 32 * t + 8 * i;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int ra = mt * 16 + g, rb = ra + 8;
                    uint32_t xa[4] = {0u, 0u, 0u, 0u}, xb[4] = {0u, 0u, 0u, 0u};
                    if (ra < M) x_pairs(X + ra * ldx + kx, xa);
                    if (rb < M) x_pairs(X + rb * ldx + kx, xb);
                    const uint32_t a0[4] = {xa[0], xb[0], xa[1], xb[1]};
                    const uint32_t a1[4] = {xa[2], xb[2], xa[3], xb[3]};
                    mma_16816(tmp[mt], a0, p[0], p[1]);
                    mma_16816(tmp[mt], a1, p[2], p[3]);
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[mt][0] = fmaf(tmp[mt][0], s0[b], acc[mt][0]);
                acc[mt][1] = fmaf(tmp[mt][1], s1[b], acc[mt][1]);
                acc[mt][2] = fmaf(tmp[mt][2], s0[b], acc[mt][2]);
                acc[mt][3] = fmaf(tmp[mt][3], s1[b], acc[mt][3]);
            }
        }
    }
    if (!waited) pdl_wait_prior_grid();

    // Sum the KQ partial tiles of each n tile.
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][mt * 4 + i][lane] = acc[mt][i];
    __syncthreads();
    if (kq != 0) return;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < KQ; ++q) sum += red[q * NT + nt][mt * 4 + i][lane];
            v[i] = sum;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = mt * 16 + g + 8 * h;
            if (row >= M) continue;
            __half* dst = Y + row * ldy + c0;
            if (c0 + 1 < N && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(v[2 * h], v[2 * h + 1]);
            } else {
                if (c0 < N) dst[0] = __float2half_rn(v[2 * h]);
                if (c0 + 1 < N) dst[1] = __float2half_rn(v[2 * h + 1]);
            }
        }
    }
}

// ---------------------------------------------------------------- decode
//
// Decode shapes (M <= 16) compute Y^T = W . X^T: the weights are the MMA's A
// operand (16 weight rows per m16n8k16) and X^T the B operand (8 batch rows
// per MMA), so a batch of one wastes 7/8 of an MMA instead of 15/16.
//
// In a chain of layers a call can only use X once the previous call has
// finished, so everything that does not need X comes first:
//  - at entry 16 lanes bulk-copy the CTA's 16 weight rows into shared memory
//    (cp.async.bulk, the whole slab in flight at once) and the CTA copies the
//    rows' group scales next to them, before the previous kernel has
//    finished;
//  - after griddepcontrol.wait each warp loads the X values of its own K
//    slice straight into MMA fragment registers.
// The arithmetic after the wait is spread over 16 warps (warp w on K slice
// w) so that the part of a call that cannot overlap the previous one stays
// short.  The per-weight work is the dequantization, exact in fp16: one lop3
// per fp16 pair does the two's-complement fix (XOR 8), the mask and the
// exponent OR at once; even k gives 1024 + (v + 8) (minus 1032 -> v), odd k
// gives 1024 + 16 (v + 8) (times 1/16 minus 72 -> v).  Group scales are
// applied in fp32 after each group's MMAs; the 16 slices' partial tiles are
// added through shared memory.
constexpr int kDecWarps = 16;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kWRowPad = 64;
constexpr size_t kDecMaxSmem = 200 * 1024;  // dynamic shared memory
constexpr int kSiteW16Bulk = 301;
constexpr int kSiteW16Drain = 302;

// Shared memory of one CTA: 16 weight rows of K/2 bytes (+ pad), the rows'
// group scales (16 x (G + 2) halves: the odd word stride spreads the rows over
// the banks), and the partial tiles of the 16 warps.
__host__ __device__ constexpr size_t dec_w_bytes(int64_t K) { return 16 * static_cast<size_t>(K / 2 + kWRowPad); }
__host__ __device__ constexpr size_t dec_s_stride(int64_t K) { return static_cast<size_t>(K / 128 + 2); }
__host__ __device__ constexpr size_t dec_smem_bytes(int64_t M, int64_t K) {
    return dec_w_bytes(K) + ((16 * dec_s_stride(K) * 2 + 15) / 16) * 16 +
           static_cast<size_t>(kDecWarps) * (M <= 8 ? 1 : 2) * 4 * 32 * 4;
}

// d = b ? (c ? ~a : a) : c, bitwise: with b = mask and c = (exponent bits
// outside the mask) | (8-bits inside it), one instruction XORs the nibbles
// with 8, keeps them and ORs in the fp16 exponent.
__device__ __forceinline__ uint32_t lop3_nib(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Exact fp16 pairs of the 8 signed nibbles of `w` (nibble j = physical k_j):
// p[0] = (k0, k4), p[1] = (k1, k5), p[2] = (k2, k6), p[3] = (k3, k7).
__device__ __forceinline__ void dequant_word_fast(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    const uint32_t e0 = lop3_nib(w, 0x000F000Fu, 0x64086408u);   // 1024 + n ^ 8
    const uint32_t e1 = lop3_nib(w, 0x00F000F0u, 0x64806480u);   // 1024 + 16 (n ^ 8)
    const uint32_t e2 = lop3_nib(w8, 0x000F000Fu, 0x64086408u);
    const uint32_t e3 = lop3_nib(w8, 0x00F000F0u, 0x64806480u);
    const __half2 c1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 c16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const __half2 cm72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
    __half2 v0 = __hsub2(*reinterpret_cast<const __half2*>(&e0), c1032);
    __half2 v1 = __hfma2(*reinterpret_cast<const __half2*>(&e1), c16th, cm72);
    __half2 v2 = __hsub2(*reinterpret_cast<const __half2*>(&e2), c1032);
    __half2 v3 = __hfma2(*reinterpret_cast<const __half2*>(&e3), c16th, cm72);
    p[0] = *reinterpret_cast<uint32_t*>(&v0);
    p[1] = *reinterpret_cast<uint32_t*>(&v1);
    p[2] = *reinterpret_cast<uint32_t*>(&v2);
    p[3] = *reinterpret_cast<uint32_t*>(&v3);
}

// X fragment of 8 consecutive k (one 16-byte load) in the pair order of
// dequant_word_fast: (x0, x4), (x1, x5), (x2, x6), (x3, x7).
__device__ __forceinline__ uint4 x_pairs(uint4 v) {
    return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                      __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

template <int MB>  // batch tiles of 8 rows: M <= 8 * MB
__global__ void __launch_bounds__(kDecThreads, 2)
    k_w4a16_dec(int M, int N, int K, const __half* __restrict__ X, int64_t ldx,
                const uint8_t* __restrict__ Wq, const __half* __restrict__ S, __half* __restrict__ Y,
                int64_t ldy, const Ctl ctl) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int gpw = (G + kDecWarps - 1) / kDecWarps;
    const int gbeg = min(G, warp * gpw), gend = min(G, gbeg + gpw);
    const int n0 = blockIdx.x * 16;
    const int rows = min(16, N - n0);
    const int wrs = K / 2 + kWRowPad;                           // bytes per staged weight row
    const int sst = static_cast<int>(dec_s_stride(K));          // halves per staged scale row
    uint8_t* ws = dsm;
    unsigned short* ss = reinterpret_cast<unsigned short*>(dsm + dec_w_bytes(K));
    float* red = reinterpret_cast<float*>(dsm + dec_w_bytes(K) + ((16 * sst * 2 + 15) / 16) * 16);
    const uint32_t bar = smem_u32(&wbar);

    if (threadIdx.x == 0) {
        failed = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        // one row per lane, issued in parallel
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows) * (K / 2));
        __syncwarp();
        if (lane < rows)
            bulk_copy_g2s(smem_u32(ws + lane * wrs), Wq + static_cast<int64_t>(n0 + lane) * (K / 2),
                          static_cast<uint32_t>(K / 2), bar);
    }
    pdl_launch_dependents();
    // group scales of the 16 rows (raw 16-bit; rows past N read as 0)
    for (int i = threadIdx.x; i < 16 * G; i += kDecThreads) {
        const int r = i / G, gi = i - r * G;
        ss[r * sst + gi] = r < rows ? ld_nc_u16(S + static_cast<int64_t>(n0 + r) * G + gi) : 0;
    }
    __syncthreads();  // scales staged

    // X may be the previous kernel's output: read it only now.
    pdl_wait_prior_grid();
    if (!bounded_wait(bar, 0u, nullptr, ctl, kSiteW16Bulk)) {
        failed = 1;
        if (lane == 0) bounded_wait(bar, 0u, nullptr, ctl, kSiteW16Drain);
    }

    float acc[MB][4];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mb][i] = 0.f;

    for (int gi = gbeg; gi < gend; ++gi) {
        // X fragments of this group: lane (g, t) holds batch row mb*8 + g at
        // k = 32t + 8i + 0..7, i = 0..3
        uint4 xf[MB][4];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
            const int m = mb * 8 + g;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                xf[mb][i] = m < M ? x_pairs(ld_x_u4(
                                        X + static_cast<int64_t>(m) * ldx + gi * kGroup + 32 * t + 8 * i))
                                  : make_uint4(0u, 0u, 0u, 0u);
        }
        uint4 w0 = make_uint4(0u, 0u, 0u, 0u);  // nibbles 0: rows past N contribute 0
        uint4 w1 = w0;
        if (g < rows) w0 = *reinterpret_cast<const uint4*>(ws + g * wrs + gi * 64 + 16 * t);
        if (g + 8 < rows) w1 = *reinterpret_cast<const uint4*>(ws + (g + 8) * wrs + gi * 64 + 16 * t);
        float tmp[MB][4];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int i = 0; i < 4; ++i) tmp[mb][i] = 0.f;
        const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w};
        const uint32_t wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t pa[4], pb[4];
            dequant_word_fast(wa[i], pa);
            dequant_word_fast(wb[i], pb);
            const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
                mma_16816(tmp[mb], a0, xf[mb][i].x, xf[mb][i].y);
                mma_16816(tmp[mb], a1, xf[mb][i].z, xf[mb][i].w);
            }
        }
        const float sc0 = __half2float(__ushort_as_half(ss[g * sst + gi]));
        const float sc1 = __half2float(__ushort_as_half(ss[(g + 8) * sst + gi]));
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
            acc[mb][0] = fmaf(tmp[mb][0], sc0, acc[mb][0]);
            acc[mb][1] = fmaf(tmp[mb][1], sc0, acc[mb][1]);
            acc[mb][2] = fmaf(tmp[mb][2], sc1, acc[mb][2]);
            acc[mb][3] = fmaf(tmp[mb][3], sc1, acc[mb][3]);
        }
    }

#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[(warp * MB * 4 + mb * 4 + i) * 32 + lane] = acc[mb][i];
    __syncthreads();
    if (warp >= MB || failed) return;
    // warp mb writes batch tile mb: lane (g, t) holds Y[mb*8 + 2t + {0,1}][n0 + g / n0 + g + 8]
    const int mb = warp;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kDecWarps; ++q) sum += red[(q * MB * 4 + mb * 4 + i) * 32 + lane];
        v[i] = sum;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int m = mb * 8 + 2 * t + j;
        if (m >= M) continue;
        if (g < rows) Y[m * ldy + n0 + g] = __float2half_rn(v[j]);
        if (g + 8 < rows) Y[m * ldy + n0 + g + 8] = __float2half_rn(v[2 + j]);
    }
}

// ------------------------------------------------- decode, M <= 8 (GEMV)
//
// A chain of decode calls (one layer after another) is bound by two things:
// streaming the packed weights, and the latency of each call after the
// previous one has finished (griddepcontrol.wait returns ~0.7 us after the
// last CTA of the previous grid has left).  This kernel is shaped so that the
// first overlaps the second:
//  - one CTA per SM, using at most half of the SM (512 threads, <= 64
//    registers, <= ~110 KB of shared memory), so the next call's CTAs are
//    resident while this call computes and their weight rows (bulk copies)
//    and scales are in flight before this call ends; the CTA owns R
//    consecutive weight rows (R = N / #SMs rounded up, at most 32) and all
//    of K;
//  - the work after the wait is cut to the arithmetic that needs X.  A
//    nibble n (offset binary, v + 8) masked into the low mantissa bits of a
//    zero-exponent fp16 word IS the fp16 subnormal n * 2^-24: no exponent
//    OR, no subtraction, so a 32-bit word of 8 weights costs one shift and
//    four lop3 (even k at bits 0-3 of each half: n * 2^-24; odd k at bits
//    4-7: 16 n * 2^-24).  Even and odd k go to separate MMAs and
//    accumulators (the odd one carries the factor 16), and the offset 8 is
//    removed by starting each group's even accumulator at
//    -8 * 2^-24 * sum(x over the group) (the sum in fp32, fixed order),
//    computed once per call when X is staged; the weights stay exact.  Every
//    product is exact (an 11-bit by 4-bit product in fp32);
//    the scale s * 2^24 (even) and s * 2^20 (odd) is applied in fp32 per
//    group, as in the other W4A16 kernels.
//  - X (M x K) is staged once into shared memory, already permuted into the
//    MMA's pair order, together with the group sums.
// With T m16 tiles per CTA, warp w works on tile w / (16 / T) and on every
// (16 / T)-th group; rows past the CTA's are computed on its last row's data
// and never stored, batch columns past M read a zero slot, so the loop has no
// predicated loads.  The warps' partial tiles are added through shared memory
// in one pass.
constexpr int kD1Warps = 16;
constexpr int kD1Threads = 32 * kD1Warps;
constexpr int kD1MaxRows = 32;                  // two m16 tiles
constexpr size_t kD1Budget = 110 * 1024;        // two calls' CTAs share an SM
constexpr int kSiteW16D1Bulk = 303;
constexpr int kSiteW16D1Drain = 304;

// Shared-memory layout of k_w4a16_gemv for R rows, M batch rows, K.
struct D1Layout {
    int64_t wrs;        // bytes per staged weight row (K/2 + 64: rows g and g+8 on other banks)
    int64_t xrs;        // 16-byte slots per staged X row (16 per group + 4)
    int64_t srs;        // floats per scale row (2 per group + 2)
    int64_t w_off, x_off, c_off, s_off, red_off, bytes;
};
inline D1Layout d1_layout(int64_t M, int64_t K, int64_t R) {
    D1Layout L;
    const int64_t G = K / 128;
    L.wrs = K / 2 + 64;
    L.xrs = G * 16 + 4;
    L.srs = 2 * G + 2;
    L.w_off = 0;
    L.x_off = L.w_off + R * L.wrs;
    L.c_off = L.x_off + (M * L.xrs + 1) * 16;  // + one zero slot
    L.s_off = L.c_off + G * 8 * 4;
    L.red_off = L.s_off + ((R * L.srs * 4 + 15) / 16) * 16;
    L.bytes = L.red_off + static_cast<int64_t>(kD1Warps) * 16 * M * 4;
    return L;
}

// The same layout narrowed for the kernel (all offsets below the budget).
struct D1Off {
    int wrs, xrs, srs, x_off, c_off, s_off, red_off;
};
inline D1Off d1_off(const D1Layout& L) {
    return D1Off{static_cast<int>(L.wrs), static_cast<int>(L.xrs), static_cast<int>(L.srs),
                 static_cast<int>(L.x_off), static_cast<int>(L.c_off), static_cast<int>(L.s_off),
                 static_cast<int>(L.red_off)};
}

// d = a . b + c (m16n8k16, fp16 inputs, fp32 accumulators), c separate from d.
__device__ __forceinline__ void mma_16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                            float c0, float c1, float c2, float c3) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// 16-byte shared-memory load by the lanes whose `pred` is set; the others
// get zeros and issue no access, so a warp whose active lanes sit in one
// quarter costs one shared-memory wavefront instead of four.
__device__ __forceinline__ uint4 lds128_if(const void* p, bool pred) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    asm("{\n.reg .pred q;\nsetp.ne.b32 q, %5, 0;\n@q ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n}"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "r"(smem_u32(p)), "r"(static_cast<int>(pred)));
    return v;
}

// (a ^ c) & b: the nibbles under mask b, XORed with 8 (two's complement ->
// offset binary), nothing else: an fp16 subnormal n * 2^-24 (or 16 n * 2^-24).
__device__ __forceinline__ uint32_t nib_sub(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x48;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// T: m16 tiles per CTA (R <= 16 T).  GPW: groups per warp when it is known
// at compile time (the group loop then unrolls: about 10% fewer cycles in the
// loop), 0 for any K.
template <int T, int GPW>
__global__ void __launch_bounds__(kD1Threads, 2)
    k_w4a16_gemv(int M, int N, int K, const __half* __restrict__ X, int64_t ldx,
                 const uint8_t* __restrict__ Wq, const __half* __restrict__ S, __half* __restrict__ Y,
                 int64_t ldy, int R, const D1Off L, const Ctl ctl) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup, K8 = K / 8;
    const int n0 = blockIdx.x * R;
    const int rows = min(R, N - n0);
    uint8_t* ws = dsm;
    uint4* xs = reinterpret_cast<uint4*>(dsm + L.x_off);
    float* cs = reinterpret_cast<float*>(dsm + L.c_off);
    float* sp = reinterpret_cast<float*>(dsm + L.s_off);
    float* red = reinterpret_cast<float*>(dsm + L.red_off);
    const uint32_t bar = smem_u32(&wbar);

    if (threadIdx.x == 0) {
        failed = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {  // the CTA's weight rows, one bulk copy per row
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows) * (K / 2));
        __syncwarp();
        for (int r = lane; r < rows; r += 32)
            bulk_copy_g2s(smem_u32(ws + r * L.wrs), Wq + static_cast<int64_t>(n0 + r) * (K / 2),
                          static_cast<uint32_t>(K / 2), bar);
    }
    pdl_launch_dependents();
    // scales in fp32, pre-multiplied by 2^24 (even k) and 2^20 (odd k)
    for (int i = threadIdx.x; i < rows * G; i += kD1Threads) {
        const int r = i / G, gi = i - r * G;
        const float sc = __half2float(__ushort_as_half(ld_nc_u16(S + static_cast<int64_t>(n0 + r) * G + gi)));
        *reinterpret_cast<float2*>(sp + r * L.srs + 2 * gi) = make_float2(sc * 16777216.f, sc * 1048576.f);
    }

    // X may be the previous kernel's output: read it only now.
    pdl_wait_prior_grid();
    // Stage X: chunk j = 8 consecutive k of row m, stored as the pairs
    // (x0,x4) (x2,x6) (x1,x5) (x3,x7) at slot (g_i * 4 + i) * 4 + t of row m,
    // where k = 128 g_i + 32 t + 8 i; 16 consecutive chunks make a group,
    // whose sum (fp32, fixed order) gives the even accumulator's start.
    for (int m = 0; m < M; ++m) {
        const __half* xr = X + static_cast<int64_t>(m) * ldx;
        uint4* xsr = xs + m * L.xrs;
        for (int cb = warp * 32; cb < K8; cb += kD1Threads) {  // whole warps: the sums shuffle
            const int c8 = cb + lane;
            const bool ok = c8 < K8;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (ok) v = ld_x_u4(xr + 8 * c8);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[q]));
                sum += f.x;
                sum += f.y;
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (ok) {
                const int gi = c8 >> 4, u = c8 & 15;
                xsr[(gi * 4 + (u & 3)) * 4 + (u >> 2)] =
                    make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.y, v.w, 0x5410),
                               __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x7632));
                if (u == 0) cs[gi * 8 + m] = -4.76837158203125e-07f * sum;  // -8 * 2^-24
            }
        }
    }
    for (int i = threadIdx.x; i < G * 8; i += kD1Threads)  // batch columns past M
        if ((i & 7) >= M) cs[i] = 0.f;
    if (threadIdx.x == 0) xs[L.xrs * M] = make_uint4(0u, 0u, 0u, 0u);
    if (!bounded_wait(bar, 0u, nullptr, ctl, kSiteW16D1Bulk)) {
        failed = 1;
        if (lane == 0) bounded_wait(bar, 0u, nullptr, ctl, kSiteW16D1Drain);
    }
    __syncthreads();  // X, group sums and (unless failed) weights staged

    // warp w: tile w / WPT, groups w % WPT, w % WPT + WPT, ...
    constexpr int WPT = kD1Warps / T;
    const int tt = warp / WPT, gw = warp - tt * WPT;
    // Rows past the CTA's are computed on the data of its last row and never
    // stored; batch columns past M read a zero slot.
    const int r0 = min(16 * tt + g, rows - 1), r1 = min(16 * tt + g + 8, rows - 1);
    const uint8_t* wrow0 = ws + r0 * L.wrs + 16 * t;
    const uint8_t* wrow1 = ws + r1 * L.wrs + 16 * t;
    const float* srow0 = sp + r0 * L.srs;
    const float* srow1 = sp + r1 * L.srs;
    // Lanes of batch columns past M read nothing (zeros): with M <= 2 only
    // the first eight lanes load X, one wavefront per load instead of four.
    const bool xlane = g < M;
    const uint4* xbase = xlane ? xs + g * L.xrs + t : xs + L.xrs * M;  // zero slot after the rows
    const int xstep = xlane ? 4 : 0, xgs = xlane ? 16 : 0;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    auto group = [&](const int gi) {
        const uint4* xrow = xbase + xgs * gi;
        const float2 cc = *reinterpret_cast<const float2*>(cs + gi * 8 + 2 * t);
        const uint4 w0 = *reinterpret_cast<const uint4*>(wrow0 + gi * 64);
        const uint4 w1 = *reinterpret_cast<const uint4*>(wrow1 + gi * 64);
        const float2 s0 = *reinterpret_cast<const float2*>(srow0 + 2 * gi);
        const float2 s1 = *reinterpret_cast<const float2*>(srow1 + 2 * gi);
        float ae[4], ao[4];
        const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w}, wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t ha = wa[i] >> 8, hb = wb[i] >> 8;
            const uint32_t ev[4] = {nib_sub(wa[i], 0x000F000Fu, 0x00080008u), nib_sub(wb[i], 0x000F000Fu, 0x00080008u),
                                    nib_sub(ha, 0x000F000Fu, 0x00080008u), nib_sub(hb, 0x000F000Fu, 0x00080008u)};
            const uint32_t od[4] = {nib_sub(wa[i], 0x00F000F0u, 0x00800080u), nib_sub(wb[i], 0x00F000F0u, 0x00800080u),
                                    nib_sub(ha, 0x00F000F0u, 0x00800080u), nib_sub(hb, 0x00F000F0u, 0x00800080u)};
            const uint4 xf = lds128_if(xrow + xstep * i, xlane);
            if (i == 0) {
                mma_16816_c(ae, ev, xf.x, xf.y, cc.x, cc.y, cc.x, cc.y);
                mma_16816_c(ao, od, xf.z, xf.w, 0.f, 0.f, 0.f, 0.f);
            } else {
                mma_16816(ae, ev, xf.x, xf.y);
                mma_16816(ao, od, xf.z, xf.w);
            }
        }
        y[0] = fmaf(s0.y, ao[0], fmaf(s0.x, ae[0], y[0]));
        y[1] = fmaf(s0.y, ao[1], fmaf(s0.x, ae[1], y[1]));
        y[2] = fmaf(s1.y, ao[2], fmaf(s1.x, ae[2], y[2]));
        y[3] = fmaf(s1.y, ao[3], fmaf(s1.x, ae[3], y[3]));
        };
    if constexpr (GPW > 0) {
#pragma unroll
        for (int j = 0; j < GPW; ++j) group(gw + j * WPT);
    } else {
        for (int gi = gw; gi < G; gi += WPT) group(gi);
    }

    // partial tiles: red[warp][row][m] (the warp's tile), batch columns < M only
    {
        float* rw = red + warp * 16 * M;
        if (2 * t < M) {
            rw[g * M + 2 * t] = y[0];
            rw[(g + 8) * M + 2 * t] = y[2];
        }
        if (2 * t + 1 < M) {
            rw[g * M + 2 * t + 1] = y[1];
            rw[(g + 8) * M + 2 * t + 1] = y[3];
        }
    }
    __syncthreads();
    if (failed) return;
    // output (m, r): sum of the WPT partials of r's tile, in warp order
    for (int m = 0; m < M; ++m)
        for (int r = threadIdx.x; r < rows; r += kD1Threads) {
            const float* pr = red + ((r >> 4) * WPT * 16 + (r & 15)) * M + m;
            float v[WPT];
#pragma unroll
            for (int w = 0; w < WPT; ++w) v[w] = pr[w * 16 * M];
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < WPT; ++w) sum += v[w];
            Y[static_cast<int64_t>(m) * ldy + n0 + r] = __float2half_rn(sum);
        }
}

// ------------------------------------- decode, 9 <= M <= 16 (batched GEMV)
//
// The co-resident shape of k_w4a16_gemv (one CTA per SM at half its
// resources, R <= 32 weight rows bulk-copied before the dependency wait) for
// batches whose X (M x K fp16) does not fit next to the weights: after the
// wait every warp reads the X fragments of its own groups straight from L2
// (prefetching the next group's while it computes this one).  Two batch tiles
// share every dequantized A fragment.  The nibbles become exact fp16 integers
// (one lop3 per pair: two's-complement fix, mask and exponent of 1024; then
// one fp16 subtract or fused multiply-add), so no group sums are needed; the
// group scale is applied in fp32 per group.  Warp w takes groups w, w + 8, ...
// for both m16 tiles; the partial tiles are added through shared memory.
constexpr int kD2Warps = 8;
constexpr int kD2Threads = 32 * kD2Warps;
constexpr int kSiteW16D2Bulk = 305;
constexpr int kSiteW16D2Drain = 306;

struct D2Off {
    int wrs, srs, s_off, red_off;
};
inline int64_t d2_bytes(int64_t M, int64_t K, int64_t R, D2Off* off) {
    const int64_t G = K / 128;
    const int64_t wrs = K / 2 + 64, srs = G + 1;
    const int64_t s_off = R * wrs;
    const int64_t red_off = s_off + ((R * srs * 4 + 15) / 16) * 16;
    const int64_t bytes = red_off + static_cast<int64_t>(kD2Warps) * 2 * 16 * M * 4;
    if (off) *off = D2Off{static_cast<int>(wrs), static_cast<int>(srs), static_cast<int>(s_off),
                          static_cast<int>(red_off)};
    return bytes;
}

// T: m16 tiles per CTA (R <= 16 T); GPW: groups per warp if known at
// compile time (the group loop unrolls), else 0.
template <int T, int GPW>
__global__ void __launch_bounds__(kD2Threads, 2)
    k_w4a16_gemv16(int M, int N, int K, const __half* __restrict__ X, int64_t ldx,
                   const uint8_t* __restrict__ Wq, const __half* __restrict__ S, __half* __restrict__ Y,
                   int64_t ldy, int R, const D2Off L, const Ctl ctl) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / kGroup;
    const int n0 = blockIdx.x * R;
    const int rows = min(R, N - n0);
    uint8_t* ws = dsm;
    float* sp = reinterpret_cast<float*>(dsm + L.s_off);
    float* red = reinterpret_cast<float*>(dsm + L.red_off);
    const uint32_t bar = smem_u32(&wbar);

    if (threadIdx.x == 0) {
        failed = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {  // the CTA's weight rows, one bulk copy per row
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows) * (K / 2));
        __syncwarp();
        for (int r = lane; r < rows; r += 32)
            bulk_copy_g2s(smem_u32(ws + r * L.wrs), Wq + static_cast<int64_t>(n0 + r) * (K / 2),
                          static_cast<uint32_t>(K / 2), bar);
    }
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < rows * G; i += kD2Threads) {
        const int r = i / G, gi = i - r * G;
        sp[r * L.srs + gi] = __half2float(__ushort_as_half(ld_nc_u16(S + static_cast<int64_t>(n0 + r) * G + gi)));
    }
    __syncthreads();  // scales staged

    // X may be the previous kernel's output: read it only now.
    pdl_wait_prior_grid();
    if (!bounded_wait(bar, 0u, nullptr, ctl, kSiteW16D2Bulk)) {
        failed = 1;
        if (lane == 0) bounded_wait(bar, 0u, nullptr, ctl, kSiteW16D2Drain);
    }
    __syncthreads();

    // rows past the CTA's are computed on its last row's data and never stored
    int roff[T][2];
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
        roff[tt][0] = min(16 * tt + g, rows - 1);
        roff[tt][1] = min(16 * tt + g + 8, rows - 1);
    }
    // X fragments: lane (g, t), batch tile mb holds row 8 mb + g at
    // k = 128 g_i + 32 t + 8 i + 0..7 as (x0,x4) (x1,x5) (x2,x6) (x3,x7)
    const bool xv0 = g < M, xv1 = 8 + g < M;
    const __half* xr0 = X + static_cast<int64_t>(xv0 ? g : 0) * ldx + 32 * t;
    const __half* xr1 = X + static_cast<int64_t>(xv1 ? 8 + g : 0) * ldx + 32 * t;
    auto load_x = [&](int gi, uint4 (&xf)[2][4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            xf[0][i] = xv0 ? x_pairs(ld_x_u4(xr0 + gi * kGroup + 8 * i))
                           : make_uint4(0u, 0u, 0u, 0u);
            xf[1][i] = xv1 ? x_pairs(ld_x_u4(xr1 + gi * kGroup + 8 * i))
                           : make_uint4(0u, 0u, 0u, 0u);
        }
    };

    float y[T][2][4];
#pragma unroll
    for (int tt = 0; tt < T; ++tt)
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int q = 0; q < 4; ++q) y[tt][mb][q] = 0.f;

    uint4 xn[2][4];
    if (warp < G) load_x(warp, xn);
    auto group = [&](const int gi) {
        uint4 xf[2][4];
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int i = 0; i < 4; ++i) xf[mb][i] = xn[mb][i];
        if (gi + kD2Warps < G) load_x(gi + kD2Warps, xn);  // next group's fragments in flight
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(ws + roff[tt][0] * L.wrs + gi * 64 + 16 * t);
            const uint4 w1 = *reinterpret_cast<const uint4*>(ws + roff[tt][1] * L.wrs + gi * 64 + 16 * t);
            const float s0 = sp[roff[tt][0] * L.srs + gi], s1 = sp[roff[tt][1] * L.srs + gi];
            float tmp[2][4];
            const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w}, wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t pa[4], pb[4];
                dequant_word_fast(wa[i], pa);
                dequant_word_fast(wb[i], pb);
                const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
                const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
                for (int mb = 0; mb < 2; ++mb) {
                    if (i == 0)
                        mma_16816_c(tmp[mb], a0, xf[mb][i].x, xf[mb][i].y, 0.f, 0.f, 0.f, 0.f);
                    else
                        mma_16816(tmp[mb], a0, xf[mb][i].x, xf[mb][i].y);
                    mma_16816(tmp[mb], a1, xf[mb][i].z, xf[mb][i].w);
                }
            }
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
                y[tt][mb][0] = fmaf(tmp[mb][0], s0, y[tt][mb][0]);
                y[tt][mb][1] = fmaf(tmp[mb][1], s0, y[tt][mb][1]);
                y[tt][mb][2] = fmaf(tmp[mb][2], s1, y[tt][mb][2]);
                y[tt][mb][3] = fmaf(tmp[mb][3], s1, y[tt][mb][3]);
            }
        }
        };
    if constexpr (GPW > 0) {
#pragma unroll
        for (int j = 0; j < GPW; ++j) group(warp + j * kD2Warps);
    } else {
        for (int gi = warp; gi < G; gi += kD2Warps) group(gi);
    }

    // partial tiles: red[warp][tile][row][m], batch rows < M only; lane (g, t)
    // holds rows g, g + 8 and batch rows 8 mb + 2t, 8 mb + 2t + 1
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
        float* rw = red + (warp * T + tt) * 16 * M;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int m = 8 * mb + 2 * t + j;
                if (m < M) {
                    rw[g * M + m] = y[tt][mb][j];
                    rw[(g + 8) * M + m] = y[tt][mb][2 + j];
                }
            }
    }
    __syncthreads();
    if (failed) return;
    // output (m, r): sum of the 8 warps' partials in warp order
    for (int o = threadIdx.x; o < rows * M; o += kD2Threads) {
        const int r = o / M, m = o - r * M;
        const float* pr = red + ((r >> 4) * 16 + (r & 15)) * M + m;
        float v[kD2Warps];
#pragma unroll
        for (int w = 0; w < kD2Warps; ++w) v[w] = pr[w * T * 16 * M];
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kD2Warps; ++w) sum += v[w];
        Y[static_cast<int64_t>(m) * ldy + n0 + r] = __float2half_rn(sum);
    }
}

static std::atomic<int> g_w4a16_pdl{1};
static std::atomic<int> g_w4a16_tc_form{0};  // 0: resident weights where they fit, 1: ring only

template <int MT, int NT>
static int launch_w4a16(int M, int N, int K, const __half* X, int64_t ldx, const uint8_t* Wq,
                        const __half* S, __half* Y, int64_t ldy, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + 8 * NT - 1) / (8 * NT)));
    cfg.blockDim = dim3(kW16Threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_w4a16_pdl.load() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return map_cuda(cudaLaunchKernelEx(&cfg, k_w4a16<MT, NT>, M, N, K, X, ldx, Wq, S, Y, ldy));
}

template <int MB>
static int launch_w4a16_dec(int M, int N, int K, const __half* X, int64_t ldx, const uint8_t* Wq,
                            const __half* S, __half* Y, int64_t ldy, size_t smem, const Ctl& ctl,
                            cudaStream_t s) {
    static std::atomic<int> attr_done{0};
    if (smem > 48 * 1024 && !attr_done.load()) {
        const cudaError_t e = cudaFuncSetAttribute(
            k_w4a16_dec<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kDecMaxSmem));
        if (e != cudaSuccess) return map_cuda(e);
        attr_done.store(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + 15) / 16));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_w4a16_pdl.load() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return map_cuda(cudaLaunchKernelEx(&cfg, k_w4a16_dec<MB>, M, N, K, X, ldx, Wq, S, Y, ldy, ctl));
}

// Rows per CTA of k_w4a16_gemv, or 0 when its staging does not fit.
static int d1_rows(int64_t M, int64_t N, int64_t K, int dev) {
    if (M > 8) return 0;
    const int64_t sms = num_sms(dev);
    int64_t R = (N + sms - 1) / sms;
    if (R > kD1MaxRows) R = kD1MaxRows;
    while (R > 1 && static_cast<size_t>(d1_layout(M, K, R).bytes) > kD1Budget) --R;
    if (static_cast<size_t>(d1_layout(M, K, R).bytes) > kD1Budget) return 0;
    return static_cast<int>(R);
}

static int launch_w4a16_gemv(int M, int N, int K, const __half* X, int64_t ldx, const uint8_t* Wq,
                             const __half* S, __half* Y, int64_t ldy, int R, const Ctl& ctl,
                             cudaStream_t s) {
    using KernelFn = void (*)(int, int, int, const __half*, int64_t, const uint8_t*, const __half*, __half*,
                              int64_t, int, D1Off, Ctl);
    const int T = R > 16 ? 2 : 1;
    const int gpw = (K / kGroup) % (kD1Warps / T) == 0 ? (K / kGroup) / (kD1Warps / T) : 0;
    KernelFn fn;
    if (T == 2)
        fn = gpw == 4 ? k_w4a16_gemv<2, 4> : gpw == 8 ? k_w4a16_gemv<2, 8> : k_w4a16_gemv<2, 0>;
    else
        fn = gpw == 2 ? k_w4a16_gemv<1, 2> : gpw == 4 ? k_w4a16_gemv<1, 4> : k_w4a16_gemv<1, 0>;
    static std::atomic<int> attr_done{0};
    if (!attr_done.load()) {
        const KernelFn all[6] = {k_w4a16_gemv<2, 4>, k_w4a16_gemv<2, 8>, k_w4a16_gemv<2, 0>,
                                 k_w4a16_gemv<1, 2>, k_w4a16_gemv<1, 4>, k_w4a16_gemv<1, 0>};
        for (KernelFn f : all) {
            const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kD1Budget));
            if (e != cudaSuccess) return map_cuda(e);
        }
        attr_done.store(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + R - 1) / R));
    cfg.blockDim = dim3(kD1Threads);
    const D1Layout lay = d1_layout(M, K, R);
    const D1Off off = d1_off(lay);
    cfg.dynamicSmemBytes = static_cast<size_t>(lay.bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_w4a16_pdl.load() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return map_cuda(cudaLaunchKernelEx(&cfg, fn, M, N, K, X, ldx, Wq, S, Y, ldy, R, off, ctl));
}

// Rows per CTA of k_w4a16_gemv16, or 0 when it does not fit.
static int d2_rows(int64_t M, int64_t N, int64_t K, int dev) {
    if (M > 16) return 0;
    const int64_t sms = num_sms(dev);
    int64_t R = (N + sms - 1) / sms;
    if (R > kD1MaxRows) R = kD1MaxRows;
    while (R > 1 && static_cast<size_t>(d2_bytes(M, K, R, nullptr)) > kD1Budget) --R;
    if (static_cast<size_t>(d2_bytes(M, K, R, nullptr)) > kD1Budget) return 0;
    return static_cast<int>(R);
}

static int launch_w4a16_gemv16(int M, int N, int K, const __half* X, int64_t ldx, const uint8_t* Wq,
                               const __half* S, __half* Y, int64_t ldy, int R, const Ctl& ctl,
                               cudaStream_t s) {
    using KernelFn = void (*)(int, int, int, const __half*, int64_t, const uint8_t*, const __half*, __half*,
                              int64_t, int, D2Off, Ctl);
    const int gpw = (K / kGroup) % kD2Warps == 0 ? (K / kGroup) / kD2Warps : 0;
    KernelFn fn;
    if (R > 16)
        fn = gpw == 4 ? k_w4a16_gemv16<2, 4> : k_w4a16_gemv16<2, 0>;
    else
        fn = gpw == 4 ? k_w4a16_gemv16<1, 4> : k_w4a16_gemv16<1, 0>;
    static std::atomic<int> attr_done{0};
    if (!attr_done.load()) {
        const KernelFn all[4] = {k_w4a16_gemv16<2, 4>, k_w4a16_gemv16<2, 0>, k_w4a16_gemv16<1, 4>,
                                 k_w4a16_gemv16<1, 0>};
        for (KernelFn f : all) {
            const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kD1Budget));
            if (e != cudaSuccess) return map_cuda(e);
        }
        attr_done.store(1);
    }
    D2Off off;
    const int64_t bytes = d2_bytes(M, K, R, &off);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + R - 1) / R));
    cfg.blockDim = dim3(kD2Threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_w4a16_pdl.load() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return map_cuda(cudaLaunchKernelEx(&cfg, fn, M, N, K, X, ldx, Wq, S, Y, ldy, R, off, ctl));
}
}  // namespace qg

#include "w4a16_tc.cuh"

namespace qg {

// Launches w4a16_tc_kernel<Cfg> for batch rows [m0, m0 + 128).
template <class Cfg>
static int launch_w4a16_tc(const CUtensorMap& tmX, const CUtensorMap& tmW, int M, int N, int K, int m0,
                           const __half* S, __half* Y, int64_t ldy, const Ctl& ctl, int dev,
                           cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(
                w4a16_tc_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
            if (e != cudaSuccess) return map_cuda(e);
            attr_set[dev] = true;
        }
    }
    W16TcParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.m0 = m0;
    p.Y = Y;
    p.ldy = ldy;
    p.S = S;
    p.ctl = ctl;
    const int tiles = (N + Cfg::BN - 1) / Cfg::BN;
    const int grid = tiles * Cfg::KSPLIT;  // a cluster per 128 output columns
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_w4a16_pdl.load() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return map_cuda(cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<Cfg>, tmX, tmW, p));
}

// Resource budgets of the instances launched above.  The GEMV kernels count
// on two CTAs per SM (the next call's CTAs start while this call's run).
#define QG_W16_BUDGET(FN, NAME, THREADS, SMEM, MIN_CTAS) \
    QG_KERNEL_BUDGET(NAME, reinterpret_cast<const void*>(FN), THREADS, SMEM, 0, 1, MIN_CTAS)
QG_W16_BUDGET((k_w4a16<1, 2>), "k_w4a16<1,2>", kW16Threads, 0, 1);
QG_W16_BUDGET((k_w4a16<2, 4>), "k_w4a16<2,4>", kW16Threads, 0, 1);
QG_W16_BUDGET((k_w4a16<4, 8>), "k_w4a16<4,8>", kW16Threads, 0, 1);
QG_W16_BUDGET((k_w4a16<8, 8>), "k_w4a16<8,8>", kW16Threads, 0, 1);
QG_W16_BUDGET((k_w4a16_dec<1>), "k_w4a16_dec<1>", kDecThreads, static_cast<int>(kDecMaxSmem), 1);
QG_W16_BUDGET((k_w4a16_dec<2>), "k_w4a16_dec<2>", kDecThreads, static_cast<int>(kDecMaxSmem), 1);
QG_W16_BUDGET((k_w4a16_gemv<2, 4>), "k_w4a16_gemv<2,4>", kD1Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv<2, 8>), "k_w4a16_gemv<2,8>", kD1Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv<2, 0>), "k_w4a16_gemv<2,0>", kD1Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv<1, 2>), "k_w4a16_gemv<1,2>", kD1Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv<1, 4>), "k_w4a16_gemv<1,4>", kD1Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv<1, 0>), "k_w4a16_gemv<1,0>", kD1Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv16<2, 4>), "k_w4a16_gemv16<2,4>", kD2Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv16<2, 0>), "k_w4a16_gemv16<2,0>", kD2Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv16<1, 4>), "k_w4a16_gemv16<1,4>", kD2Threads, static_cast<int>(kD1Budget), 2);
QG_W16_BUDGET((k_w4a16_gemv16<1, 0>), "k_w4a16_gemv16<1,0>", kD2Threads, static_cast<int>(kD1Budget), 2);
#undef QG_W16_BUDGET
QG_KERNEL_BUDGET("w4a16_tc_kernel<W16TcCfg>", reinterpret_cast<const void*>(w4a16_tc_kernel<W16TcCfg>),
                 W16TcCfg::THREADS, W16TcCfg::SMEM_BYTES, W16TcCfg::TMEM_COLS, W16TcCfg::KSPLIT, 1);
QG_KERNEL_BUDGET("w4a16_tc_kernel<W16TcResCfg>", reinterpret_cast<const void*>(w4a16_tc_kernel<W16TcResCfg>),
                 W16TcResCfg::THREADS, W16TcResCfg::SMEM_BYTES, W16TcResCfg::TMEM_COLS, W16TcResCfg::KSPLIT, 1);

}  // namespace qg

using namespace qg;

extern "C" {

int qg_set_pdl(int enable) {
    g_w4a16_pdl.store(enable ? 1 : 0);
    return QG_OK;
}

int qg_set_w4a16_tc_form(int form) {
    if (form != 0 && form != 1) return QG_ERR_INVALID_ARG;
    g_w4a16_tc_form.store(form);
    return QG_OK;
}

int w4a16_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* X, int64_t ldx, const uint8_t* Wq,
               const uint16_t* Wscale, int64_t group, uint16_t* Y, int64_t ldy, void* stream) {
    const qg::NvtxRange nvtx_range("w4a16_gemm");
    if (M < 1 || N < 1 || K < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return QG_ERR_INVALID_ARG;
    if (group != kGroup) return QG_ERR_UNSUPPORTED;
    if (K % kGroup) return QG_ERR_INVALID_ARG;
    if (!X || !Wq || !Wscale || !Y) return QG_ERR_INVALID_ARG;
    if (ldx < K || ldy < N) return QG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(Wscale) || !aligned16(Y) || ldx % 8)
        return QG_ERR_MISALIGNED;
    if (current_device() < 0) return QG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __half* Xh = reinterpret_cast<const __half*>(X);
    const __half* Sh = reinterpret_cast<const __half*>(Wscale);
    __half* Yh = reinterpret_cast<__half*>(Y);
    const int n = static_cast<int>(N), k = static_cast<int>(K);
    // Decode shapes: weight slab bulk-copied and X staged in shared memory,
    // weights as the A operand.
    // GEMV shapes: one CTA per SM, half an SM each, so consecutive calls overlap.
    if (M <= 8) {
        const int dev = current_device();
        if (dev < 0) return QG_ERR_CUDA;
        const int R = d1_rows(M, N, K, dev);
        if (R > 0) {
            const Ctl ctl = host_ctl(dev);
            if (!ctl.status) return QG_ERR_CUDA;
            return launch_w4a16_gemv(static_cast<int>(M), n, k, Xh, ldx, Wq, Sh, Yh, ldy, R, ctl, s);
        }
    }
    // Batched GEMV (X too large to stage): same co-resident shape, X from L2.
    if (M <= 16) {
        const int dev = current_device();
        if (dev < 0) return QG_ERR_CUDA;
        const int R = d2_rows(M, N, K, dev);
        if (R > 0) {
            const Ctl ctl = host_ctl(dev);
            if (!ctl.status) return QG_ERR_CUDA;
            return launch_w4a16_gemv16(static_cast<int>(M), n, k, Xh, ldx, Wq, Sh, Yh, ldy, R, ctl, s);
        }
    }
    const size_t dec_smem = dec_smem_bytes(M, K);
    if (M <= 16 && dec_smem <= kDecMaxSmem) {
        const int dev = current_device();
        if (dev < 0) return QG_ERR_CUDA;
        const Ctl ctl = host_ctl(dev);
        if (!ctl.status) return QG_ERR_CUDA;
        if (M <= 8)
            return launch_w4a16_dec<1>(static_cast<int>(M), n, k, Xh, ldx, Wq, Sh, Yh, ldy,
                                       dec_smem, ctl, s);
        return launch_w4a16_dec<2>(static_cast<int>(M), n, k, Xh, ldx, Wq, Sh, Yh, ldy, dec_smem,
                                   ctl, s);
    }
    // Larger batches: tensor cores, 128 batch rows per launch.
    if ((K / kGroup + W16TcCfg::KSPLIT - 1) / W16TcCfg::KSPLIT <= W16TcCfg::MAX_SLICE_GROUPS) {
        const int dev = current_device();
        if (dev < 0 || dev >= 64) return QG_ERR_CUDA;
        const Ctl ctl = host_ctl(dev);
        if (!ctl.status) return QG_ERR_CUDA;
        CUtensorMap tmX, tmW;
        int rc = make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, K, M, ldx * 2, W16TcCfg::BK,
                              W16TcCfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
        if (!rc) rc = make_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, K / 2, N, K / 2,
                                   W16TcCfg::BK / 2, W16TcCfg::BN, CU_TENSOR_MAP_SWIZZLE_NONE);
        // all packed rows of a K quarter resident when it holds <= 8 groups
        const bool res = g_w4a16_tc_form.load() == 0 &&
                         (K / kGroup + W16TcCfg::KSPLIT - 1) / W16TcCfg::KSPLIT <= W16TcResCfg::MAX_SLICE_GROUPS;
        for (int64_t r0 = 0; !rc && r0 < M; r0 += W16TcCfg::BM)
            rc = res ? launch_w4a16_tc<W16TcResCfg>(tmX, tmW, static_cast<int>(M), n, k, static_cast<int>(r0),
                                                    Sh, Yh, ldy, ctl, dev, s)
                     : launch_w4a16_tc<W16TcCfg>(tmX, tmW, static_cast<int>(M), n, k, static_cast<int>(r0), Sh,
                                                 Yh, ldy, ctl, dev, s);
        return rc;
    }
    // Rows are processed in chunks of up to 128 (8 m16 tiles per CTA).
    for (int64_t r0 = 0; r0 < M; r0 += 128) {
        const int m = static_cast<int>(M - r0 < 128 ? M - r0 : 128);
        const __half* Xr = Xh + r0 * ldx;
        __half* Yr = Yh + r0 * ldy;
        int rc;
        if (m <= 16)
            rc = launch_w4a16<1, 2>(m, n, k, Xr, ldx, Wq, Sh, Yr, ldy, s);
        else if (m <= 32)
            rc = launch_w4a16<2, 4>(m, n, k, Xr, ldx, Wq, Sh, Yr, ldy, s);
        else if (m <= 64)
            rc = launch_w4a16<4, 8>(m, n, k, Xr, ldx, Wq, Sh, Yr, ldy, s);
        else
            rc = launch_w4a16<8, 8>(m, n, k, Xr, ldx, Wq, Sh, Yr, ldy, s);
        if (rc) return rc;
    }
    return QG_OK;
}

}  // extern "C"

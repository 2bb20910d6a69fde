// Host-side helpers of the tcgen05 GEMM shared between translation units.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "qg_internal.h"

namespace qg {

// Encodes a 2-D tiled TMA map: `outer` rows of `inner` elements, rows
// `row_stride_bytes` apart, box of box_inner x box_outer elements.
int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int64_t inner,
                 int64_t outer, int64_t row_stride_bytes, int box_inner, int box_outer,
                 CUtensorMapSwizzle swizzle);

// Kernel choice set by qg_set_gemm_path: 0 by shape, 1 one CTA per tile,
// 2 CTA pairs.
int gemm_path();

// The caller-owned events of qg_set_profile_events (null when unset).
void profile_events(void** before, void** after);

// Encodes a 2-D TMA map over a K-major matrix (rows x k_elems, row stride in
// bytes) with the 128-byte swizzle and a box of box_k x box_rows elements.
// fp16 selects 2-byte elements, otherwise 1-byte elements.
int make_tmap_kmajor(CUtensorMap* map, bool fp16, const void* base, int64_t k_elems, int64_t rows,
                     int64_t row_stride_bytes, int box_k, int box_rows);

// fp16 tcgen05 GEMM with an fp16 epilogue: C = A . B^T (+ bias per column).
// A: M x K (lda elements), B: N x K (ldb elements), C: M x N (ldc elements).
int run_gemm_f16_tc(const __half* A, int64_t lda, const __half* B, int64_t ldb, int64_t M, int64_t N,
                    int64_t K, __half* C, int64_t ldc, const __half* bias, const Ctl& ctl,
                    cudaStream_t stream);

// int8 rows (K values, source row stride lds bytes) -> fp16 rows of K values
// (exact), destination rows K apart; one launch enqueued on `s`.  K is a
// multiple of 16.
int s8_to_f16_rows(const int8_t* src, int64_t rows, int64_t lds, __half* dst, int64_t K, int dev,
                   cudaStream_t s);

// The exact INT8 GEMM on operands already converted to fp16 (A16: M x K,
// B16: N x K, both with row stride K): C = A . B^T in int32 (ldc elements),
// with the K-chunk length qg_set_s8_chunk selects.
int run_gemm_s8_converted(const __half* A16, const __half* B16, int64_t M, int64_t N, int64_t K, int32_t* C,
                          int64_t ldc, const Ctl& ctl, cudaStream_t stream);

// Grid size for the elementwise grid-stride kernels (256 threads per block).
int conv_grid(int dev, int64_t work_items);

// Packed signed 4-bit rows (K values, low nibble = even k) of two operands
// -> one e4m3 byte per value (exact, destination row stride K bytes), one
// launch enqueued on `s`.  K is a multiple of 32.
// One operand of s4_to_e4m3_pair: rows of packed nibbles (row stride lds
// bytes) -> rows of K e4m3 bytes.
int s4_to_e4m3_rows(const uint8_t* src, int64_t rows, int64_t lds, uint8_t* dst, int64_t K, int dev,
                    cudaStream_t s);

int s4_to_e4m3_pair(const uint8_t* a, int64_t a_rows, int64_t a_lds, uint8_t* a_dst, const uint8_t* b,
                    int64_t b_rows, int64_t b_lds, uint8_t* b_dst, int64_t K, int dev, cudaStream_t s);

}  // namespace qg

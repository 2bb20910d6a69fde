/*
 * qgemm.h -- C ABI of the GB300 (sm_103a) quantized tensor-core GEMM library.
 *
 * Sources of the operations (web pages on the subject):
 *  [L4]   "Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study
 *          on NVIDIA L4" (arXiv 2608.10103), abstract: exact INT8 and INT4
 *          GEMM and the FP16 GEMM they are compared with.
 *  [SM75] "fused-int4-gemm-sm75" README: INT4 weight-only (W4A16) linear with
 *          register-level dequantization and per-group scales (group 128).
 *  [W4A4] "Warp-Specialized Kernel Implementation for W4A4 MatMul on Latest
 *          GPU Architectures", section 1: Y = (Q(X).Q(W)^T) (.) scale + L(X) + b.
 *
 * Conventions shared by every call
 *  - Matrix names follow the GEMM C = A . B, with A: M x K, B: K x N, C: M x N.
 *    A / X is stored row-major (QG_ROW_MAJOR, K contiguous).  B / W is stored
 *    K-major, i.e. column-major as a K x N matrix (QG_COL_MAJOR) which is the
 *    same bytes as an N x K row-major matrix.  C / Y is row-major.  Other
 *    layouts return QG_ERR_UNSUPPORTED.
 *  - "s4p": two signed 4-bit values per byte along K; the LOW nibble holds the
 *    even k, the HIGH nibble the odd k; each nibble is two's complement.
 *  - fp16 data is IEEE binary16 passed as uint16_t bit patterns.
 *  - Leading dimensions are in elements (in BYTES for s4p operands).
 *  - Every pointer is a DEVICE pointer owned by the caller.  The library never
 *    allocates, frees or synchronizes in these calls (qg_device_status is the
 *    one call that synchronizes).  Scratch memory, where a call needs it, is
 *    passed in as a workspace of at least qg_workspace_size() bytes.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  Calls are thread-safe.
 *  - Any M, N >= 1.  Divisibility of K is stated per call.
 *  - Alignment: every pointer 16-byte aligned; the leading dimension of every
 *    INPUT matrix times its element size a multiple of 16 bytes; otherwise
 *    QG_ERR_MISALIGNED.  Output leading dimensions only need ldc >= N (rows
 *    that start 16-byte aligned are written with vector stores).
 *  - Errors: argument errors are detected synchronously before any launch and
 *    nothing is enqueued.  A launch failure returns QG_ERR_CUDA.  Kernels bound
 *    every wait; a wait that runs out records QG_ERR_TIMEOUT in a device
 *    status word that qg_device_status() reports.  No call traps or aborts.
 *  - Per-device state (the status word's address, the no-alloc scratch
 *    address) is looked up once per device and kept for the life of the
 *    library: do not use the library on a device after cudaDeviceReset of
 *    that device in the same process.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad group/block/rank  */
    QG_ERR_UNSUPPORTED = 2,  /* layout or shape this build does not handle    */
    QG_ERR_MISALIGNED = 3,   /* pointer or leading dimension not 16B aligned  */
    QG_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required    */
    QG_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed             */
    QG_ERR_TIMEOUT = 6       /* a device-side bounded wait ran out            */
} qg_status;

typedef enum { QG_ROW_MAJOR = 0, QG_COL_MAJOR = 1 } qg_layout;

/* Operation ids for qg_workspace_size. */
typedef enum {
    QG_OP_S8 = 0, QG_OP_S4 = 1, QG_OP_F16 = 2, QG_OP_W4A16 = 3, QG_OP_W4A4 = 4, QG_OP_S8_HOST = 5,
    QG_OP_W4A4_PREPACKED = 6,  /* workspace of w4a4_gemm_prepacked */
    QG_OP_W4A4_WEIGHTS = 7     /* size of the buffer w4a4_prepack_weights fills (M unused: pass 1) */
} qg_op;

/* Human-readable name of a status code (static string, never NULL). */
const char *qg_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int qg_version(void);

/* Bytes of workspace the call `op` needs for an M x N x K problem (0 if none).
 * For QG_OP_W4A4, K is the quantized reduction dimension (the size covers a
 * low-rank term of rank up to 32). */
size_t qg_workspace_size(int op, int64_t M, int64_t N, int64_t K);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device: QG_OK, or QG_ERR_TIMEOUT if any kernel since the last
 * call gave up on a bounded wait.  A failed CUDA call returns QG_ERR_CUDA. */
int qg_device_status(void *stream);

/* As qg_device_status, and also copies the whole status word into words[6]
 * (words may be NULL): {error code, call-site tag of the role that gave up,
 * number of errors recorded, block index, phase parity that wait expected,
 * shared-memory address of the barrier it waited on}.  The tag and the last
 * two words say which role, which ring slot and which phase stalled. */
int qg_device_status_detail(int *words, void *stream);

/* Diagnostics: the code of the most recent failed CUDA call behind a
 * QG_ERR_CUDA (a cudaError_t, or minus a CUresult for a driver call such as
 * the tensor-map encoder), 0 if none; reading it clears it. */
int qg_last_cuda_error(void);

/* Sets the limit of every device-side wait, in nanoseconds (default 2e9;
 * also read once from the environment variable QG_TIMEOUT_NS).  0 restores
 * the default. */
int qg_set_timeout_ns(uint64_t ns);

/* Resource budget of one kernel instance of the library: what one CTA asks
 * of an SM and how many CTAs of it the design relies on finding resident per
 * SM (two for the W4A16 GEMV kernels and the W4A4 quantizer, whose next call
 * starts while the current one runs; one for the tensor-memory kernels, which
 * must never share an SM with a second CTA of themselves, since the tensor
 * memory of an SM is 512 columns).  `kernel` is a static string. */
typedef struct {
    const char *kernel;   /* kernel name with its template arguments */
    int threads;          /* threads per CTA */
    int smem_bytes;       /* largest dynamic shared memory a launch requests */
    int tmem_cols;        /* tensor-memory columns each CTA allocates (0 = none) */
    int cluster;          /* CTAs per thread-block cluster */
    int min_ctas_per_sm;  /* CTAs the design needs resident on one SM */
} qg_kernel_budget;

/* Number of kernel instances in the budget table (host only, no device). */
int qg_kernel_budget_count(void);

/* Copies entry `index` (0 .. count-1) into *out; host only.
 * QG_ERR_INVALID_ARG for an index out of range or a NULL out. */
int qg_kernel_budget_get(int index, qg_kernel_budget *out);

/* Needs a device: the compiled kernel's registers per thread and static
 * shared memory, and the CTAs per SM that the device would keep resident at
 * the entry's threads and dynamic shared memory (the runtime's occupancy
 * calculator; it raises the kernel's dynamic shared-memory limit to the
 * entry's size first, as the launcher does).  QG_ERR_CUDA without a device. */
int qg_kernel_budget_measure(int index, int *regs_per_thread, int *static_smem_bytes,
                             int *ctas_per_sm);

/* Self-test of the failure path (no counterpart on the pages): enqueues one
 * CTA that waits on an mbarrier nothing arrives on, with a limit of limit_ns
 * (1 .. 1e9).  The wait runs out, the kernel records QG_ERR_TIMEOUT (call-site
 * tag 900) in the device status word and returns; qg_device_status() then
 * reports QG_ERR_TIMEOUT once and clears it.  Nothing faults or traps, and the
 * context stays usable.  QG_ERR_INVALID_ARG for a limit out of range. */
int qg_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* Self-test of the three deadlock patterns of a hand-built asynchronous
 * pipeline ("Warp-Specialized Kernel Implementation for W4A4 MatMul ...",
 * section 3), staged in one CTA with every wait bounded by limit_ns
 * (1 .. 1e9):
 *   1 = incomplete arrival count (a barrier expecting two producers gets one;
 *       site tag 901),
 *   2 = phase mismatch (the consumer waits on the wrong parity, 1, of a
 *       barrier whose phase 0 has completed; tag 902),
 *   3 = dependency cycle (two roles each wait for the other's arrival first;
 *       tag 903 or 904, whichever gives up first).
 * Each ends in QG_ERR_TIMEOUT in the device status word, read back by
 * qg_device_status_detail; nothing faults or hangs and the context stays
 * usable.  QG_ERR_INVALID_ARG for another pattern or a limit out of range. */
int qg_selftest_deadlock(int pattern, uint64_t limit_ns, void *stream);

/* Testing hook: K-chunk length of qgemm_s8, in blocks of 64 (1..16, default
 * 16 = 1024).  Every chunk's fp32 partial sums stay within 2^24 for any
 * value in 1..16; shorter chunks only cost more accumulator drains. */
int qg_set_s8_chunk(int kblocks);

/* Testing hook: tensor-core GEMM kernel of gemm_f16, qgemm_s8 and qgemm_s4.
 * 0 = chosen by shape (CTA pairs with 256 x 256 tiles when M >= 256 and
 * N >= 256, else one CTA per 128 x 256 tile), 1 = always one CTA per tile,
 * 2 = always CTA pairs.  Results are identical; only speed differs. */
int qg_set_gemm_path(int path);

/* Ablation knob: route of qgemm_s4.  0 = the GEMM kernel reads the packed
 * nibbles and converts them itself where that is faster (CTA pairs, i.e.
 * M >= 256 and N >= 256, K <= 65536 and M*N*K <= 2^34; default), 1 = always
 * a conversion pass to e4m3 bytes in the workspace before the GEMM kernel.
 * Results are identical; QG_ERR_INVALID_ARG for another value. */
int qg_set_s4_path(int path);

/* Ablation knob: tile of the paired kernel behind w4a4_gemm,
 * w4a4_gemm_affine and w4a4_gemm_prepacked when M > 128.  0 = 256 x 256
 * tiles with 16 epilogue warps (default), 1 = 256 x 192 tiles with 12.  The
 * arithmetic and its order are the same, so the results are bit-identical;
 * QG_ERR_INVALID_ARG for another value. */
int qg_set_w4a4_pair_form(int form);

/* L2 cache policy of the tensor-core GEMMs behind gemm_f16, qgemm_s8 and
 * qgemm_s4 (an ablation knob; results are identical in every mode):
 *   0 = every TMA operand load evict-normal (default);
 *   1 = A tiles evict-last, B tiles evict-first: the kernels finish a group
 *       of row-blocks against every column block before the next group, so
 *       an A tile is read again in later rounds while a B tile is read by the
 *       group's row-blocks at about the same time and then not for a whole
 *       group;
 *   2 = as 1, and the output written with streaming (evict-first) stores.
 * QG_ERR_INVALID_ARG for another mode. */
int qg_set_l2_policy(int mode);

/* Programmatic dependent launch of w4a16_gemm (default on).  When on, a
 * w4a16_gemm kernel may start while the previous kernel on the stream is
 * still running: it streams Wq and Wscale at once and reads X only after
 * that kernel has completed.  Wq and Wscale must therefore not be written by
 * the kernel launched just before it on the same stream; pass 0 to turn the
 * overlap off. */
int qg_set_pdl(int enable);

/* Form of the tensor-core w4a16_gemm kernel (batches above 16 rows):
 *   0 = default: when a K quarter holds at most 8 groups (K <= 4096) every
 *       packed weight row of a CTA's quarter is loaded before the dependency
 *       wait and stays in shared memory, and only X streams through the ring;
 *   1 = X and the packed rows share one ring at every K (the form used for
 *       K > 4096).
 * Both give identical bits.  QG_ERR_INVALID_ARG for another value. */
int qg_set_w4a16_tc_form(int form);

/* Measurement hook: while `before` and `after` are non-NULL cudaEvent_t
 * handles (created by the caller), every qgemm_s8, qgemm_s4, gemm_f16 and
 * w4a4_gemm call records `before` on its stream right before launching its
 * tensor-core GEMM kernel and `after` right after it, so that kernel can be
 * timed alone.  Pass NULL, NULL to stop.  Both or neither must be NULL. */
int qg_set_profile_events(void *before, void *after);

/* [L4] Exact INT8 GEMM:  C[i][j] = sum_k A[i][k] * B[j][k]  (int32 result).
 *  A : int8, M x K row-major, lda >= K.
 *  B : int8, K-major (N x K row-major bytes), ldb >= K.
 *  C : int32, M x N row-major, ldc >= N.
 *  K : multiple of 16, K < 131072 (so every int32 result is exact).
 *  ws: workspace of qg_workspace_size(QG_OP_S8, M, N, K) bytes, 256-byte
 *      aligned, device memory; contents on entry are ignored.
 * The result is bit-exact (integer arithmetic is exact). */
int qgemm_s8(int64_t M, int64_t N, int64_t K,
             const int8_t *A, int64_t lda, int layout_a,
             const int8_t *B, int64_t ldb, int layout_b,
             int32_t *C, int64_t ldc,
             void *ws, size_t ws_bytes, void *stream);

/* qgemm_s8 without a caller-supplied workspace.  The paper has no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory: plugin hosts that pass a kernel only its inputs and outputs
 * and own every allocation, engines whose memory plan is fixed after
 * start-up, and code that must not call cudaMalloc at that point (it can
 * synchronize the device).  Arguments, layouts and results are those of
 * qgemm_s8.  The scratch is a static device array of
 * QG_S8_NOALLOC_SCRATCH_BYTES inside this library, held by every GPU that
 * loads the library until the process exits:
 *  - problems needing more than that (qg_workspace_size(QG_OP_S8, M, N, K)
 *    > QG_S8_NOALLOC_SCRATCH_BYTES, e.g. beyond M = N = K = 2048) return
 *    QG_ERR_WORKSPACE and enqueue nothing;
 *  - the first call on each device looks up the array's device address with
 *    that device current; make it before any stream capture on the device;
 *  - `stream` must belong to the current device (QG_ERR_INVALID_ARG
 *    otherwise); the looked-up address is kept for the life of the library,
 *    so do not call it on a device after cudaDeviceReset of that device;
 *  - all calls share the array and it keeps the last call's contents; no part
 *    of it needs to start at zero, but calls that overlap on the GPU (other
 *    streams, unordered host threads) race on it: serialize them.
 * It calls no allocator. */
#define QG_S8_NOALLOC_SCRATCH_BYTES (16u << 20)
int qgemm_s8_noalloc(int64_t M, int64_t N, int64_t K,
                     const int8_t *A, int64_t lda, int layout_a,
                     const int8_t *B, int64_t ldb, int layout_b,
                     int32_t *C, int64_t ldc, void *stream);

/* qgemm_s8 with A, B and C in HOST memory (no counterpart on the pages; the
 * end-to-end form of the INT8 GEMM for data that starts and ends on the host):
 *  A : int8, M x K row-major, lda >= K      (host pointer)
 *  B : int8, N x K row-major, ldb >= K      (host pointer)
 *  C : int32, M x N row-major, ldc >= N     (host pointer, written)
 *  K : multiple of 16, K < 131072.
 *  ws: device workspace of qg_workspace_size(QG_OP_S8_HOST, M, N, K) bytes,
 *      256-byte aligned (device copies of A, B, their fp16 forms and C).
 * The problem is cut into pieces (up to 8 row slices of A times up to 2 row
 * slices of B); the host-to-device copies, the conversion and GEMM of each
 * piece, and the device-to-host copies of finished pieces run on three
 * internal streams of the current device, so that they overlap.  Each slice
 * crosses the link once and is converted once.  The work is ordered after
 * what is already enqueued on `stream`, and `stream` waits for the last copy
 * back: C is complete once `stream` has been synchronized.  Page-locked host
 * memory keeps the copies asynchronous and at full link speed; pageable
 * memory is accepted (the driver stages it and the call may block).  The
 * host buffers and ws must stay valid until then.  The result is bit-exact.
 * The internal streams are shared by all calls on a device; calls from
 * several host threads are enqueued one at a time.  The call may be captured
 * into a CUDA graph (its streams fork from `stream` and join back into it);
 * while such a capture is open, make no other qgemm_s8_host call on that
 * device, since the shared streams belong to the capture until it ends. */
int qgemm_s8_host(int64_t M, int64_t N, int64_t K,
                  const int8_t *A, int64_t lda,
                  const int8_t *B, int64_t ldb,
                  int32_t *C, int64_t ldc,
                  void *ws, size_t ws_bytes, void *stream);

/* [L4] Exact INT4 GEMM on s4p operands:  C = A . B^T  (int32 result).
 *  A : s4p, M x K values, lda_bytes >= K/2.
 *  B : s4p, K-major (N x K values), ldb_bytes >= K/2.
 *  C : int32, M x N row-major, ldc >= N.
 *  K : multiple of 32, K < 262144.
 *  ws: workspace of qg_workspace_size(QG_OP_S4, M, N, K) bytes, 256-byte aligned.
 * The result is bit-exact. */
int qgemm_s4(int64_t M, int64_t N, int64_t K,
             const uint8_t *A, int64_t lda_bytes, int layout_a,
             const uint8_t *B, int64_t ldb_bytes, int layout_b,
             int32_t *C, int64_t ldc,
             void *ws, size_t ws_bytes, void *stream);

/* [L4] FP16 GEMM, fp32 accumulation, fp16 result rounded to nearest even:
 *  C = A . B^T.  A: M x K row-major, B: K-major (N x K), C: M x N row-major.
 *  K : multiple of 8.  No workspace. */
int gemm_f16(int64_t M, int64_t N, int64_t K,
             const uint16_t *A, int64_t lda, int layout_a,
             const uint16_t *B, int64_t ldb, int layout_b,
             uint16_t *C, int64_t ldc, void *stream);

/* [SM75] W4A16 weight-only linear:
 *  Y[m][n] = sum_k X[m][k] * (Wq[n][k] * Wscale[n][k / group]),
 *  fp32 accumulation, fp16 result.
 *  X      : fp16, M x K row-major, ldx >= K.
 *  Wq     : s4p, N x K values, packed contiguously (N rows of K/2 bytes).
 *  Wscale : fp16, N x (K/group), contiguous.  No zero points.
 *  group  : 128 (the only group size this build supports).
 *  Y      : fp16, M x N row-major, ldy >= N.
 *  K      : multiple of `group`.  No workspace.
 * Batches of up to 16 rows keep every weight exact (q applied as an exact
 * fp16 integer, the scale in fp32 per group).  Larger batches on the tensor
 * cores dequantize each weight to the fp16 product q * s (rounded once, at
 * most 2^-11 of the weight); |Wscale| must stay below 8188 there. */
int w4a16_gemm(int64_t M, int64_t N, int64_t K,
               const uint16_t *X, int64_t ldx,
               const uint8_t *Wq, const uint16_t *Wscale, int64_t group,
               uint16_t *Y, int64_t ldy, void *stream);

/* [W4A4] Activation quantizer Q(X) with the fused low-rank down-projection:
 *  per row m and K-block j (block elements):
 *    s = fp16(max|x| / 7)           (binary32 division, round to nearest even)
 *    q = s == 0 ? 0 : clamp(rint(x / s), -8, 7)   (binary32 division by the
 *        rounded scale, rint round-half-even)
 *  and XU = X . U rounded to fp16 (fp32 accumulation); U is the K x rank
 *  down-projection L1 of the low-rank branch.
 *  X      : fp32, M x K row-major, ldx >= K.
 *  U      : fp16, U transposed: rank x K row-major, the layout of the weight
 *           of a K -> rank linear layer (may be NULL when rank == 0).
 *  Xq     : s4p output, M x K values, contiguous (M rows of K/2 bytes).
 *  Xscale : fp16 output, M x (K/block), contiguous.
 *  XU     : fp16 output, M x rank, contiguous (ignored when rank == 0).
 *  block  : 64 (the only block size this build supports); K multiple of block.
 *  rank   : 0 or 32.
 * The same call quantizes weights (rank 0).  Xq and Xscale are bit-exact
 * with the definition above. */
int w4a4_quantize(int64_t M, int64_t K, const float *X, int64_t ldx,
                  const uint16_t *U, int64_t rank,
                  uint8_t *Xq, uint16_t *Xscale, uint16_t *XU,
                  int64_t block, void *stream);

/* [W4A4] Y = (Q(X).Q(W)^T) (.) scale + L(X) + b, with the block-wise scale
 * applied inside the K-sum:
 *  Y[m][n] = sum_j Xscale[m][j]*Wscale[n][j] * sum_{k in block j} Xq[m][k]*Wq[n][k]
 *          + sum_r XU[m][r] * V[r][n] + bias[n],
 *  fp32 accumulation, fp16 result; V is the rank x N up-projection L2 of the
 *  low-rank branch.
 *  Xq, Xscale : as produced by w4a4_quantize (M rows).
 *  Wq, Wscale : the same format for W (N rows).
 *  XU : fp16 M x rank.  V : fp16, V transposed: N x rank row-major, the
 *       layout of the weight of a rank -> N linear layer, 16-byte aligned.
 *       rank 0 or 32 (XU and V may be NULL when rank == 0).
 *  bias : fp16 N, or NULL.
 *  block : 64.  K multiple of 64.  Y : fp16 M x N row-major, ldy >= N.
 *  ws : workspace of qg_workspace_size(QG_OP_W4A4, M, N, K) bytes, 256-byte
 *       aligned. */
int w4a4_gemm(int64_t M, int64_t N, int64_t K,
              const uint8_t *Xq, const uint16_t *Xscale,
              const uint8_t *Wq, const uint16_t *Wscale, int64_t block,
              const uint16_t *XU, const uint16_t *V, int64_t rank,
              const uint16_t *bias, uint16_t *Y, int64_t ldy,
              void *ws, size_t ws_bytes, void *stream);

/* [W4A4] w4a4_gemm with the column-wise affine calibration that the page's
 * drain warps apply before writing (sections 1 and 5.2), read as the map
 * t -> alpha[n] * t + bias[n] on every output column:
 *  Y[m][n] = alpha[n] * ( sum_j Xscale[m][j]*Wscale[n][j] * sum_{k in block j} Xq[m][k]*Wq[n][k]
 *                        + sum_r XU[m][r] * V[r][n] ) + bias[n].
 *  alpha : fp16, N column multipliers, device memory, not NULL (w4a4_gemm is
 *          the case alpha = 1).  Every other argument, layout, workspace and
 *          error as in w4a4_gemm.
 * The multiplier is folded into the fp32 copy of Wscale that the call builds
 * in its workspace (an fp16 scale times an fp16 multiplier is exact in fp32),
 * so it costs no extra pass and no extra work in the GEMM kernel. */
int w4a4_gemm_affine(int64_t M, int64_t N, int64_t K,
                     const uint8_t *Xq, const uint16_t *Xscale,
                     const uint8_t *Wq, const uint16_t *Wscale, int64_t block,
                     const uint16_t *XU, const uint16_t *V, int64_t rank,
                     const uint16_t *alpha, const uint16_t *bias,
                     uint16_t *Y, int64_t ldy,
                     void *ws, size_t ws_bytes, void *stream);

/* [W4A4] The weight side of w4a4_gemm prepared once (the page's weights are
 * quantized offline; inference reuses them for every call): writes into
 * `packed` the e4m3 codes of Wq (N x K bytes) and the transposed fp32 table
 * of Wscale (with the column multiplier alpha folded in when alpha is not
 * NULL, as in w4a4_gemm_affine).
 *  Wq, Wscale, block : as in w4a4_gemm (N rows).
 *  alpha  : fp16 N column multipliers, or NULL (= 1).
 *  packed : device buffer of qg_workspace_size(QG_OP_W4A4_WEIGHTS, 1, N, K)
 *           bytes, 256-byte aligned, owned by the caller; valid once the
 *           work on `stream` has run.  Its layout is private to this library.
 * Errors as in w4a4_gemm. */
int w4a4_prepack_weights(int64_t N, int64_t K, const uint8_t *Wq, const uint16_t *Wscale,
                         int64_t block, const uint16_t *alpha,
                         void *packed, size_t packed_bytes, void *stream);

/* [W4A4] w4a4_gemm (or w4a4_gemm_affine, when alpha was given to
 * w4a4_prepack_weights) with the weights from w4a4_prepack_weights: only X
 * is converted per call.  The result is bit for bit that of w4a4_gemm on
 * the same inputs (the same kernels on the same operands).
 *  packed, packed_bytes : from w4a4_prepack_weights for these N, K.
 *  ws : workspace of qg_workspace_size(QG_OP_W4A4_PREPACKED, M, N, K) bytes,
 *       256-byte aligned.
 * Every other argument as in w4a4_gemm. */
int w4a4_gemm_prepacked(int64_t M, int64_t N, int64_t K,
                        const uint8_t *Xq, const uint16_t *Xscale,
                        const void *packed, size_t packed_bytes, int64_t block,
                        const uint16_t *XU, const uint16_t *V, int64_t rank,
                        const uint16_t *bias, uint16_t *Y, int64_t ldy,
                        void *ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* QGEMM_H */

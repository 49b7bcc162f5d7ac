/*
 * qmm.h -- C ABI of libqmm: block-quantized int4 x int8 matrix products on
 * one GB300 (sm_103a).
 *
 * The method (what every product entry computes):
 *  - Weights are Q4_0 blocks of 32 values with one fp16 scale
 *    (TinyLLaMA C++ guide, kenji.blog, section 6.1 "Arquitectura de
 *    cuantizacion por bloques"): w_i ~ Delta * q_i, q_i in [-8, 7],
 *    Delta = max|w_i| / 7 (llama.cpp guide, kenji.blog/id, section 2.2).
 *  - Activations are quantized on the fly to Q8_0-style int8 blocks of 32
 *    (Colibri page, kerneldigest.dev, "Arquitectura del Sistema"):
 *    d = max|x| / 127 kept as fp16, q = round-half-away(x / d) in [-127,127].
 *  - Each output is y = sum over blocks b of d_w[b] * d_x[b] * dot_b, where
 *    dot_b = sum_{i<32} q_w,i * q_x,i is an exact int32 (llama.cpp guide 2.2,
 *    y ~ Delta * Delta_x * sum q_i q_x,i), accumulated in fp32.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *    and allocates every buffer (the library allocates no device memory).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every entry only enqueues work on it and returns; none
 *    synchronises except qmm_last_device_error.
 *  - Shapes: W is N x K (N output rows, K reduction length), K % 32 == 0,
 *    B = K / 32 blocks per row.  Activations are M x K.
 *  - Return value: QMM_OK (0) or a nonzero qmm_status.  On an argument
 *    error nothing is launched.  Launch errors surface as QMM_ERR_CUDA from
 *    cudaGetLastError right after the launch.
 *
 * Device layout of a Q4_0 matrix ("planes", bytes identical to the page's
 * 18-byte blocks, split so each 16-byte nibble group is 16-byte aligned):
 *  - qs : uint8 [N][B][16].  Byte j of block b holds element 32b+j in its low
 *         nibble and element 32b+j+16 in its high nibble, each stored as
 *         u = q + 8 (all 16 nibble values are accepted).  Must be 16-byte
 *         aligned.
 *  - d  : uint16 [N][B], the fp16 bit pattern of each block's scale.
 *         Must be 2-byte aligned.
 * Q8_0 activations: q int8 [M][K] (16-byte aligned, row stride K) and
 * d uint16 [M][B] fp16 bit patterns (row stride B).
 */
#ifndef QMM_H_
#define QMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#define QMM_QK 32        /* values per block */
#define QMM_ABI_VERSION 2

typedef enum qmm_status {
    QMM_OK = 0,
    QMM_ERR_ARG = 1,            /* NULL pointer or negative size            */
    QMM_ERR_SHAPE = 2,          /* K % 32 != 0, empty where not allowed, too large */
    QMM_ERR_ALIGN = 3,          /* pointer misaligned for the documented layout */
    QMM_ERR_DEVICE = 4,         /* current device is not sm_103 (or no device) */
    QMM_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed     */
    QMM_ERR_TIMEOUT = 6,        /* a bounded device-side wait gave up       */
    QMM_ERR_BAD_EXPERT_ID = 7,  /* an expert id outside [0, E) was skipped  */
    QMM_ERR_WORKSPACE = 8,      /* workspace NULL or smaller than required  */
    QMM_ERR_SCRATCH_LIMIT = 9   /* larger than the library's fixed scratch  */
} qmm_status;

/* Human-readable name of a status code (static string, never NULL). */
QMM_API const char* qmm_status_string(int status);

/* QMM_ABI_VERSION of the loaded library. */
QMM_API int qmm_abi_version(void);

/* ---------------------------------------------------------------------
 * Weight preparation (set-up time, not on the decode path)
 * ------------------------------------------------------------------- */

/* Quantize fp32 weights w [N][K] (row stride ldw >= K floats) to Q4_0
 * planes, per block: amax = max|w|, d32 = amax/7 (IEEE fp32 division),
 * q = clamp(round-half-away(w/d32), -8, 7), d = fp16(d32) (round to nearest
 * even); an all-zero block gives d = 0, q = 0.  (llama.cpp guide 2.2.)
 * N == 0 is a no-op. */
QMM_API qmm_status qmm_quantize_q4_0(const float* w, int64_t N, int64_t K, int64_t ldw,
                             uint8_t* qs, uint16_t* d, void* stream);

/* Split page-format Q4_0 blocks (TinyLLaMA guide 6.1: 2-byte fp16 scale,
 * little endian, then 16 nibble bytes; 18 bytes per block, [N][B][18], on
 * the device, any alignment) into the planes above.  N == 0 is a no-op. */
QMM_API qmm_status qmm_repack_q4_0(const uint8_t* blocks, int64_t N, int64_t K,
                           uint8_t* qs, uint16_t* d, void* stream);

/* ---------------------------------------------------------------------
 * Activation quantizer
 * ------------------------------------------------------------------- */

/* Q8_0 of x [M][K] (fp32, row stride ldx >= K floats, 16-byte aligned,
 * ldx % 4 == 0): per block amax, d32 = amax/127 (IEEE division), q =
 * clamp(round-half-away(x/d32), -127, 127), d = fp16(d32); zero block ->
 * d = 0, q = 0.  Non-finite inputs, or amax/127 above 65504, are outside
 * the domain (result unspecified).  Outputs q [M][K], d [M][B].
 * M == 0 is a no-op. */
QMM_API qmm_status qmm_quantize_q8_0(const float* x, int64_t M, int64_t K, int64_t ldx,
                             int8_t* q, uint16_t* d, void* stream);

/* SwiGLU then Q8_0 (TinyLLaMA guide 4.4: SwiGLU = Swish(x W_gate) * (x W_up),
 * Swish(z) = z * sigmoid(z)): h = gate / (1 + expf(-gate)) * up in fp32,
 * then Q8_0 of each row of h as qmm_quantize_q8_0.  gate/up/h are
 * [rows][K] with row stride ld floats (16-byte aligned, ld % 4 == 0).
 * h_out may be NULL; when given it receives the fp32 h.  rows == 0 is a
 * no-op. */
QMM_API qmm_status qmm_swiglu_quantize_q8_0(const float* gate, const float* up, int64_t rows, int64_t K,
                                    int64_t ld, int8_t* q, uint16_t* d, float* h_out, void* stream);

/* ---------------------------------------------------------------------
 * Products
 * ------------------------------------------------------------------- */

/* Batch-1 GEMV (llama.cpp guide 2.1-2.2: the decode-time bottleneck):
 * y[n] = sum_b fp32(d_w[n][b]) * fp32(d_x[b]) * dot(n, b), n < N.
 * xq int8 [K] (16-byte aligned), xd uint16 [B], y fp32 [N].  N >= 1. */
QMM_API qmm_status qmm_gemv_q4_0_q8_0(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K,
                              const int8_t* xq, const uint16_t* xd, float* y, void* stream);

/* Flags of qmm_gemv_q4_0_f32. */
#define QMM_X_SWIGLU 1       /* x holds gate = x[0..K) and up = x[K..2K); the activation
                                quantized is SwiGLU(gate, up) as in qmm_swiglu_quantize_q8_0 */
#define QMM_Y_SWIGLU_PAIRS 2 /* rows interleaved gate_0, up_0, gate_1, up_1, ...: the output
                                is y[i] = Swish(g_i) * u_i, g_i = row 2i . x, u_i = row 2i+1 . x
                                (N even, y has N/2 entries, no residual; needs K % 256 == 0
                                and a 16-byte aligned w_d) */
#define QMM_CHAIN 4          /* programmatic dependent launch (see below) */

/* Batch-1 GEMV from fp32 activations: quantizes x [K] (16-byte aligned) to
 * Q8_0 exactly as qmm_quantize_q8_0 inside the same launch, then
 * y[n] = sum_b d_w[n][b] * d_x[b] * dot(n, b) (+ residual[n] when residual
 * is not NULL: the residual add of a transformer block, TinyLLaMA guide 5.2
 * graph).  SwiGLU (TinyLLaMA guide 4.4) can be fused on either side with
 * QMM_X_SWIGLU / QMM_Y_SWIGLU_PAIRS.  y must not alias x or residual.
 * xq_out [K] / xd_out [B] may be NULL; when given they receive the Q8_0
 * activation.  With QMM_CHAIN the kernel may start before the preceding
 * kernel on `stream` has finished and stream its weights meanwhile; it
 * reads x and residual only after that kernel has completed.  So the
 * weight planes must not be written by any kernel still running when this
 * call is enqueued.  The fp32 activation is staged on chip: K <= 40960. */
QMM_API qmm_status qmm_gemv_q4_0_f32(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K,
                             const float* x, const float* residual, float* y,
                             int8_t* xq_out, uint16_t* xd_out, int flags, void* stream);

/* Batch-1 GEMV of a decode chain, input and output forms chosen per call:
 *  - activation: fp32 x [K] (quantized to Q8_0 inside the launch, as in
 *    qmm_gemv_q4_0_f32, QMM_X_SWIGLU allowed) when x is not NULL, else the
 *    Q8_0 activation xq [K] (16-byte aligned) / xd [B];
 *  - output: fp32 y [N_out] (+ residual [N] when not NULL) when y is not
 *    NULL, and/or its Q8_0 encoding yq [N_out] (16-byte aligned) / yd
 *    [N_out/32] when yq and yd are not NULL -- exactly what
 *    qmm_quantize_q8_0 would make of y, so the next GEMV of a chain reads it
 *    with no quantization of its own.  N_out = N, or N/2 with
 *    QMM_Y_SWIGLU_PAIRS.  A Q8_0 output needs N_out % 32 == 0.
 * flags: QMM_X_SWIGLU, QMM_Y_SWIGLU_PAIRS, QMM_CHAIN as for
 * qmm_gemv_q4_0_f32.  Requires K % 256 == 0 and w_d 16-byte aligned (the
 * weights are streamed by the tensor-memory-access engine); K <= 40960. */
QMM_API qmm_status qmm_gemv_fused(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K,
                                  const float* x, const int8_t* xq, const uint16_t* xd,
                                  const float* residual, float* y, int8_t* yq, uint16_t* yd,
                                  int flags, void* stream);

/* Small-batch GEMM (batched decode, speculative verify -- Colibri page,
 * MTP drafts verified in one batched forward): for m < M, n < N,
 * y[m*ldy + n] = sum_b d_w[n][b] * d_x[m][b] * dot(m, n, b).
 * xq int8 [M][K], xd [M][B]; ldy >= N.  M >= 1. */
QMM_API qmm_status qmm_gemm_q4_0_q8_0(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K,
                              int64_t M, const int8_t* xq, const uint16_t* xd, float* y, int64_t ldy,
                              void* stream);

/* Device workspace bytes of qmm_gemm_q4_0_q8_0_ws for K and M: for 1..16
 * tokens one 9216 * ceil(M / 8)-byte record per 512 columns of K (rounded
 * up) plus 16 KiB of flag words (a large product is cut evenly over the SMs;
 * a row chunk cut between two CTAs is finished through y and a flag); 0
 * otherwise.  QMM_ERR_ARG for a NULL bytes or M < 0, QMM_ERR_SHAPE
 * for K <= 0 or K % 32 != 0. */
QMM_API qmm_status qmm_gemm_workspace_size(int64_t K, int64_t M, size_t* bytes);

/* qmm_gemm_q4_0_q8_0 with a caller-owned device workspace (at least
 * qmm_gemm_workspace_size bytes, 128-byte aligned, contents irrelevant and
 * overwritten; one call at a time per workspace).  Where the 16-warp
 * warp-MMA layout applies (3..16 tokens, see qmm_debug_gemm_kernel; xd
 * 16-byte aligned) a first launch forms the activation's MMA operand once
 * for the whole call into the workspace, and every CTA of the product copies
 * it from there instead of forming it itself; the results are those of
 * qmm_gemm_q4_0_q8_0 bit for bit, except where the two take different row
 * plans: a large product cut evenly over the SMs (a row chunk cut between
 * two CTAs sums its two parts separately), and a small-N, long-K product
 * whose K the plain entry splits over clusters sharing 192-row chunks (here
 * 128-row chunks); same tolerance, the same bits on every call.  Elsewhere the workspace is not used and
 * the call is qmm_gemm_q4_0_q8_0.  Host checks as qmm_gemm_q4_0_q8_0's, then
 * QMM_ERR_WORKSPACE for a workspace that is NULL, smaller than required or
 * misaligned (when the required size is not 0).  Both launches use
 * programmatic dependent launch: the product's weights stream while the
 * kernel before on `stream` finishes; xq and xd are read only after it has
 * completed. */
QMM_API qmm_status qmm_gemm_q4_0_q8_0_ws(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K,
                                         int64_t M, const int8_t* xq, const uint16_t* xd, float* y,
                                         int64_t ldy, void* workspace, size_t workspace_bytes, void* stream);

/* Which kernel qmm_gemm_q4_0_q8_0 uses for 2 or more tokens, process-wide,
 * for testing and timing the kernels on the same inputs:
 *  - QMM_GEMM_KERNEL_AUTO (the default): the fastest measured: the
 *    streaming kernel for 2 tokens, and for 3-4 tokens when N <= 4096 or
 *    K >= 8192 unless the 16-warp layout below applies; otherwise the
 *    warp-MMA kernels;
 *  - QMM_GEMM_KERNEL_MMA: the warp-MMA kernels (mma.sync, any M): up to 16
 *    tokens the 16-warp layout where its row plan qualifies (ceil(N / SMs)
 *    in 65..192 rows, xd 16-byte aligned), else the row-group kernel;
 *  - QMM_GEMM_KERNEL_MMA_GROUPS: the warp-MMA row-group kernel alone;
 *  - QMM_GEMM_KERNEL_TMEM: the tcgen05 kernel with the weight operand in
 *    tensor memory (M <= 16, K % 256 == 0, all four operand planes 16-byte
 *    aligned; otherwise the GEMM returns QMM_ERR_SHAPE);
 *  - QMM_GEMM_KERNEL_STREAM: the dp4a streaming kernel of the batch-1 GEMV,
 *    up to 8 tokens per weight pass (more tokens: more passes).
 * All compute the same fp32 result up to the order of the fp32 sums.
 * `previous` (may be NULL) receives the old setting; QMM_ERR_ARG for an
 * unknown kernel.  Not synchronised with GEMM calls on other host threads. */
#define QMM_GEMM_KERNEL_AUTO 0
#define QMM_GEMM_KERNEL_MMA 1
#define QMM_GEMM_KERNEL_TMEM 2
#define QMM_GEMM_KERNEL_STREAM 3
#define QMM_GEMM_KERNEL_MMA_GROUPS 4
QMM_API qmm_status qmm_debug_gemm_kernel(int kernel, int* previous);

/* Test hook of the failure handling of the streaming GEMV kernel (the
 * kernel of qmm_gemv_fused, qmm_gemv_fused_op, qmm_gemv_q4_0_f32 and the
 * 1-8 token qmm_gemm_q4_0_q8_0): every wait on the device is bounded, and
 * this sets the bound of the launches that follow, process-wide:
 * limit_ns in [1e3, 1e10] (the default is 2e9, two seconds).  With
 * withhold_last_copy = 1 the producer of every CTA never issues its last
 * weight copy, so the consumers' wait for it runs out: the launch ends
 * without writing the outputs that depend on it, the device error word
 * gets QMM_ERR_TIMEOUT (read with qmm_last_device_error), and the context
 * stays usable; every copy that was issued lands before the CTA ends.
 * withhold_last_copy = 0 restores normal operation.  `previous_limit_ns`
 * (may be NULL) receives the old bound.  QMM_ERR_ARG outside those ranges.
 * Not synchronised with launches on other host threads.  No counterpart on
 * the pages. */
QMM_API qmm_status qmm_debug_stream_wait(uint64_t limit_ns, int withhold_last_copy, uint64_t* previous_limit_ns);

/* Per-block integer dots, for bit-exact checking: dots[(m*N + n)*B + b] =
 * sum_{i<32} q_w * q_x, int32, computed with the product kernels' own
 * unpack and dot code.  M, N >= 1. */
QMM_API qmm_status qmm_debug_block_dots(const uint8_t* w_qs, int64_t N, int64_t K, int64_t M, const int8_t* xq,
                                int32_t* dots, void* stream);

/* ---------------------------------------------------------------------
 * One batch-1 GEMV of a decode step described by an op (a decode step's
 * projections, TinyLLaMA guide section 5 graph; each op as qmm_gemv_fused)
 * ------------------------------------------------------------------- */

/* One batch-1 GEMV op.  Pointers are device pointers; the fields mean what
 * the arguments of qmm_gemv_fused mean:
 *  - weights w_qs/w_d of N x K (K % 256 == 0, K <= 40960, both planes
 *    16-byte aligned);
 *  - activation: fp32 x [K] (16-byte aligned) when x is not NULL -- first
 *    normalized by RMSNorm (TinyLLaMA guide 4.1: x / sqrt(mean(x^2) + eps)
 *    (.) gamma, in fp32) when norm_w (gamma [K], 16-byte aligned) is not
 *    NULL -- then quantized to Q8_0 exactly as qmm_quantize_q8_0; xq/xd,
 *    when not NULL, then RECEIVE that Q8_0 activation.  With x NULL the
 *    activation is the Q8_0 xq [K] / xd [K/32];
 *  - outputs y (fp32 [N_out], + residual [N_out] when residual is not NULL)
 *    and/or yq/yd (Q8_0 of y, N_out % 32 == 0);
 *  - flags 0 or QMM_Y_SWIGLU_PAIRS (N_out = N / 2, no residual). */
typedef struct qmm_gemv_op {
    const uint8_t* w_qs;
    const uint16_t* w_d;
    int64_t N, K;
    const float* x;
    const float* norm_w;
    const int8_t* xq;
    const uint16_t* xd;
    const float* residual;
    float* y;
    int8_t* yq;
    uint16_t* yd;
    float norm_eps;
    int32_t flags;
} qmm_gemv_op;

/* One op as one launch of the streaming GEMV kernel.  flags: 0 or
 * QMM_CHAIN (programmatic dependent launch, as for qmm_gemv_q4_0_f32). */
QMM_API qmm_status qmm_gemv_fused_op(const qmm_gemv_op* op, int flags, void* stream);

/* A chain of ops in one call: ops[0..n) each as qmm_gemv_fused_op(&ops[i],
 * flags, stream), in order.  Every op is checked before anything is
 * launched; the first bad op's status is returned and nothing is launched.
 * A launch that fails returns QMM_ERR_CUDA after the launches before it.
 * n == 0 is a no-op; ops host memory, read during the call only. */
QMM_API qmm_status qmm_gemv_fused_ops(const qmm_gemv_op* ops, int32_t n, int flags, void* stream);

/* ---------------------------------------------------------------------
 * Weight-format variants of the batch-1 product
 * ------------------------------------------------------------------- */

/* Largest K of qmm_gemv_rowwise_q8_0 and of qmm_gemv_q4_0_f32_fma (the
 * activation is staged whole in shared memory). */
#define QMM_ROWWISE_MAX_K 131072
#define QMM_F32_FMA_MAX_K 49152

/* Per-row-scale int4 / int2 container (Colibri page, "Arquitectura del
 * Sistema": an int4 container with per-row scales; int4 and int2 packing).
 * The page fixes no layout; the reading taken: for row n,
 *   delta = max_k |w[n][k]| / qmax in fp32, qmax = 2^(bits-1) - 1 (the
 *     llama.cpp guide's section 2.2 rule applied to the whole row);
 *   q = clamp(round-half-away(w / delta), -2^(bits-1), qmax) (IEEE fp32
 *     division); a zero row gets delta = 0 and q = 0;
 *   codes u = q + 2^(bits-1), 8/bits per byte: element k in byte k*bits/8
 *     at bit (k mod 8/bits)*bits.
 * w fp32 [N][K] (row stride ldw >= K, 4-byte aligned) -> w_q uint8
 * [N][K*bits/8], w_s fp32 [N]; device, caller-owned.  bits is 4 or 2;
 * K % 32 == 0 (bits 4) or K % 64 == 0 (bits 2), else QMM_ERR_SHAPE.
 * N == 0 is a no-op. */
QMM_API qmm_status qmm_quantize_rowwise(const float* w, int64_t N, int64_t K, int64_t ldw, int32_t bits,
                                        uint8_t* w_q, float* w_s, void* stream);

/* y[n] = w_s[n] * sum_b d_x[b] * sum_{i<32} q_w[n][32b+i] * q_x[32b+i]
 * (batch 1): per-row codes (layout of qmm_quantize_rowwise) times a Q8_0
 * activation (xq int8 [K], xd fp16 bits [K/32]); the block dots are exact
 * int32, the combine fp32.  w_q 16-byte aligned, w_s 4, xq 16, xd 2, y 4.
 * bits 4 or 2; K % 32 == 0 (bits 4) or K % 64 == 0 (bits 2), K <=
 * QMM_ROWWISE_MAX_K, else QMM_ERR_SHAPE. */
QMM_API qmm_status qmm_gemv_rowwise_q8_0(const uint8_t* w_q, const float* w_s, int32_t bits, int64_t N, int64_t K,
                                         const int8_t* xq, const uint16_t* xd, float* y, void* stream);

/* y[n] = sum_k (d_w[n][k/32] * q_w[n][k]) * x[k] (batch 1): Q4_0 planes (the
 * layout of qmm_gemv_q4_0_q8_0) times an fp32 activation that is not
 * quantized, the dequantize-then-multiply-add flow of the TinyLLaMA guide,
 * section 6.2.  fp32 arithmetic: exact codes, one fp32 sum per 16 values,
 * the block sum times d_w added to the row's running sum.  w_qs 16-byte
 * aligned, w_d 2, x 16, y 4; K % 32 == 0 and K <= QMM_F32_FMA_MAX_K, else
 * QMM_ERR_SHAPE. */
QMM_API qmm_status qmm_gemv_q4_0_f32_fma(const uint8_t* w_qs, const uint16_t* w_d, int64_t N, int64_t K,
                                         const float* x, float* y, void* stream);

/* ---------------------------------------------------------------------
 * MoE expert-grouped GEMV (Colibri page: only the routed experts of each
 * token are applied; sigmoid router, top-k)
 * ------------------------------------------------------------------- */

/* Bytes of workspace qmm_moe_gemv needs for E experts and T*k slots. */
QMM_API qmm_status qmm_moe_workspace_size(int32_t E, int32_t T, int32_t k, size_t* bytes);

/* For every slot s = t*k + j (t < T, j < k) with expert e = ids[s]:
 *   y[s][n] = sum_b d_w(e)[n][b] * d_x[b] * dot, n < N,
 * where expert e's planes are w_qs + e*N*K/2 and w_d + e*N*B (experts
 * stored back to back), and the activation is row t of xq/xd
 * (x_per_slot == 0: xq [T][K], xd [T][B]) or row s (x_per_slot != 0:
 * xq [T*k][K], xd [T*k][B]).  y is fp32 [T*k][N].  Each distinct expert's
 * weights are streamed once per call and applied to all slots routed to it.
 * ids int32 [T][k] on the device; an id outside [0, E) is skipped (its y
 * row is left untouched) and sets the device error word, reported by
 * qmm_last_device_error as QMM_ERR_BAD_EXPERT_ID.  Duplicate ids are
 * allowed.  workspace: device, >= qmm_moe_workspace_size bytes, 16-byte
 * aligned, contents need not be initialised.  T == 0 is a no-op. */
QMM_API qmm_status qmm_moe_gemv(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                        const int32_t* ids, int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd,
                        int x_per_slot, float* y, void* workspace, size_t workspace_bytes, void* stream);

/* Limits of qmm_moe_router_topk. */
#define QMM_ROUTER_MAX_EXPERTS 1024
#define QMM_ROUTER_MAX_K 64

/* Sigmoid top-k router (Colibri page, "Arquitectura del Sistema": a
 * sigmoid router picks the experts of each token).  For each token t < T:
 *   s_e = 1 / (1 + exp(-logits[t][e])) in fp32, e < E;
 *   ids[t][0..k-1] = the k experts of largest score, in decreasing order,
 *     ties to the lower expert index (sigmoid is strictly increasing, so the
 *     comparison is made on the logits themselves);
 *   gates[t][j] = s_{ids[t][j]} / sum_{i<k} s_{ids[t][i]}, the sum taken in
 *     j order (the normalisation over the k, with no bias, is a reading: the
 *     page does not say).
 * logits fp32 [T][E], ids int32 [T][k], gates fp32 [T][k]: device, 4-byte
 * aligned, caller-owned.  1 <= k <= min(E, QMM_ROUTER_MAX_K),
 * E <= QMM_ROUTER_MAX_EXPERTS, else QMM_ERR_SHAPE.  Logits must be finite;
 * the selection equals that of the double-precision sigmoid for logits in
 * [-87, 16].  T == 0 is a no-op.
 * workspace: NULL, or device memory of at least qmm_moe_workspace_size(E, T,
 * k) bytes, 16-byte aligned, contents need not be initialised.  Given one, the
 * same launch (a single CTA, meant for decode-size T) also groups the chosen
 * slots by expert there, which is what qmm_moe_gemv_pregrouped reads; without
 * one, tokens are routed one warp each over as many CTAs as needed. */
QMM_API qmm_status qmm_moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* ids,
                                       float* gates, void* workspace, size_t workspace_bytes, void* stream);

/* The slot grouping of qmm_moe_gemv on its own: groups the T*k slots of
 * ids (int32 [T][k], device, values in [0, E)) by expert into workspace,
 * exactly the tables qmm_moe_router_topk builds there for its chosen ids.
 * For ids that do not come from the router (e.g. remapped to the slots of an
 * expert store) before qmm_moe_gemv_pregrouped, qmm_moe_gemv_pregrouped_f32
 * or qmm_moe_gemv_gate_up.  An id outside [0, E) is left out of the tables
 * and sets the device error word (QMM_ERR_BAD_EXPERT_ID).  workspace: >=
 * qmm_moe_workspace_size(E, T, k) bytes, 16-byte aligned.  T == 0 is a
 * no-op. */
QMM_API qmm_status qmm_moe_group_ids(const int32_t* ids, int32_t T, int32_t k, int32_t E, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* qmm_moe_gemv on the slot grouping that qmm_moe_router_topk left in
 * workspace for the same E, T and k (no ids argument, no grouping launch):
 * every later expert GEMV of a MoE layer (gate, up, down) reuses one
 * routing.  The workspace must not be changed in between; an expert id of
 * the grouping is always in range.  Same arguments, layouts, results and
 * errors as qmm_moe_gemv otherwise. */
QMM_API qmm_status qmm_moe_gemv_pregrouped(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                                           int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd,
                                           int x_per_slot, float* y, const void* workspace, size_t workspace_bytes,
                                           void* stream);

/* The first half of every routed expert's FFN in one launch: gate and up
 * projections, then SwiGLU (TinyLLaMA guide section 4.4: Swish(x W_gate)
 * times x W_up, Swish(z) = z sigmoid(z)), on the grouping of
 * qmm_moe_router_topk as for qmm_moe_gemv_pregrouped.  Each expert's N rows
 * interleave its two projections: row 2i is gate row i, row 2i + 1 up row i
 * (N = 2 * F, even).  For every slot s:
 *   h[s][i] = g / (1 + exp(-g)) * u,   g = y[s][2i], u = y[s][2i + 1],
 * with y as qmm_moe_gemv_pregrouped would compute it: each of g and u equals
 * bit for bit what a qmm_moe_gemv_pregrouped call over the same rows gives,
 * and h what qmm_swiglu_quantize_q8_0 writes as h_out for them.  h fp32
 * [T*k][N/2], 4-byte aligned.  The activation is the Q8_0 xq/xd as for
 * qmm_moe_gemv_pregrouped, or, when x is not NULL, fp32 rows x (same row
 * layout, 16-byte aligned) quantized inside the launch exactly as
 * qmm_quantize_q8_0 would (xq and xd are then not read).  Requires the
 * streaming path (K % 256 == 0, w_qs and w_d 16-byte aligned) and N even,
 * else QMM_ERR_SHAPE; other arguments and errors as
 * qmm_moe_gemv_pregrouped. */
QMM_API qmm_status qmm_moe_gemv_gate_up(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                                        int32_t T, int32_t k, const float* x, const int8_t* xq, const uint16_t* xd,
                                        int x_per_slot, float* h, const void* workspace, size_t workspace_bytes,
                                        void* stream);

/* qmm_moe_gemv_pregrouped with fp32 activation rows x (x_per_slot == 0:
 * [T][K], else [T*k][K]; 16-byte aligned), each quantized to Q8_0 inside
 * the launch exactly as qmm_quantize_q8_0 would, so the result equals bit
 * for bit that of qmm_moe_gemv_pregrouped on qmm_quantize_q8_0(x): the
 * expert GEMV after a SwiGLU with no quantization launch in between.
 * Requires the streaming path (K % 256 == 0, w_qs and w_d 16-byte aligned),
 * else QMM_ERR_SHAPE. */
QMM_API qmm_status qmm_moe_gemv_pregrouped_f32(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N,
                                               int64_t K, int32_t T, int32_t k, const float* x, int x_per_slot,
                                               float* y, const void* workspace, size_t workspace_bytes,
                                               void* stream);

/* y[t][n] = sum_{j=0..k-1} gates[t][j] * z[t][j][n], j ascending (fixed
 * order, deterministic).  z fp32 [T][k][N], gates fp32 [T][k], y [T][N]. */
QMM_API qmm_status qmm_moe_combine(const float* z, const float* gates, int32_t T, int32_t k, int64_t N, float* y,
                           void* stream);

/* One MoE FFN layer on fp32 activations, from router logits (Colibri page,
 * "Arquitectura del Sistema": router, routed experts, combined result;
 * TinyLLaMA guide section 4.4: SwiGLU), as four launches on stream, with
 * the results of these calls in this order:
 *   qmm_moe_router_topk(logits, T, E, k, ids, gates, workspace, ...);
 *   qmm_moe_gemv_gate_up(gu_qs, gu_d, E, 2 * F, H, T, k, x, NULL, NULL, 0, h, ...);
 *   qmm_moe_gemv_pregrouped_f32(down_qs, down_d, E, H, F, T, k, h, 1, z, ...);
 *   qmm_moe_combine(z, gates, T, k, H, y);
 * bit for bit.  gu_qs/gu_d: each expert's 2F interleaved gate/up rows of H
 * columns; down_qs/down_d: each expert's H rows of F columns; x fp32 [T][H]
 * and h fp32 [T*k][F] (16-byte aligned), z fp32 [T*k][H], y fp32 [T][H],
 * ids int32 [T][k], gates fp32 [T][k]; workspace as for
 * qmm_moe_router_topk, required.  Because the launches' order is fixed
 * here, the down launch reads the grouping and starts streaming its weights
 * before the gate/up launch has finished (the gate/up launch lets it start
 * only after the router has completed); only its activation reads wait.
 * Every check of the four calls is made before the first launch; the
 * streaming path is required for both expert tensors (H and F multiples of
 * 256, planes 16-byte aligned), else QMM_ERR_SHAPE.  The fastest measured
 * form for few routed slots (T * k * 4 <= E); with more, Q8_0 launches of
 * x and h ahead of the Q8_0-input expert GEMVs measured 2% faster. */
QMM_API qmm_status qmm_moe_layer_f32(const float* logits, int32_t T, int32_t E, int32_t k, const uint8_t* gu_qs,
                                     const uint16_t* gu_d, const uint8_t* down_qs, const uint16_t* down_d,
                                     int64_t H, int64_t F, const float* x, int32_t* ids, float* gates, float* h,
                                     float* z, float* y, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------
 * Expert hot-store (Colibri page, "Arquitectura del Sistema": a
 * least-recently-used cache of experts per layer, an optional hot store in
 * RAM or VRAM, and a prefetcher that asks ahead for the experts the next
 * layer will use).  Host memory holds every expert; the device keeps
 * n_slots of them in a slot arena that the MoE entries read: remap the
 * router's expert ids to slot ids (qmm_store_map_ids) and pass the arena
 * as the expert tensor with E = n_slots.
 * ------------------------------------------------------------------- */

/* A host-side LRU over keys 0..n_keys-1 and slots 0..n_slots-1 (the
 * policy of the store, usable on its own; no device needed).
 *  - A use request (use != 0) needs its keys now: its distinct keys must
 *    fit in the slots, else QMM_ERR_SHAPE and nothing changes.  Each
 *    distinct key counts once as a hit or a miss.  All its keys are
 *    protected from eviction until the next use request.  Keys become most
 *    recent in request order.
 *  - A prefetch (use == 0) loads absent keys into slots holding no key of
 *    the last use request (a key that finds none gets slot -1) and makes
 *    resident keys most recent.
 *  - A load takes a never-used slot (slot 0 first), else the least recently
 *    used slot that is not protected.
 * slots_out [n] (slot of each key), load_keys / load_slots [n] (the loads,
 * in order) and n_loads may each be NULL.  Keys out of range: QMM_ERR_ARG. */
typedef struct qmm_lru qmm_lru;
QMM_API qmm_status qmm_lru_create(int32_t n_keys, int32_t n_slots, qmm_lru** out);
QMM_API void qmm_lru_destroy(qmm_lru* lru);
QMM_API qmm_status qmm_lru_request(qmm_lru* lru, const int32_t* keys, int32_t n, int32_t use, int32_t* slots_out,
                                   int32_t* load_keys, int32_t* load_slots, int32_t* n_loads);
QMM_API qmm_status qmm_lru_stats(const qmm_lru* lru, int64_t* hits, int64_t* misses, int64_t* evictions,
                                 int64_t* prefetched);
/* Slot of a key, -1 when it is not resident. */
QMM_API qmm_status qmm_lru_slot_of(const qmm_lru* lru, int32_t key, int32_t* slot);

/* One plane of every expert (e.g. the nibble plane of the gate matrix):
 * expert e is `bytes` bytes at host + e * host_stride (host memory, pinned
 * for asynchronous copies; caller-owned, valid for the store's life), and
 * slot s is `bytes` bytes at dev + s * bytes (device arena of n_slots *
 * bytes, caller-owned). */
typedef struct qmm_store_plane {
    const void* host;
    int64_t host_stride;
    void* dev;
    int64_t bytes;
} qmm_store_plane;

#define QMM_STORE_MAX_PLANES 16

typedef struct qmm_store qmm_store;

/* A store of E experts in n_slots device slots (n_slots <= E), n_planes
 * planes per expert (<= QMM_STORE_MAX_PLANES).  dev_slot_of: device int32
 * [E], caller-owned, kept by the store (slot of each expert or -1); set to
 * all -1 here (synchronously).  Needs an sm_103 device (the current one). */
QMM_API qmm_status qmm_store_create(int32_t E, int32_t n_slots, const qmm_store_plane* planes, int32_t n_planes,
                                    int32_t* dev_slot_of, qmm_store** out);
/* Frees the store's host state and events (not the caller's buffers).
 * Work already enqueued stays valid. */
QMM_API void qmm_store_destroy(qmm_store* store);

/* Makes experts ids[0..n) (host array, duplicates allowed) resident for
 * work enqueued next on compute_stream: a use request of the LRU; each
 * missing expert is copied into its slot with one cudaMemcpyAsync per plane
 * on copy_stream, after the compute stream has passed the release of every
 * earlier request that used that slot; compute_stream then waits for the
 * copies, and the device slot table is updated on compute_stream.  The
 * host does not wait.  copy_stream may equal compute_stream (no overlap).
 * More distinct experts than slots: QMM_ERR_SHAPE, nothing changes. */
QMM_API qmm_status qmm_store_request(qmm_store* store, const int32_t* ids, int32_t n, void* compute_stream,
                                     void* copy_stream);
/* Marks the end of the last request's use of its slots: call after
 * enqueuing the work that reads them (on the same compute stream).  If it
 * is not called, the next request does it first. */
QMM_API qmm_status qmm_store_release(qmm_store* store, void* compute_stream);
/* Starts copying experts ids[0..n) (host array) that are absent, on
 * copy_stream, into slots holding no expert of the last request (the
 * prefetch of the page's next-layer prediction).  They become usable by the
 * next qmm_store_request, which waits for these copies. */
QMM_API qmm_status qmm_store_prefetch(qmm_store* store, const int32_t* ids, int32_t n, void* copy_stream);
/* slot_ids[i] = slot of expert ids[i] (device int32 arrays of n): the ids
 * of the expert GEMV for the slot arena.  An expert that is not resident
 * maps to -1 and sets the device error word (QMM_ERR_BAD_EXPERT_ID); the
 * MoE entries then skip that slot. */
QMM_API qmm_status qmm_store_map_ids(qmm_store* store, const int32_t* ids, int64_t n, int32_t* slot_ids,
                                     void* stream);
QMM_API qmm_status qmm_store_stats(const qmm_store* store, int64_t* hits, int64_t* misses, int64_t* evictions,
                                   int64_t* prefetched, int64_t* bytes_copied);

/* ---------------------------------------------------------------------
 * MoE expert GEMV without a caller workspace.  A library addition: the
 * pages have no counterpart (they say nothing about device memory).
 * ------------------------------------------------------------------- */

/* Size of the fixed scratch that qmm_moe_gemv_static uses in place of a
 * workspace: 256 KiB.  Enough whenever qmm_moe_workspace_size(E, T, k) is
 * at most this, e.g. E = 256 experts with up to 64,510 routed slots T*k. */
#define QMM_MOE_STATIC_SCRATCH_BYTES (256 * 1024)

/* Same computation, arguments, layouts, results and error codes as
 * qmm_moe_gemv, without the workspace arguments, and it allocates nothing:
 * the routing tables go to a fixed array inside the library (a file-scope
 * __device__ array of QMM_MOE_STATIC_SCRATCH_BYTES, 256-byte aligned, one
 * per device).
 *
 * Meant for callers that cannot allocate device memory when they call: a
 * serving loop that reserved all device memory at start-up, code that must
 * not call an allocator in the step (cudaMalloc may synchronise the device
 * and fails under memory pressure), or a plain C caller with no memory pool
 * to carve a workspace from.
 *
 *  - Limit: if qmm_moe_workspace_size(E, T, k) exceeds
 *    QMM_MOE_STATIC_SCRATCH_BYTES the call returns QMM_ERR_SCRATCH_LIMIT and
 *    launches nothing; use qmm_moe_gemv with a workspace for such sizes.
 *  - Nothing has to start at zero: every call rebuilds the tables from ids
 *    before reading them, so what an earlier call left there is never used.
 *  - Setup: the first call on a device (with that device current) looks up
 *    the scratch's device address once (cudaGetSymbolAddress) and sets the
 *    kernels' shared-memory attributes; later calls reuse both.  Make that
 *    first call before beginning a stream capture on the device.
 *  - Concurrency: every call on one device shares the one scratch.  Calls on
 *    one stream run in order and are safe.  Calls that can run at the same
 *    time on one device (streams with no ordering between them, e.g. from
 *    several host threads) race on the scratch and may write wrong outputs:
 *    order them on one stream or with events.
 *  - T == 0 is a no-op and needs no device. */
QMM_API qmm_status qmm_moe_gemv_static(const uint8_t* w_qs, const uint16_t* w_d, int32_t E, int64_t N, int64_t K,
                               const int32_t* ids, int32_t T, int32_t k, const int8_t* xq, const uint16_t* xd,
                               int x_per_slot, float* y, void* stream);

/* ---------------------------------------------------------------------
 * Errors raised on the device
 * ------------------------------------------------------------------- */

/* Synchronises `stream`, reads and clears the device error word of the
 * current device: QMM_OK, QMM_ERR_BAD_EXPERT_ID or QMM_ERR_TIMEOUT (a
 * bounded wait gave up).  QMM_ERR_CUDA if the synchronisation failed. */
QMM_API qmm_status qmm_last_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H_ */

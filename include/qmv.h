/*
 * qmv.h -- C ABI of the GB300 (sm_103a) weight-only-quantized skinny matmul library.
 *
 * The operations are the decode-time hot path of two systems described on the
 * pages this library follows:
 *  - "Machine Learning on NVIDIA CMP" (llama.cpp on throttled Ampere dies):
 *    section "TL;DR" -- decode runs through MMVQ, the quantized mat x vec whose
 *    inner loop is a 4-wide int8 dot with int32 accumulation (section "The DP2A
 *    patch"), over Q4_0 weights (section "llama.cpp results", Llama-2-7B-Q4_0).
 *  - "v100-skinny README": section "How QPN works" -- QPN2 (NVFP4 W4A16: e2m1
 *    codes, an FP8 scale per 16 weights, a global scale) and QPN8 (FP8 e4m3
 *    W8A16), weights decoded only in registers, fp16 activations; section
 *    "Native mixed-precision checkpoint path" -- per-region dispatch at M = 1..8.
 *
 * Conventions shared by every entry point
 *  - Pointers to weights, activations and outputs are DEVICE pointers on the
 *    current CUDA device, owned by the caller. The library allocates no memory
 *    and keeps no per-call state; it never frees or retains a pointer.
 *  - All arrays are row-major and little-endian. M is the number of activation
 *    rows (1..8 for the Q4_0 / Q4_K / Q8_1 calls, 1..96 for NVFP4 / FP8), N the number of
 *    weight rows (outputs per activation row), K the reduction length. Outputs y are fp32 [M][N] and fully overwritten.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default stream)
 *    and may be captured in a CUDA graph. Arguments are validated on the host
 *    before any CUDA call; an invalid call returns an error and launches nothing.
 *    Faults during execution surface at the caller's next synchronization.
 *  - M == 0 or N == 0 is a valid empty call (nothing launched). K == 0 writes
 *    zeros to y (an empty sum).
 *  - Calls are thread-safe. Calls that write overlapping outputs must not run
 *    concurrently.
 */
#ifndef QMV_H_
#define QMV_H_

#include <stdint.h>

#if defined(__GNUC__)
#define QMV_API __attribute__((visibility("default")))
#else
#define QMV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared opaquely so C callers need no CUDA header. */
typedef struct CUstream_st *qmv_stream_t;

typedef int qmv_status;
#define QMV_OK                0
#define QMV_ERR_NULL         -1  /* a required pointer is NULL */
#define QMV_ERR_SHAPE        -2  /* M outside 0..8 (0..96 NVFP4 / FP8), N or K negative, K not a multiple of the format's block */
#define QMV_ERR_ALIGN        -3  /* a pointer is not aligned to its element type (see each call) */
#define QMV_ERR_CUDA         -4  /* a CUDA runtime call failed (launch, attribute, device query) */
#define QMV_ERR_TIMEOUT      -5  /* qmv_error_flags: a bounded device-side wait gave up */

/* Human-readable name of a status code (static string, never NULL). */
QMV_API const char *qmv_status_string(qmv_status status);

/*
 * fp32 -> Q8_1 activation quantizer.
 * The pages name MMVQ's int8 activation operand (section "The DP2A patch",
 * "Machine Learning on NVIDIA CMP") but not its format; this is llama.cpp's Q8_1
 * block as this library defines it:
 *   x   fp32 [M][K], K a multiple of 32, 4-byte aligned.
 *   xq  M * (K/32) blocks of 36 bytes, [M][K/32] order, 4-byte aligned:
 *       bytes 0..1 d8 (fp16), 2..3 s8 (fp16), 4..35 q[32] (int8).
 *   Per block, in IEEE fp32 with round to nearest even: d = max|x_i| / 127;
 *   q_i = d == 0 ? 0 : clamp(round_half_away_from_zero(x_i / d), -127, 127);
 *   d8 = fp16(d); s8 = fp16(d * sum_i q_i). NaN/Inf inputs are outside the
 *   contract; |x| above 127 * 65504 makes d8 infinite.
 */
QMV_API qmv_status qmv_quantize_q8_1(const float *x, void *xq, int M, int64_t K, qmv_stream_t stream);

/*
 * Q4_0 x Q8_1 mat-vec (MMVQ), M = 1..8 activation rows.
 *   w   Q4_0 [N][K/32] blocks of 18 bytes: fp16 scale d4, then 16 bytes qs;
 *       element j of the block is qs[j] & 15, element j+16 is qs[j] >> 4;
 *       weight value d4 * (q - 8). 2-byte aligned (16-byte aligned and K a
 *       multiple of 256 select the streaming kernels: dp4a at small M, the tensor
 *       cores -- m16n8k32 int8, the nibbles as 16 (q - 8) -- from M = 5).
 *   xq  Q8_1 [M][K/32] (as written by qmv_quantize_q8_1), 4-byte aligned.
 *   y   fp32 [M][N]: y[m][n] = sum_b d4[n][b] * d8[m][b] * (S - 8 T), with the
 *       exact integer block sums S = sum_j q4_j * q8_j and T = sum_j q8_j
 *       ("The DP2A patch": 4-wide int8 dot, int32 accumulation).
 *   K must be a multiple of 32.
 */
QMV_API qmv_status qmv_q4_0_q8_1(const void *w, const void *xq, float *y, int M, int64_t N, int64_t K,
                         qmv_stream_t stream);

/*
 * Quantize + MMVQ in one kernel: the same result as qmv_quantize_q8_1(x) followed
 * by qmv_q4_0_q8_1 (bit-identical outputs; the Q8_1 blocks are built in shared
 * memory by the quantizer's own device code and never written to global memory).
 * Saves one launch and the Q8_1 round trip per call.
 *   w  Q4_0 as in qmv_q4_0_q8_1, 16-byte aligned; K a multiple of 256.
 *   x  fp32 [M][K], 16-byte aligned.   y  fp32 [M][N].
 * Returns QMV_ERR_SHAPE for shapes the streaming kernels cannot take (their
 * staged activations do not fit in shared memory; use the two-call path there)
 * and QMV_ERR_ALIGN for a misaligned w or x.
 */
QMV_API qmv_status qmv_q4_0_q8_1_fused(const void *w, const float *x, float *y, int M, int64_t N, int64_t K,
                                       qmv_stream_t stream);

/*
 * Several independent fused calls with the same M and K in ONE launch: call i
 * computes y[i] = W[i] x[i] exactly as qmv_q4_0_q8_1_fused(w[i], x[i], y[i], M,
 * N[i], K) would (bit-identical). Decode runs matrices that read the same input
 * -- the q, k, v projections of a layer, or its gate and up projections -- one
 * after another only because each is a separate call; grouping them removes the
 * dependent launches between them.
 *   count       1..8 matrices.
 *   w, x, y, N  HOST arrays of `count` entries (device pointers and row counts),
 *               read during the call only. Each x[i] may equal another x[j].
 * Errors as in qmv_q4_0_q8_1_fused, checked per matrix.
 */
QMV_API qmv_status qmv_q4_0_q8_1_fused_group(int count, const void *const *w, const float *const *x,
                                             float *const *y, const int64_t *N, int M, int64_t K,
                                             qmv_stream_t stream);

/*
 * The grouped launch on Q8_1 activations: call i computes y[i] exactly as
 * qmv_q4_0_q8_1(w[i], xq[i], y[i], M, N[i], K) would (bit-identical). With several
 * activation rows this is the faster path: qmv_quantize_q8_1 quantizes each input
 * once, where the fused entry points quantize it again in every CTA.
 *   count        1..8 matrices.
 *   w, xq, y, N  HOST arrays of `count` entries; w[i] Q4_0 16-byte aligned, xq[i]
 *                Q8_1 [M][K/32] 4-byte aligned (each may equal another xq[j]),
 *                y[i] fp32 [M][N[i]]. K a multiple of 256.
 * Errors as in qmv_q4_0_q8_1_fused_group.
 */
QMV_API qmv_status qmv_q4_0_q8_1_group(int count, const void *const *w, const void *const *xq, float *const *y,
                                       const int64_t *N, int M, int64_t K, qmv_stream_t stream);

/*
 * Q4_K x Q8_1 mat-vec, M = 1..8 activation rows: llama.cpp's K-quant super-block,
 * the format of the Q4_K_M models of "Machine Learning on NVIDIA CMP", section
 * "llama.cpp results" (the pages name it without printing the layout).
 *   w   Q4_K [N][K/256] super-blocks of 144 bytes, 16-byte aligned:
 *       bytes 0..1 d (fp16), 2..3 dmin (fp16), 4..15 eight packed 6-bit
 *       sub-block scales sc_j and minimums mn_j (j < 4: sc = p[j] & 63,
 *       mn = p[j+4] & 63; j >= 4: sc = (p[j+4] & 15) | (p[j-4] >> 6) << 4,
 *       mn = (p[j+4] >> 4) | (p[j] >> 6) << 4), 16..143 nibbles: data byte
 *       32c + e holds element 64c + e (low nibble) and 64c + 32 + e (high).
 *       Element i of sub-block j = i / 32: w = d * sc_j * q - dmin * mn_j.
 *   xq  Q8_1 [M][K/32] as written by qmv_quantize_q8_1, 4-byte aligned.
 *   y   fp32 [M][N]: y[m][n] = sum_b d8[m][b] * (d sc_j S - dmin mn_j T) over
 *       the Q8_1 blocks b (= sub-blocks), with the exact integer sums
 *       S = sum q * q8 and T = sum q8, accumulated in fp32.
 *   K a multiple of 256. The dp4a streaming kernel serves M = 1..4, the int8
 *   tensor cores (m16n8k32 on the unsigned nibbles, D = S exactly) M = 5..8; both
 *   stage the activations in shared memory, so very large K returns QMV_ERR_SHAPE.
 */
QMV_API qmv_status qmv_q4_k_q8_1(const void *w, const void *xq, float *y, int M, int64_t N, int64_t K,
                                 qmv_stream_t stream);

/* Quantize + Q4_K MMVQ in one kernel, as qmv_q4_0_q8_1_fused is for Q4_0:
 * bit-identical to qmv_quantize_q8_1 followed by qmv_q4_k_q8_1. x fp32 [M][K],
 * 16-byte aligned; other arguments and errors as in qmv_q4_k_q8_1. */
QMV_API qmv_status qmv_q4_k_q8_1_fused(const void *w, const float *x, float *y, int M, int64_t N, int64_t K,
                                       qmv_stream_t stream);

/* Grouped Q4_K launches (1..8 matrices, HOST arrays of device pointers and row
 * counts), each call i exactly as the single call on (w[i], x[i] or xq[i], y[i],
 * N[i]); matrices given the same activation pointer stage it once. */
QMV_API qmv_status qmv_q4_k_q8_1_group(int count, const void *const *w, const void *const *xq, float *const *y,
                                       const int64_t *N, int M, int64_t K, qmv_stream_t stream);
QMV_API qmv_status qmv_q4_k_q8_1_fused_group(int count, const void *const *w, const float *const *x,
                                             float *const *y, const int64_t *N, int M, int64_t K,
                                             qmv_stream_t stream);

/*
 * NVFP4 W4A16 skinny GEMM ("v100-skinny README", section "How QPN works": QPN2).
 *   codes        [N][K/2] bytes, two E2M1 codes per byte: k even in the low
 *                nibble, k odd in the high nibble (OCP MX E2M1 values).
 *   scales_e4m3  [N][K/16] bytes, one OCP E4M3 (FN) scale per 16 consecutive k.
 *   global_scale per-tensor fp32 scale g.
 *   x            fp16 [M][K] (IEEE binary16 bit patterns), 2-byte aligned.
 *   y            fp32 [M][N]: y[m][n] = g * sum_k e2m1(c[n][k]) * e4m3(s[n][k/16]) * x[m][k],
 *                accumulated in fp32 (no fp16 partial sums: the page's own fix for
 *                fp16 overflow on activation outliers).
 *   K must be a multiple of 16. codes, x 16-byte aligned and K a multiple of 256
 *   select the tensor-core streaming kernel.
 *   M = 1..16: rows 9..16 ride the same pass over the weights as rows 1..8 (a
 *   second 8-row activation tile of the tensor-core product), so the weights are
 *   read from memory once for all M rows. M = 17..96 (the chunked band of the
 *   README's "Native mixed-precision checkpoint path" dispatch table), and M = 9..16
 *   when N spans at most a third of the SMs' worth of 128-row tiles: one pass over
 *   the weights on the 5th-generation tensor cores (tcgen05.mma, weights decoded into
 *   and fp32 accumulators kept in tensor memory, M padded to a multiple of 16, K split
 *   over a thread-block cluster when the tiles leave half the SMs idle), x 16-byte
 *   aligned and scales_e4m3 16-byte aligned; otherwise balanced chunks of at most 16
 *   rows, one launch and one weight pass each.
 *   Resources of the tcgen05 path: one CTA per SM holding all 512 tensor-memory
 *   columns (a CTA of another kernel on the same SM that also allocates tensor memory
 *   waits for it), and, when K is split, a launch of thread-block clusters of 2..4
 *   CTAs. It allocates no global memory; the partial sums of a split stay in shared
 *   memory.
 */
QMV_API qmv_status qgemm_nvfp4_w4a16(const uint8_t *codes, const uint8_t *scales_e4m3, float global_scale,
                             const uint16_t *x, float *y, int M, int64_t N, int64_t K,
                             qmv_stream_t stream);

/*
 * FP8 E4M3 W8A16 skinny GEMM ("v100-skinny README", section "How QPN works": QPN8,
 * one contiguous e4m3 byte stream).
 *   w          [N][K] OCP E4M3 (FN) bytes.
 *   row_scale  fp32 [N] per-output-row scale, 4-byte aligned.
 *   x          fp16 [M][K], 2-byte aligned.
 *   y          fp32 [M][N]: y[m][n] = row_scale[n] * sum_k e4m3(w[n][k]) * x[m][k],
 *              accumulated in fp32.
 *   Any K >= 0. w, x 16-byte aligned and K a multiple of 128 select the
 *   tensor-core streaming kernel. The same bands as qgemm_nvfp4_w4a16: M = 1..16 in
 *   one pass over the weights, then (from 9 rows for launches of few tiles) one pass
 *   on the tcgen05 kernel, or chunks of at most 16 rows when it cannot be used.
 */
QMV_API qmv_status qgemm_fp8_w8a16(const uint8_t *w, const float *row_scale, const uint16_t *x, float *y,
                           int M, int64_t N, int64_t K, qmv_stream_t stream);

/*
 * Several NVFP4 (or FP8) matrices with the same M and K reading the SAME activations
 * x in ONE launch -- the gate and up projections of a layer, say: y[i] is matrix i's
 * product as the single call defines it, within the same error bound (the fp32
 * partial sums of a tile may be added in another order than in a single call).
 * The tensor-core kernel only: K a multiple of 256 (NVFP4) or
 * 128 (FP8), codes / w 16-byte aligned, scales and row scales 4-byte aligned, x
 * 16-byte aligned (QMV_ERR_SHAPE / QMV_ERR_ALIGN otherwise).
 *   count                 1..8 matrices.
 *   codes, scales_e4m3, global_scale, w, row_scale, y, N
 *                         HOST arrays of `count` entries (device pointers, scales
 *                         and row counts), read during the call only.
 */
QMV_API qmv_status qgemm_nvfp4_w4a16_group(int count, const uint8_t *const *codes,
                                           const uint8_t *const *scales_e4m3, const float *global_scale,
                                           const uint16_t *x, float *const *y, const int64_t *N, int M, int64_t K,
                                           qmv_stream_t stream);
QMV_API qmv_status qgemm_fp8_w8a16_group(int count, const uint8_t *const *w, const float *const *row_scale,
                                         const uint16_t *x, float *const *y, const int64_t *N, int M, int64_t K,
                                         qmv_stream_t stream);

/*
 * Launch overlap between consecutive calls (programmatic dependent launch),
 * process-wide, off by default. When enabled, every kernel of this library is
 * launched so that it may start while the preceding kernel on the stream is
 * still running: it reads its WEIGHTS (and scales) at once, and waits for the
 * preceding kernel to finish and flush before it reads activations or writes
 * outputs. Contract: weights must not be written by the kernel that immediately
 * precedes a call on its stream (static model weights never are; copies and
 * memsets are not kernels and keep full ordering). This hides the launch gap and
 * the pipeline ramp of a chain of small calls, such as the layers of a decode step.
 */
QMV_API void qmv_set_launch_overlap(int enable);
QMV_API int qmv_get_launch_overlap(void);

/* ---------------------------------------------------------------------------
 * Introspection (tests and benchmarks)
 * ------------------------------------------------------------------------- */

/*
 * Offset-corrected integer block dots of qmv_q4_0_q8_1, computed by the same
 * device code and the same kernel choice as the product call:
 *   dots int32 [M][N][K/32], dots[m][n][b] = S - 8 T (see qmv_q4_0_q8_1).
 * Pointers and alignment as in qmv_q4_0_q8_1.
 */
QMV_API qmv_status qmv_debug_q4_0_block_dots(const void *w, const void *xq, int32_t *dots, int M, int64_t N,
                                     int64_t K, qmv_stream_t stream);

/*
 * Raw integer sub-block dots of qmv_q4_k_q8_1 from the same device code and
 * kernel: dots int32 [M][N][K/32], dots[m][n][b] = S = sum q * q8 over the 32
 * weights of sub-block b (no minimum term). Pointers and alignment as in
 * qmv_q4_k_q8_1.
 */
QMV_API qmv_status qmv_debug_q4_k_block_dots(const void *w, const void *xq, int32_t *dots, int M, int64_t N,
                                             int64_t K, qmv_stream_t stream);

/*
 * The launch plan the Q4_0 / Q4_K heuristic picks for one call on a device given
 * by its SM count and shared-memory limits. The streaming-kernel plans need no
 * CUDA call (usable without a GPU); the tensor-core kernel's plan (M >= 5 unless
 * QMV_Q4_MMA_MIN_M / QMV_Q4K_MMA_MIN_M move the threshold) queries the current
 * device's occupancy and returns QMV_ERR_CUDA without one.
 *   q4k          0 = Q4_0 (K % 32 == 0), 1 = Q4_K (K % 256 == 0).
 *   M, N, K      as in qmv_q4_0_q8_1 (M 1..8, N >= n_inputs, K > 0); N rows in all.
 *   n_inputs     1..8 matrices of N / n_inputs rows, each with its own activation.
 *   w_align16    1 if the weights start on 16-byte boundaries, else 0.
 *   sm_count, smem_optin, smem_per_sm  the device (GB300: 152, 232448, 233472).
 *   out          HOST int64 [8]: route (a qmv_route_name index), warps per CTA,
 *                ring slots per warp, grid (CTAs), dynamic shared memory bytes,
 *                activation records in registers (0/1), lane pairs (0/1), and
 *                144-byte units per ring slot. For Q4_K a q4_0_generic route means that
 *                no kernel takes the shape (the call returns QMV_ERR_SHAPE).
 * Returns QMV_ERR_NULL for out == NULL, QMV_ERR_SHAPE for values out of range.
 */
QMV_API qmv_status qmv_debug_plan_q4(int q4k, int M, int64_t N, int64_t K, int n_inputs, int w_align16,
                                     int sm_count, int smem_optin, int smem_per_sm, int64_t *out);

/*
 * The launch plan the NVFP4 / FP8 heuristic picks for one call (count = 1) or one
 * grouped launch (count 1..8 matrices of N[i] rows, the same M and K) on a device
 * given by its limits, with no CUDA call (usable without a GPU). From 17 activation
 * rows on (from 9 when the tiles span at most a third of the SMs), the tcgen05 kernel
 * takes the call (route nvfp4_tcgen05 /
 * fp8_tcgen05: 128-row tiles, all M rows in one pass over the weights; out[3] = its
 * MMA-issuing threads, out[4] = its weight stages, out[9] = grid, out[10] = shared
 * memory, out[11] = its 64-k A buffers in tensor memory, out[12] = its activation
 * slices, out[13] = the CTAs (a cluster) that share each tile, each a range of K;
 * QMV_WQ_UMMA_MIN_M / QMV_WQ_UMMA_FEW_TILES_MIN_M move the thresholds). Below it the planner scores
 * candidate plans (warps, ring slots, activations staged in shared memory or not,
 * passes over K) by the whole-tile tail they leave on the device's CTAs; the CTAs
 * per SM of a candidate come from a model here -- the least of ctas_by_regs, the SM's
 * shared memory over the candidate's (plus 1 KB reserved per CTA), and 64 resident
 * warps -- where a launch asks the device's occupancy calculator.
 *   fp4           1 = NVFP4, 0 = FP8.
 *   M, K, N       as in qgemm_nvfp4_w4a16 / qgemm_fp8_w8a16 (M 1..96); N HOST int64
 *                 [count]. Above 16 rows the plan is that of the first (largest) of
 *                 the balanced chunks of at most 16 rows.
 *   aligned16     1 if codes / weights and x start on 16-byte boundaries.
 *   sm_count, smem_optin, smem_per_sm   the device (GB300: 152, 232448, 233472).
 *   ctas_by_regs  HOST int [3] or NULL: the CTAs per SM the registers of the kernel
 *                 variants allow -- 8 warps with one 8-row activation tile, 8 warps
 *                 with two, 16 warps. NULL takes the launch bounds' minimum {3, 2, 1}
 *                 (the compiler keeps the registers within them).
 *   out           HOST int64 [14]: route (a qmv_route_name index), chunks, rows of
 *                 the first chunk, warps, ring slots, staged (0/1), passes over K,
 *                 tiles per round, CTAs per SM, grid, dynamic shared memory bytes, A
 *                 buffers, activation slices and K splits (tcgen05 route; 0
 *                 otherwise). The generic route fills only route, chunks (8-row
 *                 launches) and rows.
 * Returns QMV_ERR_NULL for out or N NULL, QMV_ERR_SHAPE for values out of range or
 * a shape no plan fits.
 */
QMV_API qmv_status qmv_debug_plan_wq(int fp4, int M, int64_t K, int count, const int64_t *N, int aligned16,
                                     int sm_count, int smem_optin, int smem_per_sm, const int *ctas_by_regs,
                                     int64_t *out);

/*
 * Kernel-choice census: a counter per kernel route, bumped on every launch, so a
 * caller can check which kernel served each region and that no fallback ran
 * (the census of "v100-skinny README", "Native mixed-precision checkpoint path").
 * Routes are numbered 0 .. qmv_route_count()-1; counts are cumulative since the
 * last reset.
 */
QMV_API int qmv_route_count(void);
QMV_API const char *qmv_route_name(int route);
QMV_API int64_t qmv_route_launches(int route);
QMV_API void qmv_route_reset(void);

/*
 * Device-side error word of the current device: bit flags set by kernels whose
 * bounded waits gave up (they skip their work instead of hanging). Synchronizes
 * the device. Returns QMV_OK and writes the word to *flags; clear=1 resets it.
 */
QMV_API qmv_status qmv_error_flags(uint32_t *flags, int clear);

/*
 * Self-check of the bounded device-side wait that every streaming kernel uses on
 * its mbarriers: one thread waits on an mbarrier that nothing completes, so the
 * wait must give up after its bound, set the timeout bit (1) of the error word and
 * return, leaving the context usable. The bound: 0.5 s of %globaltimer time once at
 * least 1024 polls have been made (a context switched off the GPU makes no polls),
 * and at most 2^21 polls in any case.
 *   out  DEVICE int64 [2], 8-byte aligned, owned by the caller: out[0] = 1 if the
 *        wait completed (never expected), 0 if it gave up; out[1] = nanoseconds
 *        spent waiting (%globaltimer).
 * Asynchronous on `stream`. Returns QMV_ERR_NULL / QMV_ERR_ALIGN for a bad `out`,
 * QMV_ERR_CUDA if the launch fails.
 */
QMV_API qmv_status qmv_debug_wait_bound(int64_t *out, qmv_stream_t stream);

/*
 * Self-check of how a multi-warp kernel gives up (the tensor-core kernels: their
 * warps meet at a CTA-wide barrier after every round). One CTA of 8 warps; each warp
 * fills a 2-slot ring with real bulk copies, except warp `stuck_warp`, which arms its
 * mbarriers and issues nothing, so its bounded wait runs out while the others reach
 * the round's barrier. The stuck warp flags the timeout bit (1) of the error word and
 * the CTA's abort word and goes on to the barrier; after it every warp sees the
 * abort, waits (bounded) for its own copies in flight and returns: no thread is left
 * at a barrier, no copy lands in the memory of an exited CTA. Takes about two wait
 * bounds (the give-up, then the stuck warp's drain).
 *   out         DEVICE int64 [8][4], 8-byte aligned: per warp, 1 if its wait gave up;
 *               1 if it passed the barrier and saw the abort; the copies still in
 *               flight when it left the round; nanoseconds from its first wait to
 *               the barrier.
 *   stuck_warp  0..7.
 * Asynchronous on `stream`. Returns QMV_ERR_NULL / QMV_ERR_ALIGN for a bad `out`,
 * QMV_ERR_SHAPE for stuck_warp out of range, QMV_ERR_CUDA if the launch fails.
 */
QMV_API qmv_status qmv_debug_cta_abort(int64_t *out, int stuck_warp, qmv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H_ */

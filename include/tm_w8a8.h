/*
 * W8A8 GEMM: 8-bit integer weights and activations ("LMDeploy Guide: Fast
 * Mixed-Precision LLM Inference Engine": W8A8 among the precision formats
 * the engine serves, from SmoothQuant-style post-training quantisation).
 *
 * The scheme (our reading; the smoothing factors are folded into the fp16
 * weights beforehand): activations quantised per token, dynamically; weights
 * per output channel; both symmetric, in IEEE binary32 with
 * round-to-nearest-even at each step:
 *   a = max |x| over the row (column);  s = a / 127, or 1 when a == 0
 *   q = clamp(rint(x / s), -127, 127)          (one division per value)
 *   Y[m][n] = fp16( s_x[m] * s_w[n] * sum_k q_x[m][k] q_w[k][n] )
 * The integer products are exact on the tensor cores (fp16 operands holding
 * the integers, fp32 accumulation: exact while a partial sum stays below
 * 2^24); the scaling is one fp32 product per output.
 *
 * Conventions as in tm_w4a16.h: device pointers, asynchronous on `stream`
 * (a cudaStream_t, NULL = legacy default stream) unless stated otherwise,
 * no allocation outside tm_w8_pack.
 */
#ifndef TM_W8A8_H
#define TM_W8A8_H

#include <stddef.h>
#include <stdint.h>

#include "tm_w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque packed 8-bit weights (codes in the kernel's fragment order and the
 * per-channel scales), one device allocation. */
typedef struct tm_w8_packed tm_w8_packed;

/*
 * Per-token dynamic quantisation of the activations (the rule above, per row).
 *   X : device fp16 bits [M][K] row-major, 16-byte aligned; K % 16 == 0
 *   xq: device int8 [M][K], 16-byte aligned;  sx: device fp32 [M], 4-byte aligned
 * One launch; TM_ERR_INVALID_ARG on a bad shape, TM_ERR_ALIGNMENT on a
 * misaligned pointer.
 */
tm_status tm_w8a8_quantize_act(const uint16_t* X, int M, int K, int8_t* xq, float* sx, void* stream);

/*
 * Per-output-channel quantisation of fp16 weights (the rule above, per column n
 * over the K rows), producing the inputs of tm_w8_pack.
 *   W : device fp16 bits [K][N] row-major, 16-byte aligned; N % 16 == 0
 *   q : device int8 [K][N], 8-byte aligned;  sw: device fp32 [N], 4-byte aligned
 * Asynchronous on `stream`: a memset of sw and three launches (column maxima
 * through an integer atomic max, the codes, the scales); no allocation.
 */
tm_status tm_w8_quantize_weight(const uint16_t* W, int K, int N, int8_t* q, float* sw, void* stream);

/*
 * Offline repack of per-channel quantised weights into the GEMM's order.
 *   q : device int8 [K][N] row-major (codes -127..127)
 *   sw: device fp32 [N]
 *   K % 16 == 0, N % 16 == 0; K is padded to a multiple of 128 with zero codes.
 * Synchronous on the current device; the caller frees the handle with
 * tm_w8_packed_free.
 */
tm_status tm_w8_pack(const int8_t* q, const float* sw, int K, int N, tm_w8_packed** out);

/* Inverse of tm_w8_pack into device buffers with its input layouts
 * (synchronous; pack -> unpack is bit-exact). */
tm_status tm_w8_unpack(const tm_w8_packed* p, int8_t* q, float* sw);

/* K, N and the bytes of the device allocation of a handle (any out pointer may be NULL). */
tm_status tm_w8_packed_info(const tm_w8_packed* p, int* K, int* N, size_t* bytes);

/* Release a handle (NULL is ignored). */
void tm_w8_packed_free(tm_w8_packed* p);

/*
 * Y = fp16(s_x s_w^T . (q_x q_w)), one launch.
 *   xq: device int8 [M][K] (from tm_w8a8_quantize_act), 16-byte aligned
 *   sx: device fp32 [M];  Y: device fp16 [M][N] row-major, 16-byte aligned
 *   split_k: 0 automatic, else 1, 2, 4 or 8 CTAs (a thread-block cluster)
 *            sharing one output tile along K, reduced through distributed
 *            shared memory (no global workspace)
 * M up to 32 rows run on mma.sync in one row tile (decode); larger M on
 * tcgen05 (kind::f16, fp32 accumulators in tensor memory) in tiles of 128
 * output columns x 64 or 128 rows, both operands converted to exact fp16 in
 * the kernel (weights into tensor memory, X into shared memory).
 * Waits are bounded: a copy that never lands sets the device timeout bit
 * (tm_device_error), and Y is then undefined (possibly stale) until
 * tm_device_error reports the bit clear -- the status this call returned
 * describes the launch only.
 */
tm_status tm_w8a8_gemm(const int8_t* xq, const float* sx, const tm_w8_packed* p, void* Y, int M, int split_k,
                       void* stream);

/* tm_w8a8_gemm with the rows of X per CTA of the tensor-memory kernel (M > 32)
 * chosen explicitly: tile_m = 64, 128 or 256 (0 = automatic; ignored for M <= 32). */
tm_status tm_w8a8_gemm_ex(const int8_t* xq, const float* sx, const tm_w8_packed* p, void* Y, int M, int split_k,
                          int tile_m, void* stream);

/*
 * tm_w8a8_quantize_act with the codes written as exact fp16 integers
 * (-127..127) instead of int8: the X operand of tm_w8a8_gemm_f16.
 *   X   : device fp16 bits [M][K] row-major, 16-byte aligned; K % 16 == 0
 *   xq16: device fp16 bits [M][K], 16-byte aligned;  sx: device fp32 [M], 4-byte aligned
 * Same codes and scales as tm_w8a8_quantize_act, bit for bit; one launch.
 */
tm_status tm_w8a8_quantize_act_f16(const uint16_t* X, int M, int K, uint16_t* xq16, float* sx, void* stream);

/*
 * The product of tm_w8a8_gemm with the codes as fp16 integers (from
 * tm_w8a8_quantize_act_f16), for the tensor-memory kernel: X is copied into
 * shared memory by TMA as the MMA's B operand with no conversion, so the
 * kernel's converter warps handle the weights only (the int8 form converts
 * both, and its shared-memory traffic per 128-k block is ~1.4x higher).
 * Every M runs the tensor-memory kernel (use tm_w8a8_gemm with int8 codes for
 * decode, M <= 32).  split_k and tile_m as in tm_w8a8_gemm_ex; for M > 32 the
 * result equals tm_w8a8_gemm_ex's bit for bit (same products, same order).
 * Bounded waits as in tm_w8a8_gemm: after a timeout Y is undefined until
 * tm_device_error reports the bit clear.
 *   xq16: device fp16 [M][K], 16-byte aligned;  sx: fp32 [M];  Y: fp16 [M][N], 16-byte aligned
 */
tm_status tm_w8a8_gemm_f16(const uint16_t* xq16, const float* sx, const tm_w8_packed* p, void* Y, int M,
                           int split_k, int tile_m, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TM_W8A8_H */

/* W4A8-FP8 building blocks of the routed-expert layer: per-block fp8
 * quantisation of activations and the block-scaled INT4 x fp8 linear.
 *
 * "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", section "A pass
 * through the model" and its input-quantisation setting (dtype float8e4m3,
 * input_scale_group_size 128): expert inputs are e4m3 with one scale per
 * token per 128 consecutive elements; the 4-bit weights become fp8 exactly;
 * each 128-wide block's partial sum is scaled by its activation scale and
 * its weight group scale on the accumulator (section "The Humming kernels":
 * the input scales must reach the accumulator).
 *
 * Readings: OCP e4m3 (E4M3FN: bias 7, no infinities, largest finite 448);
 * scale = fp32(amax / 448) of the block's fp32 values, 1 for an all-zero
 * block; code = e4m3 value nearest to fp32(x / scale), ties to even,
 * saturated at +-448. The weights use the W4A16 layer's storage (moe_w4a16.h):
 * INT4 codes q + 8, 8 per uint32 along K, bf16 group scales per 128.
 *
 * Both calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 * default stream), launch one kernel, allocate nothing, and return
 * MOE_W4A8_OK, or MOE_W4A8_INVALID_ARG for a bad size or pointer (nothing is
 * launched), or MOE_W4A8_CUDA_ERROR if the launch fails. All pointers are
 * device pointers owned by the caller.
 */
#ifndef MOE_W4A8_H
#define MOE_W4A8_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_w4a8_status {
  MOE_W4A8_OK = 0,
  MOE_W4A8_INVALID_ARG = -1,
  MOE_W4A8_CUDA_ERROR = -5,
};

/* x: fp32 [rows, K] row-major (16-byte aligned; K a multiple of 128).
 * codes: e4m3 bytes [rows, K] (4-byte aligned); scales: fp32 [rows, K / 128].
 * rows == 0 is a no-op. */
int moe_w4a8_quantize_blocks(const float* x, int32_t rows, int32_t K, uint8_t* codes,
                             float* scales, void* stream);

/* y[r, n] = sum over 128-blocks g of w_s[n, g] * x_scales[r, g] *
 *           sum_{k in g} q[n, k] * codes[r, k]
 * codes: e4m3 [rows, K] (4-byte aligned), x_scales: fp32 [rows, K / 128];
 * w_q: uint32 [N, K / 8] (INT4, offset binary), w_s: bf16 bits [N, K / 128];
 * y: fp32 [rows, N]. K a multiple of 128, N a multiple of 16; rows == 0 is a
 * no-op. Products run on the fp8 tensor cores (fp32 accumulation within a
 * block), the block scales multiply each block's fp32 partial. */
int moe_w4a8_linear(const uint8_t* codes, const float* x_scales, int32_t rows, int32_t K,
                    const uint32_t* w_q, const uint16_t* w_s, int32_t N, float* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A8_H */

// W4A8-FP8 building blocks: per-block fp8 quantisation of activations and the
// block-scaled INT4 x fp8 linear.
//
// "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", section "A pass
// through the model" and its input-quantisation setting (dtype float8e4m3,
// input_scale_group_size 128): the 4-bit weights become fp8 exactly (the
// integers -8..7 are e4m3 values), the activations entering an expert GEMM are
// e4m3 with one scale per token per 128 consecutive elements, and the
// per-128 activation scales, like the weight group scales, are applied to each
// 128-wide block's partial sum on the accumulator (the section on the Humming
// kernels: those input scales were not being applied).
//
// Readings (the pages are silent): OCP e4m3 (bias 7, largest finite 448); a
// block's scale is fp32(amax / 448), 1 for an all-zero block; a code is the
// e4m3 value nearest to fp32(x / scale), ties to even, saturated at +-448.
//
// These are the variant's first GPU steps, not yet a layer: a quantisation
// kernel (one warp per (row, 128-block)) and a linear kernel on the legacy
// fp8 tensor-core path (mma.sync m16n8k32 e4m3, one warp per 16 output
// channels x 8 rows); the weights' group scales and the rows' block scales
// multiply each block's fp32 partial before it is added.
#include "common.cuh"
#include "moe_w4a8.h"

#include <cuda_fp8.h>

namespace moe {
namespace {

constexpr int kBlk = 128;

// two fp32 values -> two e4m3 codes (low byte: a), round to nearest even,
// saturated to the largest finite value
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// x: [rows, K] fp32 (row stride K); codes [rows, K] e4m3 bytes; scales
// [rows, K / 128] fp32. Warp w of the grid takes block (w / nb, w % nb); lane
// l its elements 4l .. 4l + 3.
__global__ void quantize_blocks_kernel(const float* __restrict__ x, int rows, int K,
                                       uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int nb = K / kBlk;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)rows * nb) return;
  const int r = (int)(wid / nb), g = (int)(wid - (long long)r * nb);
  const float4 v = *reinterpret_cast<const float4*>(x + (size_t)r * K + g * kBlk + 4 * lane);
  const float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  // non-negative floats order as their bit patterns
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const uint16_t lo = e4m3x2(__fdiv_rn(v.x, sc), __fdiv_rn(v.y, sc));
  const uint16_t hi = e4m3x2(__fdiv_rn(v.z, sc), __fdiv_rn(v.w, sc));
  *reinterpret_cast<uint32_t*>(codes + (size_t)r * K + g * kBlk + 4 * lane) =
      (uint32_t)lo | ((uint32_t)hi << 16);
  if (lane == 0) scales[(size_t)r * nb + g] = sc;
}

// four INT4 codes (offset binary, nibbles 0..3 of `bits`) -> four e4m3 bytes;
// exact, since -8..7 are e4m3 values
__device__ __forceinline__ uint32_t int4x4_to_e4m3x4(uint32_t bits) {
  const float q0 = (float)((int)(bits & 15u) - 8), q1 = (float)((int)((bits >> 4) & 15u) - 8);
  const float q2 = (float)((int)((bits >> 8) & 15u) - 8), q3 = (float)((int)((bits >> 12) & 15u) - 8);
  return (uint32_t)e4m3x2(q0, q1) | ((uint32_t)e4m3x2(q2, q3) << 16);
}

__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// y[r, n] = sum_g s_w[n, g] * s_x[r, g] * sum_{k in g} q[n, k] * c[r, k].
// One warp per tile of 16 output channels (the MMA's M, the weights) x 8 rows
// (its N). Fragment of lane (gid = lane / 4, tig = lane % 4): A rows gid and
// gid + 8, K bytes 4 tig .. 4 tig + 3 and + 16; B row-of-K 4 tig .. + 3 and
// + 16 of activation row gid; D channels gid / gid + 8, rows 2 tig, 2 tig + 1.
__global__ void linear_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ xs,
                              int rows, int K, const uint32_t* __restrict__ wq,
                              const uint16_t* __restrict__ ws, int N, float* __restrict__ y) {
  const int nb = K / kBlk;
  const int n0 = blockIdx.x * 16, r0 = blockIdx.y * 8;
  const int lane = threadIdx.x, gid = lane >> 2, tig = lane & 3;
  const int ra = r0 + gid;                       // B: activation row of this lane
  const bool ra_ok = ra < rows;
  const int rc0 = r0 + 2 * tig, rc1 = rc0 + 1;  // D: rows of this lane
  const uint32_t* w0 = wq + (size_t)(n0 + gid) * (K / 8);
  const uint32_t* w1 = wq + (size_t)(n0 + gid + 8) * (K / 8);
  const uint8_t* cb = codes + (size_t)(ra_ok ? ra : 0) * K;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int g = 0; g < nb; ++g) {
    float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kBlk / 32; ++ks) {
      const int kb = g * kBlk + ks * 32;
      // 4 INT4 codes = 16 bits of a word: K index kb + 4 tig (+ 16)
      const int wlo = (kb + 4 * tig) >> 3, shlo = ((4 * tig) & 7) * 4;
      const int whi = (kb + 16 + 4 * tig) >> 3, shhi = ((16 + 4 * tig) & 7) * 4;
      uint32_t a[4];
      a[0] = int4x4_to_e4m3x4(__ldg(w0 + wlo) >> shlo);
      a[1] = int4x4_to_e4m3x4(__ldg(w1 + wlo) >> shlo);
      a[2] = int4x4_to_e4m3x4(__ldg(w0 + whi) >> shhi);
      a[3] = int4x4_to_e4m3x4(__ldg(w1 + whi) >> shhi);
      uint32_t b[2];
      b[0] = ra_ok ? __ldg(reinterpret_cast<const uint32_t*>(cb + kb + 4 * tig)) : 0u;
      b[1] = ra_ok ? __ldg(reinterpret_cast<const uint32_t*>(cb + kb + 16 + 4 * tig)) : 0u;
      mma_e4m3_16832(part, a, b);
    }
    // the block's scales on its fp32 partial: weight group scale per channel,
    // activation block scale per row
    const float sw0 = __uint_as_float((uint32_t)__ldg(ws + (size_t)(n0 + gid) * nb + g) << 16);
    const float sw1 = __uint_as_float((uint32_t)__ldg(ws + (size_t)(n0 + gid + 8) * nb + g) << 16);
    const float sx0 = rc0 < rows ? __ldg(xs + (size_t)rc0 * nb + g) : 0.f;
    const float sx1 = rc1 < rows ? __ldg(xs + (size_t)rc1 * nb + g) : 0.f;
    acc[0] = fmaf(sw0 * sx0, part[0], acc[0]);
    acc[1] = fmaf(sw0 * sx1, part[1], acc[1]);
    acc[2] = fmaf(sw1 * sx0, part[2], acc[2]);
    acc[3] = fmaf(sw1 * sx1, part[3], acc[3]);
  }
  if (rc0 < rows) {
    y[(size_t)rc0 * N + n0 + gid] = acc[0];
    y[(size_t)rc0 * N + n0 + gid + 8] = acc[2];
  }
  if (rc1 < rows) {
    y[(size_t)rc1 * N + n0 + gid] = acc[1];
    y[(size_t)rc1 * N + n0 + gid + 8] = acc[3];
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_w4a8_quantize_blocks(const float* x, int32_t rows, int32_t K, uint8_t* codes,
                                        float* scales, void* stream) {
  if (rows < 0 || K <= 0 || K % moe::kBlk != 0) return MOE_W4A8_INVALID_ARG;
  if (rows == 0) return MOE_W4A8_OK;
  if (!x || !codes || !scales || !moe::aligned16(x) || ((uintptr_t)codes & 3u))
    return MOE_W4A8_INVALID_ARG;
  const long long warps = (long long)rows * (K / moe::kBlk);
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return MOE_W4A8_INVALID_ARG;
  moe::quantize_blocks_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      x, rows, K, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_W4A8_OK : MOE_W4A8_CUDA_ERROR;
}

extern "C" int moe_w4a8_linear(const uint8_t* codes, const float* x_scales, int32_t rows,
                               int32_t K, const uint32_t* w_q, const uint16_t* w_s, int32_t N,
                               float* y, void* stream) {
  if (rows < 0 || K <= 0 || K % moe::kBlk != 0 || N <= 0 || N % 16 != 0)
    return MOE_W4A8_INVALID_ARG;
  if (rows == 0) return MOE_W4A8_OK;
  if (!codes || !x_scales || !w_q || !w_s || !y || ((uintptr_t)codes & 3u) || ((uintptr_t)w_q & 3u))
    return MOE_W4A8_INVALID_ARG;
  const dim3 grid(N / 16, (rows + 7) / 8);
  if (grid.y > 65535u) return MOE_W4A8_INVALID_ARG;
  moe::linear_kernel<<<grid, 32, 0, (cudaStream_t)stream>>>(codes, x_scales, rows, K, w_q, w_s, N, y);
  return cudaGetLastError() == cudaSuccess ? MOE_W4A8_OK : MOE_W4A8_CUDA_ERROR;
}

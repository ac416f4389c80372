// Weighted unpermute-combine fused with the shared expert's output.
//
// out[t] = y_shared[t] + sum_j w[t, j] * y[inv[t, j]]   (fp32 sums, then bf16 RNE;
// y is fp32 from the GEMV engine, bf16 from the tensor-core engine)
//
// This stands in for the expert-parallel combine of the pages' serving setup
// ("Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", "A first cut":
// --enable-expert-parallel): on one GPU the all-to-all becomes a gather of the
// expert-sorted rows. Slots are summed in fixed order j = 0..k-1 after the
// shared expert, so a token's result does not depend on the rest of the batch.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// fp32 y: four channels per thread (16-byte loads).
__global__ void __launch_bounds__(256) combine_f32_kernel(const Dims d, const Routing r,
                                                          const float* __restrict__ y,
                                                          uint16_t* __restrict__ out) {
  const int h4 = d.H / 4;
  const long long total = (long long)d.T * h4;
  const float4* y4 = reinterpret_cast<const float4*>(y);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / h4), n4 = (int)(idx - (long long)t * h4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (d.Is > 0) acc = y4[(size_t)(d.T * d.k + t) * h4 + n4];
    for (int j = 0; j < d.k; ++j) {
      const float w = r.wts[t * d.k + j];
      const int row = r.inv[t * d.k + j];
      if (row < 0 || row >= d.T * d.k) {
        atomicOr(r.err, kErrRange);
        continue;
      }
      const float4 v = y4[(size_t)row * h4 + n4];
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(acc.x) | ((uint32_t)f32_to_bf16_bits(acc.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(acc.z) | ((uint32_t)f32_to_bf16_bits(acc.w) << 16);
    reinterpret_cast<uint2*>(out)[idx] = o;
  }
}

// bf16 y: eight channels per thread (16-byte loads), each widened exactly.
__device__ __forceinline__ void fma_bf16x8(float w, const uint4& v, float (&a)[8]) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), a[2 * i]);
    a[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xffff0000u), a[2 * i + 1]);
  }
}

__global__ void __launch_bounds__(256) combine_bf16_kernel(const Dims d, const Routing r,
                                                           const uint16_t* __restrict__ y,
                                                           uint16_t* __restrict__ out) {
  const int h8 = d.H / 8;
  const long long total = (long long)d.T * h8;
  const uint4* y8 = reinterpret_cast<const uint4*>(y);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / h8), n8 = (int)(idx - (long long)t * h8);
    float a[8];
    if (d.Is > 0) {
      const uint4 v = y8[(size_t)(d.T * d.k + t) * h8 + n8];
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[2 * i] = __uint_as_float(q[i] << 16);
        a[2 * i + 1] = __uint_as_float(q[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = 0.f;
    }
    for (int j = 0; j < d.k; ++j) {
      const float w = r.wts[t * d.k + j];
      const int row = r.inv[t * d.k + j];
      if (row < 0 || row >= d.T * d.k) {
        atomicOr(r.err, kErrRange);
        continue;
      }
      fma_bf16x8(w, y8[(size_t)row * h8 + n8], a);
    }
    uint4 o;
    o.x = (uint32_t)f32_to_bf16_bits(a[0]) | ((uint32_t)f32_to_bf16_bits(a[1]) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(a[2]) | ((uint32_t)f32_to_bf16_bits(a[3]) << 16);
    o.z = (uint32_t)f32_to_bf16_bits(a[4]) | ((uint32_t)f32_to_bf16_bits(a[5]) << 16);
    o.w = (uint32_t)f32_to_bf16_bits(a[6]) | ((uint32_t)f32_to_bf16_bits(a[7]) << 16);
    reinterpret_cast<uint4*>(out)[idx] = o;
  }
}

int combine_blocks(long long total) {
  long long blocks = (total + 255) / 256;
  return (int)(blocks > 152 * 16 ? 152 * 16 : blocks);
}

}  // namespace

cudaError_t launch_combine(const Dims& d, const Routing& r, const float* y, uint16_t* out,
                           cudaStream_t s, LaunchLog& log) {
  log.begin("combine", s);
  combine_f32_kernel<<<combine_blocks((long long)d.T * (d.H / 4)), 256, 0, s>>>(d, r, y, out);
  log.end(s);
  return cudaGetLastError();
}
cudaError_t launch_combine(const Dims& d, const Routing& r, const uint16_t* y, uint16_t* out,
                           cudaStream_t s, LaunchLog& log) {
  log.begin("combine", s);
  combine_bf16_kernel<<<combine_blocks((long long)d.T * (d.H / 8)), 256, 0, s>>>(d, r, y, out);
  log.end(s);
  return cudaGetLastError();
}

}  // namespace moe

// Weighted unpermute-combine fused with the shared expert's output.
//
// out[t] = y_shared[t] + sum_j w[t, j] * y[inv[t, j]]   (fp32, then bf16 RNE)
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

__global__ void __launch_bounds__(256) combine_kernel(const Dims d, const Routing r,
                                                      const float* __restrict__ y,
                                                      uint16_t* __restrict__ out) {
  const int h4 = d.H / 4;
  const long long total = (long long)d.T * h4;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / h4), n4 = (int)(idx - (long long)t * h4);
    const float4* y4 = reinterpret_cast<const float4*>(y);
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

}  // namespace

cudaError_t launch_combine(const Dims& d, const Routing& r, const float* y, uint16_t* out,
                           cudaStream_t s, LaunchLog& log) {
  const long long total = (long long)d.T * (d.H / 4);
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  log.begin("combine", s);
  combine_kernel<<<(int)blocks, 256, 0, s>>>(d, r, y, out);
  log.end(s);
  return cudaGetLastError();
}

}  // namespace moe

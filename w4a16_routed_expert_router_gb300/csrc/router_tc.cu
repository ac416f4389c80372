// Router logits on the tensor cores for large batches.
//
// logit[t, e] = sum_h x[t, h] * W[e, h], x bf16, W fp32 (the gate weight is
// kept in full precision; "canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP",
// table "Component precisions"). The fp32 weight is split into three bf16
// planes, W = W0 + W1 + W2 with W0 = bf16(W), W1 = bf16(W - W0),
// W2 = bf16(W - W0 - W1), which carry 24 significant bits between them; each
// product of a bf16 x with a plane is exact in fp32, so the sum of three
// kind::f16 MMAs is the fp32 dot product up to how the additions round.
//
// The tensor core's fp32 accumulation is not carried along the whole hidden
// dimension: each 64-wide K block (12 MMAs) goes into a fresh TMEM
// accumulator, and the epilogue warps add the block sums into fp32 registers
// with ordinary round-to-nearest additions, in block order. Accumulating all
// 4096 products inside the MMA drifted by several 1e-5 on N(0,1)-sized logits
// (measured against the fp64 oracle); the block-wise sums keep the error at
// the level of an fp32 loop.
//
// One CTA computes a 128-expert x 128-token tile over the whole hidden
// dimension: warp 0 streams the three plane tiles and the token tile by TMA
// (128-byte swizzle), warp 1 owns two 128-column TMEM accumulators and issues
// the MMAs, warps 2-9 (64 tokens of 32 experts each) sum the blocks and store
// fp32 logits [T, E].
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kRThreads = 10 * 32;
constexpr int kRBK = 64;                 // K per stage: one 128-byte swizzle atom
constexpr int kRStages = 3;
constexpr int kRTile = 128 * kRBK * 2;   // 16 KB: 128 rows x 64 bf16
constexpr int kRStageB = 4 * kRTile;     // three weight planes + the token tile

struct RSmem {
  uint8_t stage[kRStages][kRStageB];
  uint64_t full[kRStages], empty[kRStages];
  uint64_t acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
};
constexpr int kRSmemBytes = (int)sizeof(RSmem) + 1024;
// Each CTA allocates 256 of the SM's 512 TMEM columns: at most two CTAs may
// share an SM, which the shared-memory footprint guarantees.
static_assert(3 * kRSmemBytes > 228 * 1024, "router_tc_kernel must stay at <= 2 CTAs per SM");

__global__ void __launch_bounds__(256) router_split_kernel(const float4* __restrict__ w,
                                                           uint2* __restrict__ planes, long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = w[i];
    const float a[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[3][2];
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      float r0 = a[j], r1 = a[j + 1];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const uint16_t b0 = f32_to_bf16_bits(r0), b1 = f32_to_bf16_bits(r1);
        p[q][j >> 1] = (uint32_t)b0 | ((uint32_t)b1 << 16);
        r0 -= bf16_bits_to_f32(b0);  // exact: the remainder of a round-to-nearest
        r1 -= bf16_bits_to_f32(b1);
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) planes[q * n4 + i] = make_uint2(p[q][0], p[q][1]);
  }
}

__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                     const __grid_constant__ CUtensorMap wmap, const Dims d, float* logits,
                     unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  RSmem& s =
      *reinterpret_cast<RSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 128, e0 = blockIdx.y * 128;
  const int nkb = d.H / kRBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], 8);
    }
    mbar_init(&s.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t filled = 0, last_ph = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % kRStages;
        const uint32_t ph = (kb / kRStages) & 1;
        if (!bwait(&s.empty[st], ph ^ 1u, err)) break;
        mbar_arrive_expect_tx(&s.full[st], kRStageB);
        const uint32_t dst = smem_u32(s.stage[st]);
        for (int q = 0; q < 3; ++q)
          tma_2d(dst + q * kRTile, &wmap, &s.full[st], kb * kRBK, q * d.E + e0);
        tma_2d(dst + 3 * kRTile, &xmap, &s.full[st], kb * kRBK, t0);
        filled |= 1u << st;
        last_ph = (last_ph & ~(1u << st)) | (ph << st);
      }
      // no copy may still be landing when the CTA exits
      for (int i = 0; i < kRStages; ++i)
        if (filled & (1u << i)) mbar_wait(&s.full[i], (last_ph >> i) & 1u, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 128);
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % kRStages, ab = kb & 1;
        if (!bwait(&s.acc_empty[ab], ((kb >> 1) & 1) ^ 1u, err) ||
            !bwait(&s.full[st], (kb / kRStages) & 1, err))
          break;
        tc_fence_after();
        const uint32_t base = smem_u32(s.stage[st]);
        const uint32_t acc = tmem + ab * 128;
#pragma unroll
        for (int k = 0; k < kRBK / 16; ++k) {
          const uint64_t bd = smem_desc_sw128(base + 3 * kRTile + k * 32);
#pragma unroll
          for (int q = 0; q < 3; ++q)
            mma_bf16(acc, smem_desc_sw128(base + q * kRTile + k * 32), bd, idesc, (k | q) ? 1u : 0u);
        }
        mma_commit(&s.empty[st]);
        mma_commit(&s.acc_full[ab]);
      }
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0, err);
    }
  } else {
    // block sums: TMEM lane = expert within the tile, column = token; warp
    // 2 + i takes lane quarter i & 3 and tokens [64 (i >> 2), +64)
    const int q = warp & 3, cb = ((warp - 2) >> 2) * 64;
    const int e = e0 + q * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + cb;
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int ab = kb & 1;
      if (!warp_wait(&s.acc_full[ab], (kb >> 1) & 1, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[32];
      tmem_ld32(lane_addr + ab * 128, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] += v[j];
      tmem_ld32(lane_addr + ab * 128 + 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[32 + j] += v[j];
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.acc_empty[ab]);
    }
    if (ok && e < d.E) {
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (t0 + cb + j < d.T) logits[(size_t)(t0 + cb + j) * d.E + e] = acc[j];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_free(tmem, 256);
  }
}

}  // namespace

cudaError_t router_tc_setup() {
  return cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kRSmemBytes);
}

cudaError_t launch_router_logits_tc(const Dims& d, const float* router_w, uint16_t* planes,
                                    const CUtensorMap& xmap, const CUtensorMap& wmap, float* logits,
                                    unsigned* err, cudaStream_t s, LaunchLog& log) {
  const long long n4 = (long long)d.E * d.H / 4;
  log.begin("router_split", s);
  router_split_kernel<<<(int)((n4 + 255) / 256 < 1216 ? (n4 + 255) / 256 : 1216), 256, 0, s>>>(
      reinterpret_cast<const float4*>(router_w), reinterpret_cast<uint2*>(planes), n4);
  log.end(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  log.begin("router_logits_tc", s);
  router_tc_kernel<<<dim3((d.T + 127) / 128, (d.E + 127) / 128), kRThreads, kRSmemBytes, s>>>(
      xmap, wmap, d, logits, err);
  log.end(s);
  return cudaGetLastError();
}

}  // namespace moe

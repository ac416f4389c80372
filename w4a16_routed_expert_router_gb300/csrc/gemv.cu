// Split-K GEMV expert kernels of the W4A16 MoE layer (decode-sized batches).
//
// "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", sections "A pass
// through the model" and "Where does the time go?": below the bf16 ridge the
// expert GEMMs are memory bound, so at decode sizes the job is to stream the
// packed INT4 weights of the experts that were hit exactly once at full HBM
// bandwidth and turn them into bf16 in registers.
//
// Design (GB300):
//  * persistent CTAs (1 per SM), a static round-robin over tasks. A task is
//    (active expert, channel tile, pass of <= 16 rows of that expert).
//  * one producer warp streams the task's weight tiles with 3-D TMA into a
//    8-stage shared-memory ring (mbarrier full/empty handshake); a stage holds
//    two 16-row tiles x 8 K-groups of 128 (16 KB of packed INT4).
//  * 8 consumer warps split K: warp w takes K-group w of every stage. Each
//    lane turns its 4-bit codes into exact bf16 integers (one lop3 and one
//    bf16x2 subtract per pair) and feeds mma.sync m16n8k16 with weights as
//    the 16-row A operand and up to 8 tokens as B. The group scale is applied
//    in fp32 to the group's partial sums, so q * scale is never rounded.
//  * the K order inside one MMA is a fixed permutation of the true K order;
//    the token operand (x, or the gate/up output h) is stored in the same
//    permutation ("interleaved": within each 8 values, (0,4)(1,5)(2,6)(3,7)).
//  * cross-warp reduction in fixed warp order (deterministic, batch
//    invariant), then the epilogue: SwiGLU -> bf16 h (gate/up) or fp32 y (down).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kStageBytes = 2 * 8 * 1024;       // 2 tiles x 8 groups x (16 rows x 64 B)
constexpr int kRedFloats = 8 * 2 * 2 * 32 * 4;  // warps x tiles x token blocks x lanes x 4
constexpr int kSmemBytes = kGemvStages * kStageBytes + kRedFloats * 4 + 2 * kGemvStages * 8;

struct GemvParams {
  Dims d;
  Routing r;
  const uint16_t* scale_routed;
  const uint16_t* scale_shared;
  const uint16_t* bsrc;  // token operand, interleaved rows
  int bstride;           // elements per token-operand row
  uint16_t* hout;        // gate/up: h [rows, hstride]
  int hstride;
  float* yout;           // down: y [rows, H]
};

struct Task {
  bool shared;
  int ngroups;  // K / 128
  int rowA0;    // first row of tile 0 in the tensor map's row space
  int rowA1;    // first row of tile 1
  int r0;       // first expert-sorted row of this pass
  int nr;       // rows in this pass (1..16)
  int tile;     // channel tile index
};

template <int MODE>
__device__ __forceinline__ Task decode_task(const GemvParams& p, int tau) {
  const Dims& d = p.d;
  const int* prefix = (MODE == 1) ? p.r.task1 : p.r.task2;
  const int n_total = p.r.meta[kMetaActive];
  int lo = 0, hi = n_total - 1;  // find a with prefix[a] <= tau < prefix[a+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tau)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int a = lo;
  const int local = tau - prefix[a];
  const int e = p.r.active[a];
  Task t;
  t.shared = (e == d.E);
  const int seg0 = t.shared ? d.T * d.k : p.r.offsets[e];
  const int seg1 = t.shared ? d.T * d.k + d.T : p.r.offsets[e + 1];
  const int passes = (seg1 - seg0 + kPassRows - 1) / kPassRows;
  t.tile = local / passes;
  const int pass = local - t.tile * passes;
  t.r0 = seg0 + pass * kPassRows;
  t.nr = min(kPassRows, seg1 - t.r0);
  if (MODE == 1) {
    const int inter = t.shared ? d.Is : d.I;
    t.ngroups = d.H / kGroup;
    t.rowA0 = (t.shared ? 0 : e * 2 * inter) + t.tile * kTile1;
    t.rowA1 = t.rowA0 + inter;
  } else {
    t.ngroups = (t.shared ? d.Is : d.I) / kGroup;
    t.rowA0 = (t.shared ? 0 : e * d.H) + t.tile * kTile2;
    t.rowA1 = t.rowA0 + 16;
  }
  return t;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void named_bar_consumers() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// 8 MMA steps (128 K) of one warp for one tile pair and one token block.
// wA/wB: rows g and g+8 of the tile (4 words each); b[m]: token operand.
__device__ __forceinline__ void group_mma(const uint4& wA, const uint4& wB, const uint4* b,
                                          float* tmp) {
  tmp[0] = tmp[1] = tmp[2] = tmp[3] = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t ra = word_of(wA, m), rb = word_of(wB, m);
    uint32_t a[4];
    a[0] = int4_pair_to_bf16x2<0>(ra);
    a[1] = int4_pair_to_bf16x2<0>(rb);
    a[2] = int4_pair_to_bf16x2<1>(ra);
    a[3] = int4_pair_to_bf16x2<1>(rb);
    mma_bf16_16816(tmp, a, b[m].x, b[m].y, tmp);
    a[0] = int4_pair_to_bf16x2<2>(ra);
    a[1] = int4_pair_to_bf16x2<2>(rb);
    a[2] = int4_pair_to_bf16x2<3>(ra);
    a[3] = int4_pair_to_bf16x2<3>(rb);
    mma_bf16_16816(tmp, a, b[m].z, b[m].w, tmp);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_routed,
                const __grid_constant__ CUtensorMap tm_shared, const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + kGemvStages * kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGemvStages * kStageBytes + kRedFloats * 4);
  uint64_t* empty = full + kGemvStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntasks = p.r.meta[MODE == 1 ? kMetaTasks1 : kMetaTasks2];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemvStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_routed);
      prefetch_tmap(&tm_shared);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < ntasks && ok; tau += gridDim.x) {
        const Task t = decode_task<MODE>(p, tau);
        const CUtensorMap* tm = t.shared ? &tm_shared : &tm_routed;
        for (int g0 = 0; g0 < t.ngroups; g0 += 8) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.r.err)) {
            ok = false;
            break;
          }
          const int gcnt = min(8, t.ngroups - g0);
          mbar_arrive_expect_tx(&full[stage], gcnt * 2 * 1024);
          uint8_t* dst = stages + stage * kStageBytes;
          for (int g = 0; g < gcnt; ++g) {
            tma_load_3d(dst + g * 1024, tm, &full[stage], 0, g0 + g, t.rowA0);
            tma_load_3d(dst + (8 + g) * 1024, tm, &full[stage], 0, g0 + g, t.rowA1);
          }
          if (++stage == kGemvStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const Dims& d = p.d;
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int tau = blockIdx.x; tau < ntasks; tau += gridDim.x) {
    const Task t = decode_task<MODE>(p, tau);
    const uint16_t* scales = t.shared ? p.scale_shared : p.scale_routed;
    const int ng = t.ngroups;
    // token-operand rows of this lane (B column g of each 8-token block)
    const uint16_t* brow[2];
    bool bval[2];
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      const int j = tb * 8 + g;
      bval[tb] = j < t.nr;
      int row = t.r0 + (bval[tb] ? j : 0);
      if (MODE == 1) row = t.shared ? row - d.T * d.k : p.r.perm[row];
      brow[tb] = p.bsrc + (size_t)row * p.bstride + 32 * c;
    }
    const bool tb1 = t.nr > 8;
    float acc[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;

    const size_t s00 = (size_t)(t.rowA0 + g) * ng, s01 = s00 + (size_t)8 * ng;
    const size_t s10 = (size_t)(t.rowA1 + g) * ng, s11 = s10 + (size_t)8 * ng;

    for (int g0 = 0; g0 < ng; g0 += 8) {
      const int gi = g0 + warp;
      const bool mine = gi < ng;
      float sc[4];
      uint4 b0[4], b1[4];
      if (mine) {
        sc[0] = bf16_bits_to_f32(__ldg(scales + s00 + gi));
        sc[1] = bf16_bits_to_f32(__ldg(scales + s01 + gi));
        sc[2] = bf16_bits_to_f32(__ldg(scales + s10 + gi));
        sc[3] = bf16_bits_to_f32(__ldg(scales + s11 + gi));
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          b0[m] = bval[0] ? __ldg(reinterpret_cast<const uint4*>(brow[0] + gi * kGroup) + m)
                          : make_uint4(0, 0, 0, 0);
          b1[m] = (tb1 && bval[1])
                      ? __ldg(reinterpret_cast<const uint4*>(brow[1] + gi * kGroup) + m)
                      : make_uint4(0, 0, 0, 0);
        }
      }
      if (ok) ok = mbar_wait(&full[stage], phase, p.r.err);
      if (mine && ok) {
        const uint32_t base = smem_u32(stages + stage * kStageBytes) + warp * 1024 + g * 64 + c * 16;
        const uint4 w00 = lds128(base), w01 = lds128(base + 8 * 64);
        const uint4 w10 = lds128(base + 8 * 1024), w11 = lds128(base + 8 * 1024 + 8 * 64);
        float tmp[4];
        group_mma(w00, w01, b0, tmp);
        acc[0][0][0] = fmaf(sc[0], tmp[0], acc[0][0][0]);
        acc[0][0][1] = fmaf(sc[0], tmp[1], acc[0][0][1]);
        acc[0][0][2] = fmaf(sc[1], tmp[2], acc[0][0][2]);
        acc[0][0][3] = fmaf(sc[1], tmp[3], acc[0][0][3]);
        group_mma(w10, w11, b0, tmp);
        acc[1][0][0] = fmaf(sc[2], tmp[0], acc[1][0][0]);
        acc[1][0][1] = fmaf(sc[2], tmp[1], acc[1][0][1]);
        acc[1][0][2] = fmaf(sc[3], tmp[2], acc[1][0][2]);
        acc[1][0][3] = fmaf(sc[3], tmp[3], acc[1][0][3]);
        if (tb1) {
          group_mma(w00, w01, b1, tmp);
          acc[0][1][0] = fmaf(sc[0], tmp[0], acc[0][1][0]);
          acc[0][1][1] = fmaf(sc[0], tmp[1], acc[0][1][1]);
          acc[0][1][2] = fmaf(sc[1], tmp[2], acc[0][1][2]);
          acc[0][1][3] = fmaf(sc[1], tmp[3], acc[0][1][3]);
          group_mma(w10, w11, b1, tmp);
          acc[1][1][0] = fmaf(sc[2], tmp[0], acc[1][1][0]);
          acc[1][1][1] = fmaf(sc[2], tmp[1], acc[1][1][1]);
          acc[1][1][2] = fmaf(sc[3], tmp[2], acc[1][1][2]);
          acc[1][1][3] = fmaf(sc[3], tmp[3], acc[1][1][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kGemvStages) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- deterministic cross-warp reduction and epilogue
    float4* redw = reinterpret_cast<float4*>(red);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j)
        redw[((warp * 2 + i) * 2 + j) * 32 + lane] =
            make_float4(acc[i][j][0], acc[i][j][1], acc[i][j][2], acc[i][j][3]);
    named_bar_consumers();
    {
      const int row = threadIdx.x >> 4, tok = threadIdx.x & 15;
      const int tb = tok >> 3, col = tok & 7;
      const int ln = (row & 7) * 4 + (col >> 1), q = (row >> 3) * 2 + (col & 1);
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        v0 += red[(((w * 2 + 0) * 2 + tb) * 32 + ln) * 4 + q];
        v1 += red[(((w * 2 + 1) * 2 + tb) * 32 + ln) * 4 + q];
      }
      if (tok < t.nr) {
        const size_t orow = (size_t)(t.r0 + tok);
        if (MODE == 1) {
          const int n = t.tile * kTile1 + row;
          const int pos = (n & ~7) | ((n & 3) << 1) | ((n >> 2) & 1);
          p.hout[orow * p.hstride + pos] = f32_to_bf16_bits(silu(v0) * v1);
        } else {
          const int n = t.tile * kTile2 + row;
          p.yout[orow * d.H + n] = v0;
          p.yout[orow * d.H + n + 16] = v1;
        }
      }
    }
    named_bar_consumers();
  }
}

GemvParams make_params(const Dims& d, const Routing& r, const GemvWeights& w) {
  GemvParams p;
  p.d = d;
  p.r = r;
  p.scale_routed = w.scale_routed;
  p.scale_shared = w.scale_shared;
  p.bsrc = nullptr;
  p.bstride = 0;
  p.hout = nullptr;
  p.hstride = 0;
  p.yout = nullptr;
  return p;
}

}  // namespace

cudaError_t gemv_setup(int* ctas_per_sm) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes)) != cudaSuccess)
    return e;
  int n1 = 0, n2 = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, gemv_kernel<1>, kGemvThreads,
                                                         kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n2, gemv_kernel<2>, kGemvThreads,
                                                         kSmemBytes)) != cudaSuccess)
    return e;
  *ctas_per_sm = n1 < n2 ? n1 : n2;
  return cudaSuccess;
}

cudaError_t launch_gemv_gate_up(const Dims& d, const Routing& r, const GemvWeights& w,
                                const uint16_t* xg, uint16_t* h, int hstride, int grid,
                                cudaStream_t s, LaunchLog& log) {
  GemvParams p = make_params(d, r, w);
  p.bsrc = xg;
  p.bstride = d.H;
  p.hout = h;
  p.hstride = hstride;
  log.begin("gemv_gate_up_swiglu", s);
  gemv_kernel<1><<<grid, kGemvThreads, kSmemBytes, s>>>(w.tm_routed, w.tm_shared, p);
  log.end(s);
  return cudaGetLastError();
}

cudaError_t launch_gemv_down(const Dims& d, const Routing& r, const GemvWeights& w,
                             const uint16_t* h, int hstride, float* y, int grid, cudaStream_t s,
                             LaunchLog& log) {
  GemvParams p = make_params(d, r, w);
  p.bsrc = h;
  p.bstride = hstride;
  p.yout = y;
  log.begin("gemv_down", s);
  gemv_kernel<2><<<grid, kGemvThreads, kSmemBytes, s>>>(w.tm_routed, w.tm_shared, p);
  log.end(s);
  return cudaGetLastError();
}

}  // namespace moe

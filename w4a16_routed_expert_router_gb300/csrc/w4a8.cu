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
#include "kernels.h"
#include "moe_w4a8.h"

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

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const uint16_t* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// x: [rows, K] fp32 or bf16 (row stride K); codes [rows, K] e4m3 bytes;
// scales [rows, K / 128] fp32. Warp w of the grid takes block (w / nb, w % nb);
// lane l its elements 4l .. 4l + 3.
template <typename In>
__global__ void quantize_blocks_kernel(const In* __restrict__ x, int rows, int K,
                                       uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int nb = K / kBlk;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)rows * nb) return;
  const int r = (int)(wid / nb), g = (int)(wid - (long long)r * nb);
  const float4 v = load4(x + (size_t)r * K + g * kBlk + 4 * lane);
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

// ------------------------------------------------------------ the layer
// One 16-channel x 8-row tile of the block-scaled product over the 128-blocks
// g = g0, g0 + gstep, ... < nb: A the INT4 weight rows wr0 (channel gid) and
// wr1 (gid + 8) with their bf16 group scales ws0 / ws1, B this lane's
// activation row (codes, or null: a padding row), D rows scaled by sx0 / sx1
// (null: padding).
__device__ __forceinline__ void tile_16x8(const uint32_t* wr0, const uint32_t* wr1,
                                          const uint16_t* ws0, const uint16_t* ws1, int nb, int g0,
                                          int gstep, const uint8_t* brow, const float* sx0,
                                          const float* sx1, int tig, float (&acc)[4]) {
  for (int g = g0; g < nb; g += gstep) {
    float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kBlk / 32; ++ks) {
      const int kb = g * kBlk + ks * 32;
      const int wlo = (kb + 4 * tig) >> 3, shlo = ((4 * tig) & 7) * 4;
      const int whi = (kb + 16 + 4 * tig) >> 3, shhi = ((16 + 4 * tig) & 7) * 4;
      uint32_t a[4];
      a[0] = int4x4_to_e4m3x4(__ldg(wr0 + wlo) >> shlo);
      a[1] = int4x4_to_e4m3x4(__ldg(wr1 + wlo) >> shlo);
      a[2] = int4x4_to_e4m3x4(__ldg(wr0 + whi) >> shhi);
      a[3] = int4x4_to_e4m3x4(__ldg(wr1 + whi) >> shhi);
      uint32_t b[2];
      b[0] = brow ? *reinterpret_cast<const uint32_t*>(brow + kb + 4 * tig) : 0u;
      b[1] = brow ? *reinterpret_cast<const uint32_t*>(brow + kb + 16 + 4 * tig) : 0u;
      mma_e4m3_16832(part, a, b);
    }
    const float w0 = __uint_as_float((uint32_t)__ldg(ws0 + g) << 16);
    const float w1 = __uint_as_float((uint32_t)__ldg(ws1 + g) << 16);
    const float x0 = sx0 ? sx0[g] : 0.f, x1 = sx1 ? sx1[g] : 0.f;
    acc[0] = fmaf(w0 * x0, part[0], acc[0]);
    acc[1] = fmaf(w0 * x1, part[1], acc[1]);
    acc[2] = fmaf(w1 * x0, part[2], acc[2]);
    acc[3] = fmaf(w1 * x1, part[3], acc[3]);
  }
}

struct W4a8Layer {
  Dims d;
  Routing r;
  W4a8Weights w;
  const uint8_t* xc;  // e4m3 x [T, H] (token order)
  const float* xs;    // [T, H / 128]
  float* hf;          // fp32 h [rows, hst] (expert-sorted rows)
  const uint8_t* hc;  // e4m3 h [rows, hst]
  const float* hs;    // [rows, hst / 128]
  int hst;
  float* y;           // fp32 [rows, H]
};

__device__ __forceinline__ int passes8(int rows) { return (rows + kPassRows - 1) / kPassRows; }

// The expert tasks of the W4A16 GEMV engine (the routing lists their prefix
// per active expert): the shared expert's first, then (expert, channel tile,
// 8-row pass) in expert order. MODE 1: 16 gate + 16 up channels; MODE 2: 32
// output channels. One block of kSplit warps per task (grid-stride): warp w
// takes the 128-blocks w, w + kSplit, ... of K; warp 0 adds the warps'
// partials in warp order and writes the result.
constexpr int kSplit = 4;
template <int MODE>
__global__ void __launch_bounds__(kSplit * 32) grouped_kernel(const W4a8Layer L) {
  __shared__ float red[kSplit][32][8];
  const Dims& d = L.d;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int ct_sh = MODE == 1 ? d.Is / kTile1 : d.H / kTile2;
  const int n_sh = d.Is > 0 ? ct_sh * passes8(d.T) : 0;
  const int n_act = L.r.meta[kMetaActive];
  const int total = n_sh + L.r.meta[MODE == 1 ? kMetaTasks1 : kMetaTasks2];
  const int* pre = MODE == 1 ? L.r.task1 : L.r.task2;
  for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
    bool sh;
    int e, seg0, seg1, local;
    if (tau < n_sh) {
      sh = true;
      e = d.E;
      seg0 = d.T * d.k;
      seg1 = seg0 + d.T;
      local = tau;
    } else {
      sh = false;
      const int tr = tau - n_sh;
      int lo = 0, hi = n_act - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(pre + mid) <= tr) lo = mid;
        else hi = mid - 1;
      }
      e = __ldg(L.r.active + lo);
      seg0 = __ldg(L.r.offsets + e);
      seg1 = __ldg(L.r.offsets + e + 1);
      local = tr - __ldg(pre + lo);
    }
    const int passes = passes8(seg1 - seg0);
    const int tile = local / passes, pass = local - tile * passes;
    const int r0 = seg0 + pass * kPassRows, nr = min(kPassRows, seg1 - r0);
    const int inter = sh ? d.Is : d.I;
    // this lane's B row and the rows of its D values (expert-sorted row space)
    const int rb = r0 + gid, rc0 = r0 + 2 * tig, rc1 = rc0 + 1;
    const bool vb = gid < nr, v0 = 2 * tig < nr, v1 = 2 * tig + 1 < nr;
    if (MODE == 1) {
      // activations: x codes of the row's token
      auto tok = [&](int row) { return sh ? row - d.T * d.k : __ldg(L.r.perm + row); };
      const int nbx = d.H / kBlk;
      const uint8_t* brow = vb ? L.xc + (size_t)tok(rb) * d.H : nullptr;
      const float* s0 = v0 ? L.xs + (size_t)tok(rc0) * nbx : nullptr;
      const float* s1 = v1 ? L.xs + (size_t)tok(rc1) * nbx : nullptr;
      const uint32_t* wq = sh ? L.w.sh_w13_q : L.w.w13_q;
      const uint16_t* wsc = sh ? L.w.sh_w13_s : L.w.w13_s;
      const int rowg = (sh ? 0 : e * 2 * inter) + tile * kTile1, rowu = rowg + inter;
      const int kw = d.H / 8;
      float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
      tile_16x8(wq + (size_t)(rowg + gid) * kw, wq + (size_t)(rowg + gid + 8) * kw,
                wsc + (size_t)(rowg + gid) * nbx, wsc + (size_t)(rowg + gid + 8) * nbx, nbx, warp,
                kSplit, brow, s0, s1, tig, g);
      tile_16x8(wq + (size_t)(rowu + gid) * kw, wq + (size_t)(rowu + gid + 8) * kw,
                wsc + (size_t)(rowu + gid) * nbx, wsc + (size_t)(rowu + gid + 8) * nbx, nbx, warp,
                kSplit, brow, s0, s1, tig, u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        red[warp][lane][i] = g[i];
        red[warp][lane][4 + i] = u[i];
      }
      __syncthreads();
      if (warp == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          g[i] = red[0][lane][i];
          u[i] = red[0][lane][4 + i];
        }
        for (int w = 1; w < kSplit; ++w)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            g[i] += red[w][lane][i];
            u[i] += red[w][lane][4 + i];
          }
      }
      const int c0 = tile * kTile1 + gid;
      auto hv = [](float gg, float uu) { return gg / (1.0f + __expf(-gg)) * uu; };
      if (warp == 0 && v0) {
        L.hf[(size_t)rc0 * L.hst + c0] = hv(g[0], u[0]);
        L.hf[(size_t)rc0 * L.hst + c0 + 8] = hv(g[2], u[2]);
      }
      if (warp == 0 && v1) {
        L.hf[(size_t)rc1 * L.hst + c0] = hv(g[1], u[1]);
        L.hf[(size_t)rc1 * L.hst + c0 + 8] = hv(g[3], u[3]);
      }
      __syncthreads();  // red is rewritten by the next task
    } else {
      // activations: this row's h codes (already in expert-sorted order)
      const int nbh = L.hst / kBlk, nbk = inter / kBlk;
      const uint8_t* brow = vb ? L.hc + (size_t)rb * L.hst : nullptr;
      const float* s0 = v0 ? L.hs + (size_t)rc0 * nbh : nullptr;
      const float* s1 = v1 ? L.hs + (size_t)rc1 * nbh : nullptr;
      const uint32_t* wq = sh ? L.w.sh_w2_q : L.w.w2_q;
      const uint16_t* wsc = sh ? L.w.sh_w2_s : L.w.w2_s;
      const int kw = inter / 8;
      float acc[2][4] = {};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int row = (sh ? 0 : e * d.H) + tile * kTile2 + 16 * half;
        tile_16x8(wq + (size_t)(row + gid) * kw, wq + (size_t)(row + gid + 8) * kw,
                  wsc + (size_t)(row + gid) * nbk, wsc + (size_t)(row + gid + 8) * nbk, nbk, warp,
                  kSplit, brow, s0, s1, tig, acc[half]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        red[warp][lane][i] = acc[0][i];
        red[warp][lane][4 + i] = acc[1][i];
      }
      __syncthreads();
      if (warp == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[0][i] = red[0][lane][i];
          acc[1][i] = red[0][lane][4 + i];
        }
        for (int w = 1; w < kSplit; ++w)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[0][i] += red[w][lane][i];
            acc[1][i] += red[w][lane][4 + i];
          }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int c0 = tile * kTile2 + 16 * half + gid;
          if (v0) {
            L.y[(size_t)rc0 * d.H + c0] = acc[half][0];
            L.y[(size_t)rc0 * d.H + c0 + 8] = acc[half][2];
          }
          if (v1) {
            L.y[(size_t)rc1 * d.H + c0] = acc[half][1];
            L.y[(size_t)rc1 * d.H + c0 + 8] = acc[half][3];
          }
        }
      }
      __syncthreads();  // red is rewritten by the next task
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_w4a8_experts(const Dims& d, const Routing& r, const W4a8Weights& w,
                                const uint16_t* x, uint8_t* xc, float* xs, float* hf, uint8_t* hc,
                                float* hs, int hst, float* y, int grid, cudaStream_t s,
                                LaunchLog& log) {
  cudaError_t e;
  const int rows = d.T * d.k + (d.Is > 0 ? d.T : 0);
  log.begin("w4a8_quantize_x", s);
  {
    const long long warps = (long long)d.T * (d.H / kBlk);
    quantize_blocks_kernel<uint16_t><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(
        x, d.T, d.H, xc, xs);
  }
  log.end(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  W4a8Layer L{d, r, w, xc, xs, hf, hc, hs, hst, y};
  // four 4-warp blocks per SM, all resident (up to 108 registers a thread)
  grid *= 4;
  log.begin("w4a8_gate_up_swiglu", s);
  grouped_kernel<1><<<grid, kSplit * 32, 0, s>>>(L);
  log.end(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  log.begin("w4a8_quantize_h", s);
  {
    const long long warps = (long long)rows * (hst / kBlk);
    quantize_blocks_kernel<float><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(
        hf, rows, hst, hc, hs);
  }
  log.end(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  log.begin("w4a8_down", s);
  grouped_kernel<2><<<grid, kSplit * 32, 0, s>>>(L);
  log.end(s);
  return cudaGetLastError();
}

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
  moe::quantize_blocks_kernel<float><<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
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

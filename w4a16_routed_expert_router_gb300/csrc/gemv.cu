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
//    (expert, channel tile, pass of <= 8 rows of that expert's segment). The
//    shared expert's tasks come first: they need no routing, so with
//    programmatic dependent launch they start while the router still runs.
//  * one producer thread fills a 6-stage shared-memory ring: per stage 3-D TMA
//    loads of two 16-row weight tiles x 8 K-groups of 128 (16 KB of INT4), a
//    2-D TMA load of their bf16 group scales, and 1-D bulk copies of the
//    matching activation chunk of every row of the pass (x for gate/up, h for
//    down), all counted on one mbarrier.
//  * 8 consumer warps split K: warp w takes K-group w of every stage. Each
//    lane turns its 4-bit codes into exact bf16 integers (lop3 into the bf16
//    mantissa, one bf16x2 subtract) and feeds mma.sync m16n8k16 with weights as
//    the 16-row A operand and the pass's (up to 8) rows as B. The group scale
//    is applied in fp32 to the group's partial sums, so q * scale is never
//    rounded.
//  * the K order inside one MMA is a fixed permutation of the true K order;
//    the activation operand is put in the same order ("interleaved": within
//    each 8 values (0,4)(1,5)(2,6)(3,7)): x in registers, h by the gate/up
//    epilogue when it stores h.
//  * cross-warp reduction in fixed warp order (deterministic and batch
//    invariant); gate/up epilogue SwiGLU -> bf16 h; down epilogue fp32 y and,
//    for small batches, the combine: the last task to finish a channel tile
//    (atomic ticket, no waiting) writes out = y_shared + sum_j w_j y_j there.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRows = kPassRows;                   // rows (B columns) per task
constexpr int kWBytes = 2 * 8 * 1024;              // 2 tiles x 8 groups x 16 rows x 64 B
constexpr int kSBytes = 2 * 16 * 8 * 2;            // 2 tiles x 16 rows x 8 groups bf16
constexpr int kXStride = 8 * 256 + 64;             // one row's 8 groups (bf16) + pad
constexpr int kXOff = kWBytes + kSBytes;
constexpr int kStageBytes = ((kXOff + kRows * kXStride) + 1023) / 1024 * 1024;
constexpr int kRedBytes = 8 * 2 * 32 * 16;         // warps x tiles x lanes x float4
constexpr int kSmemBytes = kGemvStages * kStageBytes + kRedBytes + 2 * kGemvStages * 8 + 16;

struct GemvParams {
  Dims d;
  Routing r;
  const uint16_t* scale_routed;  // for the consumers when scales are not TMA'd
  const uint16_t* scale_shared;
  const uint16_t* bsrc;          // activation rows: x [T, H] (gate/up) or h (down)
  int bstride;                   // elements per activation row
  uint16_t* hout;                // gate/up: h [rows, hstride], interleaved
  int hstride;
  float* yout;                   // down: y [rows, H]
  uint16_t* out;                 // down with fused combine: out [T, H]
  int* tile_cnt;                 // down with fused combine: [H / kTile2] tickets
  int scale_tma;                 // 1: scales come with the stage
  int fuse_combine;
};

struct Task {
  bool shared;
  int ngroups;  // K / 128
  int rowA0;    // first row of tile 0 in the weight tensor's row space
  int rowA1;    // first row of tile 1
  int r0;       // first expert-sorted row of this pass
  int nr;       // rows in this pass (1..kRows)
  int tile;     // channel tile index
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int passes_of(int rows) { return (rows + kRows - 1) / kRows; }

template <int MODE>
__device__ __forceinline__ int tiles_of(const Dims& d, bool shared) {
  return MODE == 1 ? (shared ? d.Is : d.I) / kTile1 : d.H / kTile2;
}

// Tasks of the shared expert: they come first and need no routing.
template <int MODE>
__device__ __forceinline__ int shared_tasks(const Dims& d) {
  return d.Is > 0 ? tiles_of<MODE>(d, true) * passes_of(d.T) : 0;
}

template <int MODE>
__device__ __forceinline__ Task make_task(const Dims& d, bool shared, int e, int seg0, int seg1,
                                          int local) {
  Task t;
  t.shared = shared;
  const int passes = passes_of(seg1 - seg0);
  t.tile = local / passes;
  const int pass = local - t.tile * passes;
  t.r0 = seg0 + pass * kRows;
  t.nr = min(kRows, seg1 - t.r0);
  if (MODE == 1) {
    const int inter = shared ? d.Is : d.I;
    t.ngroups = d.H / kGroup;
    t.rowA0 = (shared ? 0 : e * 2 * inter) + t.tile * kTile1;
    t.rowA1 = t.rowA0 + inter;
  } else {
    t.ngroups = (shared ? d.Is : d.I) / kGroup;
    t.rowA0 = (shared ? 0 : e * d.H) + t.tile * kTile2;
    t.rowA1 = t.rowA0 + 16;
  }
  return t;
}

template <int MODE>
__device__ __forceinline__ Task shared_task(const Dims& d, int tau) {
  return make_task<MODE>(d, true, d.E, d.T * d.k, d.T * d.k + d.T, tau);
}

// Routed task tau (counted after the shared ones): binary search of the
// active expert whose task range holds tau.
template <int MODE>
__device__ __forceinline__ Task routed_task(const GemvParams& p, int tau) {
  const int* prefix = (MODE == 1) ? p.r.task1 : p.r.task2;
  const int n_act = p.r.meta[kMetaActive];
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(prefix + mid) <= tau)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int e = __ldg(p.r.active + lo);
  return make_task<MODE>(p.d, false, e, __ldg(p.r.offsets + e), __ldg(p.r.offsets + e + 1),
                         tau - __ldg(prefix + lo));
}

// Activation row of expert-sorted row r: a token of x (gate/up) or a row of h.
template <int MODE>
__device__ __forceinline__ const uint16_t* act_row(const GemvParams& p, const Task& t, int r) {
  int row = r;
  if (MODE == 1) row = t.shared ? r - p.d.T * p.d.k : __ldg(p.r.perm + r);
  return p.bsrc + (size_t)row * p.bstride;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void named_bar_consumers() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// 8 MMA steps (128 K) of one warp for one 16-row tile: rows g and g+8 come
// from wA and wB (4 words each), b[m] is the activation operand. Two
// accumulator chains (even / odd word) shorten the MMA dependency chain.
__device__ __forceinline__ void group_mma(const uint4& wA, const uint4& wB, const uint4* b,
                                          float* out) {
  float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    float* t = (m & 1) ? t1 : t0;
    const uint32_t ra = word_of(wA, m), rb = word_of(wB, m);
    uint32_t a[4];
    a[0] = int4_pair_to_bf16x2<0>(ra);
    a[1] = int4_pair_to_bf16x2<0>(rb);
    a[2] = int4_pair_to_bf16x2<1>(ra);
    a[3] = int4_pair_to_bf16x2<1>(rb);
    mma_bf16_16816(t, a, b[m].x, b[m].y, t);
    a[0] = int4_pair_to_bf16x2<2>(ra);
    a[1] = int4_pair_to_bf16x2<2>(rb);
    a[2] = int4_pair_to_bf16x2<3>(ra);
    a[3] = int4_pair_to_bf16x2<3>(rb);
    mma_bf16_16816(t, a, b[m].z, b[m].w, t);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = t0[i] + t1[i];
}

template <int MODE>
__device__ __forceinline__ uint32_t stage_bytes(const Task& t, int gcnt, bool scale_tma) {
  return gcnt * 2 * 1024 + (scale_tma ? kSBytes : 0) + t.nr * gcnt * 256;
}

// Producer: weights and scales of one stage (no dependency on earlier kernels).
__device__ __forceinline__ void issue_weights(uint8_t* st, uint64_t* bar, const CUtensorMap* tm,
                                              const CUtensorMap* ts, const Task& t, int g0,
                                              int gcnt, bool scale_tma) {
  for (int g = 0; g < gcnt; ++g) {
    tma_load_3d(st + g * 1024, tm, bar, 0, g0 + g, t.rowA0);
    tma_load_3d(st + (8 + g) * 1024, tm, bar, 0, g0 + g, t.rowA1);
  }
  if (scale_tma) {
    tma_load_2d(smem_u32(st + kWBytes), ts, bar, g0, t.rowA0);
    tma_load_2d(smem_u32(st + kWBytes + 256), ts, bar, g0, t.rowA1);
  }
}

// Producer: activation chunks of one stage (depends on earlier kernels).
template <int MODE>
__device__ __forceinline__ void issue_acts(const GemvParams& p, uint8_t* st, uint64_t* bar,
                                           const Task& t, int g0, int gcnt) {
  for (int j = 0; j < t.nr; ++j)
    bulk_copy(smem_u32(st + kXOff + j * kXStride), act_row<MODE>(p, t, t.r0 + j) + g0 * kGroup,
              gcnt * 256, bar);
}

template <int MODE>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_routed,
                const __grid_constant__ CUtensorMap tm_shared,
                const __grid_constant__ CUtensorMap ts_routed,
                const __grid_constant__ CUtensorMap ts_shared, const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + kGemvStages * kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGemvStages * kStageBytes + kRedBytes);
  uint64_t* empty = full + kGemvStages;
  int* flag = reinterpret_cast<int*>(empty + kGemvStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Dims& d = p.d;
  const bool scale_tma = p.scale_tma != 0;
  const int n_sh = shared_tasks<MODE>(d);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemvStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    prefetch_tmap(&tm_routed);
    prefetch_tmap(&tm_shared);
    int stage = 0;
    uint32_t phase = 0;
    bool waited = false;
    // Stages whose weights went out before the dependency wait and whose
    // activations (h of the previous kernel, for the down pass) are pending.
    int pend_n = 0;
    int pend_stage[kGemvStages], pend_g0[kGemvStages];
    Task pend_task[kGemvStages];
    int ntasks = -1;
    for (int tau = blockIdx.x;; tau += gridDim.x) {
      const bool sh = tau < n_sh;
      if (!sh && !waited) {
        // flush pending activation copies after the dependency resolves
        pdl_wait();
        waited = true;
        for (int i = 0; i < pend_n; ++i) {
          const Task& pt = pend_task[i];
          issue_acts<MODE>(p, stages + pend_stage[i] * kStageBytes, &full[pend_stage[i]], pt,
                           pend_g0[i], min(8, pt.ngroups - pend_g0[i]));
        }
        pend_n = 0;
      }
      if (!sh) {
        if (ntasks < 0) ntasks = n_sh + ((MODE == 1) ? p.r.meta[kMetaTasks1] : p.r.meta[kMetaTasks2]);
        if (tau >= ntasks) break;
      }
      const Task t = sh ? shared_task<MODE>(d, tau) : routed_task<MODE>(p, tau - n_sh);
      const CUtensorMap* tm = t.shared ? &tm_shared : &tm_routed;
      const CUtensorMap* ts = t.shared ? &ts_shared : &ts_routed;
      bool stop = false;
      for (int g0 = 0; g0 < t.ngroups; g0 += 8) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, p.r.err)) {
          stop = true;
          break;
        }
        const int gcnt = min(8, t.ngroups - g0);
        uint8_t* st = stages + stage * kStageBytes;
        mbar_arrive_expect_tx(&full[stage], stage_bytes<MODE>(t, gcnt, scale_tma));
        issue_weights(st, &full[stage], tm, ts, t, g0, gcnt, scale_tma);
        // gate/up reads x (an input): never waits. down reads h: its copies
        // wait for the gate/up kernel; until then the stage is remembered.
        if (MODE == 1 || waited) {
          issue_acts<MODE>(p, st, &full[stage], t, g0, gcnt);
        } else if (pend_n < kGemvStages) {
          pend_stage[pend_n] = stage;
          pend_g0[pend_n] = g0;
          pend_task[pend_n] = t;
          ++pend_n;
        }
        if (++stage == kGemvStages) {
          stage = 0;
          phase ^= 1u;
        }
        // the ring is full of pending stages: resolve the dependency now
        if (MODE == 2 && !waited && pend_n == kGemvStages) {
          pdl_wait();
          waited = true;
          for (int i = 0; i < pend_n; ++i) {
            const Task& pt = pend_task[i];
            issue_acts<MODE>(p, stages + pend_stage[i] * kStageBytes, &full[pend_stage[i]], pt,
                             pend_g0[i], min(8, pt.ngroups - pend_g0[i]));
          }
          pend_n = 0;
        }
      }
      if (stop) break;
    }
    if (!waited) {
      pdl_wait();
      for (int i = 0; i < pend_n; ++i) {
        const Task& pt = pend_task[i];
        issue_acts<MODE>(p, stages + pend_stage[i] * kStageBytes, &full[pend_stage[i]], pt,
                         pend_g0[i], min(8, pt.ngroups - pend_g0[i]));
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  bool waited = false;
  int ntasks = -1;
  for (int tau = blockIdx.x;; tau += gridDim.x) {
    const bool sh = tau < n_sh;
    if (!sh) {
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      if (ntasks < 0) ntasks = n_sh + ((MODE == 1) ? p.r.meta[kMetaTasks1] : p.r.meta[kMetaTasks2]);
      if (tau >= ntasks) break;
    }
    const Task t = sh ? shared_task<MODE>(d, tau) : routed_task<MODE>(p, tau - n_sh);
    const int ng = t.ngroups;
    const uint16_t* scales = t.shared ? p.scale_shared : p.scale_routed;
    const size_t s00 = (size_t)(t.rowA0 + g) * ng, s01 = s00 + (size_t)8 * ng;
    const size_t s10 = (size_t)(t.rowA1 + g) * ng, s11 = s10 + (size_t)8 * ng;
    const bool has_row = g < t.nr;
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = 0.f;

    for (int g0 = 0; g0 < ng; g0 += 8) {
      const int gi = g0 + warp;
      const bool mine = gi < ng;
      float sc[4];
      if (mine && !scale_tma) {
        sc[0] = bf16_bits_to_f32(__ldg(scales + s00 + gi));
        sc[1] = bf16_bits_to_f32(__ldg(scales + s01 + gi));
        sc[2] = bf16_bits_to_f32(__ldg(scales + s10 + gi));
        sc[3] = bf16_bits_to_f32(__ldg(scales + s11 + gi));
      }
      if (ok) ok = mbar_wait(&full[stage], phase, p.r.err);
      if (mine && ok) {
        const uint32_t st = smem_u32(stages + stage * kStageBytes);
        const uint32_t wa = st + warp * 1024 + g * 64 + c * 16;
        const uint4 w00 = lds128(wa), w01 = lds128(wa + 8 * 64);
        const uint4 w10 = lds128(wa + 8 * 1024), w11 = lds128(wa + 8 * 1024 + 8 * 64);
        if (scale_tma) {
          const uint32_t sa = st + kWBytes + g * 16 + warp * 2;
          sc[0] = bf16_bits_to_f32(lds16(sa));
          sc[1] = bf16_bits_to_f32(lds16(sa + 8 * 16));
          sc[2] = bf16_bits_to_f32(lds16(sa + 256));
          sc[3] = bf16_bits_to_f32(lds16(sa + 256 + 8 * 16));
        }
        uint4 b[4];
        if (has_row) {
          const uint32_t xa = st + kXOff + g * kXStride + warp * 256 + c * 64;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            b[m] = lds128(xa + m * 16);
            if (MODE == 1) b[m] = interleave8(b[m]);
          }
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) b[m] = make_uint4(0u, 0u, 0u, 0u);
        }
        float tmp[4];
        group_mma(w00, w01, b, tmp);
        acc[0][0] = fmaf(sc[0], tmp[0], acc[0][0]);
        acc[0][1] = fmaf(sc[0], tmp[1], acc[0][1]);
        acc[0][2] = fmaf(sc[1], tmp[2], acc[0][2]);
        acc[0][3] = fmaf(sc[1], tmp[3], acc[0][3]);
        group_mma(w10, w11, b, tmp);
        acc[1][0] = fmaf(sc[2], tmp[0], acc[1][0]);
        acc[1][1] = fmaf(sc[2], tmp[1], acc[1][1]);
        acc[1][2] = fmaf(sc[3], tmp[2], acc[1][2]);
        acc[1][3] = fmaf(sc[3], tmp[3], acc[1][3]);
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
    redw[(warp * 2 + 0) * 32 + lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    redw[(warp * 2 + 1) * 32 + lane] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
    named_bar_consumers();
    if (MODE == 1) {
      if (threadIdx.x < 16 * kRows) {
        const int row = threadIdx.x >> 3, tok = threadIdx.x & 7;
        const int ln = (row & 7) * 4 + (tok >> 1), q = (row >> 3) * 2 + (tok & 1);
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          v0 += red[((w * 2 + 0) * 32 + ln) * 4 + q];
          v1 += red[((w * 2 + 1) * 32 + ln) * 4 + q];
        }
        if (tok < t.nr) {
          const int n = t.tile * kTile1 + row;
          const int pos = (n & ~7) | ((n & 3) << 1) | ((n >> 2) & 1);
          p.hout[(size_t)(t.r0 + tok) * p.hstride + pos] = f32_to_bf16_bits(silu(v0) * v1);
        }
      }
    } else {
      const int tl = threadIdx.x >> 7, row = (threadIdx.x >> 3) & 15, tok = threadIdx.x & 7;
      const int ln = (row & 7) * 4 + (tok >> 1), q = (row >> 3) * 2 + (tok & 1);
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += red[((w * 2 + tl) * 32 + ln) * 4 + q];
      if (tok < t.nr) p.yout[(size_t)(t.r0 + tok) * d.H + t.tile * kTile2 + tl * 16 + row] = v;
    }
    if (MODE == 2 && p.fuse_combine) {
      // last task to finish this channel tile combines it for every token
      if (!waited) {  // routing results are read below
        pdl_wait();
        waited = true;
      }
      __threadfence();
      named_bar_consumers();
      if (threadIdx.x == 0) {
        const int per_tile = (n_sh + p.r.meta[kMetaTasks2]) / (d.H / kTile2);
        *flag = (atomicAdd(&p.tile_cnt[t.tile], 1) == per_tile - 1);
      }
      named_bar_consumers();
      if (*flag) {
        __threadfence();
        const int n0 = t.tile * kTile2;
        for (int i = threadIdx.x; i < d.T * kTile2; i += 256) {
          const int tok = i / kTile2, n = n0 + (i - tok * kTile2);
          float a = d.Is > 0 ? __ldcg(p.yout + (size_t)(d.T * d.k + tok) * d.H + n) : 0.f;
          for (int j = 0; j < d.k; ++j) {
            const float w = __ldcg(p.r.wts + tok * d.k + j);
            const int row = __ldcg(p.r.inv + tok * d.k + j);
            a = fmaf(w, __ldcg(p.yout + (size_t)row * d.H + n), a);
          }
          p.out[(size_t)tok * d.H + n] = f32_to_bf16_bits(a);
        }
        if (threadIdx.x == 0) p.tile_cnt[t.tile] = 0;
      }
    }
    named_bar_consumers();
  }
}

GemvParams make_params(const Dims& d, const Routing& r, const GemvWeights& w) {
  GemvParams p{};
  p.d = d;
  p.r = r;
  p.scale_routed = w.scale_routed;
  p.scale_shared = w.scale_shared;
  p.scale_tma = w.scale_tma;
  return p;
}

template <int MODE>
cudaError_t launch(const GemvParams& p, const GemvWeights& w, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<MODE>, w.tm_routed, w.tm_shared, w.ts_routed,
                            w.ts_shared, p);
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
                                const uint16_t* x, uint16_t* h, int hstride, int grid,
                                cudaStream_t s, LaunchLog& log) {
  GemvParams p = make_params(d, r, w);
  p.bsrc = x;
  p.bstride = d.H;
  p.hout = h;
  p.hstride = hstride;
  log.begin("gemv_gate_up_swiglu", s);
  cudaError_t e = launch<1>(p, w, grid, s);
  log.end(s);
  return e;
}

cudaError_t launch_gemv_down(const Dims& d, const Routing& r, const GemvWeights& w,
                             const uint16_t* h, int hstride, float* y, uint16_t* out,
                             int* tile_cnt, int grid, cudaStream_t s, LaunchLog& log) {
  GemvParams p = make_params(d, r, w);
  p.bsrc = h;
  p.bstride = hstride;
  p.yout = y;
  p.out = out;
  p.tile_cnt = tile_cnt;
  p.fuse_combine = out != nullptr;
  log.begin(out ? "gemv_down_combine" : "gemv_down", s);
  cudaError_t e = launch<2>(p, w, grid, s);
  log.end(s);
  return e;
}

}  // namespace moe

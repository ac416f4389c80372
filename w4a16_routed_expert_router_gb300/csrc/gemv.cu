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
//  * one producer warp decodes the tasks (from a shared-memory copy of the
//    routing metadata) and fills a 6-stage ring: per stage 3-D TMA loads of two
//    16-row weight tiles x 8 K-groups of 128 (16 KB of INT4), a 2-D TMA load of
//    their bf16 group scales, and 1-D bulk copies of the matching activation
//    chunk of every row of the pass (x for gate/up, h for down), all counted
//    on one mbarrier, plus a stage descriptor telling the consumers what the
//    stage holds.
//  * 8 consumer warps split K: warp w takes K-group w of every stage. Each
//    lane turns its 4-bit codes into exact bf16 integers and feeds mma.sync
//    m16n8k16 with weights as the 16-row A operand and the pass's rows as B.
//    The group scale is applied in fp32 to the group's partial sums, so
//    q * scale is never rounded.
//  * the K order inside one MMA is a fixed permutation of the true K order;
//    the activation operand is put in the same order ("interleaved": within
//    each 8 values (0,4)(1,5)(2,6)(3,7)): x in registers, h by the gate/up
//    epilogue when it stores h.
//  * cross-warp reduction in fixed warp order (deterministic and batch
//    invariant); gate/up epilogue SwiGLU -> bf16 h; down epilogue fp32 y and,
//    for small batches, the combine: the last task to finish a channel tile
//    (atomic ticket, no waiting) writes out = y_shared + sum_j w_j y_j there.
//  * every wait is an mbarrier wait bounded in time (no named barriers), so a
//    broken hand-off ends the kernel with an error flag instead of a hang.
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

enum DescFlags { kFirst = 1, kLast = 2, kEnd = 4, kShared = 8 };

// What one stage holds; written by the producer before the stage's arrive.
struct Desc {
  int flags, g0, gcnt, ngroups, tile, r0, nr, rowA0, rowA1, pad[3];
};

enum Bar { kBarRedFull = 0, kBarRedEmpty, kBarYDone, kBarFlag, kNumBars };

struct Smem {
  uint8_t stage[kGemvStages][kStageBytes];
  float4 red[8 * 2 * 32];
  Desc desc[kGemvStages];
  int active[kMaxExperts + 2];
  int prefix[kMaxExperts + 2];
  int offsets[kMaxExperts + 2];
  uint64_t full[kGemvStages];
  uint64_t empty[kGemvStages];
  uint64_t bar[kNumBars];
  int flag;
};
constexpr int kSmemBytes = (int)sizeof(Smem);

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

// Tasks of the shared expert: they come first and need no routing.
template <int MODE>
__device__ __forceinline__ int shared_tasks(const Dims& d) {
  if (d.Is == 0) return 0;
  return (MODE == 1 ? d.Is / kTile1 : d.H / kTile2) * passes_of(d.T);
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

// Routed task tau (counted after the shared ones), decoded from the
// shared-memory copy of the active-expert list and its task prefix.
template <int MODE>
__device__ __forceinline__ Task routed_task(const Smem& s, const Dims& d, int n_act, int tau) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.prefix[mid] <= tau)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int e = s.active[lo];
  return make_task<MODE>(d, false, e, s.offsets[e], s.offsets[e + 1], tau - s.prefix[lo]);
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

// Activation row of expert-sorted row r: a token of x (gate/up) or a row of h.
template <int MODE>
__device__ __forceinline__ const uint16_t* act_row(const GemvParams& p, const Task& t, int r) {
  int row = r;
  if (MODE == 1) row = t.shared ? r - p.d.T * p.d.k : __ldg(p.r.perm + r);
  return p.bsrc + (size_t)row * p.bstride;
}

template <int MODE>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_routed,
                const __grid_constant__ CUtensorMap tm_shared,
                const __grid_constant__ CUtensorMap ts_routed,
                const __grid_constant__ CUtensorMap ts_shared, const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Dims& d = p.d;
  const bool scale_tma = p.scale_tma != 0;
  const int n_sh = shared_tasks<MODE>(d);
  unsigned* err = p.r.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGemvStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 8);
    }
    mbar_init(&s.bar[kBarRedFull], 8);
    mbar_init(&s.bar[kBarRedEmpty], 8);
    mbar_init(&s.bar[kBarYDone], 8);
    mbar_init(&s.bar[kBarFlag], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_routed);
      prefetch_tmap(&tm_shared);
    }
    int stage = 0;
    uint32_t phase = 0;
    bool waited = false, stop = false;
    int n_act = 0, n_routed = 0;
    // stages whose activations (h of the previous kernel) wait for the dependency
    int pn = 0;
    int p_stage[kGemvStages], p_g0[kGemvStages];
    Task p_task[kGemvStages];

    auto resolve = [&]() {
      pdl_wait();
      waited = true;
      n_act = p.r.meta[kMetaActive];
      n_routed = p.r.meta[MODE == 1 ? kMetaTasks1 : kMetaTasks2];
      const int* pre = (MODE == 1) ? p.r.task1 : p.r.task2;
      for (int i = lane; i <= n_act; i += 32) {
        s.prefix[i] = pre[i];
        if (i < n_act) s.active[i] = p.r.active[i];
      }
      for (int i = lane; i <= d.E; i += 32) s.offsets[i] = p.r.offsets[i];
      __syncwarp();
      for (int i = 0; i < pn; ++i) {
        const Task& t = p_task[i];
        if (lane < t.nr)
          bulk_copy(smem_u32(s.stage[p_stage[i]] + kXOff + lane * kXStride),
                    act_row<MODE>(p, t, t.r0 + lane) + p_g0[i] * kGroup,
                    min(8, t.ngroups - p_g0[i]) * 256, &s.full[p_stage[i]]);
      }
      pn = 0;
    };

    for (int tau = blockIdx.x; !stop; tau += gridDim.x) {
      const bool sh = tau < n_sh;
      if (!sh && !waited) resolve();
      if (!sh && tau >= n_sh + n_routed) break;
      const Task t = sh ? make_task<MODE>(d, true, d.E, d.T * d.k, d.T * d.k + d.T, tau)
                        : routed_task<MODE>(s, d, n_act, tau - n_sh);
      const CUtensorMap* tm = t.shared ? &tm_shared : &tm_routed;
      const CUtensorMap* ts = t.shared ? &ts_shared : &ts_routed;
      const uint16_t* arow = nullptr;
      if ((MODE == 1 || waited) && lane < t.nr) arow = act_row<MODE>(p, t, t.r0 + lane);
      for (int g0 = 0; g0 < t.ngroups; g0 += 8) {
        const int gcnt = min(8, t.ngroups - g0);
        uint8_t* st = s.stage[stage];
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&s.empty[stage], phase ^ 1u, err);
          if (ok) {
            Desc& ds = s.desc[stage];
            ds.flags = (g0 == 0 ? kFirst : 0) | (g0 + 8 >= t.ngroups ? kLast : 0) |
                       (t.shared ? kShared : 0);
            ds.g0 = g0;
            ds.gcnt = gcnt;
            ds.ngroups = t.ngroups;
            ds.tile = t.tile;
            ds.r0 = t.r0;
            ds.nr = t.nr;
            ds.rowA0 = t.rowA0;
            ds.rowA1 = t.rowA1;
            mbar_arrive_expect_tx(&s.full[stage],
                                  gcnt * 2 * 1024 + (scale_tma ? kSBytes : 0) + t.nr * gcnt * 256);
            for (int g = 0; g < gcnt; ++g) {
              tma_load_3d(st + g * 1024, tm, &s.full[stage], 0, g0 + g, t.rowA0);
              tma_load_3d(st + (8 + g) * 1024, tm, &s.full[stage], 0, g0 + g, t.rowA1);
            }
            if (scale_tma) {
              tma_load_2d(smem_u32(st + kWBytes), ts, &s.full[stage], g0, t.rowA0);
              tma_load_2d(smem_u32(st + kWBytes + 256), ts, &s.full[stage], g0, t.rowA1);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          stop = true;
          break;
        }
        if (MODE == 1 || waited) {
          if (lane < t.nr)
            bulk_copy(smem_u32(st + kXOff + lane * kXStride), arow + g0 * kGroup, gcnt * 256,
                      &s.full[stage]);
        } else {
          p_stage[pn] = stage;
          p_g0[pn] = g0;
          p_task[pn] = t;
          ++pn;
        }
        if (++stage == kGemvStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (MODE == 2 && !waited && pn == kGemvStages) resolve();
      }
    }
    if (!waited) resolve();
    // end-of-work marker for the consumers
    if (lane == 0 && !stop && mbar_wait(&s.empty[stage], phase ^ 1u, err)) {
      s.desc[stage].flags = kEnd;
      mbar_arrive(&s.full[stage]);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const uint32_t stage0 = smem_u32(s.stage[0]);
  const uint32_t w_off = warp * 1024 + g * 64 + c * 16;
  const uint32_t s_off = kWBytes + g * 16 + warp * 2;
  const uint32_t x_off = kXOff + g * kXStride + warp * 256 + c * 64;
  int stage = 0;
  uint32_t phase = 0, tphase = 0;
  bool waited = false;
  float acc[2][4] = {};
  for (;;) {
    if (!mbar_wait(&s.full[stage], phase, err)) break;
    const Desc ds = s.desc[stage];
    if (ds.flags & kEnd) break;
    if (ds.flags & kFirst) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][i] = acc[1][i] = 0.f;
    }
    if (warp < ds.gcnt) {
      const int gi = ds.g0 + warp;
      const uint32_t st = stage0 + stage * kStageBytes;
      const uint4 w00 = lds128(st + w_off), w01 = lds128(st + w_off + 8 * 64);
      const uint4 w10 = lds128(st + w_off + 8 * 1024), w11 = lds128(st + w_off + 8 * 1024 + 8 * 64);
      float sc[4];
      if (scale_tma) {
        sc[0] = bf16_bits_to_f32(lds16(st + s_off));
        sc[1] = bf16_bits_to_f32(lds16(st + s_off + 8 * 16));
        sc[2] = bf16_bits_to_f32(lds16(st + s_off + 256));
        sc[3] = bf16_bits_to_f32(lds16(st + s_off + 256 + 8 * 16));
      } else {
        const uint16_t* scl = (ds.flags & kShared) ? p.scale_shared : p.scale_routed;
        const int ng = ds.ngroups;
        sc[0] = bf16_bits_to_f32(__ldg(scl + (size_t)(ds.rowA0 + g) * ng + gi));
        sc[1] = bf16_bits_to_f32(__ldg(scl + (size_t)(ds.rowA0 + g + 8) * ng + gi));
        sc[2] = bf16_bits_to_f32(__ldg(scl + (size_t)(ds.rowA1 + g) * ng + gi));
        sc[3] = bf16_bits_to_f32(__ldg(scl + (size_t)(ds.rowA1 + g + 8) * ng + gi));
      }
      uint4 b[4];
      if (g < ds.nr) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          b[m] = lds128(st + x_off + m * 16);
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
    // the stage's next fill is an async-proxy write (TMA, bulk copy): order
    // this thread's generic reads of it before the release
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[stage]);
    if (++stage == kGemvStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (!(ds.flags & kLast)) continue;

    // ---- end of a task: deterministic cross-warp reduction and epilogue
    if (!mbar_wait(&s.bar[kBarRedEmpty], tphase ^ 1u, err)) break;
    s.red[(warp * 2 + 0) * 32 + lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    s.red[(warp * 2 + 1) * 32 + lane] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.bar[kBarRedFull]);
    if (!mbar_wait(&s.bar[kBarRedFull], tphase, err)) break;
    const float* red = reinterpret_cast<const float*>(s.red);
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
        if (tok < ds.nr) {
          const int n = ds.tile * kTile1 + row;
          const int pos = (n & ~7) | ((n & 3) << 1) | ((n >> 2) & 1);
          p.hout[(size_t)(ds.r0 + tok) * p.hstride + pos] = f32_to_bf16_bits(silu(v0) * v1);
        }
      }
    } else {
      const int tl = threadIdx.x >> 7, row = (threadIdx.x >> 3) & 15, tok = threadIdx.x & 7;
      const int ln = (row & 7) * 4 + (tok >> 1), q = (row >> 3) * 2 + (tok & 1);
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += red[((w * 2 + tl) * 32 + ln) * 4 + q];
      if (tok < ds.nr) p.yout[(size_t)(ds.r0 + tok) * d.H + ds.tile * kTile2 + tl * 16 + row] = v;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.bar[kBarRedEmpty]);

    if (MODE == 2 && p.fuse_combine) {
      // the last task to finish this channel tile combines it for every token
      if (!waited) {  // routing results are read below
        pdl_wait();
        waited = true;
      }
      if (lane == 0) mbar_arrive(&s.bar[kBarYDone]);
      if (threadIdx.x == 0) {
        if (mbar_wait(&s.bar[kBarYDone], tphase, err)) {
          __threadfence();
          const int per_tile = (n_sh + p.r.meta[kMetaTasks2]) / (d.H / kTile2);
          s.flag = (atomicAdd(&p.tile_cnt[ds.tile], 1) == per_tile - 1);
        } else {
          s.flag = 0;
        }
        mbar_arrive(&s.bar[kBarFlag]);
      }
      if (!mbar_wait(&s.bar[kBarFlag], tphase, err)) break;
      if (s.flag) {
        __threadfence();
        const int n0 = ds.tile * kTile2;
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
        if (threadIdx.x == 0) p.tile_cnt[ds.tile] = 0;
      }
    }
    tphase ^= 1u;
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

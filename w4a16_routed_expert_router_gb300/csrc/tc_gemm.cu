// Tensor-core (tcgen05 / TMEM) grouped W4A16 expert GEMMs for large batches.
//
// "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", "A pass through the
// model": above the ridge (about 146-250 FLOP per byte on the pages' GH200,
// a few hundred rows per expert) the expert GEMMs are compute bound; the
// weight-only approach turns the 4-bit weights into bf16 and runs bf16 tensor
// cores. Here that is the 5th-generation tensor core: tcgen05.mma with both
// operands in shared memory and the fp32 accumulator in tensor memory.
//
// Formulation ("swap AB"): for one expert, D[channel, row] = sum_k W[channel, k]
// * X[row, k]. The dequantised weights are the M = 128 A operand, the expert's
// rows (tokens) the N <= 256 B operand, so an expert with 190 rows wastes at
// most 15 columns instead of a half-empty 128-row tile.
//
// A task is (expert, N-tile of <= 256 rows, channel tile); gate/up tasks hold
// 128 gate + 128 up channels (two accumulators, SwiGLU in the epilogue), down
// tasks 2 x 128 output channels. Tasks run in (expert, N-tile, channel tile)
// order over persistent CTAs (one per SM), so concurrent CTAs share the same
// activation rows and weights in L2.
//
// Warp roles per CTA:
//   warp 0     TMA producer of the weights: per 64-wide K block the two 128-row
//              INT4 tiles (4 KB each, 32-byte swizzle) into a ring that the
//              dequantisers free as soon as they have read a stage.
//   warp 1     TMEM owner (allocates all 512 columns) and MMA issuer: 4 K-steps
//              x 2 tiles of tcgen05.mma kind::f16 (bf16 x bf16 -> fp32) per K
//              block; commits release the activation and bf16 stages, the
//              task's last one the accumulator.
//   warp 2     TMA producer of the activations (64-row boxes, 128-byte swizzle)
//              into four 32 KB stages: an activation tile takes about a
//              microsecond to arrive, three MMA K blocks' worth at full N.
//   warps 3-10 dequantisers, one weight row per thread: INT4 -> bf16 (q * scale,
//              one rounding) written in the canonical K-major 128-byte-swizzled
//              layout tcgen05 reads; each thread fetches its row's group scale
//              one group ahead with a plain load.
//   warps 11-26 epilogue: tcgen05.ld of the accumulator (four warps per TMEM
//              lane quarter, 16-column chunks), SwiGLU -> bf16 h, or bf16 y (the
//              combine reads y once; bf16 halves both sides of that round trip).
// The activation operand (x rows in expert order, or h) is stored with each 8
// consecutive values in the order (0,4)(1,5)(2,6)(3,7); the dequantiser emits
// the weights in that same order, so no shuffle is needed on either side.
// Every wait is an mbarrier wait bounded in time; a timeout sets the device
// error flag and the kernel winds down (MMAs drained, TMEM freed).
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kThreads = 27 * 32;
constexpr int kDqWarp0 = 3, kEpiWarp0 = 11;
constexpr int kBK = 64;                               // K per block (one 128-byte swizzle atom)
constexpr int kWStages = 4;
// Four activation stages: an activation tile takes about a microsecond to
// arrive, three MMA K blocks' worth at full N; tasks with few rows finish a K
// block sooner (4 stages against 3: zipf2048 gate/up 1.096 -> 1.075 ms,
// prefill8192 1.347 -> 1.338 ms; 2 stages: 1.19 and 1.64 ms).
constexpr int kBStages = 4;
constexpr int kAbfStages = 2;
constexpr int kInt4Tile = 128 * kBK / 2;              // 4 KB: 128 rows x 64 codes
constexpr int kWB = 2 * kInt4Tile;                    // 8 KB
constexpr int kBTile = kTcN * kBK * 2;                // 32 KB: 256 rows x 64 bf16
constexpr int kAbfTile = 128 * kBK * 2;               // 16 KB
constexpr int kAbfB = 2 * kAbfTile;                   // 32 KB

struct TcTask {
  int valid;
  int shared;
  int rowA0, rowA1;      // weight rows of tile 0 / tile 1 (tensor-map row space)
  int tile1;             // tile 1 present
  int ngroups, nkb;      // K / 128, K / 64
  int n, nmma, nbox;     // rows, MMA N (multiple of 16), 64-row B boxes
  int brow0;             // first activation row (xperm / h row space)
  int chan0;             // first output channel
};

struct Smem {
  uint8_t b[kBStages][kBTile];
  uint8_t abf[kAbfStages][kAbfB];
  uint8_t w[kWStages][kWB];
  uint64_t w_full[kWStages], w_empty[kWStages];
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t abf_full[kAbfStages], abf_empty[kAbfStages];
  uint64_t acc_full, acc_empty, drain;
  uint32_t tmem_base;
};
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;  // + alignment slack
// A CTA holds all 512 TMEM columns for its whole life, so a second CTA on the
// same SM would wait in tcgen05.alloc until the first one exits. The shared-
// memory footprint keeps the kernel at one CTA per SM (228 KB of shared memory
// per SM), and the host refuses a launch shape with more.
static_assert(2 * kSmemBytes > 228 * 1024, "tc_gemm_kernel must stay at one CTA per SM");

struct TcParams {
  Dims d;
  Routing r;
  const uint16_t* scale_routed;  // [rows, K/128] bf16
  const uint16_t* scale_shared;
  uint16_t* hout;                // gate/up: h [T*k + T, hstride], interleaved
  int hstride;
  uint16_t* yout;                // down: y [T*k + T, H] bf16
};

// q * scale for the two codes of int4_pair_to_bf16x2 (one bf16 rounding)
template <int J>
__device__ __forceinline__ uint32_t dq_pair(uint32_t word, __nv_bfloat162 s2) {
  const uint32_t q = int4_pair_to_bf16x2<J>(word);
  __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&q), s2);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ tasks
template <int MODE>
__device__ __forceinline__ int channel_tiles(const Dims& d, bool shared) {
  return MODE == 1 ? (shared ? d.Is : d.I) / 128 : d.H / 256;
}

template <int MODE>
__device__ __forceinline__ int shared_tc_tasks(const Dims& d) {
  if (d.Is == 0) return 0;
  return channel_tiles<MODE>(d, true) * ((d.T + kTcN - 1) / kTcN);
}

template <int MODE>
__device__ TcTask decode_task(const TcParams& p, int tau, int n_sh, int n_act) {
  const Dims& d = p.d;
  TcTask t{};
  int e, seg0, seg1, local;
  bool sh = tau < n_sh;
  if (sh) {
    e = d.E;
    seg0 = d.T * d.k;
    seg1 = seg0 + d.T;
    local = tau;
  } else {
    const int* pre = MODE == 1 ? p.r.task3 : p.r.task4;
    const int tr = tau - n_sh;
    int lo = 0, hi = n_act - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(pre + mid) <= tr)
        lo = mid;
      else
        hi = mid - 1;
    }
    e = __ldg(p.r.active + lo);
    seg0 = __ldg(p.r.offsets + e);
    seg1 = __ldg(p.r.offsets + e + 1);
    local = tr - __ldg(pre + lo);
  }
  const int ct = channel_tiles<MODE>(d, sh);
  const int ntile = local / ct, ctile = local - ntile * ct;
  t.valid = 1;
  t.shared = sh;
  t.brow0 = seg0 + ntile * kTcN;
  t.n = min(kTcN, seg1 - t.brow0);
  t.nmma = (t.n + 15) & ~15;
  t.nbox = (t.nmma + 63) / 64;
  const int inter = sh ? d.Is : d.I;
  if (MODE == 1) {
    t.ngroups = d.H / kGroup;
    t.rowA0 = (sh ? 0 : e * 2 * inter) + ctile * 128;
    t.rowA1 = t.rowA0 + inter;
    t.tile1 = 1;
    t.chan0 = ctile * 128;
  } else {
    t.ngroups = inter / kGroup;
    t.rowA0 = (sh ? 0 : e * d.H) + ctile * 256;
    t.rowA1 = t.rowA0 + 128;
    t.tile1 = 1;
    t.chan0 = ctile * 256;
  }
  t.nkb = t.ngroups * 2;
  return t;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap wq_r, const __grid_constant__ CUtensorMap wq_s,
                   const __grid_constant__ CUtensorMap bmap, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Dims& d = p.d;
  unsigned* err = p.r.err;
  const int n_sh = shared_tc_tasks<MODE>(d);
  const int n_act = p.r.meta[kMetaActive];
  const int ntasks = n_sh + p.r.meta[MODE == 1 ? kMetaTc1 : kMetaTc2];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(&s.w_full[i], 1);
      mbar_init(&s.w_empty[i], 8);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&s.b_full[i], 1);
      mbar_init(&s.b_empty[i], 1);
    }
    for (int i = 0; i < kAbfStages; ++i) {
      mbar_init(&s.abf_full[i], 8);
      mbar_init(&s.abf_empty[i], 1);
    }
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 16);
    mbar_init(&s.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- weight producer
    if (lane == 0) {
      prefetch_tmap(&wq_r);
      prefetch_tmap(&wq_s);
      int stage = 0;
      uint32_t ph = 0, filled = 0, last_ph = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < ntasks && ok; tau += gridDim.x) {
        const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
        const CUtensorMap* wq = t.shared ? &wq_s : &wq_r;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!bwait(&s.w_empty[stage], ph ^ 1u, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.w_full[stage], kWB);
          tma_2d(smem_u32(s.w[stage]), wq, &s.w_full[stage], kb * 8, t.rowA0);
          tma_2d(smem_u32(s.w[stage] + kInt4Tile), wq, &s.w_full[stage], kb * 8, t.rowA1);
          filled |= 1u << stage;
          last_ph = (last_ph & ~(1u << stage)) | (ph << stage);
          if (++stage == kWStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      // wind down: no TMA copy may still be landing when the CTA exits
      for (int i = 0; i < kWStages; ++i)
        if (filled & (1u << i)) mbar_wait(&s.w_full[i], (last_ph >> i) & 1u, err);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- activation producer
    if (lane == 0) {
      prefetch_tmap(&bmap);
      int stage = 0;
      uint32_t ph = 0, filled = 0, last_ph = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < ntasks && ok; tau += gridDim.x) {
        const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!bwait(&s.b_empty[stage], ph ^ 1u, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.b_full[stage], t.nbox * 64 * kBK * 2);
          for (int bx = 0; bx < t.nbox; ++bx)
            tma_2d(smem_u32(s.b[stage] + bx * 64 * kBK * 2), &bmap, &s.b_full[stage], kb * kBK,
                   t.brow0 + bx * 64);
          filled |= 1u << stage;
          last_ph = (last_ph & ~(1u << stage)) | (ph << stage);
          if (++stage == kBStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      for (int i = 0; i < kBStages; ++i)
        if (filled & (1u << i)) mbar_wait(&s.b_full[i], (last_ph >> i) & 1u, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int bstage = 0, astage = 0;
      uint32_t bph = 0, aph = 0;
      int it = 0;
      for (int tau = blockIdx.x; tau < ntasks; tau += gridDim.x, ++it) {
        const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
        const uint32_t idesc = idesc_bf16(128, t.nmma);
        // the accumulator must have been drained by the previous epilogue
        if (!bwait(&s.acc_empty, (it & 1) ^ 1u, err)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!bwait(&s.b_full[bstage], bph, err) || !bwait(&s.abf_full[astage], aph, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(s.abf[astage]);
          const uint32_t b0 = smem_u32(s.b[bstage]);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t bd = smem_desc_sw128(b0 + k * 32);
            mma_bf16(tmem, smem_desc_sw128(a0 + k * 32), bd, idesc, (kb | k) ? 1u : 0u);
            mma_bf16(tmem + 256, smem_desc_sw128(a0 + kAbfTile + k * 32), bd, idesc,
                     (kb | k) ? 1u : 0u);
          }
          mma_commit(&s.b_empty[bstage]);
          mma_commit(&s.abf_empty[astage]);
          if (++bstage == kBStages) {
            bstage = 0;
            bph ^= 1u;
          }
          if (++astage == kAbfStages) {
            astage = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&s.acc_full);
      }
      // wind down: every MMA this thread issued has completed before exit
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0, err);
    }
  } else if (warp < kEpiWarp0) {
    // ---------------------------------------------------------------- dequantisers
    const int t256 = threadIdx.x - kDqWarp0 * 32;  // 0..255
    const int tile = t256 >> 7, row = t256 & 127;
    // 32-byte swizzle of the INT4 tile: the two 16-byte halves of a row swap
    // places on row bit 2
    const uint32_t half0 = (uint32_t)((row >> 2) & 1) << 4;
    int wstage = 0, astage = 0;
    uint32_t wph = 0, aph = 0;
    // this row's scales; `scn` holds the next group's scale, loaded one group
    // (two K blocks) before it is needed, across task boundaries too
    auto scale_row = [&](const TcTask& t) {
      const int arow = (tile ? t.rowA1 : t.rowA0) + row;
      return (t.shared ? p.scale_shared : p.scale_routed) + (size_t)arow * t.ngroups;
    };
    int tau = blockIdx.x;
    TcTask t{};
    const uint16_t* gs = nullptr;
    uint16_t scn = 0;
    if (tau < ntasks) {
      t = decode_task<MODE>(p, tau, n_sh, n_act);
      gs = scale_row(t);
      scn = __ldg(gs);
    }
    bool ok = true;
    for (; tau < ntasks && ok; tau += gridDim.x) {
      const int tau_next = tau + gridDim.x;
      TcTask tn{};
      const uint16_t* gsn = nullptr;
      if (tau_next < ntasks) {
        tn = decode_task<MODE>(p, tau_next, n_sh, n_act);
        gsn = scale_row(tn);
      }
      __nv_bfloat162 s2;
      for (int kb = 0; kb < t.nkb; ++kb) {
        if ((kb & 1) == 0) {
          const uint32_t sb = scn;
          *reinterpret_cast<uint32_t*>(&s2) = sb | (sb << 16);
          const int g = kb >> 1;
          if (g + 1 < t.ngroups)
            scn = __ldg(gs + g + 1);
          else if (gsn)
            scn = __ldg(gsn);
        }
        if (!warp_wait(&s.w_full[wstage], wph, err)) {
          ok = false;
          break;
        }
        const uint32_t wsrc = smem_u32(s.w[wstage] + tile * kInt4Tile + row * 32);
        uint32_t words[8];
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(words[0]), "=r"(words[1]), "=r"(words[2]), "=r"(words[3])
                     : "r"(wsrc + half0));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(words[4]), "=r"(words[5]), "=r"(words[6]), "=r"(words[7])
                     : "r"(wsrc + (half0 ^ 16u)));
        if (!warp_wait(&s.abf_empty[astage], aph ^ 1u, err)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(s.abf[astage] + tile * kAbfTile + row * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          sts128(dst + ((j ^ (row & 7)) << 4), dq_pair<0>(words[j], s2), dq_pair<1>(words[j], s2),
                 dq_pair<2>(words[j], s2), dq_pair<3>(words[j], s2));
        // one proxy fence for both directions: the bf16 stores become visible
        // to the tensor core's async proxy, and the generic reads of the
        // weight stage are ordered before its next TMA fill, so the weight
        // stage is released only here. (Released right after the reads,
        // without a fence, about one forward in six at 2048 Zipf-routed tokens
        // had a few K blocks of some 32-row quarters dequantised from the
        // next fill's weights.)
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s.w_empty[wstage]);
          mbar_arrive(&s.abf_full[astage]);
        }
        if (++wstage == kWStages) {
          wstage = 0;
          wph ^= 1u;
        }
        if (++astage == kAbfStages) {
          astage = 0;
          aph ^= 1u;
        }
      }
      t = tn;
      gs = gsn;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                      // TMEM lane quarter this warp may access
    const int cg = (warp - kEpiWarp0) >> 2;      // 16-column chunks cg, cg + 4, ...
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int ch = q * 32 + lane;                // channel within a 128-row tile
    int it = 0;
    for (int tau = blockIdx.x; tau < ntasks; tau += gridDim.x, ++it) {
      const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
      if (!warp_wait(&s.acc_full, it & 1, err)) break;
      tc_fence_after();
      for (int c0 = cg * 16; c0 < t.n; c0 += 64) {
        float v0[16], v1[16];
        tmem_ld16(tmem + lane_base + c0, v0);
        tmem_ld16(tmem + lane_base + 256 + c0, v1);
        const int cn = t.n - c0;
        if (MODE == 1) {
          const int n = t.chan0 + ch;
          const int pos = (n & ~7) | ((n & 3) << 1) | ((n >> 2) & 1);
          uint16_t* hp = p.hout + (size_t)(t.brow0 + c0) * p.hstride + pos;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < cn) {
              const float g = v0[j];
              hp[(size_t)j * p.hstride] = f32_to_bf16_bits(__fdividef(g, 1.0f + __expf(-g)) * v1[j]);
            }
        } else {
          uint16_t* yr = p.yout + (size_t)(t.brow0 + c0) * d.H + t.chan0 + ch;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < cn) {
              yr[(size_t)j * d.H] = f32_to_bf16_bits(v0[j]);
              yr[(size_t)j * d.H + 128] = f32_to_bf16_bits(v1[j]);
            }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_free(tmem, 512);
  }
}

template <int MODE>
cudaError_t launch(const TcParams& p, const TcWeights& w, const CUtensorMap& bmap, int grid,
                   cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE>, w.wq_r, w.wq_s, bmap, p);
}

}  // namespace

cudaError_t tc_setup(int* ctas_per_sm) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(tc_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(tc_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes)) != cudaSuccess)
    return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, tc_gemm_kernel<1>, kThreads,
                                                       kSmemBytes);
}

cudaError_t launch_tc_gate_up(const Dims& d, const Routing& r, const TcWeights& w,
                              const CUtensorMap& xmap, uint16_t* h, int hstride, int grid,
                              cudaStream_t s, LaunchLog& log) {
  TcParams p{};
  p.d = d;
  p.r = r;
  p.scale_routed = w.scale_routed;
  p.scale_shared = w.scale_shared;
  p.hout = h;
  p.hstride = hstride;
  log.begin("tc_gate_up_swiglu", s);
  cudaError_t e = launch<1>(p, w, xmap, grid, s);
  log.end(s);
  return e;
}

cudaError_t launch_tc_down(const Dims& d, const Routing& r, const TcWeights& w,
                           const CUtensorMap& hmap, uint16_t* y, int grid, cudaStream_t s,
                           LaunchLog& log) {
  TcParams p{};
  p.d = d;
  p.r = r;
  p.scale_routed = w.scale_routed;
  p.scale_shared = w.scale_shared;
  p.yout = y;
  log.begin("tc_down", s);
  cudaError_t e = launch<2>(p, w, hmap, grid, s);
  log.end(s);
  return e;
}

}  // namespace moe

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
//   warp 0     TMA producer: per 64-wide K block, the two 128-row INT4 weight
//              tiles (4 KB each) and the activation rows (64-row boxes with
//              128-byte swizzle); per task the tiles' bf16 group scales.
//   warp 1     TMEM owner (allocates all 512 columns) and MMA issuer: 4 K-steps
//              x 2 tiles of tcgen05.mma kind::f16 (bf16 x bf16 -> fp32) per K
//              block, commits release the stages, the last one the accumulator.
//   warps 2-9  dequantisers: INT4 -> bf16 (q * scale, one rounding) written in
//              the canonical K-major 128-byte-swizzled layout tcgen05 reads.
//   warps 10-13 epilogue: tcgen05.ld of the accumulator, SwiGLU -> bf16 h, or
//              fp32 y.
// The activation operand (x rows in expert order, or h) is stored with each 8
// consecutive values in the order (0,4)(1,5)(2,6)(3,7); the dequantiser emits
// the weights in that same order, so no shuffle is needed on either side.
// Every wait is an mbarrier wait bounded in time; a timeout sets the device
// error flag and the kernel winds down (MMAs drained, TMEM freed).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 14 * 32;
constexpr int kBK = 64;                               // K per block (one 128-byte swizzle atom)
constexpr int kRawStages = 3;
constexpr int kAbfStages = 2;
constexpr int kInt4Tile = 128 * kBK / 2;              // 4 KB: 128 rows x 64 codes
constexpr int kBTile = kTcN * kBK * 2;                // 32 KB: 256 rows x 64 bf16
constexpr int kRawB = 2 * kInt4Tile + kBTile;         // 40 KB
constexpr int kAbfTile = 128 * kBK * 2;               // 16 KB
constexpr int kAbfB = 2 * kAbfTile;                   // 32 KB
constexpr int kScaleB = 2 * 128 * 32 * 2;             // 2 tiles x 128 rows x <= 32 groups bf16

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
  uint8_t raw[kRawStages][kRawB];
  uint8_t abf[kAbfStages][kAbfB];
  uint8_t scl[2][kScaleB];
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  uint64_t abf_full[kAbfStages], abf_empty[kAbfStages];
  uint64_t scl_full[2], scl_empty[2];
  uint64_t acc_full, acc_empty, drain;
  uint32_t tmem_base;
};
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;  // + alignment slack

struct TcParams {
  Dims d;
  Routing r;
  const uint16_t* scale_routed;  // [rows, K/128] bf16 (global loads when !scale_tma)
  const uint16_t* scale_shared;
  int scale_tma;
  uint16_t* hout;                // gate/up: h [T*k + T, hstride], interleaved
  int hstride;
  float* yout;                   // down: y [T*k + T, H]
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                       int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ bool aborted(const unsigned* err) {
  return (*reinterpret_cast<const volatile unsigned*>(err) & kErrTimeout) != 0;
}

// bounded mbarrier wait that also gives up once the grid recorded a timeout
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (aborted(err)) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

// the same wait by every lane of a warp, with one verdict for the warp (the
// tcgen05.ld that follows is warp-collective)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  const bool ok = bwait(bar, parity, err);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand:
// start address, stride between 8-row groups 1024 B, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t desc = 0;
  desc |= (uint64_t)((addr >> 4) & 0x3FFF);          // start address
  desc |= (uint64_t)(1) << 16;                       // leading byte offset (unused here)
  desc |= (uint64_t)((1024 >> 4) & 0x3FFF) << 32;    // stride byte offset
  desc |= (uint64_t)1 << 46;                         // descriptor version
  desc |= (uint64_t)2 << 61;                         // SWIZZLE_128B
  return desc;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  return (1u << 4)                       // D format fp32
         | (1u << 7)                     // A format bf16
         | (1u << 10)                    // B format bf16
         | ((uint32_t)(n >> 3) << 17)    // N / 8
         | ((uint32_t)(m >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t e) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(e)
               : "memory");
}

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
                   const __grid_constant__ CUtensorMap ws_r, const __grid_constant__ CUtensorMap ws_s,
                   const __grid_constant__ CUtensorMap bmap, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Dims& d = p.d;
  unsigned* err = p.r.err;
  const bool scale_tma = p.scale_tma != 0;
  const int n_sh = shared_tc_tasks<MODE>(d);
  const int n_act = p.r.meta[kMetaActive];
  const int ntasks = n_sh + p.r.meta[MODE == 1 ? kMetaTc1 : kMetaTc2];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(&s.raw_full[i], 1);
      mbar_init(&s.raw_empty[i], 1);
    }
    for (int i = 0; i < kAbfStages; ++i) {
      mbar_init(&s.abf_full[i], 8);
      mbar_init(&s.abf_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.scl_full[i], 1);
      mbar_init(&s.scl_empty[i], 8);
    }
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 4);
    mbar_init(&s.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    // the whole tensor memory of this SM: two 256-column fp32 accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s.tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&wq_r);
      prefetch_tmap(&bmap);
      int stage = 0;
      uint32_t ph = 0;
      int it = 0;
      // phase of the last fill of each stage / scale slot, for the wind-down
      uint32_t last_ph = 0, filled = 0;
      uint32_t scl_last = 0, scl_filled = 0;
      for (int tau = blockIdx.x; tau < ntasks; tau += gridDim.x, ++it) {
        const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
        const int slot = it & 1;
        if (!bwait(&s.scl_empty[slot], ((it >> 1) & 1) ^ 1u, err)) break;
        const CUtensorMap* wq = t.shared ? &wq_s : &wq_r;
        const CUtensorMap* ws = t.shared ? &ws_s : &ws_r;
        if (scale_tma) {
          mbar_arrive_expect_tx(&s.scl_full[slot], 2 * 128 * t.ngroups * 2);
          tma_2d(smem_u32(s.scl[slot]), ws, &s.scl_full[slot], 0, t.rowA0);
          tma_2d(smem_u32(s.scl[slot] + 128 * t.ngroups * 2), ws, &s.scl_full[slot], 0, t.rowA1);
          scl_filled |= 1u << slot;
          scl_last = (scl_last & ~(1u << slot)) | (((it >> 1) & 1u) << slot);
        } else {
          mbar_arrive(&s.scl_full[slot]);
        }
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!bwait(&s.raw_empty[stage], ph ^ 1u, err)) {
            ok = false;
            break;
          }
          uint8_t* st = s.raw[stage];
          mbar_arrive_expect_tx(&s.raw_full[stage], 2 * kInt4Tile + t.nbox * 64 * kBK * 2);
          tma_2d(smem_u32(st), wq, &s.raw_full[stage], kb * 8, t.rowA0);
          tma_2d(smem_u32(st + kInt4Tile), wq, &s.raw_full[stage], kb * 8, t.rowA1);
          for (int bx = 0; bx < t.nbox; ++bx)
            tma_2d(smem_u32(st + 2 * kInt4Tile + bx * 64 * kBK * 2), &bmap, &s.raw_full[stage],
                   kb * kBK, t.brow0 + bx * 64);
          filled |= 1u << stage;
          last_ph = (last_ph & ~(1u << stage)) | (ph << stage);
          if (++stage == kRawStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      // wind down: no TMA copy may still be landing in shared memory when
      // the CTA exits (all of them have landed on a normal exit)
      for (int i = 0; i < kRawStages; ++i)
        if (filled & (1u << i)) mbar_wait(&s.raw_full[i], (last_ph >> i) & 1u, err);
      for (int i = 0; i < 2; ++i)
        if (scl_filled & (1u << i)) mbar_wait(&s.scl_full[i], (scl_last >> i) & 1u, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int rstage = 0, astage = 0;
      uint32_t rph = 0, aph = 0;
      int it = 0;
      for (int tau = blockIdx.x; tau < ntasks; tau += gridDim.x, ++it) {
        const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
        const uint32_t idesc = idesc_bf16(128, t.nmma);
        // the accumulator must have been drained by the previous epilogue
        if (!bwait(&s.acc_empty, (it & 1) ^ 1u, err)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!bwait(&s.raw_full[rstage], rph, err) || !bwait(&s.abf_full[astage], aph, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(s.abf[astage]);
          const uint32_t b0 = smem_u32(s.raw[rstage] + 2 * kInt4Tile);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t bd = smem_desc_sw128(b0 + k * 32);
            mma_bf16(tmem, smem_desc_sw128(a0 + k * 32), bd, idesc, (kb | k) ? 1u : 0u);
            mma_bf16(tmem + 256, smem_desc_sw128(a0 + kAbfTile + k * 32), bd, idesc,
                     (kb | k) ? 1u : 0u);
          }
          mma_commit(&s.raw_empty[rstage]);
          mma_commit(&s.abf_empty[astage]);
          if (++rstage == kRawStages) {
            rstage = 0;
            rph ^= 1u;
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
  } else if (warp < 10) {
    // ---------------------------------------------------------------- dequantisers
    const int t256 = threadIdx.x - 64;  // 0..255
    const int tile = t256 >> 7, row = t256 & 127;
    int rstage = 0, astage = 0;
    uint32_t rph = 0, aph = 0;
    int it = 0;
    bool ok = true;
    for (int tau = blockIdx.x; tau < ntasks && ok; tau += gridDim.x, ++it) {
      const int slot = it & 1;
      const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
      if (!warp_wait(&s.scl_full[slot], (it >> 1) & 1, err)) break;
      const int arow = (tile ? t.rowA1 : t.rowA0) + row;
      const uint16_t* gscale =
          (t.shared ? p.scale_shared : p.scale_routed) + (size_t)arow * t.ngroups;
      const uint8_t* sscale = s.scl[slot] + tile * 128 * t.ngroups * 2 + row * t.ngroups * 2;
      for (int kb = 0; kb < t.nkb; ++kb) {
        if (!warp_wait(&s.raw_full[rstage], rph, err) ||
            !warp_wait(&s.abf_empty[astage], aph ^ 1u, err)) {
          ok = false;
          break;
        }
        const uint16_t sb = scale_tma ? *reinterpret_cast<const uint16_t*>(sscale + (kb >> 1) * 2)
                                      : __ldg(gscale + (kb >> 1));
        __nv_bfloat162 s2;
        *reinterpret_cast<uint32_t*>(&s2) = (uint32_t)sb | ((uint32_t)sb << 16);
        const uint4* src = reinterpret_cast<const uint4*>(s.raw[rstage] + tile * kInt4Tile + row * 32);
        const uint4 w0 = src[0], w1 = src[1];
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t dst = smem_u32(s.abf[astage] + tile * kAbfTile + row * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          sts128(dst + ((j ^ (row & 7)) << 4), dq_pair<0>(words[j], s2), dq_pair<1>(words[j], s2),
                 dq_pair<2>(words[j], s2), dq_pair<3>(words[j], s2));
        // generic-proxy stores -> visible to the tensor core's async proxy
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.abf_full[astage]);
        if (++rstage == kRawStages) {
          rstage = 0;
          rph ^= 1u;
        }
        if (++astage == kAbfStages) {
          astage = 0;
          aph ^= 1u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.scl_empty[slot]);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int ch = q * 32 + lane;           // channel within a 128-row tile
    int it = 0;
    for (int tau = blockIdx.x; tau < ntasks; tau += gridDim.x, ++it) {
      const TcTask t = decode_task<MODE>(p, tau, n_sh, n_act);
      if (!warp_wait(&s.acc_full, it & 1, err)) break;
      tc_fence_after();
      for (int c0 = 0; c0 < t.n; c0 += 32) {
        float v0[32], v1[32];
        tmem_ld32(tmem + lane_base + c0, v0);
        tmem_ld32(tmem + lane_base + 256 + c0, v1);
        const int cn = t.n - c0;
        if (MODE == 1) {
          const int n = t.chan0 + ch;
          const int pos = (n & ~7) | ((n & 3) << 1) | ((n >> 2) & 1);
          uint16_t* hp = p.hout + (size_t)(t.brow0 + c0) * p.hstride + pos;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < cn) hp[(size_t)j * p.hstride] = f32_to_bf16_bits(silu(v0[j]) * v1[j]);
        } else {
          float* yr = p.yout + (size_t)(t.brow0 + c0) * d.H + t.chan0 + ch;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < cn) {
              yr[(size_t)j * d.H] = v0[j];
              yr[(size_t)j * d.H + 128] = v1[j];
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
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
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE>, w.wq_r, w.wq_s, w.ws_r, w.ws_s, bmap, p);
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
  p.scale_tma = w.scale_tma;
  p.hout = h;
  p.hstride = hstride;
  log.begin("tc_gate_up_swiglu", s);
  cudaError_t e = launch<1>(p, w, xmap, grid, s);
  log.end(s);
  return e;
}

cudaError_t launch_tc_down(const Dims& d, const Routing& r, const TcWeights& w,
                           const CUtensorMap& hmap, float* y, int grid, cudaStream_t s,
                           LaunchLog& log) {
  TcParams p{};
  p.d = d;
  p.r = r;
  p.scale_routed = w.scale_routed;
  p.scale_shared = w.scale_shared;
  p.scale_tma = w.scale_tma;
  p.yout = y;
  log.begin("tc_down", s);
  cudaError_t e = launch<2>(p, w, hmap, grid, s);
  log.end(s);
  return e;
}

}  // namespace moe

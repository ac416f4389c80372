// Decode-sized forward (T <= kSmallT tokens) as ONE persistent cooperative
// kernel: router, gate/up + SwiGLU, down, weighted combine with the shared
// expert.
//
// At decode sizes the layer is a stream of INT4 weights: about 91 MB of
// expert weights plus the 4 MB fp32 router at one token ("Throughputmaxxing:
// DeepSeek-V4-Flash on Isambard-AI", "A pass through the model": below the
// ridge the expert GEMMs are memory bound; "Where does the time go?": the
// act+quant bucket is hundreds of tiny launches). Every kernel boundary costs
// a ramp-up and a tail of the memory pipeline, so the whole layer runs as one
// task stream that never stops fetching weights:
//
//   [gate/up shared | gate/up routed | down shared | down routed]
//
// (above 4 tokens the shared down tasks move ahead of the routed ones, see
// task_at). CTA b takes tasks b, b + G, b + 2G, ... (G = one CTA per SM). A
// task covers
// two 16-row weight tiles (16 gate + 16 up channels, or 32 down channels) of
// one expert over all of K, for one pass of <= 8 rows of that expert.
//
// Warp roles (one CTA per SM):
//  * 4 router warps: every CTA scores one or two experts for all tokens
//    (fp32; the epilogue warps, idle until the first task ends, help: 8 warps
//    hold a K slice of both router rows in registers and stream the tokens),
//    publishes the logits, waits until every CTA has (a counter), then
//    computes the whole routing itself in shared memory (top-k, histogram,
//    scan, stable permutation, task lists). Computing it redundantly per CTA
//    keeps the critical path at two global round trips, and it overlaps the
//    shared expert's work, which needs no routing.
//  * 8 consumer warps stream stages from the start: warp w takes K-group w of
//    both tiles in each 8-group sub-stage (the activation fragments serve
//    both; one MMA chain per tile); exact INT4 -> bf16 in registers (lop3
//    into the mantissa, a bf16x2 subtract), mma.sync m16n8k16 with the
//    weights as A and up to 8 rows as B, group scales applied in fp32. At the
//    end of a task each warp drops its partial sums into a slot and moves on.
//    Every stage reads its activation rows (the interleaved x that the CTAs
//    owning a token prepare once per forward, or h) in one layout, so all
//    stages share one code path.
//  * 1 weight producer warp: fills a ring of stages with a descriptor per
//    stage; it only ever waits for free stages, so the weight stream never
//    stops on a dependency. The shared expert's gate/up tasks it decodes
//    itself; from the first routed task on it reads records that the router
//    warps decoded next to the routing. A stage holds the weights plus room
//    for the pass's activation rows (min(T, 8)). Up to 4 rows, and when every
//    K is a multiple of 1024, a stage is 16 K-groups (32 KB of weights in one
//    TMA box, its scales in another): 4 stages at one token (128 KB in flight
//    per SM). Otherwise a stage is 8 K-groups (16 rows x 512 B per tile,
//    128-byte swizzled when K is a multiple of 256): 5 stages at 64 tokens.
//    Every handoff (descriptor, barrier waits and arrivals, TMA issues) is
//    per stage, so the wide stage halves them per byte.
//  * 1 activation warp: in ring order, copies each stage's activation rows
//    (interleaved x for gate/up, h for down) into the stage (1-D bulk copies). Down tasks
//    need the h rows of their (expert, pass): it polls the completion counters
//    of every active (expert, pass) at once (lanes in parallel, one round trip)
//    and keeps the finished ones in a shared-memory bitmap.
//  * 4 epilogue warps, one per slot: fixed-order reduction of the 16 partial
//    sums, SwiGLU -> bf16 h (then a release-add on the (expert, pass)
//    counter) or fp32 y (then an acq_rel ticket per channel tile; the task
//    that completes a tile combines it for every token:
//    out = y_shared + sum_j w_j y_j in slot order). Fences and atomics stay
//    off the consumers' path.
//  * Every wait is bounded in time and gives up once any wait of the grid has
//    timed out (device error flag), so a broken hand-off cannot hang the GPU.
//    The grid is launched cooperatively so all CTAs are co-resident; every
//    CTA finishes all its gate/up tasks before the down tasks that depend on
//    them, so waits on counters always make progress. The last CTA to exit
//    resets the counters.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kCW = 8;                       // consumer warps (one per K group, both tiles)
constexpr int kEW = 4;                       // epilogue warps (= slots)
constexpr int kRW = 4;                       // router warps
constexpr int kProd = kCW;                   // weight producer warp index
constexpr int kActs = kCW + 1;               // activation warp index
constexpr int kEpi0 = kCW + 2;               // first epilogue warp
constexpr int kRtr0 = kEpi0 + kEW;           // first router warp
constexpr int kThreads = (kCW + 2 + kEW + kRW) * 32;
constexpr int kSW = kRW + kEW;               // warps that score experts (router + epilogue)
constexpr int kR = 8;                        // rows per pass (MMA N)
// above this many tokens the grid ranks them (one token per CTA) instead of
// every CTA ranking all of them
constexpr int kLocalRankT = 8;
constexpr int kMaxS = 12;                    // ring stages at most (the count depends on T)
constexpr int kWB = 2 * 16 * 512;            // sub-stage: 2 tiles x 16 rows x 512 B (8 K-groups)
constexpr int kSB = 2 * 16 * 16;             // sub-stage: 2 tiles x 16 rows x 8 bf16 scales
constexpr int kXSub = 8 * 256;               // one activation row of a sub-stage (8 groups bf16)
constexpr int kMaxSub = 2;                   // sub-stages per stage at most
constexpr int kGateRows = 4;                 // up to this many tokens the shared expert's
                                             // stream waits for the router's loads
constexpr int kSmemMax = 227 * 1024;         // opt-in shared memory of one CTA
constexpr int kMaxPass = (kSmallT + kR - 1) / kR;  // passes per expert at most
constexpr int kPairs = (kMaxExperts + 1) * kMaxPass;  // (expert, pass) counters
constexpr int kItems = kSmallT * kMaxTopK;
constexpr int kMaxRecs = 512;                // a CTA's tasks after routing, kept as decoded records

// Stage descriptor flags. The consumers read only this word of a stage's
// descriptor: the K groups of the stage sit in bits 8-12, the activation rows
// in bits 13-16 and the offset of those rows in the activation pool, in
// 128-byte units, in bits 17-26.
// kPre: a gate/up stage, whose activation rows are the interleaved x.
enum { kFirst = 1, kLast = 2, kEnd = 4, kShared = 8, kDown = 16, kPre = 32, kSwz = 64 };
__host__ __device__ constexpr int stage_key(int flags, int gcnt, int nr, int act) {
  return flags | (gcnt << 8) | (nr << 13) | ((act >> 7) << 17);
}
// Bytes of one activation row of a stage of gcnt K groups (64 bytes off a
// multiple of 128: the consumers' reads are conflict-free).
__host__ __device__ constexpr int act_stride(int gcnt) { return gcnt * 256 + 64; }

struct Desc {
  int flags, g0, gcnt, ngroups, tile, r0, nr, rowA0, rowA1, cnt, act, pad;  // cnt: (expert, pass)
};

struct Smem {
  float4 red[kEW][16 * 32];             // task-end partial sums (K group x tile), one slot per epilogue warp
  float part[2][kSW][kSmallT];          // router: per-warp partial logits of 2 experts
  float bias_s[kMaxExperts];
  Desc slot_desc[kEW];
  Desc desc[kMaxS];
  int ids_s[kItems];
  float wts_s[kItems];
  int perm_s[kItems];
  int inv_s[kItems];
  int counts_s[kMaxExperts];
  int run_s[kMaxExperts];               // router: running row count per expert
  int active[kMaxExperts + 2];
  int pre1[kMaxExperts + 2];
  int pre2[kMaxExperts + 2];
  int offsets[kMaxExperts + 2];
  int4 scan[kRW];
  int meta[4];                          // n_act, routed gate/up tasks, routed down tasks
  uint2 trec[kMaxRecs];                 // this CTA's tasks from its first routed one on (task_record)
  int nrec;                             // records in trec, or -1 (too many: decode on the fly)
  int apos[kMaxS];                      // producer: pool position of each in-flight stage's rows
  uint64_t full[kMaxS];
  uint64_t empty[kMaxS];
  uint64_t desc_ready[kMaxS];           // weight producer -> activation warp
  unsigned pair_done[(kPairs + 31) / 32];  // finished (expert, pass) gate/up work
  uint64_t slot_full[kEW];
  uint64_t slot_free[kEW];
  uint64_t route_ready;                 // routing in shared memory (router warp 0)
  uint64_t rec_ready;                   // task records (router warps 1-3)
  uint64_t scored;                      // this CTA's logits published
  int flag;
};

// The stage ring follows the fixed part of shared memory: nst stages of
// stage_bytes each, sized at launch for the batch (a stage holds the weight
// and scale boxes plus min(T, kR) activation rows).
constexpr int kStageOff = (int)((sizeof(Smem) + 1023) / 1024 * 1024);

struct DecodeParams {
  Dims d;
  Routing r;
  const uint16_t* x;            // [T, H] bf16
  const float* router_w;        // [E, H]
  const float* router_bias;     // [E]
  const uint16_t* s13_routed;   // scales, for the consumers when not TMA'd
  const uint16_t* s13_shared;
  const uint16_t* s2_routed;
  const uint16_t* s2_shared;
  uint16_t* xi;                 // [T, H] bf16: x interleaved, chunks transposed (chunk_t)
  uint16_t* h;                  // [rows, hstride] bf16, interleaved, chunks transposed
  int hstride;
  uint16_t* y;                  // [rows, H] bf16: each expert's down output
  uint16_t* out;                // [T, H] bf16
  int* done1;                   // [(E + 1) * kMaxPass] gate/up tasks done per (expert, pass)
  int* tile_cnt;                // [H / 32] down tasks done per channel tile
  unsigned* sync;               // [4]: logits ticket, x-interleave ticket, exit ticket, ranked tokens
  int scale_tma;
  int nst;                      // ring stages
  int stage_bytes;              // weight and scale bytes per stage (a multiple of 1024)
  int nsub;                     // sub-stages (8 K-groups each) per stage
  int pool_off;                 // the activation pool, after the ring (bytes from its start)
  int pool_bytes;
};

struct Task {
  bool down, shared;
  int e, ngroups, rowA0, rowA1, r0, nr, tile, pass, cnt_target;
};

__device__ __forceinline__ int passes_of(int rows) { return (rows + kR - 1) / kR; }

// named barrier of the router warps
__device__ __forceinline__ void rbar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool aborted(const unsigned* err) {
  return (*reinterpret_cast<const volatile unsigned*>(err) & kErrTimeout) != 0;
}

// mbarrier wait bounded in time that also gives up once the grid aborted.
__device__ __forceinline__ bool dwait(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (aborted(err)) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *p >= target (acquire). false on timeout / abort.
__device__ __forceinline__ bool wait_counter(const int* p, int target, unsigned* err) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    __nanosleep(32);
    if (ld_acquire(p) >= target) return true;
    if (aborted(err)) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// generic shared-memory accesses of this thread before later async-proxy
// (TMA, bulk copy) accesses of the same bytes, e.g. reads of a stage before
// the release that lets the next fill overwrite it
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                       int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                       int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_5d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                       int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4)
      : "memory");
}

__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                       int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// One TMA copy brings both 16-row weight tiles of a stage (8 K-groups each),
// one more their group scales. A matrix whose rows are a whole number of
// 128-byte segments (K a multiple of 256) is viewed in 128-byte segments and
// fetched with the 128-byte swizzle: 16-byte chunk q of the 128-byte line at
// byte offset o of the stage lands at chunk q ^ ((o >> 7) & 7). Rows 512 bytes
// apart then differ in bit 2 of the swizzle, so the two rows read by a quarter
// warp fall in opposite halves of the banks. Other matrices use plain
// row-major boxes (512 bytes per row). Either way tile 0 sits in the first
// 8 KB of the stage and tile 1 in the second, and the scales of tile 0 / 1 in
// the first / second 256 bytes after them.
//   gate/up (the gate rows of a tile and the up rows of the same channels,
//   I' rows apart): a box over {row segment, segments, 16 rows, 2 halves};
//   down (32 consecutive rows): a box over {row segment, segments, 32 rows}.
__device__ __forceinline__ bool swizzled_k(int K) { return K % 256 == 0; }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// Activation rows the consumers read with the transposed addressing (the
// interleaved x of routed gate/up stages, and h) store 16-byte chunk w of each
// K group (w = 4c + m: lane column c, MMA step m) at position 4m + c.
__device__ __forceinline__ int chunk_t(int w) { return ((w & 3) << 2) | (w >> 2); }

// The 8 MMA steps of one K group of one tile, accumulated in one chain (the
// group's partial sum, scaled once afterwards): each code pair becomes bf16
// q exactly (lop3 into the mantissa, then a bf16x2 subtract).
__device__ __forceinline__ void stage_mma(const uint4& wA, const uint4& wB, const uint4 (&b)[4],
                                          float (&t)[4]) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
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
}

// ------------------------------------------------------------ task decode
struct Counts {
  int sh1, r1, sh2, r2, n_act;
};

__device__ __forceinline__ Task make_task(const Dims& d, bool down, bool shared, int e, int seg0,
                                          int seg1, int local) {
  Task t;
  t.down = down;
  t.shared = shared;
  t.e = e;
  const int passes = passes_of(seg1 - seg0);
  t.tile = local / passes;
  t.pass = local - t.tile * passes;
  t.r0 = seg0 + t.pass * kR;
  t.nr = min(kR, seg1 - t.r0);
  const int inter = shared ? d.Is : d.I;
  if (!down) {
    t.ngroups = d.H / kGroup;
    t.rowA0 = (shared ? 0 : e * 2 * inter) + t.tile * kTile1;
    t.rowA1 = t.rowA0 + inter;
    t.cnt_target = 0;
  } else {
    t.ngroups = inter / kGroup;
    t.rowA0 = (shared ? 0 : e * d.H) + t.tile * kTile2;
    t.rowA1 = t.rowA0 + 16;
    t.cnt_target = inter / kTile1;  // gate/up tiles of this (expert, pass)
  }
  return t;
}

__device__ __forceinline__ int find_active(const int* pre, int n_act, int tau) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= tau)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Task tau of the concatenated list [gate/up shared | gate/up routed | down
// shared | down routed], or t.ngroups == 0 when tau is past its end. Only the
// first part needs no routing; every CTA takes all its gate/up tasks before
// its down tasks, and the shared down work sits between the two routed halves
// so that the routed gate/up stream starts as soon as the routing is known.
// Above kGateRows tokens the shared expert's down tasks come right after its
// gate/up tasks, inside the routing window: their stages hold a full pass of
// 8 activation rows each, so the pool takes them one at a time, which the
// routing hides but the routed stream would not. At smaller batches they sit
// between the routed halves, where their h is long ready.
__device__ __forceinline__ bool shared_down_first(const Dims& d) { return d.T > kGateRows; }
__device__ __forceinline__ int pre_routing_tasks(const Dims& d, const Counts& c) {
  return c.sh1 + (shared_down_first(d) ? c.sh2 : 0);
}

__device__ __forceinline__ Task task_at(const Smem& s, const Dims& d, const Counts& c, int tau) {
  const int sh0 = d.T * d.k, sh1 = d.T * d.k + d.T;
  const bool early = shared_down_first(d);
  if (tau < c.sh1) return make_task(d, false, true, d.E, sh0, sh1, tau);
  tau -= c.sh1;
  if (early) {
    if (tau < c.sh2) return make_task(d, true, true, d.E, sh0, sh1, tau);
    tau -= c.sh2;
  }
  if (tau < c.r1) {
    const int a = find_active(s.pre1, c.n_act, tau);
    const int e = s.active[a];
    return make_task(d, false, false, e, s.offsets[e], s.offsets[e + 1], tau - s.pre1[a]);
  }
  tau -= c.r1;
  if (!early) {
    if (tau < c.sh2) return make_task(d, true, true, d.E, sh0, sh1, tau);
    tau -= c.sh2;
  }
  if (tau < c.r2) {
    const int a = find_active(s.pre2, c.n_act, tau);
    const int e = s.active[a];
    return make_task(d, true, false, e, s.offsets[e], s.offsets[e + 1], tau - s.pre2[a]);
  }
  Task t{};
  t.ngroups = 0;
  return t;
}

// A task in two words: expert (9 bits), tile (12), pass (3), down, shared;
// first row (16), rows (16).
__device__ __forceinline__ uint2 task_record(const Task& t) {
  return make_uint2((uint32_t)t.e | ((uint32_t)t.tile << 9) | ((uint32_t)t.pass << 21) |
                        ((uint32_t)t.down << 24) | ((uint32_t)t.shared << 25),
                    (uint32_t)t.r0 | ((uint32_t)t.nr << 16));
}

__device__ __forceinline__ Task task_of_record(const Dims& d, uint2 r) {
  Task t;
  t.e = (int)(r.x & 511u);
  t.tile = (int)((r.x >> 9) & 4095u);
  t.pass = (int)((r.x >> 21) & 7u);
  t.down = ((r.x >> 24) & 1u) != 0;
  t.shared = ((r.x >> 25) & 1u) != 0;
  t.r0 = (int)(r.y & 0xffffu);
  t.nr = (int)(r.y >> 16);
  const int inter = t.shared ? d.Is : d.I;
  if (!t.down) {
    t.ngroups = d.H / kGroup;
    t.rowA0 = (t.shared ? 0 : t.e * 2 * inter) + t.tile * kTile1;
    t.rowA1 = t.rowA0 + inter;
    t.cnt_target = 0;
  } else {
    t.ngroups = inter / kGroup;
    t.rowA0 = (t.shared ? 0 : t.e * d.H) + t.tile * kTile2;
    t.rowA1 = t.rowA0 + 16;
    t.cnt_target = inter / kTile1;
  }
  return t;
}

// ------------------------------------------------------------ router
constexpr int kPer = kMaxExperts / 32;  // logits per lane

// Order-preserving key of a finite float (larger float -> larger key; key 0
// stays below every float and marks a taken candidate).
__device__ __forceinline__ unsigned fkey(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token whose logits lane l holds for experts l, l + 32, ...;
// lanes 0..k-1 return the chosen expert (descending sel, ties -> lower index)
// and its renormalised unbiased score. A round is two warp reductions: the
// largest selection key, then the lowest expert index among the lanes holding
// it. The sorted-list version (topk.cuh) gives the same results in ~0.6x the
// time; rank_spread uses it, but inlined here it moves the register
// allocation of the whole kernel and costs the one-token forward 2-3 us, so
// the in-line ranking keeps this one.
__device__ __forceinline__ void warp_topk(const float (&lg)[kPer], const float* bias, int E, int k,
                                          int lane, int* out_id, float* out_w) {
  float sc[kPer];
  unsigned key[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      sc[i] = __frcp_rn(1.0f + expf(-lg[i]));  // = 1 / (1 + e^-l), correctly rounded
      key[i] = fkey(sc[i] + bias[e]);
    } else {
      sc[i] = 0.f;
      key[i] = 0u;
    }
  }
  // this lane's best remaining candidate (lowest i among equal keys)
  auto local_best = [&](unsigned& bk, int& bi) {
    bk = key[0];
    bi = 0;
#pragma unroll
    for (int i = 1; i < kPer; ++i)
      if (key[i] > bk) {
        bk = key[i];
        bi = i;
      }
  };
  unsigned bk;
  int bi;
  local_best(bk, bi);
  float chosen_s = 0.f;
  int chosen_e = -1;
  for (int j = 0; j < k; ++j) {
    const unsigned m = __reduce_max_sync(0xffffffffu, bk);
    const unsigned cand = bk == m ? (unsigned)(lane + 32 * bi) : 0xffffffffu;
    const unsigned win = __reduce_min_sync(0xffffffffu, cand);
    const int wl = (int)(win & 31u), wi = (int)(win >> 5);
    float ws = 0.f;
    if (lane == wl) {
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (i == wi) {
          ws = sc[i];
          key[i] = 0u;
        }
      local_best(bk, bi);
    }
    ws = __shfl_sync(0xffffffffu, ws, wl);
    if (lane == j) {
      chosen_e = (int)win;
      chosen_s = ws;
    }
  }
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, chosen_s, j);
  *out_id = chosen_e;
  *out_w = chosen_s / sum;
}

__device__ __forceinline__ void load_logits(const float* row, int E, int lane, float (&lg)[kPer]) {
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? __ldcg(row + e) : 0.f;
  }
}

// Exclusive scan of four ints over the 128 router threads (t = router thread).
__device__ __forceinline__ int4 rscan4(int4 v, int t, int4* scr, int4* total) {
  const int lane = t & 31, warp = t >> 5;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, inc.x, o), b = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int c = __shfl_up_sync(0xffffffffu, inc.z, o), e = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) {
      inc.x += a;
      inc.y += b;
      inc.z += c;
      inc.w += e;
    }
  }
  if (lane == 31) scr[warp] = inc;
  rbar();
  int4 base = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
  for (int w = 0; w < kRW; ++w) {
    const int4 s = scr[w];
    if (w < warp) {
      base.x += s.x;
      base.y += s.y;
      base.z += s.z;
      base.w += s.w;
    }
    tot.x += s.x;
    tot.y += s.y;
    tot.z += s.z;
    tot.w += s.w;
  }
  rbar();
  *total = tot;
  return make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z,
                   base.w + inc.w - v.w);
}

// Warps that score experts: the router warps, joined by the epilogue warps
// when the batch is tiny (they are free until the first task ends, which
// takes longer than scoring a few tokens; at larger batches scoring would hold
// them up).
__device__ __forceinline__ int scoring_warps(const Dims& d) {
  return d.T <= 4 ? kSW : (d.T <= kLocalRankT ? kRW : kSW + kCW);
}

// named barrier of the scoring warps
constexpr int kTB = 4;  // tokens per x load batch in the scoring loop

__device__ __forceinline__ void sbar(int nsw) {
  asm volatile("bar.sync 2, %0;" ::"r"(nsw * 32) : "memory");
}

// Logits of this CTA's experts (e = b and b + G, for all tokens) by the nsw
// scoring warps. K is cut into kSW slices whatever the batch size, so a
// token's logits do not depend on the batch; scoring warp w takes slices w,
// w + nsw, ... Per slice each lane keeps its share of both router rows in
// registers (up to 4 float4 each; larger slices go in chunks) and streams the
// tokens' x through, two tokens per round trip; the slice partials are summed
// in slice order.
__device__ __noinline__ void score_experts_impl(Smem& s, const Dims d, const float* router_w, const uint16_t* x,
                                               float* logits, int sw) {
  const int nsw = scoring_warps(d);
  const int lane = threadIdx.x & 31, tid = sw * 32 + lane;
  // more warps than slices: the warps of a slice split its token batches; a
  // (slice, token) partial is computed the same way whichever warp takes it
  const int share = nsw > kSW ? nsw / kSW : 1;
  const int sl_first = nsw > kSW ? sw % kSW : sw, sl_step = nsw > kSW ? kSW : nsw;
  const int t_first = (nsw > kSW ? sw / kSW : 0) * kTB;
  const int kw = d.H / kSW;   // K slice (a multiple of 16)
  const int nf = kw / 4;      // float4 of the slice
  for (int eb = blockIdx.x; eb < d.E; eb += 2 * gridDim.x) {
    const int e0 = eb, e1 = eb + gridDim.x;
    const bool has1 = e1 < d.E;
    for (int sl = sl_first; sl < kSW; sl += sl_step)
    for (int f0 = 0; f0 < nf; f0 += 128) {
      const float4* w0 = reinterpret_cast<const float4*>(router_w + (size_t)e0 * d.H + sl * kw);
      const float4* w1 = reinterpret_cast<const float4*>(router_w + (size_t)(has1 ? e1 : e0) * d.H +
                                                         sl * kw);
      float4 v0[4], v1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = f0 + u * 32 + lane;
        const bool ok = f < nf;
        v0[u] = ok ? __ldg(w0 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        v1[u] = ok && has1 ? __ldg(w1 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int t0 = t_first; t0 < d.T; t0 += share * kTB) {
        uint2 xv[kTB][4];
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
          const int t = min(t0 + j, d.T - 1);
          const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)t * d.H + sl * kw);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int f = f0 + u * 32 + lane;
            xv[j][u] = f < nf ? __ldg(xr + f) : make_uint2(0u, 0u);
          }
        }
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
          const int t = t0 + j;
          if (t >= d.T) break;
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint2 xw = xv[j][u];
            const float x0 = __uint_as_float(xw.x << 16), x1 = __uint_as_float(xw.x & 0xffff0000u);
            const float x2 = __uint_as_float(xw.y << 16), x3 = __uint_as_float(xw.y & 0xffff0000u);
            a0 = fmaf(x0, v0[u].x, a0);
            a0 = fmaf(x1, v0[u].y, a0);
            a0 = fmaf(x2, v0[u].z, a0);
            a0 = fmaf(x3, v0[u].w, a0);
            a1 = fmaf(x0, v1[u].x, a1);
            a1 = fmaf(x1, v1[u].y, a1);
            a1 = fmaf(x2, v1[u].z, a1);
            a1 = fmaf(x3, v1[u].w, a1);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            a0 += __shfl_xor_sync(0xffffffffu, a0, o);
            a1 += __shfl_xor_sync(0xffffffffu, a1, o);
          }
          if (lane == 0) {
            s.part[0][sl][t] = f0 == 0 ? a0 : s.part[0][sl][t] + a0;
            s.part[1][sl][t] = f0 == 0 ? a1 : s.part[1][sl][t] + a1;
          }
        }
      }
    }
    sbar(nsw);
    if (tid < 2 * d.T) {
      const int slot = tid / d.T, t = tid - slot * d.T;
      if (slot == 0 || has1) {
        float v = 0.f;
        for (int w = 0; w < kSW; ++w) v += s.part[slot][w][t];
        logits[(size_t)t * d.E + (slot ? e1 : e0)] = v;
      }
    }
    sbar(nsw);
  }
}

// The scoring is compiled out of line: the main kernel's register allocation
// then serves the stage loops alone (decode1 46.2 -> 44.3 us median over four
// interleaved runs; decode64 753 -> 755 us).
__device__ __forceinline__ void score_experts(Smem& s, const DecodeParams& p, int sw) {
  score_experts_impl(s, p.d, p.router_w, p.x, p.r.logits, sw);
}

// Ranking spread over the grid, above kLocalRankT tokens: CTA b ranks tokens
// b, b + G, ... (one router warp per token), publishes their ids and weights,
// and reads everybody's back once all T tokens are ranked (a second grid
// counter). Every CTA ranking all tokens itself would take T / 4 rankings per
// router warp. Out of line on purpose: inlined, it changed the register
// allocation of the whole kernel and cost the one-token forward about 4 us.
__device__ __noinline__ bool rank_spread(const float* logits, int* ids, float* wts, unsigned* err,
                                         unsigned* counter, const float* bias, int T, int E, int k,
                                         int* s_ids, float* s_wts, int* s_counts, int* s_flag) {
  const int tid = threadIdx.x - kRtr0 * 32, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, b = blockIdx.x;
  for (int t = b + warp * G; t < T; t += kRW * G) {
    float lg[kPer];
    load_logits(logits + (size_t)t * E, E, lane, lg);
    int id;
    float w;
    warp_topk_sorted<kMaxTopK>(lg, bias, E, k, lane, &id, &w);
    if (lane < k) {
      if (id < 0 || id >= E) {
        atomicOr(err, kErrRange);
        id = 0;
      }
      ids[t * k + lane] = id;
      wts[t * k + lane] = w;
    }
  }
  rbar();
  if (tid == 0) {
    const int mine = b < T ? (T - b + G - 1) / G : 0;
    if (mine > 0) {
      __threadfence();
      atomicAdd(counter, (unsigned)mine);
    }
    *s_flag = wait_counter(reinterpret_cast<const int*>(counter), T, err) ? 1 : 0;
  }
  rbar();
  if (!*s_flag) return false;
  for (int i = tid; i < T * k; i += kRW * 32) {
    const int id = __ldcg(ids + i);
    s_ids[i] = id;
    s_wts[i] = __ldcg(wts + i);
    atomicAdd(&s_counts[id], 1);
  }
  return true;
}

// Router warps: score this CTA's experts, wait for every CTA's logits, then
// compute the whole routing in shared memory. Returns false on timeout.
__device__ bool router_phase(Smem& s, const DecodeParams& p) {
  const Dims& d = p.d;
  const int tid = threadIdx.x - kRtr0 * 32, lane = tid & 31, warp = tid >> 5;
  score_experts(s, p, warp);
  // publish this CTA's logits and wait for everybody's; the bias (needed only
  // for the ranking) arrives meanwhile
  if (tid == 0) {
    __threadfence();
    atomicAdd(&p.sync[0], 1u);
    mbar_arrive(&s.scored);
  }
  for (int e = tid; e < d.E; e += kRW * 32) s.bias_s[e] = __ldg(p.router_bias + e);
  rbar();
  if (tid == 0) {
    s.flag = wait_counter(reinterpret_cast<const int*>(p.sync), (int)gridDim.x, p.r.err) ? 1 : 0;
  }
  for (int e = tid; e < kMaxExperts; e += kRW * 32) s.counts_s[e] = 0;
  rbar();  // thread 0 acquired the counter; the barrier orders everybody's reads after it
  if (!s.flag) return false;

  if (d.T > kLocalRankT) {
    if (!rank_spread(p.r.logits, p.r.ids, p.r.wts, p.r.err, p.sync + 3, s.bias_s, d.T, d.E, d.k,
                     s.ids_s, s.wts_s, s.counts_s, &s.flag))
      return false;
  } else {
    // ---- the routing of every token, in shared memory (the next token's
    // logits are in flight while this one is ranked)
    float lg[kPer], nx[kPer];
    if (warp < d.T) load_logits(p.r.logits + (size_t)warp * d.E, d.E, lane, nx);
    for (int t = warp; t < d.T; t += kRW) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) lg[i] = nx[i];
      if (t + kRW < d.T) load_logits(p.r.logits + (size_t)(t + kRW) * d.E, d.E, lane, nx);
      int id;
      float w;
      warp_topk(lg, s.bias_s, d.E, d.k, lane, &id, &w);
      if (lane < d.k) {
        if (id < 0 || id >= d.E) {
          atomicOr(p.r.err, kErrRange);
          id = 0;
        }
        s.ids_s[t * d.k + lane] = id;
        s.wts_s[t * d.k + lane] = w;
        atomicAdd(&s.counts_s[id], 1);
      }
    }
  }
  rbar();
  {
    // two experts per thread: e = 2 tid, 2 tid + 1
    int c2[2], ps[2];
    int4 v = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = 2 * tid + i;
      c2[i] = (e < d.E) ? s.counts_s[e] : 0;
      ps[i] = passes_of(c2[i]);
      v.x += c2[i];
      v.y += c2[i] > 0 ? 1 : 0;
      v.z += ps[i] * (d.I / kTile1);
      v.w += ps[i] * (d.H / kTile2);
    }
    int4 tot;
    int4 ex = rscan4(v, tid, s.scan, &tot);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = 2 * tid + i;
      if (e < d.E) {
        s.offsets[e] = ex.x;
        if (c2[i] > 0) {
          s.active[ex.y] = e;
          s.pre1[ex.y] = ex.z;
          s.pre2[ex.y] = ex.w;
        }
      }
      ex.x += c2[i];
      ex.y += c2[i] > 0 ? 1 : 0;
      ex.z += ps[i] * (d.I / kTile1);
      ex.w += ps[i] * (d.H / kTile2);
    }
    if (tid == 0) {
      s.offsets[d.E] = tot.x;
      s.pre1[tot.y] = tot.z;
      s.pre2[tot.y] = tot.w;
      s.meta[0] = tot.y;
      s.meta[1] = tot.z;
      s.meta[2] = tot.w;
    }
  }
  rbar();
  const int n = d.T * d.k;
  if (warp > 0) {
    // this CTA's tasks from its first routed one on (tau = first, first + G,
    // ...), decoded into records by the other router warps while warp 0
    // builds the permutation; the weight producer reads one record per task
    Counts c;
    c.sh1 = d.Is > 0 ? (d.Is / kTile1) * passes_of(d.T) : 0;
    c.sh2 = d.Is > 0 ? (d.H / kTile2) * passes_of(d.T) : 0;
    c.n_act = s.meta[0];
    c.r1 = s.meta[1];
    c.r2 = s.meta[2];
    const int b = blockIdx.x, G = gridDim.x;
    const int total = c.sh1 + c.r1 + c.sh2 + c.r2;
    const int npre = pre_routing_tasks(d, c);
    const int first = npre <= b ? b : b + ((npre - b + G - 1) / G) * G;
    const int nrec = first < total ? (total - first + G - 1) / G : 0;
    if (tid == 32) s.nrec = nrec <= kMaxRecs ? nrec : -1;
    if (nrec <= kMaxRecs)
      for (int j = tid - 32; j < nrec; j += (kRW - 1) * 32)
        s.trec[j] = task_record(task_at(s, d, c, first + j * G));
    asm volatile("bar.sync 3, %0;" ::"n"((kRW - 1) * 32) : "memory");
    if (tid == 32) mbar_arrive(&s.rec_ready);  // the producer decodes on the fly until then
  }
  if (warp == 0) {
    // stable placement, 32 items at a time: rank among equal experts in the
    // chunk by __match_any_sync, plus the expert's running count
    for (int e = lane; e < d.E; e += 32) s.run_s[e] = s.offsets[e];
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int i = c0 + lane;
      const bool valid = i < n;
      const int e = valid ? s.ids_s[i] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lt);
      if (valid) {
        const int pos = s.run_s[e] + rank;
        s.perm_s[pos] = i / d.k;
        s.inv_s[i] = pos;
      }
      __syncwarp();
      if (valid && rank == 0) s.run_s[e] += __popc(peers);
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&s.route_ready);
  }
  rbar();
  // one CTA also writes the routing out (the get-routing hook reads it)
  if (blockIdx.x == 0) {
    for (int i = tid; i < n; i += kRW * 32) {
      if (d.T <= kLocalRankT) {  // else the ranking CTAs wrote them
        p.r.ids[i] = s.ids_s[i];
        p.r.wts[i] = s.wts_s[i];
      }
      p.r.perm[i] = s.perm_s[i];
      p.r.inv[i] = s.inv_s[i];
    }
    for (int e = tid; e <= d.E; e += kRW * 32) {
      p.r.offsets[e] = s.offsets[e];
      if (e < d.E) p.r.counts[e] = s.counts_s[e];
    }
    for (int a = tid; a <= s.meta[0]; a += kRW * 32) {
      if (a < s.meta[0]) p.r.active[a] = s.active[a];
      p.r.task1[a] = s.pre1[a];
      p.r.task2[a] = s.pre2[a];
    }
    if (tid == 0) {
      p.r.meta[kMetaActive] = s.meta[0];
      p.r.meta[kMetaTasks1] = s.meta[1];
      p.r.meta[kMetaTasks2] = s.meta[2];
    }
  }
  return true;
}

// ------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm13r, const __grid_constant__ CUtensorMap tm13s,
                  const __grid_constant__ CUtensorMap tm2r, const __grid_constant__ CUtensorMap tm2s,
                  const __grid_constant__ CUtensorMap ts13r, const __grid_constant__ CUtensorMap ts13s,
                  const __grid_constant__ CUtensorMap ts2r, const __grid_constant__ CUtensorMap ts2s,
                  const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  uint8_t* const stage_base = smem_raw + kStageOff;
  const int nst = p.nst, sb = p.stage_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Dims& d = p.d;
  unsigned* err = p.r.err;
  const bool scale_tma = p.scale_tma != 0;
  // swizzled weight boxes need 1024-byte aligned stages; every thread of every
  // CTA sees the same address, so all of them leave before any barrier
  if (smem_u32(stage_base) & 1023u) {
    if (threadIdx.x == 0) atomicOr(err, kErrLayout);
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nst; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kCW);
      mbar_init(&s.desc_ready[i], 1);
    }
    for (int i = 0; i < (kPairs + 31) / 32; ++i) s.pair_done[i] = 0u;
    for (int i = 0; i < kEW; ++i) {
      mbar_init(&s.slot_full[i], kCW);
      mbar_init(&s.slot_free[i], 1);
    }
    mbar_init(&s.route_ready, 1);
    mbar_init(&s.rec_ready, 1);
    mbar_init(&s.scored, 1);
    fence_mbar_init();
  }
  __syncthreads();

  Counts cnt;
  cnt.sh1 = d.Is > 0 ? (d.Is / kTile1) * passes_of(d.T) : 0;
  cnt.sh2 = d.Is > 0 ? (d.H / kTile2) * passes_of(d.T) : 0;
  cnt.r1 = cnt.r2 = cnt.n_act = 0;

  if (warp == kProd) {
    // ---------------------------------------------------------------- weight producer
    // One lane decodes the CTA's tasks in order and fills the ring. Only the
    // shared expert's gate/up tasks need no routing; the first routed task
    // waits for this CTA's routing (shared memory).
    if (lane == 0) {
      prefetch_tmap(&tm13r);
      prefetch_tmap(&tm13s);
      prefetch_tmap(&tm2r);
      prefetch_tmap(&tm2s);
      bool known = false, stop = false;
      int stage = 0;
      uint32_t phase = 0;
      const int nsub = p.nsub, gps = 8 * nsub;  // K groups per stage
      int rec = 0;     // tasks since the first routed one
      int nrec = -2;   // records: -2 not ready yet, -1 none (too many), else their count
      // The activation pool is a FIFO in stage order: a stage's rows take
      // [apos, apos + need) of an unbounded byte sequence, stored at that
      // position modulo the pool (an allocation never wraps), and are freed
      // when the stage is released. q counts stages, rel the released ones.
      int q = 0, rel = 0, head = 0;
      const int P = p.pool_bytes;
      if (d.T <= kGateRows) dwait(&s.scored, 0, err);  // small batch: the router's loads go first
      for (int tau = blockIdx.x; !stop; tau += gridDim.x) {
        if (tau >= pre_routing_tasks(d, cnt) && !known) {
          if (!dwait(&s.route_ready, 0, err)) break;
          cnt.n_act = s.meta[0];
          cnt.r1 = s.meta[1];
          cnt.r2 = s.meta[2];
          known = true;
        }
        Task t;
        if (known) {
          if (nrec == -2 && mbar_try_wait(&s.rec_ready, 0)) nrec = s.nrec;
          if (nrec >= 0) {
            if (rec >= nrec) break;  // past the last task
            t = task_of_record(d, s.trec[rec]);
          } else {
            t = task_at(s, d, cnt, tau);
          }
          ++rec;
        } else {
          t = task_at(s, d, cnt, tau);
        }
        if (t.ngroups == 0) break;  // past the last task
        const CUtensorMap* tm = t.down ? (t.shared ? &tm2s : &tm2r) : (t.shared ? &tm13s : &tm13r);
        const CUtensorMap* ts = t.down ? (t.shared ? &ts2s : &ts2r) : (t.shared ? &ts13s : &ts13r);
        const bool swz = swizzled_k(t.ngroups * kGroup);
        const int half = t.shared ? 0 : 2 * t.e;  // gate half of the expert (up: half + 1)
        for (int g0 = 0; g0 < t.ngroups; g0 += gps) {
          const int gcnt = min(gps, t.ngroups - g0);
          if (!dwait(&s.empty[stage], phase ^ 1u, err)) {
            stop = true;
            break;
          }
          rel = max(rel, q - nst + 1);  // the slot's previous stage is released
          // room for nr activation rows in the pool: wait for the oldest
          // stages' releases until they fit (a stage's release is the phase
          // of its slot's empty barrier that completes when it is consumed)
          const int need = (t.nr * act_stride(gcnt) + 127) & ~127;
          int apos = head;
          if (apos % P + need > P) apos += P - apos % P;
          while (rel < q && apos + need - s.apos[rel % nst] > P) {
            if (!dwait(&s.empty[rel % nst], (uint32_t)(rel / nst) & 1u, err)) {
              stop = true;
              break;
            }
            ++rel;
          }
          if (stop) break;
          s.apos[stage] = apos;
          head = apos + need;
          Desc& ds = s.desc[stage];
          const bool pre = !t.down;  // gate/up: the interleaved x rows
          ds.flags = stage_key((g0 == 0 ? kFirst : 0) | (g0 + gps >= t.ngroups ? kLast : 0) |
                                   (t.shared ? kShared : 0) | (t.down ? kDown : 0) |
                                   (pre ? kPre : 0) | (swz ? kSwz : 0),
                               gcnt, t.nr, apos % P);
          ds.act = apos % P;
          ds.g0 = g0;
          ds.gcnt = gcnt;
          ds.ngroups = t.ngroups;
          ds.tile = t.tile;
          ds.r0 = t.r0;
          ds.nr = t.nr;
          ds.rowA0 = t.rowA0;
          ds.rowA1 = t.rowA1;
          ds.cnt = t.e * kMaxPass + t.pass;
          // a box always delivers its full size (out-of-range parts are
          // zero-filled); the activation warp copies nr rows into the pool
          mbar_arrive_expect_tx(&s.full[stage], nsub * (kWB + (scale_tma ? kSB : 0)) + t.nr * gcnt * 256);
          const uint32_t st = smem_u32(stage_base + (size_t)stage * sb), ss = st + nsub * kWB;
          if (nsub == 2) {
            // wide views: 16 K groups of both tiles in one box
            if (!t.down) {
              tma_5d(st, tm, &s.full[stage], 0, 0, t.tile * kTile1, g0 / 8, half);
              if (scale_tma) tma_4d(ss, ts, &s.full[stage], 0, t.tile * kTile1, g0 / 8, half);
            } else {
              tma_5d(st, tm, &s.full[stage], 0, 0, 0, g0 / 8, t.rowA0 / 16);
              if (scale_tma) tma_4d(ss, ts, &s.full[stage], 0, 0, g0 / 8, t.rowA0 / 16);
            }
          } else if (!t.down) {
            if (swz)
              tma_4d(st, tm, &s.full[stage], 0, g0 / 2, t.tile * kTile1, half);
            else
              tma_3d(st, tm, &s.full[stage], g0 * 16, t.tile * kTile1, half);
            if (scale_tma) tma_3d(ss, ts, &s.full[stage], g0, t.tile * kTile1, half);
          } else {
            if (swz)
              tma_3d(st, tm, &s.full[stage], 0, g0 / 2, t.rowA0);
            else
              tma_2d(st, tm, &s.full[stage], g0 * 16, t.rowA0);
            if (scale_tma) tma_2d(ss, ts, &s.full[stage], g0, t.rowA0);
          }
          mbar_arrive(&s.desc_ready[stage]);
          ++q;
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!stop && dwait(&s.empty[stage], phase ^ 1u, err)) {
        s.desc[stage].flags = kEnd;
        mbar_arrive(&s.full[stage]);
        mbar_arrive(&s.desc_ready[stage]);
      }
    }
    __syncwarp();
  } else if (warp == kActs) {
    // ---------------------------------------------------------------- activation rows
    // First this CTA's share of the tokens (t = b, b + G, ...): the
    // interleaved copy of x that every CTA's gate/up stages read, published on
    // its own counter. It needs no routing, so the shared expert's gate/up
    // stages can complete while the router works.
    {
      const int h8 = d.H / 8;  // 16-byte chunks of a row; 16 per K group
      for (int t = blockIdx.x; t < d.T; t += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * d.H);
        uint4* dst = reinterpret_cast<uint4*>(p.xi + (size_t)t * d.H);
        for (int c0 = 0; c0 < h8; c0 += 32 * 8) {
          uint4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int cidx = c0 + u * 32 + lane;
            if (cidx < h8) v[u] = __ldg(src + cidx);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int cidx = c0 + u * 32 + lane;
            if (cidx < h8) dst[(cidx & ~15) | chunk_t(cidx & 15)] = interleave8(v[u]);
          }
        }
      }
      __threadfence();
      __syncwarp();
      if (lane == 0 && (int)blockIdx.x < d.T) atomicAdd(&p.sync[1], 1u);
    }
    int stage = 0;
    uint32_t phase = 0;
    bool pre_ready = false;
    // is the gate/up work of (expert, pass) `want` finished anywhere in the
    // grid? One acquire load of its counter (lane 0), remembered in the CTA's
    // bitmap. Polling every active pair at once cost the first down stage at
    // 64 tokens a chain of ~49 dependent acquire loads per lane.
    auto pair_ready = [&](int want) -> bool {
      int ok = 0;
      if (lane == 0) {
        const int target = (want / kMaxPass == d.E ? d.Is : d.I) / kTile1;
        ok = ld_acquire(p.done1 + want) >= target ? 1 : 0;
        if (ok) s.pair_done[want >> 5] |= 1u << (want & 31);
      }
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    for (;;) {
      if (!__all_sync(0xffffffffu, dwait(&s.desc_ready[stage], phase, err))) break;
      const Desc ds = s.desc[stage];
      if (ds.flags & kEnd) break;
      const bool down = (ds.flags & kDown) != 0;
      // lane 0 writes the bitmap: its view decides, for the whole warp
      if (down && !__shfl_sync(0xffffffffu, (s.pair_done[ds.cnt >> 5] >> (ds.cnt & 31)) & 1u, 0)) {
        // wait for the gate/up work of this (expert, pass) anywhere in the grid
        const uint64_t t0 = global_ns();
        bool got = pair_ready(ds.cnt);
        while (!got) {
          __nanosleep(128);
          if (aborted(err)) break;
          if (global_ns() - t0 > kWaitLimitNs) {
            if (lane == 0) atomicOr(err, kErrTimeout);
            break;
          }
          got = pair_ready(ds.cnt);
        }
        if (!got) break;
      }
      if (down) {
        // every lane that copies h orders its copies after the acquires above
        __syncwarp();
        fence_proxy_async();
      }
      if ((ds.flags & kPre) && !pre_ready) {
        // the interleaved x comes from other CTAs' generic stores, published
        // on its own counter by the CTAs that own a token
        int ok = 1;
        if (lane == 0)
          ok = wait_counter(reinterpret_cast<const int*>(p.sync + 1), min(d.T, (int)gridDim.x), err) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        fence_proxy_async();
        pre_ready = true;
      }
      if (lane < ds.nr) {
        const int r = ds.r0 + lane;
        const uint32_t slot =
            smem_u32(stage_base + p.pool_off + ds.act + lane * act_stride(ds.gcnt));
        const uint16_t* src;
        if (!down) {
          const int tok = (ds.flags & kShared) ? r - d.T * d.k : s.perm_s[r];
          src = p.xi + (size_t)tok * d.H;
        } else {
          src = p.h + (size_t)r * p.hstride;
        }
        bulk_copy(slot, src + ds.g0 * kGroup, ds.gcnt * 256, &s.full[stage]);
      }
      if (++stage == nst) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp < kCW) {
    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    const int gw = warp;  // K group of the stage; both 16-row tiles
    const uint32_t stage0 = smem_u32(stage_base);
    const uint32_t w_off = g * 512 + gw * 64 + c * 16;
    // the same 16 bytes in a swizzled tile (rows g and g + 8 share the pattern)
    const uint32_t seg = (uint32_t)gw >> 1;
    const uint32_t w_off_s =
        g * 512 + seg * 128 + (((((uint32_t)(gw & 1) << 2) | c) ^ (seg | ((uint32_t)(g & 1) << 2))) << 4);
    // a stage is [tile][sub-stage][16 rows][512 B] of weights, then the
    // scales [tile][sub-stage][16 rows][8]; the activation rows are in the pool
    const int nsub = p.nsub;
    const uint32_t tstride = nsub * (kWB / 2), sstride = nsub * (kSB / 2);  // per tile
    const uint32_t s_off = nsub * kWB + g * 16 + gw * 2;
    const uint32_t pool0 = stage0 + p.pool_off;
    const uint32_t xt_off = gw * 256 + c * 16;  // + row g of the stage's rows: transposed (xi, h)
    int stage = 0;
    uint32_t phase = 0;
    int tseq = 0;  // tasks finished (the same sequence for all consumer warps)
    // above kLocalRankT tokens the consumers score experts first: the shared
    // expert's 8-row stages come one at a time until the routing is known
    if (scoring_warps(d) > kSW) score_experts(s, p, kSW + warp);
    float acc[2][4] = {};
    for (;;) {
      if (!dwait(&s.full[stage], phase, err)) break;
      const int key = s.desc[stage].flags;  // one shared-memory word per stage
      if (key & kEnd) break;
      if (key & kFirst) {
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[0][i] = acc[1][i] = 0.f;
      }
      const int gcnt = (key >> 8) & 31, nr = (key >> 13) & 15;
      const uint32_t xrow = pool0 + (((uint32_t)key >> 17) << 7) + g * act_stride(gcnt);  // row g
      // sub-stage j: K groups 8 j .. 8 j + 7 of the stage; this warp takes group 8 j + gw
#pragma unroll
      for (int j = 0; j < kMaxSub; ++j) {
        if (j >= nsub || 8 * j + gw >= gcnt) break;
        const uint32_t st = stage0 + stage * sb + j * (kWB / 2);  // + tile: this sub-stage's weights
        const uint32_t sj = stage0 + stage * sb + j * 256;  // + s_off: its scales
        const uint32_t xj = xrow + j * kXSub;  // + xt_off: its activations
        const uint32_t wo = (key & kSwz) ? w_off_s : w_off;
        uint4 wA[2], wB[2];
        float sc[2][2];  // [tile][row g / g + 8]
#pragma unroll
        for (int tl = 0; tl < 2; ++tl) {
          wA[tl] = lds128(st + tl * tstride + wo);
          wB[tl] = lds128(st + tl * tstride + wo + 8 * 512);
          if (scale_tma) {
            sc[tl][0] = bf16_bits_to_f32(lds16(sj + tl * sstride + s_off));
            sc[tl][1] = bf16_bits_to_f32(lds16(sj + tl * sstride + s_off + 8 * 16));
          } else {
            const Desc& dd = s.desc[stage];
            const uint16_t* scl = (key & kDown) ? ((key & kShared) ? p.s2_shared : p.s2_routed)
                                                : ((key & kShared) ? p.s13_shared : p.s13_routed);
            const int row = (tl ? dd.rowA1 : dd.rowA0) + g;
            const int grp = dd.g0 + 8 * j + gw;
            sc[tl][0] = bf16_bits_to_f32(__ldg(scl + (size_t)row * dd.ngroups + grp));
            sc[tl][1] = bf16_bits_to_f32(__ldg(scl + (size_t)(row + 8) * dd.ngroups + grp));
          }
        }
        // activation rows (interleaved x, or h) store chunk 4c + m of a K
        // group at 4m + c: the 4 lanes of a row read 64 contiguous bytes per
        // step (no bank conflicts)
        uint4 b[4];
        if (g < nr) {
#pragma unroll
          for (int m = 0; m < 4; ++m) b[m] = lds128(xj + xt_off + m * 64);
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) b[m] = make_uint4(0u, 0u, 0u, 0u);
        }
        // 2 tiles x 8 MMA steps, one chain per tile (the x fragments are
        // shared by both tiles)
        float t4[2][4] = {};
        stage_mma(wA[0], wB[0], b, t4[0]);
        stage_mma(wA[1], wB[1], b, t4[1]);
#pragma unroll
        for (int tl = 0; tl < 2; ++tl) {
          acc[tl][0] = fmaf(sc[tl][0], t4[tl][0], acc[tl][0]);
          acc[tl][1] = fmaf(sc[tl][0], t4[tl][1], acc[tl][1]);
          acc[tl][2] = fmaf(sc[tl][1], t4[tl][2], acc[tl][2]);
          acc[tl][3] = fmaf(sc[tl][1], t4[tl][3], acc[tl][3]);
        }
      }
      // the stage is refilled by TMA and bulk copies (async proxy) once
      // released: order this thread's generic reads of it before that
      fence_proxy_async_smem();
      if (key & kLast) {
        // end of a task: hand the partial sums to the slot's epilogue warp;
        // the stage's descriptor is copied before the stage is released
        const int b = tseq % kEW;
        const uint32_t use = (uint32_t)(tseq / kEW);
        if (!dwait(&s.slot_free[b], (use & 1u) ^ 1u, err)) break;
        if (warp == 0 && lane == 0) s.slot_desc[b] = s.desc[stage];
        s.red[b][warp * 32 + lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        s.red[b][(8 + warp) * 32 + lane] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s.empty[stage]);
          mbar_arrive(&s.slot_full[b]);
        }
        ++tseq;
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[stage]);
      }
      if (++stage == nst) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // end of work: one end marker per epilogue warp
    for (int j = 0; j < kEW; ++j) {
      const int b = (tseq + j) % kEW;
      const uint32_t use = (uint32_t)((tseq + j) / kEW);
      if (!dwait(&s.slot_free[b], (use & 1u) ^ 1u, err)) break;
      if (warp == 0 && lane == 0) s.slot_desc[b].flags = kEnd;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.slot_full[b]);
    }
  } else if (warp >= kRtr0) {
    // ---------------------------------------------------------------- router
    router_phase(s, p);
  } else {
    // ---------------------------------------------------------------- epilogue
    if (scoring_warps(d) > kRW) score_experts(s, p, kRW + (warp - kEpi0));
    const int b = warp - kEpi0;  // this warp's slot
    const int g = lane >> 2, c = lane & 3;
    int routed_down = -1;
    for (uint32_t use = 0;; ++use) {
      if (!dwait(&s.slot_full[b], use & 1u, err)) break;
      const Desc ds = s.slot_desc[b];
      if (ds.flags & kEnd) break;
      const float4* red = s.red[b];
      const bool down = (ds.flags & kDown) != 0;
      // lane L holds the fragment (rows g, g+8) x (tokens 2c, 2c+1) of both tiles
      float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 a = red[w * 32 + lane], q = red[(8 + w) * 32 + lane];
        v0.x += a.x;
        v0.y += a.y;
        v0.z += a.z;
        v0.w += a.w;
        v1.x += q.x;
        v1.y += q.y;
        v1.z += q.z;
        v1.w += q.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.slot_free[b]);  // partial sums consumed
      const float f0[4] = {v0.x, v0.y, v0.z, v0.w}, f1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = g + 8 * (q >> 1), tok = 2 * c + (q & 1);
        if (tok >= ds.nr) continue;
        const size_t orow = (size_t)(ds.r0 + tok);
        if (!down) {
          const int n = ds.tile * kTile1 + row;
          // interleaved within 8, 16-byte chunks transposed within the K group
          const int pos = (n & ~127) | (chunk_t((n >> 3) & 15) << 3) | ((n & 3) << 1) | ((n >> 2) & 1);
          p.h[orow * p.hstride + pos] = f32_to_bf16_bits(silu(f0[q]) * f1[q]);
        } else {
          uint16_t* yr = p.y + orow * d.H + ds.tile * kTile2;
          yr[row] = f32_to_bf16_bits(f0[q]);
          yr[16 + row] = f32_to_bf16_bits(f1[q]);
        }
      }
      // each lane publishes its own h / y stores before the warp's release-add
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      __syncwarp();
      int tile_last = 0;
      if (lane == 0) {
        if (!down) {
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.done1 + ds.cnt) : "memory");
        } else {
          // A shared-expert down task can finish before the routing exists;
          // then it is not a tile's last (every tile has routed down tasks,
          // and they need the routing), so it only counts itself.
          if (routed_down < 0 && mbar_try_wait(&s.route_ready, 0)) routed_down = s.meta[2];
          int old;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                       : "=r"(old)
                       : "l"(p.tile_cnt + ds.tile)
                       : "memory");
          tile_last = routed_down >= 0 && old == (cnt.sh2 + routed_down) / (d.H / kTile2) - 1;
        }
      }
      tile_last = __shfl_sync(0xffffffffu, tile_last, 0);
      if (tile_last) {
        // this task completed a channel tile: combine it for every token
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        // lane (t8, q): channels n0 + 8q .. + 7 of tokens t8, t8 + 8, ...; all
        // (k + 1) rows of a token are loaded before any is summed (the loop is
        // bound by the latency of these L2 reads), the sum in slot order as
        // everywhere
        const int n = ds.tile * kTile2 + 8 * (lane & 3);
        const uint4* yv = reinterpret_cast<const uint4*>(p.y + n);
        const size_t rs = (size_t)d.H / 8;  // 16-byte chunks per y row
        for (int tok = lane >> 2; tok < d.T; tok += 8) {
          uint4 v[kMaxTopK];
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j)
            if (j < d.k) v[j] = __ldcg(yv + (size_t)s.inv_s[tok * d.k + j] * rs);
          float a[8];
          {
            const uint4 sh = d.Is > 0 ? __ldcg(yv + (size_t)(d.T * d.k + tok) * rs) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t q4[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              a[2 * i] = __uint_as_float(q4[i] << 16);
              a[2 * i + 1] = __uint_as_float(q4[i] & 0xffff0000u);
            }
          }
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j) {
            if (j >= d.k) break;
            const float w = s.wts_s[tok * d.k + j];
            const uint32_t q4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              a[2 * i] = fmaf(w, __uint_as_float(q4[i] << 16), a[2 * i]);
              a[2 * i + 1] = fmaf(w, __uint_as_float(q4[i] & 0xffff0000u), a[2 * i + 1]);
            }
          }
          uint4 o;
          o.x = (uint32_t)f32_to_bf16_bits(a[0]) | ((uint32_t)f32_to_bf16_bits(a[1]) << 16);
          o.y = (uint32_t)f32_to_bf16_bits(a[2]) | ((uint32_t)f32_to_bf16_bits(a[3]) << 16);
          o.z = (uint32_t)f32_to_bf16_bits(a[4]) | ((uint32_t)f32_to_bf16_bits(a[5]) << 16);
          o.w = (uint32_t)f32_to_bf16_bits(a[6]) | ((uint32_t)f32_to_bf16_bits(a[7]) << 16);
          *reinterpret_cast<uint4*>(p.out + (size_t)tok * d.H + n) = o;
        }
        if (lane == 0) p.tile_cnt[ds.tile] = 0;
      }
    }
  }

  // ---- the last CTA out resets the grid's counters for the next forward
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s.flag = (atomicAdd(&p.sync[2], 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (s.flag) {
    __threadfence();
    for (int i = threadIdx.x; i < (d.E + 1) * kMaxPass; i += blockDim.x) p.done1[i] = 0;
    for (int i = threadIdx.x; i < d.H / kTile2; i += blockDim.x) p.tile_cnt[i] = 0;
    if (threadIdx.x == 0) {
      p.sync[0] = 0u;
      p.sync[1] = 0u;
      p.sync[3] = 0u;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      p.sync[2] = 0u;
    }
  }
}

}  // namespace

// Ring geometry for a batch of T tokens. A stage holds only weights and
// scales: 16 K groups (two sub-stages, 32 KB of weights) when the wide views
// exist, else 8. The activation rows of the stages in flight share one FIFO
// pool after the ring, sized for about two rows per stage (a pass holds up to
// min(T, 8) rows; at 64 tokens most passes of a routed expert hold one or
// two) and at least one full pass, two above kGateRows tokens (the shared
// expert's full passes come first there; three 32 KB stages and two passes
// beat four stages and one at 64 tokens, 748 against 760 us).
static void ring_of(int T, bool wide, int* nst, int* stage_bytes, int* nsub, int* pool_off,
                    int* pool_bytes) {
  const int rows = T < kR ? (T < 1 ? 1 : T) : kR;
  *nsub = wide ? kMaxSub : 1;
  const int gps = 8 * *nsub;
  *stage_bytes = (*nsub * (kWB + kSB) + 1023) / 1024 * 1024;
  const int maxact = (rows * act_stride(gps) + 127) & ~127;
  const int typ = ((rows < 2 ? rows : 2) * act_stride(gps) + 127) & ~127;
  const int avail = kSmemMax - kStageOff;
  int n = avail / (*stage_bytes + typ);
  if (n > kMaxS) n = kMaxS;
  // above kGateRows tokens the pool holds two full passes, so that two of the
  // shared expert's 8-row stages are in flight before the routing is known
  const int passes_in_pool = T > kGateRows ? 2 : 1;
  while (n > 1 && avail - n * *stage_bytes < passes_in_pool * maxact) --n;
  *nst = n;
  *pool_off = n * *stage_bytes;
  *pool_bytes = avail - *pool_off;
  if (*pool_bytes > (1 << 17)) *pool_bytes = 1 << 17;  // the stage key holds offsets below 128 KB
  *pool_bytes &= ~127;
}

cudaError_t decode_setup(int* ctas_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemMax);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_kernel, kThreads,
                                                       kSmemMax);
}

size_t decode_counter_ints(int E, int H) { return (size_t)(E + 1) * kMaxPass + H / kTile2 + 4; }

cudaError_t launch_decode(const Dims& d, const Routing& r, const DecodeWeights& w, const uint16_t* x,
                          uint16_t* xi, uint16_t* h, int hstride, uint16_t* y, uint16_t* out,
                          int* counters, int grid, cudaStream_t s, LaunchLog& log) {
  DecodeParams p{};
  p.d = d;
  p.r = r;
  p.x = x;
  p.router_w = w.router_w;
  p.router_bias = w.router_bias;
  p.s13_routed = w.s13_routed;
  p.s13_shared = w.s13_shared;
  p.s2_routed = w.s2_routed;
  p.s2_shared = w.s2_shared;
  p.xi = xi;
  p.h = h;
  p.hstride = hstride;
  p.y = y;
  p.out = out;
  p.done1 = counters;
  p.tile_cnt = counters + (size_t)(d.E + 1) * kMaxPass;
  p.sync = reinterpret_cast<unsigned*>(p.tile_cnt + d.H / kTile2);
  p.scale_tma = w.scale_tma;
  ring_of(d.T, w.wide != 0, &p.nst, &p.stage_bytes, &p.nsub, &p.pool_off, &p.pool_bytes);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kStageOff + p.pool_off + p.pool_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  log.begin("decode_fused", s);
  cudaError_t e =
      p.nsub == 2 ? cudaLaunchKernelEx(&cfg, decode_kernel, w.wtm13r, w.wtm13s, w.wtm2r, w.wtm2s,
                                       w.wts13r, w.wts13s, w.wts2r, w.wts2s, p)
                  : cudaLaunchKernelEx(&cfg, decode_kernel, w.tm13r, w.tm13s, w.tm2r, w.tm2s,
                                       w.ts13r, w.ts13s, w.ts2r, w.ts2s, p);
  log.end(s);
  return e;
}

}  // namespace moe

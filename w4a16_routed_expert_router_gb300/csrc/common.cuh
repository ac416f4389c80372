// Shared device-side definitions of the W4A16 MoE layer (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kGroup = 128;           // K-group of one bf16 scale
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;
constexpr uint32_t kErrTimeout = 0x1u;
constexpr uint32_t kErrRange = 0x2u;
constexpr uint32_t kErrLayout = 0x4u;

// Layer sizes as seen by every kernel.
struct Dims {
  int T;    // tokens of this forward
  int H;    // hidden
  int E;    // routed experts
  int k;    // top-k
  int I;    // routed intermediate
  int Is;   // shared intermediate (0: no shared expert)
};

// Routing results and bookkeeping written by the router kernels and read by
// the expert kernels (all in the handle's workspace).
struct Routing {
  float* logits;      // [T, E] fp32
  int* ids;           // [T, k]
  float* wts;         // [T, k]
  int* counts;        // [E]
  int* offsets;       // [E + 1] exclusive prefix of counts
  int* perm;          // [T*k] token of each expert-sorted row
  int* inv;           // [T*k] row of each (token, slot)
  int* active;        // [E + 1] active experts, ascending, shared (== E) last
  int* meta;          // [kMetaWords]: see Meta*
  int* task1;         // [E + 2] prefix of gate/up GEMV tasks per active expert
  int* task2;         // [E + 2] prefix of down GEMV tasks per active expert
  int* task3;         // [E + 2] prefix of gate/up tensor-core tasks per active expert
  int* task4;         // [E + 2] prefix of down tensor-core tasks per active expert
  uint16_t* xperm;    // [T*k + T, H] x rows in expert order (+ shared rows), interleaved
  int* blockcnt;      // [nblk, E] per-CTA expert counts (large-T routing)
  int* blockbase;     // [nblk, E] first row of each CTA's items per expert
  unsigned* tickets;  // [kTickets] last-block-done counters (self-resetting)
  unsigned* err;      // device error flag bits
};

enum Meta {
  kMetaActive = 0,
  kMetaTasks1 = 1,
  kMetaTasks2 = 2,
  kMetaTc1 = 3,
  kMetaTc2 = 4,
  kMetaWords = 8
};

// Tensor-core expert path: an N-tile holds up to kTcN rows of one expert; a
// gate/up task covers 128 gate + 128 up channels, a down task 2 x 128 output
// channels.
constexpr int kTcN = 256;
enum Ticket { kTicketRouter = 0, kTicketTopk = 1, kTickets = 4 };

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test, but the thread may be suspended (up to about a microsecond)
// until the phase completes instead of returning at once: waiting warps then
// leave the issue slots to the warps that have work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after about two seconds of
// global time, records a timeout in the device error flag and returns false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((i & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Warp-level bf16 MMA m16n8k16, fp32 accumulate: d = a * b + c.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1, const float* c) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// Two 4-bit codes -> two exact bf16 integers q = u - 8.
// Codes j and j+4 of a word (bits 4j.. and 4j+16..) are moved into the low
// mantissa bits of two bf16 values of exponent 2^7, giving 128 + u exactly
// (the bf16 spacing at 128 is 1); subtracting 136 leaves u - 8.
template <int J>
__device__ __forceinline__ uint32_t int4_pair_to_bf16x2(uint32_t word) {
  uint32_t v;
  const uint32_t w = word >> (4 * J);
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(v) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
  b = __hsub2(b, off);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Reorder 8 consecutive bf16 values (x0..x7, packed in 4 words) into the
// operand order of the GEMV MMA: (x0,x4) (x1,x5) (x2,x6) (x3,x7).
__device__ __forceinline__ uint4 interleave8(uint4 v) {
  uint4 r;
  r.x = __byte_perm(v.x, v.z, 0x5410);
  r.y = __byte_perm(v.x, v.z, 0x7632);
  r.z = __byte_perm(v.y, v.w, 0x5410);
  r.w = __byte_perm(v.y, v.w, 0x7632);
  return r;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

}  // namespace moe

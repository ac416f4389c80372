// Router of the W4A16 MoE layer: fp32 logits, sigmoid + bias top-k selection,
// renormalised combine weights, per-expert histogram, exclusive scan and the
// stable token permutation that gives every expert a contiguous row segment.
//
// "canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP", table "Component
// precisions": the router bias ffn.gate.bias is fp32, so the router runs in
// fp32 end to end. "What does everyone get wrong about optimizing DeepSeek V4
// Flash ...", section "Sparse architecture": six of 256 routed experts are
// active per token.
//
// Two paths:
//  * small T (<= kSmallT tokens): one kernel. Every CTA streams a slice of the
//    fp32 router weight (the only large read at decode sizes); the CTA that
//    finishes last (atomic ticket, no waiting) does top-k, histogram, scan,
//    placement and the expert task lists for all tokens.
//  * large T: a tiled fp32 logits kernel, a top-k kernel (warp per token, CTA
//    histograms, last CTA scans), and a placement kernel that ranks each
//    CTA's items stably with warp match/ballot.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

namespace {

// Expert kernels' task decomposition: gate/up tasks cover 16 channels of
// gate and 16 of up; down tasks cover 32 output channels; one task handles up
// to kPassRows rows of an expert's segment.
__device__ __forceinline__ int passes_for(int rows) { return (rows + kPassRows - 1) / kPassRows; }

constexpr int kPer = kMaxExperts / 32;  // logits per lane

// The logits of one token into registers: lane l takes experts l, l+32, ...
__device__ __forceinline__ void load_row(const float* logit_row, int E, int lane,
                                         float (&lg)[kPer]) {
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? __ldcg(logit_row + e) : 0.f;
  }
}

// Warp-wide top-k of one token whose logits lane l holds for experts l, l+32,
// ...: warp_topk_sorted (topk.cuh); returns in lanes 0..k-1 the chosen expert
// (descending sel, ties -> lower index) and its renormalised unbiased score.
__device__ __forceinline__ void warp_topk_regs(const float (&lg)[kPer], const float* bias, int E,
                                               int k, int lane, int* out_id, float* out_w) {
  warp_topk_sorted<kMaxTopK>(lg, bias, E, k, lane, out_id, out_w);
}

// The same, reading the token's logits from a row in memory.
__device__ __forceinline__ void warp_topk(const float* logit_row, const float* bias, int E, int k,
                                          int lane, int* out_id, float* out_w) {
  float lg[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? logit_row[e] : 0.f;
  }
  warp_topk_regs(lg, bias, E, k, lane, out_id, out_w);
}

// Exclusive scan of four values per thread across a 256-thread block;
// scratch >= 8 int4. Returns the exclusive prefix, *total the block sums.
__device__ __forceinline__ int4 block_scan4_256(int4 v, int4* scratch, int4* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  int4 base = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int4 s = scratch[w];
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
  *total = tot;
  return make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z,
                   base.w + inc.w - v.w);
}

// From final per-expert row counts (shared, [E]): offsets (exclusive scan,
// also left in offs_s), counts, the ascending list of active routed experts
// and the prefix of their expert-kernel tasks, and the meta words. One
// 256-thread block. The shared expert's tasks are not listed: the expert
// kernels put them first.
__device__ void finish_counts(const Dims& d, const int* counts_s, int* offs_s, const Routing& r,
                              int4* scratch) {
  const int e = threadIdx.x;
  const int c = (e < d.E) ? counts_s[e] : 0;
  const int p = passes_for(c);
  const int4 v = make_int4(c, c > 0 ? 1 : 0, p * (d.I / kTile1), p * (d.H / kTile2));
  int4 tot;
  const int4 ex = block_scan4_256(v, scratch, &tot);
  // tensor-core tasks: N-tiles of kTcN rows x channel tiles
  const int nt = (c + kTcN - 1) / kTcN;
  const int4 v2 = make_int4(nt * (d.I / 128), nt * (d.H / 256), 0, 0);
  __syncthreads();
  int4 tot2;
  const int4 ex2 = block_scan4_256(v2, scratch, &tot2);
  if (e < d.E) {
    offs_s[e] = ex.x;
    r.offsets[e] = ex.x;
    r.counts[e] = c;
    if (c > 0) {
      r.active[ex.y] = e;
      r.task1[ex.y] = ex.z;
      r.task2[ex.y] = ex.w;
      if (r.task3) {
        r.task3[ex.y] = ex2.x;
        r.task4[ex.y] = ex2.y;
      }
    }
  }
  if (threadIdx.x == 0) {
    r.offsets[d.E] = tot.x;
    r.task1[tot.y] = tot.z;
    r.task2[tot.y] = tot.w;
    r.meta[kMetaActive] = tot.y;
    r.meta[kMetaTasks1] = tot.z;
    r.meta[kMetaTasks2] = tot.w;
    if (r.task3) {
      r.task3[tot.y] = tot2.x;
      r.task4[tot.y] = tot2.y;
    }
    r.meta[kMetaTc1] = tot2.x;
    r.meta[kMetaTc2] = tot2.y;
  }
  __syncthreads();
}

}  // namespace

// ----------------------------------------------------------------- small T
// grid: ceil(E / 2) CTAs x 256 threads. Warps 0-3 score expert 2b, warps 4-7
// expert 2b+1, each warp a quarter of H. Requires T <= kSmallT, H % 512 == 0.
__global__ void __launch_bounds__(256, 1) route_small_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ router_w,
                                                          const float* __restrict__ bias, Dims d,
                                                          Routing r) {
  __shared__ float part[8][kSmallT];
  __shared__ int ids_s[kSmallT * kMaxTopK];
  __shared__ int counts_s[kMaxExperts];
  __shared__ int offs_s[kMaxExperts];
  __shared__ int4 scratch[8];
  __shared__ float lbuf[8][kMaxExperts];
  __shared__ unsigned last;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 2 + (warp >> 2);
  const int q = warp & 3;
  const int kq = d.H / 4;  // K range of one warp

  // let the expert kernel start its shared-expert work right away
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (e < d.E) {
    const float4* wrow = reinterpret_cast<const float4*>(router_w + (size_t)e * d.H + q * kq);
    const int nf = kq / 4;  // float4 per warp
    for (int t = 0; t < d.T; ++t) {
      const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)t * d.H + q * kq);
      float acc = 0.f;
      for (int f0 = 0; f0 < nf; f0 += 32 * 8) {
        float4 wv[8];
        uint2 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int f = f0 + u * 32 + lane;
          if (f < nf) {
            wv[u] = __ldg(wrow + f);
            xv[u] = __ldg(xr + f);
          } else {
            wv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            xv[u] = make_uint2(0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc = fmaf(__uint_as_float(xv[u].x << 16), wv[u].x, acc);
          acc = fmaf(__uint_as_float(xv[u].x & 0xffff0000u), wv[u].y, acc);
          acc = fmaf(__uint_as_float(xv[u].y << 16), wv[u].z, acc);
          acc = fmaf(__uint_as_float(xv[u].y & 0xffff0000u), wv[u].w, acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) part[warp][t] = acc;
    }
  }
  __syncthreads();
  if (threadIdx.x < 2 * d.T) {
    const int sub = threadIdx.x / d.T, t = threadIdx.x % d.T;
    const int ee = blockIdx.x * 2 + sub;
    if (ee < d.E) {
      const float v = ((part[4 * sub][t] + part[4 * sub + 1][t]) + part[4 * sub + 2][t]) +
                      part[4 * sub + 3][t];
      r.logits[(size_t)t * d.E + ee] = v;
    }
  }

  // ---- the last CTA to finish finishes the routing of all tokens
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = (atomicAdd(&r.tickets[kTicketRouter], 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  if (threadIdx.x < kMaxExperts) counts_s[threadIdx.x] = 0;
  __syncthreads();
  for (int t = warp; t < d.T; t += 8) {
    const float* lrow = r.logits + (size_t)t * d.E;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int ee = lane + 32 * i;
      if (ee < d.E) lbuf[warp][ee] = __ldcg(lrow + ee);
    }
    __syncwarp();
    int id;
    float w;
    warp_topk(lbuf[warp], bias, d.E, d.k, lane, &id, &w);
    __syncwarp();
    if (lane < d.k) {
      if (id < 0 || id >= d.E) {
        atomicOr(r.err, kErrRange);
        id = 0;
      }
      r.ids[t * d.k + lane] = id;
      r.wts[t * d.k + lane] = w;
      ids_s[t * d.k + lane] = id;
      atomicAdd(&counts_s[id], 1);
    }
  }
  __syncthreads();
  finish_counts(d, counts_s, offs_s, r, scratch);
  // stable placement: rank of item i among earlier items of the same expert
  const int n = d.T * d.k;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int ei = ids_s[i];
    int rank = 0;
    for (int j = 0; j < i; ++j) rank += (ids_s[j] == ei);
    const int pos = offs_s[ei] + rank;
    r.perm[pos] = i / d.k;
    r.inv[i] = pos;
  }
  if (threadIdx.x == 0) r.tickets[kTicketRouter] = 0u;
}

// ----------------------------------------------------------------- large T
// logits[T, E] = x[T, H] . Wr[E, H]^T in fp32: 64x64 tiles, K chunks of 32,
// 4x4 outputs per thread.
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ router_w,
                                                            Dims d, Routing r) {
  __shared__ float xs[32][64 + 4];
  __shared__ float ws[32][64 + 4];
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  float acc[4][4] = {};
  for (int k0 = 0; k0 < d.H; k0 += 32) {
    // load 64 tokens x 32 k of x (bf16 -> f32) and 64 experts x 32 k of Wr
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int row = i >> 5, kk = i & 31;
      const int t = t0 + row, ee = e0 + row;
      xs[kk][row] = (t < d.T) ? bf16_bits_to_f32(x[(size_t)t * d.H + k0 + kk]) : 0.f;
      ws[kk][row] = (ee < d.E) ? router_w[(size_t)ee * d.H + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = xs[kk][ty * 4 + i];
        b[i] = ws[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= d.T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ee = e0 + tx * 4 + j;
      if (ee < d.E) r.logits[(size_t)t * d.E + ee] = acc[i][j];
    }
  }
}

// Top-k for kTopkTokens tokens per CTA (8 warps), CTA expert histogram; the
// last CTA computes counts, offsets, each CTA's first row per expert and the
// task lists.
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ bias, Dims d,
                                                          Routing r) {
  __shared__ int hist[kMaxExperts];
  __shared__ int counts_s[kMaxExperts];
  __shared__ int offs_s[kMaxExperts];
  __shared__ float bias_s[kMaxExperts];
  __shared__ int4 scratch[8];
  __shared__ unsigned last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kMaxExperts; i += blockDim.x) {
    hist[i] = 0;
    bias_s[i] = i < d.E ? bias[i] : 0.f;
  }
  __syncthreads();
  // each warp ranks every 8th token of the CTA's range; the next token's
  // logits are in flight while this one is ranked
  const int t0 = blockIdx.x * kTopkTokens, t1 = min(d.T, t0 + kTopkTokens);
  float nx[kPer];
  if (t0 + warp < t1) load_row(r.logits + (size_t)(t0 + warp) * d.E, d.E, lane, nx);
  for (int t = t0 + warp; t < t1; t += 8) {
    float lg[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) lg[i] = nx[i];
    if (t + 8 < t1) load_row(r.logits + (size_t)(t + 8) * d.E, d.E, lane, nx);
    int id;
    float w;
    warp_topk_regs(lg, bias_s, d.E, d.k, lane, &id, &w);
    if (lane < d.k) {
      if (id < 0 || id >= d.E) {
        atomicOr(r.err, kErrRange);
        id = 0;
      }
      r.ids[t * d.k + lane] = id;
      r.wts[t * d.k + lane] = w;
      atomicAdd(&hist[id], 1);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < d.E; i += blockDim.x)
    r.blockcnt[(size_t)blockIdx.x * d.E + i] = hist[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = (atomicAdd(&r.tickets[kTicketTopk], 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int nblk = gridDim.x;
  const int e = threadIdx.x;
  // the per-CTA counts, 8 loads in flight at a time
  int c = 0;
  if (e < d.E) {
    int b = 0;
    for (; b + 8 <= nblk; b += 8) {
      int v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = __ldcg(r.blockcnt + (size_t)(b + q) * d.E + e);
#pragma unroll
      for (int q = 0; q < 8; ++q) c += v[q];
    }
    for (; b < nblk; ++b) c += __ldcg(r.blockcnt + (size_t)b * d.E + e);
  }
  if (e < kMaxExperts) counts_s[e] = c;
  __syncthreads();
  finish_counts(d, counts_s, offs_s, r, scratch);
  if (e < d.E) {
    int run = offs_s[e];
    int b = 0;
    for (; b + 8 <= nblk; b += 8) {
      int v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = __ldcg(r.blockcnt + (size_t)(b + q) * d.E + e);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        r.blockbase[(size_t)(b + q) * d.E + e] = run;
        run += v[q];
      }
    }
    for (; b < nblk; ++b) {
      r.blockbase[(size_t)b * d.E + e] = run;
      run += __ldcg(r.blockcnt + (size_t)b * d.E + e);
    }
  }
  if (threadIdx.x == 0) r.tickets[kTicketTopk] = 0u;
}

// Stable placement of one CTA's items (tokens [t0, t0 + kTopkTokens), items in
// (token, slot) order). Items are ranked chunk by chunk: within a warp by
// __match_any_sync, across warps by a per-warp count table.
__global__ void __launch_bounds__(256) route_place_kernel(const uint16_t* __restrict__ x, Dims d,
                                                          Routing r) {
  __shared__ int run[kMaxExperts];
  __shared__ int wcnt[8][kMaxExperts];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < d.E; i += blockDim.x)
    run[i] = r.blockbase[(size_t)blockIdx.x * d.E + i];
  for (int i = threadIdx.x; i < 8 * kMaxExperts; i += blockDim.x) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const int i0 = blockIdx.x * kTopkTokens * d.k;
  const int i1 = min(d.T, (blockIdx.x + 1) * kTopkTokens) * d.k;
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = i0; c0 < i1; c0 += 256) {
    const int i = c0 + threadIdx.x;
    const bool valid = i < i1;
    int e = valid ? r.ids[i] : -1;
    if (valid && (e < 0 || e >= d.E)) {
      atomicOr(r.err, kErrRange);
      e = 0;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    if (valid && rank == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int pos = run[e] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w][e];
      r.perm[pos] = i / d.k;
      r.inv[i] = pos;
    }
    __syncthreads();
    for (int ee = threadIdx.x; ee < d.E; ee += blockDim.x) {
      int s = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        s += wcnt[w][ee];
        wcnt[w][ee] = 0;
      }
      run[ee] += s;
    }
    __syncthreads();
  }
  if (r.xperm) {
    // the tensor-core operand: x[t] in the interleaved order at each of its
    // k expert-sorted rows and at its shared-expert row T*k + t (one warp per
    // token, each 16-byte chunk read once and written k + 1 times)
    const int h8 = d.H / 8;
    const int tend = min(d.T, (blockIdx.x + 1) * kTopkTokens);
    for (int t = blockIdx.x * kTopkTokens + warp; t < tend; t += 8) {
      // lane j < k holds the row of slot j, lane k the shared row
      int myrow = 0;
      if (lane < d.k) myrow = r.inv[t * d.k + lane];
      else if (lane == d.k) myrow = d.T * d.k + t;
      const int nd = d.k + (d.Is > 0 ? 1 : 0);
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d.H);
      for (int c0 = 0; c0 < h8; c0 += 4 * 32) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u * 32 + lane;
          if (c < h8) v[u] = interleave8(__ldg(src + c));
        }
        for (int j = 0; j < nd; ++j) {
          uint4* dst = reinterpret_cast<uint4*>(r.xperm + (size_t)__shfl_sync(0xffffffffu, myrow, j) * d.H);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < h8) dst[c] = v[u];
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ launcher
cudaError_t launch_route(const Dims& d, const Routing& r, const uint16_t* x, const float* router_w,
                         const float* bias, cudaStream_t s, LaunchLog& log, bool logits_ready) {
  if (d.T <= kSmallT && !r.xperm) {
    log.begin("route_small", s);
    route_small_kernel<<<(d.E + 1) / 2, 256, 0, s>>>(x, router_w, bias, d, r);
    log.end(s);
    return cudaGetLastError();
  }
  const int nblk = (d.T + kTopkTokens - 1) / kTopkTokens;
  if (!logits_ready) {
    log.begin("router_logits", s);
    router_logits_kernel<<<dim3((d.T + 63) / 64, (d.E + 63) / 64), 256, 0, s>>>(x, router_w, d, r);
    log.end(s);
  }
  log.begin("router_topk", s);
  router_topk_kernel<<<nblk, 256, 0, s>>>(bias, d, r);
  log.end(s);
  log.begin("route_place", s);
  route_place_kernel<<<nblk, 256, 0, s>>>(x, d, r);
  log.end(s);
  return cudaGetLastError();
}

}  // namespace moe

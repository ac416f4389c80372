// Internal interface between the C-ABI layer and the kernel translation units.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kSmallT = 64;       // <= this many tokens: single-kernel router
constexpr int kTopkTokens = 64;   // tokens per CTA in the large-T router
constexpr int kPassRows = 8;      // expert rows per GEMV task (one 8-column MMA block)
constexpr int kTile1 = 16;        // gate (and up) channels per gate/up GEMV task
constexpr int kTile2 = 32;        // output channels per down GEMV task
constexpr int kGemvStages = 6;    // TMA pipeline depth of the GEMV kernels
constexpr int kGemvThreads = 288; // 8 consumer warps + 1 TMA producer warp

// Records the kernels one forward launches (and their CUDA events when
// profiling is on).
struct LaunchLog {
  static constexpr int kMax = 16;
  int n = 0;
  const char* names[kMax];
  cudaEvent_t* events = nullptr;  // 2 * kMax events, or null
  void begin(const char* name, cudaStream_t s) {
    if (n < kMax) {
      names[n] = name;
      if (events) cudaEventRecord(events[2 * n], s);
    }
  }
  void end(cudaStream_t s) {
    if (n < kMax) {
      if (events) cudaEventRecord(events[2 * n + 1], s);
      ++n;
    }
  }
};

// Expert weights of one GEMV pass (gate/up or down).
struct GemvWeights {
  const uint16_t* scale_routed;
  const uint16_t* scale_shared;
  CUtensorMap tm_routed;   // packed INT4 weights, 3-D view (see encode_int4_map)
  CUtensorMap tm_shared;
  CUtensorMap ts_routed;   // bf16 group scales, 2-D view, when scale_tma
  CUtensorMap ts_shared;
  int scale_tma;           // K / 128 is a multiple of 8: scales ride in the TMA stage
};

// logits_ready: r.logits already holds this batch's logits (tensor-core router)
cudaError_t launch_route(const Dims& d, const Routing& r, const uint16_t* x, const float* router_w,
                         const float* bias, cudaStream_t s, LaunchLog& log,
                         bool logits_ready = false);
// Router logits for large batches on the tensor cores: splits router_w into
// three bf16 planes [3, E, H] (planes) and multiplies them with x. xmap: 2-D
// bf16 view {H, T} of x, wmap: {H, 3E} of planes, both box {64, 128} with
// 128-byte swizzle.
cudaError_t router_tc_setup();
cudaError_t launch_router_logits_tc(const Dims& d, const float* router_w, uint16_t* planes,
                                    const CUtensorMap& xmap, const CUtensorMap& wmap, float* logits,
                                    unsigned* err, cudaStream_t s, LaunchLog& log);

cudaError_t gemv_setup(int* ctas_per_sm);
cudaError_t launch_gemv_gate_up(const Dims& d, const Routing& r, const GemvWeights& w,
                                const uint16_t* x, uint16_t* h, int hstride, int grid,
                                cudaStream_t s, LaunchLog& log);
// out != nullptr: fuse the combine (small batches); else only y is written.
cudaError_t launch_gemv_down(const Dims& d, const Routing& r, const GemvWeights& w,
                             const uint16_t* h, int hstride, float* y, uint16_t* out,
                             int* tile_cnt, int grid, cudaStream_t s, LaunchLog& log);
// Decode-sized forward (T <= kSmallT) as one cooperative persistent kernel.
struct DecodeWeights {
  const float* router_w;
  const float* router_bias;
  const uint16_t* s13_routed;
  const uint16_t* s13_shared;
  const uint16_t* s2_routed;
  const uint16_t* s2_shared;
  // views of the packed weights, 8 K-groups of 16 rows per box: 3-D
  // {32 words, K/256, rows} with the 128-byte swizzle when K % 256 == 0, else
  // 2-D {K/8 words, rows}
  CUtensorMap tm13r, tm13s, tm2r, tm2s;
  // 2-D views of the scales {K/128, rows}, box {8, 16} (when scale_tma)
  CUtensorMap ts13r, ts13s, ts2r, ts2s;
  int scale_tma;
  // wide views (when every K is a multiple of 1024): one box brings 16
  // K-groups of both 16-row tiles, one more their scales
  CUtensorMap wtm13r, wtm13s, wtm2r, wtm2s, wts13r, wts13s, wts2r, wts2s;
  int wide;
};
cudaError_t decode_setup(int* ctas_per_sm);
size_t decode_counter_ints(int E, int H);
// xi: [T, H] bf16 scratch, x interleaved with its 16-byte chunks transposed
// within each K group, written by the kernel itself.
cudaError_t launch_decode(const Dims& d, const Routing& r, const DecodeWeights& w, const uint16_t* x,
                          uint16_t* xi, uint16_t* h, int hstride, uint16_t* y, uint16_t* out,
                          int* counters, int grid, cudaStream_t s, LaunchLog& log);

// Tensor-core (tcgen05) expert GEMMs for large batches.
struct TcWeights {
  const uint16_t* scale_routed;  // bf16 group scales [rows, K/128]
  const uint16_t* scale_shared;
  // 2-D views {K/8 words, rows} of the packed weights, box {8 words, 128 rows},
  // 32-byte swizzle
  CUtensorMap wq_r, wq_s;
};
cudaError_t tc_setup(int* ctas_per_sm);
// gate/up + SwiGLU: xmap is a 2-D bf16 view {H, rows} of Routing::xperm with
// box {64, 64} and 128-byte swizzle; writes h rows (interleaved order)
cudaError_t launch_tc_gate_up(const Dims& d, const Routing& r, const TcWeights& w,
                              const CUtensorMap& xmap, uint16_t* h, int hstride, int grid,
                              cudaStream_t s, LaunchLog& log);
// down: hmap is the same kind of view {hstride, rows} of h; writes y rows in bf16
cudaError_t launch_tc_down(const Dims& d, const Routing& r, const TcWeights& w,
                           const CUtensorMap& hmap, uint16_t* y, int grid, cudaStream_t s,
                           LaunchLog& log);

// W4A8-FP8 experts (csrc/w4a8.cu): x quantised to e4m3 per token per 128
// (xc, xs), gate/up + SwiGLU into fp32 h (hf [rows, hst]), h quantised (hc,
// hs), down into fp32 y [rows, H]; the tasks are the GEMV engine's (task1 /
// task2 of the routing). The combine follows (launch_combine, fp32 y).
struct W4a8Weights {
  const uint32_t* w13_q;
  const uint16_t* w13_s;
  const uint32_t* w2_q;
  const uint16_t* w2_s;
  const uint32_t* sh_w13_q;
  const uint16_t* sh_w13_s;
  const uint32_t* sh_w2_q;
  const uint16_t* sh_w2_s;
};
cudaError_t launch_w4a8_experts(const Dims& d, const Routing& r, const W4a8Weights& w,
                                const uint16_t* x, uint8_t* xc, float* xs, float* hf, uint8_t* hc,
                                float* hs, int hst, float* y, int grid, cudaStream_t s,
                                LaunchLog& log);

// y fp32 (the GEMV engine's) or bf16 (the tensor-core engine's)
cudaError_t launch_combine(const Dims& d, const Routing& r, const float* y, uint16_t* out,
                           cudaStream_t s, LaunchLog& log);
cudaError_t launch_combine(const Dims& d, const Routing& r, const uint16_t* y, uint16_t* out,
                           cudaStream_t s, LaunchLog& log);

}  // namespace moe

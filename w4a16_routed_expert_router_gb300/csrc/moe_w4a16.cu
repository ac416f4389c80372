// C ABI of the W4A16 MoE layer: argument validation, workspace, tensor maps,
// dispatch of the router / expert / combine kernels.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/moe_w4a16.h"
#include "kernels.h"

using namespace moe;

struct moe_w4a16_handle {
  moe_w4a16_config cfg;
  int device = 0;
  int num_sms = 0;
  int gemv_grid = 0;
  int decode_grid = 0;
  int tc_grid = 0;
  bool tc_ok = false;           // shapes the tensor-core experts support
  int* counters = nullptr;      // decode kernel completion counters (self-resetting)
  void* ws = nullptr;
  size_t ws_bytes = 0;
  Routing r{};
  int* tile_cnt = nullptr;      // [H / 32] combine tickets of the down kernel
  uint16_t* h = nullptr;
  int hstride = 0;
  float* y = nullptr;
  uint16_t* x_dev = nullptr;    // forward_host staging
  uint16_t* out_dev = nullptr;
  int last_T = 0;
  // forward_host with pinned buffers replays one CUDA graph (copy in, forward,
  // copy out), recorded for these buffers, this token count and these weights
  cudaStream_t capture_stream = nullptr;
  cudaGraphExec_t host_graph = nullptr;
  const void* hg_x = nullptr;
  const void* hg_out = nullptr;
  int hg_T = -1;
  moe_w4a16_weights hg_w{};
  LaunchLog log;
  cudaEvent_t events[2 * LaunchLog::kMax];
  bool events_made = false;
  // tensor-map cache keyed by the tensor pointers it was encoded for:
  // 0 w13_q, 1 w2_q, 2 sh_w13_q, 3 sh_w2_q (3-D, 1-group boxes), 4 w13_s, 5 w2_s,
  // 6 sh_w13_s, 7 sh_w2_s (scales) of the GEMV engine, 12..15 the weights in
  // 128-row boxes (tensor-core experts); 8..11 unused
  static constexpr int kMaps = 16;
  const void* map_keys[kMaps] = {};
  CUtensorMap maps[kMaps];
  // tensor maps of the decode kernel, encoded for the weight pointers in
  // dec_key (see encode_decode_maps)
  moe_w4a16_weights dec_key{};
  bool dec_ready = false;
  DecodeWeights dec{};
  // views of the workspace's activation operands for the tensor-core experts
  CUtensorMap xmap, hmap;
  // tensor-core router: bf16 planes of router_w and the view of this call's x
  uint16_t* planes = nullptr;
  CUtensorMap wmap_router, xmap_router;
  const void* xmap_key = nullptr;
  int xmap_rows = 0;
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Page-locked (or registered) host memory: copies from it can be captured.
bool is_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int validate_config(const moe_w4a16_config* c) {
  if (!c) return MOE_W4A16_ERR_INVALID_ARG;
  if (c->flags & ~(MOE_W4A16_FLAG_FORCE_GEMV | MOE_W4A16_FLAG_FORCE_TC | MOE_W4A16_FLAG_PROFILE |
                   MOE_W4A16_FLAG_W4A8))
    return MOE_W4A16_ERR_INVALID_ARG;
  if ((c->flags & MOE_W4A16_FLAG_FORCE_GEMV) && (c->flags & MOE_W4A16_FLAG_FORCE_TC))
    return MOE_W4A16_ERR_INVALID_ARG;
  if ((c->flags & MOE_W4A16_FLAG_W4A8) &&
      (c->flags & (MOE_W4A16_FLAG_FORCE_GEMV | MOE_W4A16_FLAG_FORCE_TC)))
    return MOE_W4A16_ERR_INVALID_ARG;
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) return MOE_W4A16_ERR_INVALID_ARG;
  if (c->group_size != kGroup) return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden < 128 || c->hidden > 16384 || c->hidden % 128) return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  if (c->inter < 128 || c->inter > 16384 || c->inter % 128) return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  if (c->shared_inter < 0 || c->shared_inter > 16384 || c->shared_inter % 128)
    return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  if (c->num_experts < 1 || c->num_experts > kMaxExperts) return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  // W4A8 experts keep fp32 h in the y buffer: h is at most H wide
  if ((c->flags & MOE_W4A16_FLAG_W4A8) && (c->inter > c->hidden || c->shared_inter > c->hidden))
    return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  if (c->top_k < 1 || c->top_k > kMaxTopK || c->top_k > c->num_experts)
    return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  // row counts of the stacked expert tensors must fit the int32 row indices
  if ((long long)c->num_experts * 2 * c->inter >= (1LL << 31) ||
      (long long)c->num_experts * c->hidden >= (1LL << 31))
    return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  return MOE_W4A16_OK;
}

struct Layout {
  size_t off[32];
  size_t total;
};

// Workspace carve-up; the order is the order of the fields filled in create().
Layout plan(const moe_w4a16_config& c) {
  const size_t Tm = c.max_tokens, E = c.num_experts, k = c.top_k, H = c.hidden;
  const size_t rows = Tm * k + Tm;
  const size_t hstride = c.inter > c.shared_inter ? c.inter : c.shared_inter;
  const size_t nblk = (Tm + kTopkTokens - 1) / kTopkTokens;
  const size_t sizes[] = {
      Tm * E * 4,            // 0 logits
      Tm * k * 4,            // 1 ids
      Tm * k * 4,            // 2 wts
      E * 4,                 // 3 counts
      (E + 1) * 4,           // 4 offsets
      (E + 1) * 4,           // 5 active
      kMetaWords * 4,        // 6 meta
      (E + 2) * 4,           // 7 task1
      (E + 2) * 4,           // 8 task2
      Tm * k * 4,            // 9 perm
      Tm * k * 4,            // 10 inv
      nblk * E * 4,          // 11 blockcnt
      nblk * E * 4,          // 12 blockbase
      kTickets * 4,          // 13 tickets
      4,                     // 14 err
      (size_t)H / 32 * 4,    // 15 tile_cnt
      rows * hstride * 2,    // 16 h
      rows * H * 4,          // 17 y
      Tm * H * 2,            // 18 x_dev
      Tm * H * 2,            // 19 out_dev
      decode_counter_ints(c.num_experts, c.hidden) * 4,  // 20 decode counters
      rows * H * 2,          // 21 xperm
      (E + 2) * 4,           // 22 task3
      (E + 2) * 4,           // 23 task4
      3 * E * H * 2,         // 24 router planes
  };
  Layout L;
  size_t o = 0;
  for (size_t i = 0; i < sizeof(sizes) / sizeof(sizes[0]); ++i) {
    L.off[i] = o;
    o += align256(sizes[i]);
  }
  L.total = o;
  return L;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_W4A16_OK;
  fprintf(stderr, "moe_w4a16: CUDA error %s\n", cudaGetErrorString(e));
  return MOE_W4A16_ERR_CUDA;
}

// 3-D view {16 words of one K-group, K-groups, rows} of a packed INT4 tensor
// [rows, K/8] uint32, box {16, 1, 16}: one 128-wide K-group of 16 rows.
int encode_int4_map(CUtensorMap* m, const void* base, long long rows, int K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_W4A16_ERR_CUDA;
  cuuint64_t dims[3] = {16, (cuuint64_t)(K / kGroup), (cuuint64_t)rows};
  cuuint64_t strides[2] = {64, (cuuint64_t)K / 2};  // bytes: group, row
  cuuint32_t box[3] = {16, 1, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "moe_w4a16: cuTensorMapEncodeTiled failed (%d)\n", (int)r);
    return MOE_W4A16_ERR_CUDA;
  }
  return MOE_W4A16_OK;
}

// 2-D view {K/128 groups, rows} of bf16 group scales [rows, K/128], box
// {8, 16}: 8 groups of 16 rows. Needs K/128 to be a multiple of 8 (16-byte
// row stride).
int encode_scale_map(CUtensorMap* m, const void* base, long long rows, int K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_W4A16_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)(K / kGroup), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K / kGroup) * 2};
  cuuint32_t box[2] = {8, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "moe_w4a16: cuTensorMapEncodeTiled (scales) failed (%d)\n", (int)r);
    return MOE_W4A16_ERR_CUDA;
  }
  return MOE_W4A16_OK;
}

int encode_2d(CUtensorMap* m, CUtensorMapDataType type, int esize, const void* base,
              long long cols, long long rows, int box0, int box1, CUtensorMapSwizzle swz,
              CUtensorMapL2promotion l2, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_W4A16_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
  cuuint32_t box[2] = {(cuuint32_t)box0, (cuuint32_t)box1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "moe_w4a16: cuTensorMapEncodeTiled (%s) failed (%d)\n", what, (int)r);
    return MOE_W4A16_ERR_CUDA;
  }
  return MOE_W4A16_OK;
}

int encode_nd(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
              const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
              CUtensorMapSwizzle swz, CUtensorMapL2promotion l2, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_W4A16_ERR_CUDA;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, type, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (what) fprintf(stderr, "moe_w4a16: cuTensorMapEncodeTiled (%s) failed (%d)\n", what, (int)r);
    return MOE_W4A16_ERR_CUDA;
  }
  return MOE_W4A16_OK;
}

// Decode-kernel views: one box per stage brings both 16-row weight tiles of a
// task (8 K-groups each), one more their group scales.
//  gate/up, w13 [E', 2I', K/8] (K = H; E' = E, or 1 for the shared expert):
//    K % 256 == 0: {32 words, K/256 segments, I' rows, 2E' halves}, box
//                  {32, 4, 16, 2}, 128-byte swizzle
//    otherwise:    {K/8 words, I' rows, 2E' halves}, box {128, 16, 2}
//    scales [E', 2I', K/128]: {K/128, I', 2E'}, box {8, 16, 2}
//  down, w2 [E'H rows, K/8] (K = I'):
//    K % 256 == 0: {32 words, K/256 segments, rows}, box {32, 4, 32},
//                  128-byte swizzle
//    otherwise:    {K/8 words, rows}, box {128, 32}
//    scales [rows, K/128]: {K/128, rows}, box {8, 32}
// The scale views need K/128 to be a multiple of 8 (16-byte row stride); the
// caller only encodes them then.
int encode_decode_w13(CUtensorMap* m, const void* base, int halves, int inter, int K) {
  if (K % 256 == 0) {
    const cuuint64_t dims[4] = {32, (cuuint64_t)(K / 256), (cuuint64_t)inter, (cuuint64_t)halves};
    const cuuint64_t str[3] = {128, (cuuint64_t)K / 2, (cuuint64_t)inter * (K / 2)};
    const cuuint32_t box[4] = {32, 4, 16, 2};
    return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, base, dims, str, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "decode w13");
  }
  const cuuint64_t dims[3] = {(cuuint64_t)(K / 8), (cuuint64_t)inter, (cuuint64_t)halves};
  const cuuint64_t str[2] = {(cuuint64_t)K / 2, (cuuint64_t)inter * (K / 2)};
  const cuuint32_t box[3] = {128, 16, 2};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "decode w13");
}
int encode_decode_w2(CUtensorMap* m, const void* base, long long rows, int K) {
  if (K % 256 == 0) {
    const cuuint64_t dims[3] = {32, (cuuint64_t)(K / 256), (cuuint64_t)rows};
    const cuuint64_t str[2] = {128, (cuuint64_t)K / 2};
    const cuuint32_t box[3] = {32, 4, 32};
    return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, base, dims, str, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "decode w2");
  }
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)K / 2};
  const cuuint32_t box[2] = {128, 32};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "decode w2");
}
int encode_decode_s13(CUtensorMap* m, const void* base, int halves, int inter, int K) {
  const cuuint64_t dims[3] = {(cuuint64_t)(K / kGroup), (cuuint64_t)inter, (cuuint64_t)halves};
  const cuuint64_t str[2] = {(cuuint64_t)(K / kGroup) * 2, (cuuint64_t)inter * (K / kGroup) * 2};
  const cuuint32_t box[3] = {8, 16, 2};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "decode w13 scales");
}
int encode_decode_s2(CUtensorMap* m, const void* base, long long rows, int K) {
  const cuuint64_t dims[2] = {(cuuint64_t)(K / kGroup), (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)(K / kGroup) * 2};
  const cuuint32_t box[2] = {8, 32};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "decode w2 scales");
}

// Wide decode views (every K a multiple of 1024): a stage of 16 K-groups in
// one box, laid out as [tile][half of the 16 groups][16 rows][512 B], each
// 8 KB block with the 128-byte swizzle of the narrow views. The group-half
// dimension (stride 512 B) sits between the rows and the tiles, so the rows
// of a block stay 512 bytes apart.
//  gate/up: {32 words, 4 segments, I' rows, K/1024, 2E' halves}, box {32, 4, 16, 2, 2}
//  down:    {32 words, 4 segments, 16 rows, K/1024, E'H/16 tiles}, box {32, 4, 16, 2, 2}
//  scales:  {8 groups, I' rows, K/1024, 2E' halves}, box {8, 16, 2, 2};
//           {8 groups, 16 rows, K/1024, E'H/16 tiles}, box {8, 16, 2, 2}: laid out
//           [tile][half of the 16 groups][16 rows][8] like the weights, rows
//           16 bytes apart as in the narrow views (conflict-free reads)
// An encode the driver refuses leaves the caller on the narrow views.
int encode_decode_w13_wide(CUtensorMap* m, const void* base, int halves, int inter, int K) {
  const cuuint64_t dims[5] = {32, 4, (cuuint64_t)inter, (cuuint64_t)(K / 1024), (cuuint64_t)halves};
  const cuuint64_t str[4] = {128, (cuuint64_t)K / 2, 512, (cuuint64_t)inter * (K / 2)};
  const cuuint32_t box[5] = {32, 4, 16, 2, 2};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, nullptr);
}
int encode_decode_w2_wide(CUtensorMap* m, const void* base, long long rows, int K) {
  const cuuint64_t dims[5] = {32, 4, 16, (cuuint64_t)(K / 1024), (cuuint64_t)(rows / 16)};
  const cuuint64_t str[4] = {128, (cuuint64_t)K / 2, 512, (cuuint64_t)16 * (K / 2)};
  const cuuint32_t box[5] = {32, 4, 16, 2, 2};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, nullptr);
}
int encode_decode_s13_wide(CUtensorMap* m, const void* base, int halves, int inter, int K) {
  const cuuint64_t ng = (cuuint64_t)(K / kGroup);
  const cuuint64_t dims[4] = {8, (cuuint64_t)inter, (cuuint64_t)(K / 1024), (cuuint64_t)halves};
  const cuuint64_t str[3] = {ng * 2, 16, (cuuint64_t)inter * ng * 2};
  const cuuint32_t box[4] = {8, 16, 2, 2};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, nullptr);
}
int encode_decode_s2_wide(CUtensorMap* m, const void* base, long long rows, int K) {
  const cuuint64_t ng = (cuuint64_t)(K / kGroup);
  const cuuint64_t dims[4] = {8, 16, (cuuint64_t)(K / 1024), (cuuint64_t)(rows / 16)};
  const cuuint64_t str[3] = {ng * 2, 16, 16 * ng * 2};
  const cuuint32_t box[4] = {8, 16, 2, 2};
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, base, dims, str, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, nullptr);
}

// Scales ride in the decode kernel's TMA stages when every K has a multiple
// of 8 groups (16-byte rows of scales); otherwise the consumers read them.
bool decode_scale_tma(const moe_w4a16_config& c) {
  return (c.hidden / kGroup) % 8 == 0 && (c.inter / kGroup) % 8 == 0 &&
         (c.shared_inter == 0 || (c.shared_inter / kGroup) % 8 == 0);
}

// Every input of the decode kernel that depends on the weights only.
int encode_decode_maps(DecodeWeights* dw, const moe_w4a16_config& c, const moe_w4a16_weights* w) {
  const bool has_sh = c.shared_inter > 0;
  const bool scale_tma = decode_scale_tma(c);
  const long long r2 = (long long)c.num_experts * c.hidden;
  int st;
  dw->router_w = w->router_w;
  dw->router_bias = w->router_bias;
  dw->s13_routed = w->w13_s;
  dw->s13_shared = has_sh ? w->sh_w13_s : w->w13_s;
  dw->s2_routed = w->w2_s;
  dw->s2_shared = has_sh ? w->sh_w2_s : w->w2_s;
  dw->scale_tma = scale_tma;
  if ((st = encode_decode_w13(&dw->tm13r, w->w13_q, 2 * c.num_experts, c.inter, c.hidden)) != MOE_W4A16_OK ||
      (st = encode_decode_w2(&dw->tm2r, w->w2_q, r2, c.inter)) != MOE_W4A16_OK)
    return st;
  dw->tm13s = dw->tm13r;
  dw->tm2s = dw->tm2r;
  if (has_sh && ((st = encode_decode_w13(&dw->tm13s, w->sh_w13_q, 2, c.shared_inter, c.hidden)) != MOE_W4A16_OK ||
                 (st = encode_decode_w2(&dw->tm2s, w->sh_w2_q, c.hidden, c.shared_inter)) != MOE_W4A16_OK))
    return st;
  // without TMA-borne scales the scale maps are never used: copies of the
  // weight maps keep the parameter block defined
  dw->ts13r = dw->tm13r;
  dw->ts2r = dw->tm2r;
  dw->ts13s = dw->tm13s;
  dw->ts2s = dw->tm2s;
  if (scale_tma) {
    if ((st = encode_decode_s13(&dw->ts13r, w->w13_s, 2 * c.num_experts, c.inter, c.hidden)) != MOE_W4A16_OK ||
        (st = encode_decode_s2(&dw->ts2r, w->w2_s, r2, c.inter)) != MOE_W4A16_OK)
      return st;
    dw->ts13s = dw->ts13r;
    dw->ts2s = dw->ts2r;
    if (has_sh && ((st = encode_decode_s13(&dw->ts13s, w->sh_w13_s, 2, c.shared_inter, c.hidden)) != MOE_W4A16_OK ||
                   (st = encode_decode_s2(&dw->ts2s, w->sh_w2_s, c.hidden, c.shared_inter)) != MOE_W4A16_OK))
      return st;
  }
  // the wide views, when every K allows them (else, or when the driver
  // refuses one, the kernel keeps to the narrow ones)
  dw->wide = 0;
  const bool wide_k = c.hidden % 1024 == 0 && c.inter % 1024 == 0 && (!has_sh || c.shared_inter % 1024 == 0);
  if (wide_k) {
    bool ok = encode_decode_w13_wide(&dw->wtm13r, w->w13_q, 2 * c.num_experts, c.inter, c.hidden) == MOE_W4A16_OK &&
              encode_decode_w2_wide(&dw->wtm2r, w->w2_q, r2, c.inter) == MOE_W4A16_OK;
    dw->wtm13s = dw->wtm13r;
    dw->wtm2s = dw->wtm2r;
    if (ok && has_sh)
      ok = encode_decode_w13_wide(&dw->wtm13s, w->sh_w13_q, 2, c.shared_inter, c.hidden) == MOE_W4A16_OK &&
           encode_decode_w2_wide(&dw->wtm2s, w->sh_w2_q, c.hidden, c.shared_inter) == MOE_W4A16_OK;
    dw->wts13r = dw->wtm13r;
    dw->wts2r = dw->wtm2r;
    dw->wts13s = dw->wtm13s;
    dw->wts2s = dw->wtm2s;
    if (ok && scale_tma) {
      ok = encode_decode_s13_wide(&dw->wts13r, w->w13_s, 2 * c.num_experts, c.inter, c.hidden) == MOE_W4A16_OK &&
           encode_decode_s2_wide(&dw->wts2r, w->w2_s, r2, c.inter) == MOE_W4A16_OK;
      dw->wts13s = dw->wts13r;
      dw->wts2s = dw->wts2r;
      if (ok && has_sh)
        ok = encode_decode_s13_wide(&dw->wts13s, w->sh_w13_s, 2, c.shared_inter, c.hidden) == MOE_W4A16_OK &&
             encode_decode_s2_wide(&dw->wts2s, w->sh_w2_s, c.hidden, c.shared_inter) == MOE_W4A16_OK;
    }
    dw->wide = ok ? 1 : 0;
  }
  return MOE_W4A16_OK;
}

// Tensor-core operands. Packed INT4 [rows, K/8] uint32 in boxes of 8 words x
// 128 rows (one 64-wide K block of a 128-channel tile, 32-byte swizzle: the
// two 16-byte halves of a row swap places on row bit 2); a bf16 activation
// matrix [rows, cols] in boxes of 64 x 64 (or 128) rows with the 128-byte
// swizzle the tensor core reads.
int encode_int4_map_tc(CUtensorMap* m, const void* base, long long rows, int K) {
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, base, K / 8, rows, 8, 128,
                   CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "int4 tiles");
}
int encode_act_map_tc(CUtensorMap* m, const void* base, long long cols, long long rows,
                      int box_rows = 64) {
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, 64, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "activations");
}

int get_map(moe_w4a16_handle* h, int slot, const void* base, long long rows, int K) {
  if (h->map_keys[slot] == base && base) return MOE_W4A16_OK;
  const int st = slot < 4    ? encode_int4_map(&h->maps[slot], base, rows, K)
                 : slot < 8  ? encode_scale_map(&h->maps[slot], base, rows, K)
                             : encode_int4_map_tc(&h->maps[slot], base, rows, K);
  if (st == MOE_W4A16_OK) h->map_keys[slot] = base;
  return st;
}

int validate_weights(const moe_w4a16_config& c, const moe_w4a16_weights* w) {
  if (!w) return MOE_W4A16_ERR_INVALID_ARG;
  const void* req[] = {w->router_w, w->router_bias, w->w13_q, w->w13_s, w->w2_q, w->w2_s};
  for (const void* p : req) {
    if (!p) return MOE_W4A16_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_W4A16_ERR_MISALIGNED;
  }
  if (c.shared_inter > 0) {
    const void* sh[] = {w->sh_w13_q, w->sh_w13_s, w->sh_w2_q, w->sh_w2_s};
    for (const void* p : sh) {
      if (!p) return MOE_W4A16_ERR_INVALID_ARG;
      if (!aligned16(p)) return MOE_W4A16_ERR_MISALIGNED;
    }
  }
  return MOE_W4A16_OK;
}

}  // namespace

extern "C" {

const char* moe_w4a16_status_string(int s) {
  switch (s) {
    case MOE_W4A16_OK: return "ok";
    case MOE_W4A16_ERR_INVALID_ARG: return "invalid argument";
    case MOE_W4A16_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_W4A16_ERR_TOO_MANY_TOKENS: return "num_tokens exceeds max_tokens";
    case MOE_W4A16_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_W4A16_ERR_CUDA: return "CUDA error";
    case MOE_W4A16_ERR_DEVICE: return "device error flag set";
    case MOE_W4A16_ERR_NO_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

int moe_w4a16_pack_int4(const int8_t* q, int64_t rows, int64_t K, uint32_t* out) {
  if (!q || !out || rows < 0 || K <= 0 || K % 8) return MOE_W4A16_ERR_INVALID_ARG;
  const int64_t n = rows * K;
  for (int64_t i = 0; i < n; ++i)
    if (q[i] < -8 || q[i] > 7) return MOE_W4A16_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; i += 8) {
    uint32_t w = 0;
    for (int j = 0; j < 8; ++j) w |= (uint32_t)(q[i + j] + 8) << (4 * j);
    out[i / 8] = w;
  }
  return MOE_W4A16_OK;
}

int moe_w4a16_workspace_bytes(const moe_w4a16_config* cfg, size_t* bytes) {
  const int st = validate_config(cfg);
  if (st != MOE_W4A16_OK) return st;
  if (!bytes) return MOE_W4A16_ERR_INVALID_ARG;
  *bytes = plan(*cfg).total;
  return MOE_W4A16_OK;
}

int moe_w4a16_create(const moe_w4a16_config* cfg, int device, moe_w4a16_handle** out) {
  if (!out) return MOE_W4A16_ERR_INVALID_ARG;
  *out = nullptr;
  int st = validate_config(cfg);
  if (st != MOE_W4A16_OK) return st;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev <= 0) {
    cudaGetLastError();
    return MOE_W4A16_ERR_NO_DEVICE;
  }
  if (device < 0 || device >= ndev) return MOE_W4A16_ERR_INVALID_ARG;
  cudaDeviceProp prop;
  if ((st = cuda_status(cudaGetDeviceProperties(&prop, device))) != MOE_W4A16_OK) return st;
  if (prop.major != 10 || prop.minor != 3) return MOE_W4A16_ERR_NO_DEVICE;
  if ((st = cuda_status(cudaSetDevice(device))) != MOE_W4A16_OK) return st;

  moe_w4a16_handle* h = new (std::nothrow) moe_w4a16_handle();
  if (!h) return MOE_W4A16_ERR_CUDA;
  h->cfg = *cfg;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  int per_sm = 0;
  if ((st = cuda_status(gemv_setup(&per_sm))) != MOE_W4A16_OK || per_sm < 1) {
    delete h;
    return st != MOE_W4A16_OK ? st : MOE_W4A16_ERR_CUDA;
  }
  h->gemv_grid = h->num_sms * per_sm;
  int dec_per_sm = 0;
  if ((st = cuda_status(decode_setup(&dec_per_sm))) != MOE_W4A16_OK || dec_per_sm < 1) {
    delete h;
    return st != MOE_W4A16_OK ? st : MOE_W4A16_ERR_CUDA;
  }
  h->decode_grid = h->num_sms * dec_per_sm;
  // tensor-core experts: down tiles are 256 output channels wide
  h->tc_ok = cfg->hidden % 256 == 0;
  if ((cfg->flags & MOE_W4A16_FLAG_FORCE_TC) && !h->tc_ok) {
    delete h;
    return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;
  }
  int tc_per_sm = 0;
  if ((st = cuda_status(router_tc_setup())) != MOE_W4A16_OK) {
    delete h;
    return st;
  }
  // the tensor-core experts keep all of an SM's TMEM per CTA: exactly one
  // resident CTA per SM, one persistent CTA per SM in the grid
  if ((st = cuda_status(tc_setup(&tc_per_sm))) != MOE_W4A16_OK || tc_per_sm != 1) {
    delete h;
    return st != MOE_W4A16_OK ? st : MOE_W4A16_ERR_CUDA;
  }
  h->tc_grid = h->num_sms;

  const Layout L = plan(*cfg);
  if ((st = cuda_status(cudaMalloc(&h->ws, L.total))) != MOE_W4A16_OK) {
    delete h;
    return st;
  }
  h->ws_bytes = L.total;
  cudaMemset(h->ws, 0, L.total);
  uint8_t* b = static_cast<uint8_t*>(h->ws);
  Routing& r = h->r;
  r.logits = reinterpret_cast<float*>(b + L.off[0]);
  r.ids = reinterpret_cast<int*>(b + L.off[1]);
  r.wts = reinterpret_cast<float*>(b + L.off[2]);
  r.counts = reinterpret_cast<int*>(b + L.off[3]);
  r.offsets = reinterpret_cast<int*>(b + L.off[4]);
  r.active = reinterpret_cast<int*>(b + L.off[5]);
  r.meta = reinterpret_cast<int*>(b + L.off[6]);
  r.task1 = reinterpret_cast<int*>(b + L.off[7]);
  r.task2 = reinterpret_cast<int*>(b + L.off[8]);
  r.perm = reinterpret_cast<int*>(b + L.off[9]);
  r.inv = reinterpret_cast<int*>(b + L.off[10]);
  r.blockcnt = reinterpret_cast<int*>(b + L.off[11]);
  r.blockbase = reinterpret_cast<int*>(b + L.off[12]);
  r.tickets = reinterpret_cast<unsigned*>(b + L.off[13]);
  r.err = reinterpret_cast<unsigned*>(b + L.off[14]);
  h->tile_cnt = reinterpret_cast<int*>(b + L.off[15]);
  h->h = reinterpret_cast<uint16_t*>(b + L.off[16]);
  h->hstride = cfg->inter > cfg->shared_inter ? cfg->inter : cfg->shared_inter;
  h->y = reinterpret_cast<float*>(b + L.off[17]);
  h->x_dev = reinterpret_cast<uint16_t*>(b + L.off[18]);
  h->out_dev = reinterpret_cast<uint16_t*>(b + L.off[19]);
  h->counters = reinterpret_cast<int*>(b + L.off[20]);
  r.xperm = reinterpret_cast<uint16_t*>(b + L.off[21]);
  r.task3 = reinterpret_cast<int*>(b + L.off[22]);
  r.task4 = reinterpret_cast<int*>(b + L.off[23]);
  h->planes = reinterpret_cast<uint16_t*>(b + L.off[24]);
  if (h->tc_ok) {
    const long long rows = (long long)cfg->max_tokens * (cfg->top_k + 1);
    if ((st = encode_act_map_tc(&h->xmap, r.xperm, cfg->hidden, rows)) != MOE_W4A16_OK ||
        (st = encode_act_map_tc(&h->hmap, h->h, h->hstride, rows)) != MOE_W4A16_OK ||
        (st = encode_act_map_tc(&h->wmap_router, h->planes, cfg->hidden, 3LL * cfg->num_experts,
                                128)) != MOE_W4A16_OK) {
      moe_w4a16_destroy(h);
      return st;
    }
  }

  if (cfg->flags & MOE_W4A16_FLAG_PROFILE) {
    for (int i = 0; i < 2 * LaunchLog::kMax; ++i) cudaEventCreate(&h->events[i]);
    h->events_made = true;
  }
  if ((st = cuda_status(cudaDeviceSynchronize())) != MOE_W4A16_OK) {
    moe_w4a16_destroy(h);
    return st;
  }
  *out = h;
  return MOE_W4A16_OK;
}

int moe_w4a16_destroy(moe_w4a16_handle* h) {
  if (!h) return MOE_W4A16_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  if (h->events_made)
    for (int i = 0; i < 2 * LaunchLog::kMax; ++i) cudaEventDestroy(h->events[i]);
  if (h->host_graph) cudaGraphExecDestroy(h->host_graph);
  if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  if (h->ws) cudaFree(h->ws);
  delete h;
  return MOE_W4A16_OK;
}

int moe_w4a16_forward(moe_w4a16_handle* h, const uint16_t* x, int32_t T, const moe_w4a16_weights* w,
                      uint16_t* out, void* stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  const moe_w4a16_config& c = h->cfg;
  if (T < 0) return MOE_W4A16_ERR_INVALID_ARG;
  if (T > c.max_tokens) return MOE_W4A16_ERR_TOO_MANY_TOKENS;
  int st = validate_weights(c, w);
  if (st != MOE_W4A16_OK) return st;
  h->log.n = 0;
  h->log.events = h->events_made ? h->events : nullptr;
  if (T == 0) {
    h->last_T = 0;
    return MOE_W4A16_OK;
  }
  if (!x || !out) return MOE_W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return MOE_W4A16_ERR_MISALIGNED;
  {
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), oa = reinterpret_cast<uintptr_t>(out);
    const uintptr_t n = (uintptr_t)T * c.hidden * 2;
    if (xa < oa + n && oa < xa + n) return MOE_W4A16_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) cudaSetDevice(h->device);

  Dims d{T, c.hidden, c.num_experts, c.top_k, c.inter, c.shared_inter};
  cudaError_t e;
  if (c.flags & MOE_W4A16_FLAG_W4A8) {
    // W4A8-FP8 experts at every batch size: the GEMV engine's routing (no
    // gather), e4m3 x codes and scales in the xperm buffer, fp32 h in y, e4m3
    // h codes and scales in the h buffer, fp32 y, the combine
    Routing rg = h->r;
    rg.xperm = nullptr;
    rg.task3 = rg.task4 = nullptr;
    if ((e = launch_route(d, rg, x, w->router_w, w->router_bias, s, h->log)) != cudaSuccess)
      return cuda_status(e);
    const int hst = h->hstride;
    const int rows = T * c.top_k + (c.shared_inter > 0 ? T : 0);
    uint8_t* xc = reinterpret_cast<uint8_t*>(h->r.xperm);
    float* xs = reinterpret_cast<float*>(xc + align256((size_t)T * c.hidden));
    uint8_t* hc = reinterpret_cast<uint8_t*>(h->h);
    float* hs = reinterpret_cast<float*>(hc + align256((size_t)rows * hst));
    W4a8Weights ww{reinterpret_cast<const uint32_t*>(w->w13_q), w->w13_s,
                   reinterpret_cast<const uint32_t*>(w->w2_q), w->w2_s,
                   reinterpret_cast<const uint32_t*>(w->sh_w13_q), w->sh_w13_s,
                   reinterpret_cast<const uint32_t*>(w->sh_w2_q), w->sh_w2_s};
    if ((e = launch_w4a8_experts(d, h->r, ww, x, xc, xs, h->y, hc, hs, hst, h->y, h->gemv_grid, s,
                                 h->log)) != cudaSuccess)
      return cuda_status(e);
    if ((e = launch_combine(d, h->r, h->y, out, s, h->log)) != cudaSuccess) return cuda_status(e);
    h->last_T = T;
    return MOE_W4A16_OK;
  }
  if (T <= kSmallT && !(c.flags & MOE_W4A16_FLAG_FORCE_TC)) {
    // decode sizes: the whole layer in one cooperative persistent kernel
    if (!h->dec_ready || memcmp(&h->dec_key, w, sizeof(*w)) != 0) {
      h->dec_ready = false;
      if ((st = encode_decode_maps(&h->dec, c, w)) != MOE_W4A16_OK) return st;
      h->dec_key = *w;
      h->dec_ready = true;
    }
    const DecodeWeights& dw = h->dec;
    if ((e = launch_decode(d, h->r, dw, x, h->r.xperm, h->h, h->hstride,
                           reinterpret_cast<uint16_t*>(h->y), out,
                           h->counters, h->decode_grid, s, h->log)) != cudaSuccess)
      return cuda_status(e);
    h->last_T = T;
    return MOE_W4A16_OK;
  }
  const bool has_sh = c.shared_inter > 0;
  // scales ride in the TMA stages when every K has a multiple of 8 groups
  const bool scale_tma = decode_scale_tma(c);
  const long long r13 = (long long)c.num_experts * 2 * c.inter, r2 = (long long)c.num_experts * c.hidden;
  if ((st = get_map(h, 0, w->w13_q, r13, c.hidden)) != MOE_W4A16_OK) return st;
  if ((st = get_map(h, 1, w->w2_q, r2, c.inter)) != MOE_W4A16_OK) return st;
  if (has_sh) {
    if ((st = get_map(h, 2, w->sh_w13_q, 2LL * c.shared_inter, c.hidden)) != MOE_W4A16_OK) return st;
    if ((st = get_map(h, 3, w->sh_w2_q, c.hidden, c.shared_inter)) != MOE_W4A16_OK) return st;
  }
  if (scale_tma) {
    if ((st = get_map(h, 4, w->w13_s, r13, c.hidden)) != MOE_W4A16_OK) return st;
    if ((st = get_map(h, 5, w->w2_s, r2, c.inter)) != MOE_W4A16_OK) return st;
    if (has_sh) {
      if ((st = get_map(h, 6, w->sh_w13_s, 2LL * c.shared_inter, c.hidden)) != MOE_W4A16_OK)
        return st;
      if ((st = get_map(h, 7, w->sh_w2_s, c.hidden, c.shared_inter)) != MOE_W4A16_OK) return st;
    }
  }
  GemvWeights g1, g2;
  g1.tm_routed = h->maps[0];
  g1.tm_shared = has_sh ? h->maps[2] : h->maps[0];
  g1.ts_routed = scale_tma ? h->maps[4] : h->maps[0];
  g1.ts_shared = scale_tma && has_sh ? h->maps[6] : g1.ts_routed;
  g1.scale_routed = w->w13_s;
  g1.scale_shared = has_sh ? w->sh_w13_s : w->w13_s;
  g1.scale_tma = scale_tma;
  g2.tm_routed = h->maps[1];
  g2.tm_shared = has_sh ? h->maps[3] : h->maps[1];
  g2.ts_routed = scale_tma ? h->maps[5] : h->maps[1];
  g2.ts_shared = scale_tma && has_sh ? h->maps[7] : g2.ts_routed;
  g2.scale_routed = w->w2_s;
  g2.scale_shared = has_sh ? w->sh_w2_s : w->w2_s;
  g2.scale_tma = scale_tma;

  const bool use_tc = h->tc_ok && !(c.flags & MOE_W4A16_FLAG_FORCE_GEMV);
  if (use_tc) {
    // tensor-core experts: routing also gathers x into expert order
    if ((st = get_map(h, 12, w->w13_q, r13, c.hidden)) != MOE_W4A16_OK) return st;
    if ((st = get_map(h, 13, w->w2_q, r2, c.inter)) != MOE_W4A16_OK) return st;
    if (has_sh) {
      if ((st = get_map(h, 14, w->sh_w13_q, 2LL * c.shared_inter, c.hidden)) != MOE_W4A16_OK)
        return st;
      if ((st = get_map(h, 15, w->sh_w2_q, c.hidden, c.shared_inter)) != MOE_W4A16_OK) return st;
    }
    TcWeights t1, t2;
    t1.wq_r = h->maps[12];
    t1.wq_s = has_sh ? h->maps[14] : h->maps[12];
    t1.scale_routed = w->w13_s;
    t1.scale_shared = has_sh ? w->sh_w13_s : w->w13_s;
    t2.wq_r = h->maps[13];
    t2.wq_s = has_sh ? h->maps[15] : h->maps[13];
    t2.scale_routed = w->w2_s;
    t2.scale_shared = has_sh ? w->sh_w2_s : w->w2_s;
    if (h->xmap_key != x || h->xmap_rows != T) {
      if ((st = encode_act_map_tc(&h->xmap_router, x, c.hidden, T, 128)) != MOE_W4A16_OK) return st;
      h->xmap_key = x;
      h->xmap_rows = T;
    }
    if ((e = launch_router_logits_tc(d, w->router_w, h->planes, h->xmap_router, h->wmap_router,
                                     h->r.logits, h->r.err, s, h->log)) != cudaSuccess)
      return cuda_status(e);
    if ((e = launch_route(d, h->r, x, w->router_w, w->router_bias, s, h->log, true)) != cudaSuccess)
      return cuda_status(e);
    if ((e = launch_tc_gate_up(d, h->r, t1, h->xmap, h->h, h->hstride, h->tc_grid, s, h->log)) !=
        cudaSuccess)
      return cuda_status(e);
    // y in bf16: half the bytes of its round trip through HBM (written here, read
    // once by the combine); one more rounding per expert output, inside the
    // layer's output tolerance
    uint16_t* ybf = reinterpret_cast<uint16_t*>(h->y);
    if ((e = launch_tc_down(d, h->r, t2, h->hmap, ybf, h->tc_grid, s, h->log)) != cudaSuccess)
      return cuda_status(e);
    if ((e = launch_combine(d, h->r, ybf, out, s, h->log)) != cudaSuccess) return cuda_status(e);
    h->last_T = T;
    return MOE_W4A16_OK;
  }
  Routing rg = h->r;  // the GEMV experts read x in token order
  rg.xperm = nullptr;
  rg.task3 = rg.task4 = nullptr;
  if ((e = launch_route(d, rg, x, w->router_w, w->router_bias, s, h->log)) != cudaSuccess)
    return cuda_status(e);
  if ((e = launch_gemv_gate_up(d, h->r, g1, x, h->h, h->hstride, h->gemv_grid, s, h->log)) !=
      cudaSuccess)
    return cuda_status(e);
  if ((e = launch_gemv_down(d, h->r, g2, h->h, h->hstride, h->y, nullptr, h->tile_cnt,
                            h->gemv_grid, s, h->log)) != cudaSuccess)
    return cuda_status(e);
  if ((e = launch_combine(d, h->r, h->y, out, s, h->log)) != cudaSuccess) return cuda_status(e);
  h->last_T = T;
  return MOE_W4A16_OK;
}

int moe_w4a16_forward_host(moe_w4a16_handle* h, const uint16_t* x_host, int32_t T,
                           const moe_w4a16_weights* w, uint16_t* out_host, void* stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  if (T < 0) return MOE_W4A16_ERR_INVALID_ARG;
  if (T > h->cfg.max_tokens) return MOE_W4A16_ERR_TOO_MANY_TOKENS;
  if (T > 0 && (!x_host || !out_host)) return MOE_W4A16_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = (size_t)T * h->cfg.hidden * 2;
  int st;
  if (T > 0 && !(h->cfg.flags & MOE_W4A16_FLAG_PROFILE) && is_pinned(x_host) && is_pinned(out_host)) {
    // one graph launch instead of three API calls per forward
    cudaSetDevice(h->device);
    if ((st = validate_weights(h->cfg, w)) != MOE_W4A16_OK) return st;
    if (!h->host_graph || h->hg_x != x_host || h->hg_out != out_host || h->hg_T != T ||
        memcmp(&h->hg_w, w, sizeof(*w)) != 0) {
      if (h->host_graph) {
        cudaGraphExecDestroy(h->host_graph);
        h->host_graph = nullptr;
      }
      if (!h->capture_stream &&
          (st = cuda_status(cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking))) !=
              MOE_W4A16_OK)
        return st;
      cudaStream_t c = h->capture_stream;
      if ((st = cuda_status(cudaStreamBeginCapture(c, cudaStreamCaptureModeThreadLocal))) !=
          MOE_W4A16_OK)
        return st;
      cudaError_t e = cudaMemcpyAsync(h->x_dev, x_host, n, cudaMemcpyHostToDevice, c);
      int fst = e == cudaSuccess ? moe_w4a16_forward(h, h->x_dev, T, w, h->out_dev, c) : MOE_W4A16_OK;
      if (e == cudaSuccess && fst == MOE_W4A16_OK)
        e = cudaMemcpyAsync(out_host, h->out_dev, n, cudaMemcpyDeviceToHost, c);
      cudaGraph_t g = nullptr;
      const cudaError_t ee = cudaStreamEndCapture(c, &g);
      if (fst != MOE_W4A16_OK || e != cudaSuccess || ee != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return fst != MOE_W4A16_OK ? fst : cuda_status(e != cudaSuccess ? e : ee);
      }
      e = cudaGraphInstantiate(&h->host_graph, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) {
        h->host_graph = nullptr;
        return cuda_status(e);
      }
      h->hg_x = x_host;
      h->hg_out = out_host;
      h->hg_T = T;
      h->hg_w = *w;
    }
    if ((st = cuda_status(cudaGraphLaunch(h->host_graph, s))) != MOE_W4A16_OK) return st;
    h->last_T = T;
    return cuda_status(cudaStreamSynchronize(s));
  }
  if (T > 0) {
    cudaSetDevice(h->device);
    if ((st = cuda_status(cudaMemcpyAsync(h->x_dev, x_host, n, cudaMemcpyHostToDevice, s))) !=
        MOE_W4A16_OK)
      return st;
  }
  if ((st = moe_w4a16_forward(h, h->x_dev, T, w, h->out_dev, stream)) != MOE_W4A16_OK) return st;
  if (T > 0) {
    if ((st = cuda_status(cudaMemcpyAsync(out_host, h->out_dev, n, cudaMemcpyDeviceToHost, s))) !=
        MOE_W4A16_OK)
      return st;
  }
  return cuda_status(cudaStreamSynchronize(s));
}

int moe_w4a16_get_routing(moe_w4a16_handle* h, int32_t* ids, float* wts, int32_t* offsets,
                          int32_t* perm, int32_t* inv, void* stream) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tk = (size_t)h->last_T * h->cfg.top_k * 4;
  cudaError_t e = cudaSuccess;
  if (ids && tk && e == cudaSuccess) e = cudaMemcpyAsync(ids, h->r.ids, tk, cudaMemcpyDeviceToDevice, s);
  if (wts && tk && e == cudaSuccess) e = cudaMemcpyAsync(wts, h->r.wts, tk, cudaMemcpyDeviceToDevice, s);
  if (perm && tk && e == cudaSuccess)
    e = cudaMemcpyAsync(perm, h->r.perm, tk, cudaMemcpyDeviceToDevice, s);
  if (inv && tk && e == cudaSuccess) e = cudaMemcpyAsync(inv, h->r.inv, tk, cudaMemcpyDeviceToDevice, s);
  if (offsets && e == cudaSuccess) {
    if (h->last_T > 0)
      e = cudaMemcpyAsync(offsets, h->r.offsets, (h->cfg.num_experts + 1) * 4,
                          cudaMemcpyDeviceToDevice, s);
    else
      e = cudaMemsetAsync(offsets, 0, (h->cfg.num_experts + 1) * 4, s);
  }
  return cuda_status(e);
}

int moe_w4a16_check_device_errors(moe_w4a16_handle* h, uint32_t* flags) {
  if (!h) return MOE_W4A16_ERR_INVALID_ARG;
  cudaSetDevice(h->device);
  int st;
  if ((st = cuda_status(cudaDeviceSynchronize())) != MOE_W4A16_OK) return st;
  uint32_t v = 0;
  if ((st = cuda_status(cudaMemcpy(&v, h->r.err, 4, cudaMemcpyDeviceToHost))) != MOE_W4A16_OK)
    return st;
  if (v && (st = cuda_status(cudaMemset(h->r.err, 0, 4))) != MOE_W4A16_OK) return st;
  if (flags) *flags = v;
  return v ? MOE_W4A16_ERR_DEVICE : MOE_W4A16_OK;
}

int moe_w4a16_last_launches(moe_w4a16_handle* h, int32_t* count, const char** names, float* ms,
                            int32_t capacity) {
  if (!h || capacity < 0) return MOE_W4A16_ERR_INVALID_ARG;
  const int n = h->log.n;
  if (count) *count = n;
  for (int i = 0; i < n && i < capacity; ++i) {
    if (names) names[i] = h->log.names[i];
    if (ms) {
      ms[i] = -1.f;
      if (h->events_made) {
        float v = 0.f;
        if (cudaEventElapsedTime(&v, h->events[2 * i], h->events[2 * i + 1]) == cudaSuccess) ms[i] = v;
        else cudaGetLastError();
      }
    }
  }
  return MOE_W4A16_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------
// Forward without device allocation.
//
// Some callers cannot call cudaMalloc: code that runs while a stream is being
// captured into a CUDA graph (allocation is not allowed there), plugins that
// must live inside a memory budget owned by a host framework, and latency-
// critical paths that cannot afford the allocator's synchronisation. For them
// the decode-sized forward runs on a fixed scratch array that the library
// declares itself: every GPU that loads the library holds it until exit.
// ------------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(6) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  int grid = 0;
};
constexpr int kMaxDevices = 64;
NoAllocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

struct NoAllocLayout {
  size_t off[24];
  size_t total;
};

NoAllocLayout noalloc_plan(const moe_w4a16_config& c, int T) {
  const size_t E = c.num_experts, k = c.top_k, H = c.hidden, Tz = T;
  const size_t rows = Tz * k + Tz;
  const size_t hstride = c.inter > c.shared_inter ? c.inter : c.shared_inter;
  const size_t sizes[] = {
      Tz * E * 4,                                        // 0 logits
      Tz * k * 4,                                        // 1 ids
      Tz * k * 4,                                        // 2 wts
      E * 4,                                             // 3 counts
      (E + 1) * 4,                                       // 4 offsets
      (E + 1) * 4,                                       // 5 active
      kMetaWords * 4,                                    // 6 meta
      (E + 2) * 4,                                       // 7 task1
      (E + 2) * 4,                                       // 8 task2
      Tz * k * 4,                                        // 9 perm
      Tz * k * 4,                                        // 10 inv
      0,                                                 // 11 (the error word sits at offset 0)
      decode_counter_ints(c.num_experts, c.hidden) * 4,  // 12 counters
      rows * hstride * 2,                                // 13 h
      rows * H * 2,                                      // 14 y (bf16)
      Tz * H * 2,                                        // 15 x interleaved
  };
  NoAllocLayout L;
  size_t o = 256;  // the first 256 bytes: the device error word, at a fixed offset
  for (size_t i = 0; i < sizeof(sizes) / sizeof(sizes[0]); ++i) {
    L.off[i] = o;
    o += align256(sizes[i]);
  }
  L.total = o;
  return L;
}

}  // namespace

extern "C" int moe_w4a16_noalloc_check_errors(void* stream, uint32_t* flags) {
  if (!flags) return MOE_W4A16_ERR_INVALID_ARG;
  *flags = 0;
  int dev = -1, st;
  if ((st = cuda_status(cudaGetDevice(&dev))) != MOE_W4A16_OK) return st;
  if (dev < 0 || dev >= kMaxDevices) return MOE_W4A16_ERR_NO_DEVICE;
  NoAllocDevice nd;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    nd = g_noalloc[dev];
  }
  if (!nd.ready) return MOE_W4A16_OK;  // no call on this device yet
  if ((st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)))) != MOE_W4A16_OK)
    return st;
  unsigned v = 0;
  if ((st = cuda_status(cudaMemcpy(&v, nd.scratch, sizeof(v), cudaMemcpyDeviceToHost))) !=
      MOE_W4A16_OK)
    return st;
  *flags = v;
  return MOE_W4A16_OK;
}

extern "C" int moe_w4a16_forward_noalloc(const moe_w4a16_config* cfg, const uint16_t* x,
                                         int32_t T, const moe_w4a16_weights* w, uint16_t* out,
                                         void* stream) {
  int st = validate_config(cfg);
  if (st != MOE_W4A16_OK) return st;
  const moe_w4a16_config& c = *cfg;
  if (c.flags & MOE_W4A16_FLAG_W4A8) return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;  // handles only
  if (T < 0) return MOE_W4A16_ERR_INVALID_ARG;
  if (T > MOE_W4A16_NOALLOC_MAX_TOKENS) return MOE_W4A16_ERR_TOO_MANY_TOKENS;
  if ((st = validate_weights(c, w)) != MOE_W4A16_OK) return st;
  if (T == 0) return MOE_W4A16_OK;
  if (!x || !out) return MOE_W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return MOE_W4A16_ERR_MISALIGNED;
  {
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), oa = reinterpret_cast<uintptr_t>(out);
    const uintptr_t n = (uintptr_t)T * c.hidden * 2;
    if (xa < oa + n && oa < xa + n) return MOE_W4A16_ERR_INVALID_ARG;
  }
  const NoAllocLayout L = noalloc_plan(c, T);
  if (L.total > kNoAllocScratchBytes) return MOE_W4A16_ERR_UNSUPPORTED_SHAPE;

  int dev = -1;
  if ((st = cuda_status(cudaGetDevice(&dev))) != MOE_W4A16_OK) return st;
  if (dev < 0 || dev >= kMaxDevices) return MOE_W4A16_ERR_NO_DEVICE;
  NoAllocDevice nd;
  {
    // one-time set-up per device, with that device current: resolve the
    // device address of the scratch array (the host-side symbol is only a
    // stand-in) and configure the decode kernel
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice& gd = g_noalloc[dev];
    if (!gd.ready) {
      cudaDeviceProp prop;
      if ((st = cuda_status(cudaGetDeviceProperties(&prop, dev))) != MOE_W4A16_OK) return st;
      if (prop.major != 10 || prop.minor != 3) return MOE_W4A16_ERR_NO_DEVICE;
      void* ptr = nullptr;
      if ((st = cuda_status(cudaGetSymbolAddress(&ptr, g_noalloc_scratch))) != MOE_W4A16_OK)
        return st;
      int per_sm = 0;
      if ((st = cuda_status(decode_setup(&per_sm))) != MOE_W4A16_OK) return st;
      if (per_sm < 1) return MOE_W4A16_ERR_CUDA;
      gd.scratch = static_cast<unsigned char*>(ptr);
      gd.grid = prop.multiProcessorCount * per_sm;
      gd.ready = true;
    }
    nd = gd;
  }

  unsigned char* b = nd.scratch;
  Routing r;
  r.logits = reinterpret_cast<float*>(b + L.off[0]);
  r.ids = reinterpret_cast<int*>(b + L.off[1]);
  r.wts = reinterpret_cast<float*>(b + L.off[2]);
  r.counts = reinterpret_cast<int*>(b + L.off[3]);
  r.offsets = reinterpret_cast<int*>(b + L.off[4]);
  r.active = reinterpret_cast<int*>(b + L.off[5]);
  r.meta = reinterpret_cast<int*>(b + L.off[6]);
  r.task1 = reinterpret_cast<int*>(b + L.off[7]);
  r.task2 = reinterpret_cast<int*>(b + L.off[8]);
  r.perm = reinterpret_cast<int*>(b + L.off[9]);
  r.inv = reinterpret_cast<int*>(b + L.off[10]);
  r.blockcnt = nullptr;
  r.blockbase = nullptr;
  r.tickets = nullptr;
  r.task3 = nullptr;
  r.task4 = nullptr;
  r.xperm = nullptr;
  r.err = reinterpret_cast<unsigned*>(b);
  int* counters = reinterpret_cast<int*>(b + L.off[12]);
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(b + L.off[13]);
  uint16_t* ybuf = reinterpret_cast<uint16_t*>(b + L.off[14]);
  uint16_t* xibuf = reinterpret_cast<uint16_t*>(b + L.off[15]);
  const int hstride = c.inter > c.shared_inter ? c.inter : c.shared_inter;

  // tensor maps, encoded on the host for this call
  DecodeWeights dw;
  if ((st = encode_decode_maps(&dw, c, w)) != MOE_W4A16_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: clear the counters and
  // the error word this call relies on starting at zero
  if ((st = cuda_status(cudaMemsetAsync(counters, 0,
                                        decode_counter_ints(c.num_experts, c.hidden) * 4, s))) !=
      MOE_W4A16_OK)
    return st;
  if ((st = cuda_status(cudaMemsetAsync(r.err, 0, 4, s))) != MOE_W4A16_OK) return st;
  Dims d{T, c.hidden, c.num_experts, c.top_k, c.inter, c.shared_inter};
  LaunchLog log;
  return cuda_status(
      launch_decode(d, r, dw, x, xibuf, hbuf, hstride, ybuf, out, counters, nd.grid, s, log));
}

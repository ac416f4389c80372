// Warp-wide top-k of one token's router scores, shared by the decode kernel
// and the large-batch routing kernels.
//
// "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", "A pass through the
// model" (the router picks six of the 256 routed experts per token) and
// "canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP", "Component precisions" (fp32
// gate bias): the score of expert e is s = sigmoid(logit), the selection key
// s + bias[e]; the k largest keys win, in descending order, equal keys by the
// lower expert index; the combine weights are the winners' unbiased s
// renormalised over the k of them, summed in slot order.
//
// Lane l holds experts l, l + 32, ..., l + 32 (kTopkPer - 1). Each lane first
// sorts its entries (Batcher's odd-even merge sort of 8, 19 comparators, all
// in registers); a round is then two warp reductions (the largest key, then the
// lowest expert index holding it) and a branch-free shift of the winner lane's
// list. Rescanning the winner lane's entries every round instead took about
// 1.7x as long for k = 6 of 256.
#pragma once

#include <cstdint>

namespace moe {

constexpr int kTopkPer = 8;  // entries per lane: up to 256 experts

// order-preserving map of a float to an unsigned key (larger float, larger key)
__device__ __forceinline__ unsigned topk_key(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// compare-exchange: the larger key first, equal keys by the lower index
__device__ __forceinline__ void topk_cx(unsigned& ka, int& ia, float& sa, unsigned& kb, int& ib,
                                        float& sb) {
  const bool sw = kb > ka || (kb == ka && ib < ia);
  const unsigned tk = sw ? kb : ka;
  kb = sw ? ka : kb;
  ka = tk;
  const int ti = sw ? ib : ia;
  ib = sw ? ia : ib;
  ia = ti;
  const float ts = sw ? sb : sa;
  sb = sw ? sa : sb;
  sa = ts;
}

// lg: this lane's logits (experts lane + 32 i); bias: [E] (any memory space);
// k <= kMaxK. Lanes 0..k-1 return the chosen expert and its weight.
template <int kMaxK>
__device__ __forceinline__ void warp_topk_sorted(const float (&lg)[kTopkPer], const float* bias,
                                                 int E, int k, int lane, int* out_id,
                                                 float* out_w) {
  float sc[kTopkPer];
  unsigned key[kTopkPer];
  int ix[kTopkPer];
#pragma unroll
  for (int i = 0; i < kTopkPer; ++i) {
    const int e = lane + 32 * i;
    ix[i] = e;
    if (e < E) {
      sc[i] = __frcp_rn(1.0f + expf(-lg[i]));  // = 1 / (1 + e^-l), correctly rounded
      key[i] = topk_key(sc[i] + bias[e]);
    } else {
      sc[i] = 0.f;
      key[i] = 0u;  // below every float's key
    }
  }
#define MOE_TOPK_CX(a, b) topk_cx(key[a], ix[a], sc[a], key[b], ix[b], sc[b])
  MOE_TOPK_CX(0, 1); MOE_TOPK_CX(2, 3); MOE_TOPK_CX(4, 5); MOE_TOPK_CX(6, 7);
  MOE_TOPK_CX(0, 2); MOE_TOPK_CX(1, 3); MOE_TOPK_CX(4, 6); MOE_TOPK_CX(5, 7);
  MOE_TOPK_CX(1, 2); MOE_TOPK_CX(5, 6);
  MOE_TOPK_CX(0, 4); MOE_TOPK_CX(1, 5); MOE_TOPK_CX(2, 6); MOE_TOPK_CX(3, 7);
  MOE_TOPK_CX(2, 4); MOE_TOPK_CX(3, 5);
  MOE_TOPK_CX(1, 2); MOE_TOPK_CX(3, 4); MOE_TOPK_CX(5, 6);
#undef MOE_TOPK_CX
  float chosen_s = 0.f;
  int chosen_e = -1;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      const unsigned m = __reduce_max_sync(0xffffffffu, key[0]);
      const unsigned cand = key[0] == m ? (unsigned)ix[0] : 0xffffffffu;
      const unsigned win = __reduce_min_sync(0xffffffffu, cand);
      const int wl = (int)(win & 31u);  // expert e lives in lane e % 32
      const bool me = lane == wl;
      const float ws = __shfl_sync(0xffffffffu, sc[0], wl);
#pragma unroll
      for (int i = 0; i < kTopkPer - 1; ++i) {
        key[i] = me ? key[i + 1] : key[i];
        ix[i] = me ? ix[i + 1] : ix[i];
        sc[i] = me ? sc[i + 1] : sc[i];
      }
      key[kTopkPer - 1] = me ? 0u : key[kTopkPer - 1];
      ix[kTopkPer - 1] = me ? 0x7fffffff : ix[kTopkPer - 1];
      if (lane == j) {
        chosen_e = (int)win;
        chosen_s = ws;
      }
    }
  }
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, chosen_s, j);
  *out_id = chosen_e;
  *out_w = chosen_s / sum;
}

}  // namespace moe

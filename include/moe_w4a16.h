/*
 * moe_w4a16.h -- C ABI of a GB300 (sm_103a) mixture-of-experts FFN layer with
 * W4A16 routed experts.
 *
 * The layer (one DeepSeek-V4-Flash-shaped MoE FFN):
 *   - "What does everyone get wrong about optimizing DeepSeek V4 Flash on H100,
 *     H200, B200, GB300, RTX PRO 6000, and Strix Halo?", section "Sparse
 *     architecture": one shared expert plus 256 routed experts per layer, six
 *     routed experts active per token.
 *   - "canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP", table "Base model":
 *     hidden size 4096, top-K 6; table "Component precisions": routed experts
 *     are INT4 with group_size 128, symmetric, activations bf16 (W4A16); the
 *     router bias ffn.gate.bias is fp32.
 *   - "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", section "A pass
 *     through the model": the forward pass is dominated by the MoE expert
 *     GEMMs; weight-only kernels turn the 4-bit weights into bf16 and run bf16
 *     tensor cores.
 *
 * What one forward computes, for tokens t in [0, T):
 *   logit[t,e] = sum_h x[t,h] * router_w[e,h]                (fp32)
 *   s = sigmoid(logit); sel = s + router_bias                  (fp32)
 *   ids[t,0..k) = the k experts with the largest sel, in descending order
 *                 (equal values: lower expert index first)
 *   w[t,j]      = s[t,ids[t,j]] / sum_j' s[t,ids[t,j']]        (bias not used)
 *   for each routed expert and for the shared expert, with W = (u - 8) * scale:
 *     h = silu(x W1^T) * (x W3^T);  y = h W2^T
 *   out[t] = y_shared[t] + sum_j w[t,j] * y_{ids[t,j]}[t]      (bf16, RNE)
 *
 * Storage formats (all row-major, K contiguous):
 *   x, out        bf16 bit patterns (uint16) [T, H]
 *   router_w      fp32 [E, H];  router_bias fp32 [E]
 *   w13_q         uint32 [E, 2I, H/8]: 8 four-bit codes per word along K, code
 *                 j of a word at bits 4j..4j+3, code u encodes q = u - 8.
 *                 Rows [0, I) of each expert are the gate projection W1, rows
 *                 [I, 2I) the up projection W3.
 *   w13_s         bf16 [E, 2I, H/128]: one scale per row and 128-wide K group.
 *   w2_q, w2_s    uint32 [E, H, I/8], bf16 [E, H, I/128]   (down projection)
 *   sh_*          the shared expert, same formats without the E axis and with
 *                 intermediate size Is (config.shared_inter).
 *
 * Ownership: the caller owns every tensor; the handle owns its workspace
 * (device memory sized for config.max_tokens at create time) and never frees
 * or keeps caller pointers beyond a call. A handle is bound to one device and
 * is not thread-safe: use it from one host thread and one stream at a time.
 *
 * Errors: every entry point returns MOE_W4A16_OK (0) or a negative status.
 * Invalid arguments are rejected on the host before anything is launched.
 * Kernels check their own index ranges and bounded waits and record failures
 * in a device flag, read by moe_w4a16_check_device_errors.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_w4a16_status {
  MOE_W4A16_OK = 0,
  MOE_W4A16_ERR_INVALID_ARG = -1,       /* null pointer, bad count, bad flag     */
  MOE_W4A16_ERR_UNSUPPORTED_SHAPE = -2, /* sizes outside the supported ranges    */
  MOE_W4A16_ERR_TOO_MANY_TOKENS = -3,   /* num_tokens > config.max_tokens        */
  MOE_W4A16_ERR_MISALIGNED = -4,        /* a pointer is not 16-byte aligned      */
  MOE_W4A16_ERR_CUDA = -5,              /* a CUDA runtime/driver call failed     */
  MOE_W4A16_ERR_DEVICE = -6,            /* a kernel recorded an error flag       */
  MOE_W4A16_ERR_NO_DEVICE = -7          /* no usable sm_103 device               */
};

/* config.flags */
/* Expert paths: up to 64 tokens, one fused split-K GEMV kernel; above that,
 * tcgen05 tensor-core GEMMs when hidden % 256 == 0, else split-K GEMVs. */
#define MOE_W4A16_FLAG_FORCE_GEMV 0x1u   /* > 64 tokens: split-K GEMV experts     */
#define MOE_W4A16_FLAG_FORCE_TC 0x2u     /* tensor-core experts at every size     */
                                         /* (create fails if hidden % 256 != 0)   */
#define MOE_W4A16_FLAG_PROFILE 0x4u      /* time each kernel with CUDA events     */
/* W4A8-FP8 experts ("Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", "A
 * pass through the model": e4m3 activations, one scale per token per 128
 * elements, applied with the weight group scales to each 128-block's partial
 * sum; include/moe_w4a8.h states the readings). The same weights and routing;
 * the expert GEMMs quantise x and h to e4m3 and run on the fp8 tensor cores
 * (mma.sync). Not with the FORCE flags; needs inter and shared_inter <= hidden;
 * handles only (forward_noalloc refuses it). */
#define MOE_W4A16_FLAG_W4A8 0x8u

/* device error flag bits (moe_w4a16_check_device_errors) */
#define MOE_W4A16_DEVERR_TIMEOUT 0x1u    /* a bounded wait gave up                */
#define MOE_W4A16_DEVERR_RANGE 0x2u      /* an index left its range               */
#define MOE_W4A16_DEVERR_LAYOUT 0x4u     /* shared memory not aligned as required */

typedef struct moe_w4a16_config {
  int32_t hidden;        /* H: multiple of 128, <= 16384                         */
  int32_t num_experts;   /* E: 1..256 routed experts                             */
  int32_t top_k;         /* k: 1..min(8, E)                                      */
  int32_t inter;         /* I: routed intermediate size, multiple of 128         */
  int32_t shared_inter;  /* Is: shared intermediate size, multiple of 128, 0=none */
  int32_t group_size;    /* must be 128                                          */
  int32_t max_tokens;    /* workspace is sized for this many tokens (>= 1)       */
  uint32_t flags;        /* MOE_W4A16_FLAG_*                                     */
} moe_w4a16_config;

/* Device pointers to the layer's weights, 16-byte aligned, caller-owned. */
typedef struct moe_w4a16_weights {
  const float* router_w;      /* [E, H]        fp32                            */
  const float* router_bias;   /* [E]           fp32                            */
  const uint32_t* w13_q;      /* [E, 2I, H/8]  packed INT4                      */
  const uint16_t* w13_s;      /* [E, 2I, H/128] bf16 scales                     */
  const uint32_t* w2_q;       /* [E, H, I/8]   packed INT4                      */
  const uint16_t* w2_s;       /* [E, H, I/128] bf16 scales                      */
  const uint32_t* sh_w13_q;   /* [2Is, H/8]    (NULL when shared_inter == 0)    */
  const uint16_t* sh_w13_s;   /* [2Is, H/128]                                   */
  const uint32_t* sh_w2_q;    /* [H, Is/8]                                      */
  const uint16_t* sh_w2_s;    /* [H, Is/128]                                    */
} moe_w4a16_weights;

typedef struct moe_w4a16_handle moe_w4a16_handle;

/* Bytes of device workspace a handle with this config allocates.
 * No passage defines it: a sizing query of this library. */
int moe_w4a16_workspace_bytes(const moe_w4a16_config* cfg, size_t* bytes);

/* Validate cfg, bind to `device` (must be compute capability 10.3), allocate
 * the workspace and return a handle in *out. Synchronous.
 * The sizes it accepts are the layer of "What does everyone get wrong about
 * optimizing DeepSeek V4 Flash ...", section "Sparse architecture" (256
 * routed + 1 shared expert, top-6) and "canada-quant/DeepSeek-V4-Flash-W4A16-
 * FP8-MTP", table "Base model" (hidden 4096), generalised to any sizes in the
 * ranges of moe_w4a16_config; group_size 128 is the card's "Component
 * precisions" table. */
int moe_w4a16_create(const moe_w4a16_config* cfg, int device, moe_w4a16_handle** out);

/* Free the workspace and the handle (synchronises the device). NULL is OK.
 * No passage defines it: resource release. */
int moe_w4a16_destroy(moe_w4a16_handle* h);

/* One forward pass on `stream` (a cudaStream_t; NULL = legacy default
 * stream): the whole layer as written at the top of this header, i.e. the MoE
 * FFN of "What does everyone get wrong ...", section "Sparse architecture",
 * with the W4A16 experts of the model card's "Component precisions" table,
 * run as weight-only kernels that turn the 4-bit weights into bf16 for bf16
 * tensor cores ("Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", "A pass
 * through the model"). x and out are device pointers to bf16 [num_tokens, H];
 * out may not alias x. Asynchronous: nothing is synchronised, and the call can be
 * captured into a CUDA graph (the weights struct is read on the host during
 * the call). num_tokens == 0 is a successful no-op. */
int moe_w4a16_forward(moe_w4a16_handle* h, const uint16_t* x, int32_t num_tokens,
                      const moe_w4a16_weights* w, uint16_t* out, void* stream);

/* The same forward with HOST activations: copies x_host (bf16 [T, H]) to the
 * device, runs the forward, copies the result to out_host and synchronises
 * `stream`. The computation is moe_w4a16_forward's; the host copies have no
 * passage (an end-to-end convenience of this library). Host buffers should be pinned for asynchronous copies. With pinned
 * buffers (and without FLAG_PROFILE) the copy-forward-copy sequence is
 * recorded once into a CUDA graph owned by the handle and replayed while the
 * buffers, num_tokens and the weight pointers stay the same; a change records
 * it again. Calls must not overlap (the handle is single-stream). */
int moe_w4a16_forward_host(moe_w4a16_handle* h, const uint16_t* x_host, int32_t num_tokens,
                           const moe_w4a16_weights* w, uint16_t* out_host, void* stream);

/* Copy the routing of the last forward into caller device buffers (any may be
 * NULL). The routing is the top-6 expert choice of "What does everyone get
 * wrong ...", section "Sparse architecture", scored as the header's top
 * comment states with the fp32 bias of the model card's "Component
 * precisions" table; the offsets and permutation are the per-expert grouping
 * of an indexed grouped GEMM ("Throughputmaxxing ...", "The Humming
 * kernels"). Buffers: topk_ids int32 [T, k], topk_w fp32 [T, k], offsets int32 [E + 1]
 * (exclusive prefix of per-expert row counts), perm int32 [T*k] (token of
 * each expert-sorted row; rows of one expert in ascending token order), inv
 * int32 [T*k] (row of each (token, slot)). Asynchronous on `stream`. */
int moe_w4a16_get_routing(moe_w4a16_handle* h, int32_t* topk_ids, float* topk_w,
                          int32_t* offsets, int32_t* perm, int32_t* inv, void* stream);

/* Synchronise the handle's device, return the device error flag bits
 * (MOE_W4A16_DEVERR_*) in *flags and clear them. Returns
 * MOE_W4A16_ERR_DEVICE when any bit was set.
 * No passage defines it: error reporting of this library. */
int moe_w4a16_check_device_errors(moe_w4a16_handle* h, uint32_t* flags);

/* Number of kernels the last forward launched, and (with FLAG_PROFILE) their
 * names and durations in milliseconds, read after the stream has finished.
 * names[i] points to static strings. Either array may be NULL.
 * Measurement hook: the per-kernel breakdown follows "Throughputmaxxing ...",
 * section "Where does the time go?" (time per kernel bucket against its
 * roofline). */
int moe_w4a16_last_launches(moe_w4a16_handle* h, int32_t* count, const char** names,
                            float* ms, int32_t capacity);

/* Forward without any device allocation (no handle, no workspace).
 *
 * Not a step of the layer itself: the pages have no counterpart. It exists
 * for callers that cannot call cudaMalloc -- code running while a stream is
 * captured into a CUDA graph, plugins confined to a memory budget owned by a
 * host framework, latency-critical paths that cannot afford the allocator.
 * Scratch is a fixed 6 MiB array declared by the library as a __device__
 * variable; every GPU that loads the library holds it until the process
 * exits. Limits: num_tokens <= MOE_W4A16_NOALLOC_MAX_TOKENS, and the layer's
 * scratch (routing, h, y, counters) must fit the array; larger requests
 * return MOE_W4A16_ERR_TOO_MANY_TOKENS or MOE_W4A16_ERR_UNSUPPORTED_SHAPE
 * without launching anything.
 *
 * The first call on a device does a one-time set-up there (it resolves the
 * array's device address and configures the kernel); make that first call
 * before any stream capture. Every call uses the same array and leaves its
 * contents behind, so calls that overlap on the GPU (other streams, other
 * host threads) race with each other; the call clears the counters it needs
 * at zero on `stream` itself. cfg->max_tokens and cfg->flags are ignored;
 * x, out and the weights are device pointers as for moe_w4a16_forward.
 * The call returns once the work is enqueued; the device error word of the
 * last call is read with moe_w4a16_noalloc_check_errors. The set-up is kept
 * for the life of the process: after cudaDeviceReset on a device, this entry
 * point must not be called on it again. */
#define MOE_W4A16_NOALLOC_MAX_TOKENS 16
int moe_w4a16_forward_noalloc(const moe_w4a16_config* cfg, const uint16_t* x, int32_t num_tokens,
                              const moe_w4a16_weights* w, uint16_t* out, void* stream);

/* Device error flags of the last moe_w4a16_forward_noalloc call on the
 * current device (the same bits as moe_w4a16_check_device_errors; 0 when the
 * kernel's bounded waits all completed). No passage defines it. Synchronises
 * `stream` (the stream that call used), then reads the word at the fixed
 * start of the scratch array. *flags = 0 if no such call was made on this
 * device. Returns MOE_W4A16_ERR_INVALID_ARG for a null flags pointer, a CUDA
 * status for a failed synchronisation or copy. */
int moe_w4a16_noalloc_check_errors(void* stream, uint32_t* flags);

/* Pack signed 4-bit weights into the storage format of w13_q / w2_q.
 *
 * q: host int8 [rows, K], row-major, every value in [-8, 7]; out: host
 * uint32 [rows, K/8]. Element kk of a row goes to word kk/8, code kk%8 (bits
 * 4*(kk%8) .. +3) as u = q + 8, which is the layout the header describes for
 * the packed tensors ("canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP", table
 * "Component precisions": INT4, symmetric, group 128). Synchronous, no
 * device work; the caller owns both buffers. Returns
 * MOE_W4A16_ERR_INVALID_ARG for null pointers, rows < 0, K not a positive
 * multiple of 8, or a value outside [-8, 7]; nothing is written then. */
int moe_w4a16_pack_int4(const int8_t* q, int64_t rows, int64_t K, uint32_t* out);

/* Static description of a status code. No passage defines it. */
const char* moe_w4a16_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A16_H */

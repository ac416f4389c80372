"""fp64 CPU oracle of one W4A16 routed-expert MoE FFN layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code, header, table or helper with the CUDA
path and imports nothing from it; it works on the storage-format arrays that
``moe_synth`` draws.

What the layer computes (the pages fix the structure; the arithmetic they leave
open is read in its plainest form, and each reading is named where it is used):

* "What does everyone get wrong about optimizing DeepSeek V4 Flash ...",
  section "Sparse architecture": each MoE layer has one shared expert and 256
  routed experts, six routed experts active per token.
* "canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP", table "Base model": hidden
  4096, top-K = 6; table "Component precisions": routed experts are INT4,
  group_size 128, symmetric (W4A16), and the router bias ``ffn.gate.bias`` is
  kept in FP32.
* "Throughputmaxxing: DeepSeek-V4-Flash on Isambard-AI", section "A pass
  through the model": a weight-only kernel turns the 4-bit weights into bf16
  and multiplies them with bf16 activations (A16).

Readings (the pages are silent): sigmoid scores, bias used for selection only,
selected scores renormalised to sum to 1 (no extra scaling factor); SwiGLU
expert FFN ``silu(gate) * up`` then down; shared expert unweighted and added;
offset-binary nibble codes, 8 per uint32 along K; bf16 group scales multiply
the integer. Everything is computed in fp64 without intermediate rounding.

Parity status per function: every function below is pinned by the CPU tests in
``tests/test_oracle.py`` (hand-built bit patterns, brute-force top-k, closed
forms, direct-loop FFN, invariances). No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

GROUP = 128


# ---------------------------------------------------------------- storage types
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16): the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def unpack_int4(words) -> np.ndarray:
    """Integer weights q in [-8, 7] from packed uint32 words.

    Model card "canada-quant/DeepSeek-V4-Flash-W4A16-FP8-MTP", "Component
    precisions": symmetric INT4. Reading: code u = q + 8 (offset binary), 8
    codes per word along K, code j of a word at bits 4j..4j+3. Output shape is
    the input shape with the last axis multiplied by 8.
    """
    w = np.asarray(words, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    u = (w[..., None] >> shifts) & np.uint32(0xF)
    q = u.astype(np.int16) - 8
    return q.reshape(*w.shape[:-1], w.shape[-1] * 8).astype(np.int8)


def dequant(words, scale_bits, group: int = GROUP) -> np.ndarray:
    """fp64 weight W[n, kk] = q[n, kk] * scale[n, kk // group]."""
    q = unpack_int4(words).astype(np.float64)
    s = bf16_to_f64(scale_bits)
    n, k = q.shape
    if s.shape != (n, k // group):
        raise ValueError(f"scale shape {s.shape} != {(n, k // group)}")
    return (q.reshape(n, k // group, group) * s[:, :, None]).reshape(n, k)


# --------------------------------------------------------------------- routing
def router_logits(x_bits, router_w) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * Wr[e, h] in fp64 (x bf16, Wr fp32 exact)."""
    x = bf16_to_f64(x_bits)
    w = np.asarray(router_w, dtype=np.float32).astype(np.float64)
    return x @ w.T


def sigmoid(z) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def select_topk(logits, bias, k: int):
    """Top-k routing: sigmoid scores, bias for selection, renormalised weights.

    ``sel = sigmoid(logit) + bias`` (the fp32 router bias of the model card's
    "Component precisions" table); the k experts with the largest ``sel`` are
    taken in descending order, equal values ordered by lower expert index; the
    combine weights are the unbiased scores of the chosen experts divided by
    their sum. Returns (ids int32 [T, k], weights fp64 [T, k], sel fp64 [T, E]).
    """
    s = sigmoid(logits)
    sel = s + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    T, E = sel.shape
    # stable sort of -sel: equal values keep ascending expert index
    order = np.argsort(-sel, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    chosen = np.take_along_axis(s, ids.astype(np.int64), axis=1)
    weights = chosen / chosen.sum(axis=1, keepdims=True) if T else chosen
    return ids, weights, sel


def selection_margin(logits, bias, k: int) -> np.ndarray:
    """Gap between the k-th and (k+1)-th largest selection score of each token."""
    s = sigmoid(logits)
    sel = s + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    part = -np.sort(-sel, axis=1)
    return part[:, k - 1] - part[:, k]


def expert_counts(ids, num_experts: int):
    """Row count of each expert and the exclusive prefix sum (length E + 1)."""
    counts = np.bincount(np.asarray(ids, dtype=np.int64).ravel(),
                         minlength=num_experts).astype(np.int32)
    offsets = np.zeros(num_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return counts, offsets


def stable_permutation(ids, offsets):
    """Rows of each expert's segment list its (token, slot) pairs by ascending token.

    Returns ``perm`` int32 [T*k] (token of each row) and ``inv`` int32 [T, k]
    (row of each (token, slot)). Pure-Python loop: the definition written out.
    """
    ids = np.asarray(ids)
    T, k = ids.shape if ids.ndim == 2 else (0, 0)
    fill = np.array(offsets[:-1], dtype=np.int64, copy=True)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            r = int(fill[e])
            fill[e] += 1
            perm[r] = t
            inv[t, j] = r
    return perm, inv


# ------------------------------------------------------------------ expert FFN
def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu_expert(x_rows, w13, w2) -> np.ndarray:
    """One expert on fp64 rows: ``(silu(x W1^T) * (x W3^T)) W2^T``.

    ``w13`` is fp64 [2I, H] with gate rows first, ``w2`` fp64 [H, I].
    """
    inter = w13.shape[0] // 2
    g = x_rows @ w13[:inter].T
    u = x_rows @ w13[inter:].T
    return (silu(g) * u) @ w2.T


def expert_dense(weights: dict, group: int = GROUP):
    """Dequantised fp64 (w13, w2) of one expert from its storage-format dict."""
    return (dequant(weights["w13_q"], weights["w13_s"], group),
            dequant(weights["w2_q"], weights["w2_s"], group))


# -------------------------------------------------------------------- the layer
def route(x_bits, router_w, router_b, num_experts: int, k: int) -> dict:
    logits = router_logits(x_bits, router_w)
    ids, weights, _ = select_topk(logits, router_b, k)
    counts, offsets = expert_counts(ids, num_experts)
    perm, inv = stable_permutation(ids, offsets)
    return {"logits": logits, "ids": ids, "weights": weights, "counts": counts,
            "offsets": offsets, "perm": perm, "inv": inv}


def moe_forward(x_bits, router_w, router_b, experts, shared, k: int,
                group: int = GROUP, token_subset=None) -> dict:
    """The whole layer in fp64.

    ``experts`` is a sequence of storage-format dicts (one per routed expert),
    ``shared`` the shared expert's dict or None. Routing is computed for every
    token; the output ``out`` (fp64 [len(subset), H]) only for ``token_subset``
    (all tokens by default), which lets full-size workloads be checked on a
    sample of tokens.

    out[t] = shared(x[t]) + sum_j w[t, j] * expert_{ids[t, j]}(x[t])
    """
    E = len(experts)
    r = route(x_bits, router_w, router_b, E, k)
    T = r["ids"].shape[0]
    subset = np.arange(T) if token_subset is None else np.asarray(token_subset, dtype=np.int64)
    x = bf16_to_f64(x_bits)[subset]
    out = np.zeros_like(x)
    if shared is not None and subset.size:
        w13, w2 = expert_dense(shared, group)
        out += swiglu_expert(x, w13, w2)
    ids = r["ids"][subset]
    wts = r["weights"][subset]
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        w13, w2 = expert_dense(experts[int(e)], group)
        y = swiglu_expert(x[rows], w13, w2)
        out[rows] += wts[rows, slots][:, None] * y
    r["out"] = out
    r["subset"] = subset
    return r

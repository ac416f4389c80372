"""fp64 CPU oracle of the W4A8-FP8 variant of the routed-expert layer.

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: only ``tests/`` may import it.
It shares nothing with the CUDA path.

What the variant computes ("Throughputmaxxing: DeepSeek-V4-Flash on
Isambard-AI", section "A pass through the model", and the input-quantisation
setting printed there: dtype float8e4m3, input_scale_group_size 128): the
4-bit weights are turned into fp8 exactly (the integers -8..7 are e4m3
values), the activations entering each expert GEMM are fp8 e4m3 with one scale
per token per 128 consecutive elements, the products run in fp8 and the
per-128 activation scales, like the weight group scales, are applied to each
128-wide block's partial sum (the page's Humming fix: those input scales were
not being applied on the accumulator).

Readings (the pages are silent): e4m3 is the OCP "E4M3FN" format (bias 7, no
infinities, largest finite 448); a block's scale is fp32(amax / 448), or 1 for
an all-zero block; a code is the e4m3 value nearest to fp32(x / scale), ties to
the even code, saturated at +-448; the SwiGLU output h is quantised the same
way per row and 128 channels before the down projection, from its fp32 value;
routing, the shared expert's presence and the combine are those of the W4A16
layer (``moe_oracle``).

Parity status: ``e4m3_round``, ``quantize_blocks`` and ``w4a8_linear`` are
pinned by ``tests/test_oracle_w4a8.py`` (brute force over all 256 e4m3 codes,
hand-built ties and saturation, exact blocks, equality with the W4A16 weights
on exactly representable inputs, a planted missing-scale bug, power-of-two
invariance). ``swiglu_expert_w4a8`` and ``moe_forward_w4a8`` are pinned by an
independent brute-force composition on the tiny layer (its own nibble and
bf16 decoding, nearest-code search over the enumerated e4m3 table, per-block
scaled fp64 sums, every (token, slot) expert evaluated alone; the routing is
the W4A16 oracle's, pinned by its own tests), and a variant without the fp8
step on h is shown to differ.

There is no W4A8 CUDA path yet; this oracle is the first step of that variant.
"""
from __future__ import annotations

import numpy as np

from oracle import moe_oracle as mo

BLOCK = 128
E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6          # smallest normal binade 2^-6


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 value of fp64 inputs, ties to even, saturated at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    # spacing of the e4m3 grid around a: 2^(e - 3) in binade 2^e, 2^-9 below
    # the smallest normal binade
    _, ex = np.frexp(np.where(a > 0, a, 1.0))   # a = m 2^ex, m in [0.5, 1): binade 2^(ex - 1)
    e = np.maximum(ex.astype(np.float64) - 1.0, _MIN_NORMAL_EXP)
    step = np.exp2(e - 3)
    q = np.rint(a / step) * step           # a / step is exact; rint is half-even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def quantize_blocks(x, block: int = BLOCK):
    """Per-row, per-block e4m3 quantisation of fp32-valued activations.

    x: [rows, K] (values representable in fp32). Returns (codes, scales):
    codes fp64 [rows, K] on the e4m3 grid, scales fp64 [rows, K / block] holding
    fp32 values, so that x ~= codes * scale of its block.
    """
    x32 = np.asarray(x, dtype=np.float32)
    rows, K = x32.shape
    assert K % block == 0
    xb = x32.reshape(rows, K // block, block)
    amax = np.max(np.abs(xb), axis=2)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    ratio = (xb / scale[:, :, None]).astype(np.float32)      # fp32 division, correctly rounded
    codes = e4m3_round(ratio.astype(np.float64))
    return codes.reshape(rows, K), scale.astype(np.float64)


def w4a8_linear(codes, scales, q_w, s_w, block: int = BLOCK) -> np.ndarray:
    """y[r, n] = sum over blocks g of s_w[n, g] * scales[r, g] *
    sum_{k in g} q_w[n, k] * codes[r, k] (fp64, exact products)."""
    rows, K = codes.shape
    N = q_w.shape[0]
    G = K // block
    cb = codes.reshape(rows, G, block)
    qb = q_w.astype(np.float64).reshape(N, G, block)
    part = np.einsum("rgk,ngk->rng", cb, qb)                # block partial sums
    return np.einsum("rng,ng,rg->rn", part, s_w, scales)


def swiglu_expert_w4a8(x_rows, weights: dict, block: int = BLOCK) -> np.ndarray:
    """One expert: gate/up on e4m3 x, SwiGLU, down on e4m3 h."""
    q13 = mo.unpack_int4(weights["w13_q"])
    s13 = mo.bf16_to_f64(weights["w13_s"])
    q2 = mo.unpack_int4(weights["w2_q"])
    s2 = mo.bf16_to_f64(weights["w2_s"])
    inter = q13.shape[0] // 2
    xc, xs = quantize_blocks(x_rows, block)
    gu = w4a8_linear(xc, xs, q13, s13, block)
    h = mo.silu(gu[:, :inter]) * gu[:, inter:]
    hc, hs = quantize_blocks(h.astype(np.float32), block)
    return w4a8_linear(hc, hs, q2, s2, block)


def moe_forward_w4a8(x_bits, router_w, router_b, experts, shared, k: int,
                     block: int = BLOCK, token_subset=None) -> dict:
    """The layer with W4A8 experts: routing and combine as in ``moe_oracle``."""
    E = len(experts)
    r = mo.route(x_bits, router_w, router_b, E, k)
    T = r["ids"].shape[0]
    subset = np.arange(T) if token_subset is None else np.asarray(token_subset, dtype=np.int64)
    x = mo.bf16_to_f64(x_bits)[subset]
    out = np.zeros_like(x)
    if shared is not None and subset.size:
        out += swiglu_expert_w4a8(x, shared, block)
    ids = r["ids"][subset]
    wts = r["weights"][subset]
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        y = swiglu_expert_w4a8(x[rows], experts[int(e)], block)
        out[rows] += wts[rows, slots][:, None] * y
    r["out"] = out
    r["subset"] = subset
    return r

"""Seeded synthetic inputs for the W4A16 routed-expert MoE layer.

This module is shared by the oracle-side tests and by the GPU-side tests and
benchmark. It holds no arithmetic of the layer itself: it draws random
numbers, rounds draws to the storage types (bf16 bit patterns, fp32), and
lays them out in the storage format the layer consumes. Every step that
needs the layer's routing (the score-margin guard and the Zipf bias fit) takes
that computation as a callback from the caller.

Storage format (one reading of the model card "canada-quant/DeepSeek-V4-Flash-
W4A16-FP8-MTP", table "Component precisions": routed experts are "W4A16 INT4,
group_size=128, symmetric"):

* packed weights: uint32 words, 8 four-bit codes per word along the reduction
  (K) axis; code ``kk`` of a row sits at bits ``4*(kk % 8) .. 4*(kk % 8)+3`` of
  word ``kk // 8``. A code ``u`` in [0, 15] stands for the integer ``q = u - 8``
  in [-8, 7] (offset binary). Rows are output channels, K is contiguous.
* scales: bf16 bit patterns (uint16), one per row and per 128-wide group of
  K, row-major ``[N, K / 128]``; the weight is ``q * scale``.
* gate/up projection ``w13``: rows ``[0, I)`` are the gate projection, rows
  ``[I, 2I)`` the up projection.

Because every code is uniform on [0, 15], a uniformly random uint32 word is
exactly a word of 8 independent uniform codes, so weights are drawn as words.
"""
from __future__ import annotations

import dataclasses
import os
from typing import Callable, Optional

import numpy as np

GROUP = 128

# Stream tags: every tensor gets its own counter-keyed PCG64 stream so that a
# single expert (or a single token row) can be regenerated on its own.
_TAG_ROUTER_W = 1
_TAG_ROUTER_B = 2
_TAG_W13_Q = 3
_TAG_W13_S = 4
_TAG_W2_Q = 5
_TAG_W2_S = 6
_TAG_X = 7
_TAG_X_RESAMPLE = 8
_TAG_CAL = 9
_TAG_ZIPF_RANK = 10


@dataclasses.dataclass(frozen=True)
class MoeShape:
    """Sizes of one MoE FFN layer and the seeds of its synthetic inputs."""

    name: str
    tokens: int          # T
    hidden: int          # H
    experts: int         # E (routed)
    top_k: int           # k
    inter: int           # I, routed-expert intermediate size
    shared_inter: int    # Is, shared-expert intermediate size (0: none)
    layer_seed: int      # seeds all weights of the layer
    token_seed: int      # seeds the activations
    zipf_s: Optional[float] = None  # router bias fitted to Zipf(s) popularity
    group: int = GROUP

    def with_tokens(self, tokens: int, name: Optional[str] = None) -> "MoeShape":
        return dataclasses.replace(self, tokens=tokens, name=name or self.name)


# The five workloads: a tiny layer that the oracle runs in well under a
# second, and four workloads on one DeepSeek-V4-Flash-shaped layer (256 routed
# experts, top-6, one shared expert, hidden 4096; the expert intermediate size
# 2048 is a synthetic choice) -- decode at 1 and 64 tokens, an 8192-token
# prefill chunk, and 2048 decode tokens with Zipf(1.1)-skewed routing.
CONFIGS = {
    "tiny16": MoeShape("tiny16", 16, 256, 8, 2, 128, 128, 1000, 1000),
    "decode1": MoeShape("decode1", 1, 4096, 256, 6, 2048, 2048, 1001, 1001),
    "decode64": MoeShape("decode64", 64, 4096, 256, 6, 2048, 2048, 1001, 1002),
    "prefill8192": MoeShape("prefill8192", 8192, 4096, 256, 6, 2048, 2048, 1001, 1003),
    "zipf2048": MoeShape("zipf2048", 2048, 4096, 256, 6, 2048, 2048, 1001, 1004, zipf_s=1.1),
    # profiler-sized stand-in for prefill8192: the same expert shape and about
    # the same rows per expert (1536 * 6 / 48 = 192), a sixth of the weights
    "prefill1536e48": MoeShape("prefill1536e48", 1536, 4096, 48, 6, 2048, 2048, 1001, 1005),
}
CONFIG_ORDER = ["tiny16", "decode1", "decode64", "prefill8192", "zipf2048", "prefill1536e48"]

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "tests", "golden")


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _words(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)


def _scales(rng: np.random.Generator, rows: int, k: int, group: int) -> np.ndarray:
    # bf16 group scales uniform in [0.5, 1.5] / (8 * sqrt(K)), K = reduction size
    u = rng.uniform(0.5, 1.5, size=(rows, k // group)).astype(np.float64)
    return f32_to_bf16_bits((u / (8.0 * np.sqrt(k))).astype(np.float32))


def expert_weights(shape: MoeShape, e: int) -> dict:
    """Packed weights of routed expert ``e`` (``e == shape.experts``: shared).

    Returns ``w13_q`` uint32 [2I', H/8], ``w13_s`` uint16 [2I', H/128],
    ``w2_q`` uint32 [H, I'/8], ``w2_s`` uint16 [H, I'/128] with I' = I for a
    routed expert and Is for the shared one.
    """
    H = shape.hidden
    inter = shape.shared_inter if e == shape.experts else shape.inter
    s = shape.layer_seed
    return {
        "w13_q": _words(_rng(s, _TAG_W13_Q, e), (2 * inter, H // 8)),
        "w13_s": _scales(_rng(s, _TAG_W13_S, e), 2 * inter, H, shape.group),
        "w2_q": _words(_rng(s, _TAG_W2_Q, e), (H, inter // 8)),
        "w2_s": _scales(_rng(s, _TAG_W2_S, e), H, inter, shape.group),
    }


def router_weights(shape: MoeShape) -> np.ndarray:
    """fp32 router weight [E, H], N(0, 1/sqrt(H)) (std 1/16 at H = 256)."""
    rng = _rng(shape.layer_seed, _TAG_ROUTER_W)
    w = rng.standard_normal((shape.experts, shape.hidden)) / np.sqrt(shape.hidden)
    return w.astype(np.float32)


def router_bias(shape: MoeShape) -> np.ndarray:
    """fp32 router bias [E]: N(0, 0.01), or the stored Zipf fit for skewed layers."""
    if shape.zipf_s is not None:
        return load_zipf_bias(shape)
    rng = _rng(shape.layer_seed, _TAG_ROUTER_B)
    return (rng.standard_normal(shape.experts) * 0.01).astype(np.float32)


def tokens(shape: MoeShape, n: Optional[int] = None) -> np.ndarray:
    """bf16 bit patterns [T, H] of N(0, 1) draws rounded to nearest-even."""
    n = shape.tokens if n is None else n
    rng = _rng(shape.token_seed, _TAG_X)
    return f32_to_bf16_bits(rng.standard_normal((n, shape.hidden)).astype(np.float32))


def resample_token_row(shape: MoeShape, t: int, attempt: int) -> np.ndarray:
    rng = _rng(shape.token_seed, _TAG_X_RESAMPLE, t, attempt)
    return f32_to_bf16_bits(rng.standard_normal(shape.hidden).astype(np.float32))


def guard_margins(shape: MoeShape, x_bits: np.ndarray,
                  margin_fn: Callable[[np.ndarray], np.ndarray],
                  min_margin: float = 1e-3, max_attempts: int = 200) -> np.ndarray:
    """Redraw every token row whose k-th/(k+1)-th selection-score gap is small.

    ``margin_fn(rows)`` returns, for bf16 token rows, the gap between the k-th
    and (k+1)-th largest selection scores; it is supplied by the caller. Rows
    are redrawn one by one from a stream keyed by (token seed, row, attempt),
    so the result does not depend on which other rows needed a redraw.
    """
    x = np.array(x_bits, copy=True)
    bad = np.nonzero(margin_fn(x) < min_margin)[0]
    attempt = 0
    while bad.size:
        if attempt >= max_attempts:
            raise RuntimeError(f"margin guard: {bad.size} rows still below {min_margin}")
        for t in bad:
            x[t] = resample_token_row(shape, int(t), attempt)
        m = margin_fn(x[bad])
        bad = bad[m < min_margin]
        attempt += 1
    return x


def calibration_tokens(shape: MoeShape, n: int = 2048) -> np.ndarray:
    """A token draw independent of the workload's, used to fit the Zipf bias."""
    rng = _rng(shape.token_seed, _TAG_CAL)
    return f32_to_bf16_bits(rng.standard_normal((n, shape.hidden)).astype(np.float32))


def zipf_targets(shape: MoeShape, n_tokens: int) -> np.ndarray:
    """Target per-expert row counts: Zipf(s) over a seeded random expert ranking.

    Expected count of the rank-r expert is T*k*r^-s / sum_r r^-s, capped at the
    token count (top-k picks distinct experts, so no expert exceeds T rows).
    """
    E = shape.experts
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** -shape.zipf_s
    p /= p.sum()
    counts = np.minimum(n_tokens * shape.top_k * p, 0.97 * n_tokens)
    order = _rng(shape.layer_seed, _TAG_ZIPF_RANK).permutation(E)
    target = np.empty(E)
    target[order] = counts
    return target


def fit_zipf_bias(shape: MoeShape, count_fn: Callable[[np.ndarray], np.ndarray],
                  n_tokens: int, iters: int = 1200, lr: float = 0.05) -> np.ndarray:
    """Fit an fp32 router bias so that routed row counts follow ``zipf_targets``.

    ``count_fn(bias)`` returns per-expert row counts of the calibration draw
    routed with that bias (supplied by the caller). The update is a fixed
    number of multiplicative steps on the count ratio, done in log space with
    a decaying step: ``bias += lr / (1 + i / 200) * log((target + 1) / (count + 1))``
    at step i, clipped to [-2, 2].
    """
    target = zipf_targets(shape, n_tokens)
    b = np.zeros(shape.experts, dtype=np.float64)
    for i in range(iters):
        c = count_fn(b.astype(np.float32))
        step = lr / (1.0 + i / 200.0)
        b = np.clip(b + step * np.log((target + 1.0) / (c + 1.0)), -2.0, 2.0)
    return b.astype(np.float32)


def zipf_bias_path(shape: MoeShape) -> str:
    return os.path.join(GOLDEN_DIR, f"{shape.name}_router_bias.txt")


def load_zipf_bias(shape: MoeShape) -> np.ndarray:
    path = zipf_bias_path(shape)
    words = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                words.append(int(line.split()[0], 16))
    b = np.array(words, dtype=np.uint32).view(np.float32)
    if b.size != shape.experts:
        raise ValueError(f"{path}: {b.size} values, expected {shape.experts}")
    return b


@dataclasses.dataclass
class LayerInputs:
    """All inputs of one forward call, in storage format (numpy, host)."""

    shape: MoeShape
    x: np.ndarray            # uint16 bf16 bits [T, H]
    router_w: np.ndarray     # float32 [E, H]
    router_b: np.ndarray     # float32 [E]
    experts: list            # per routed expert: dict from expert_weights
    shared: Optional[dict]   # dict from expert_weights, or None

    def stacked(self, key: str) -> np.ndarray:
        return np.stack([w[key] for w in self.experts])


def make_layer(shape: MoeShape, margin_fn: Optional[Callable] = None,
               x: Optional[np.ndarray] = None) -> LayerInputs:
    """Build one layer's inputs. With ``margin_fn`` the token rows are guarded."""
    xb = tokens(shape) if x is None else x
    if margin_fn is not None and xb.shape[0]:
        xb = guard_margins(shape, xb, margin_fn)
    experts = [expert_weights(shape, e) for e in range(shape.experts)]
    shared = expert_weights(shape, shape.experts) if shape.shared_inter else None
    return LayerInputs(shape, xb, router_weights(shape), router_bias(shape), experts, shared)

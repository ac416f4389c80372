"""Shared helpers of the GPU parity tests: guarded inputs, oracle references,
running the CUDA path through the C ABI, and the acceptance checks.

Acceptance (fixed for this layer): routing bit-exact (expert ids, per-expert
offsets, permutation and its inverse); combine weights within fp32 rounding;
outputs with max|err| <= 2e-2 * max|ref| + 1e-3 and relative Frobenius
error <= 5e-3 against the fp64 oracle.
"""
from __future__ import annotations

import functools

import numpy as np

import moe_synth as ms
from oracle import moe_oracle as mo

MAX_ERR_REL = 2e-2
MAX_ERR_ABS = 1e-3
FROB_REL = 5e-3


def margin_fn(shape: ms.MoeShape, router_w, router_b):
    def fn(rows):
        return mo.selection_margin(mo.router_logits(rows, router_w), router_b, shape.top_k)
    return fn


@functools.lru_cache(maxsize=2)
def _weights(layer_seed, hidden, experts, top_k, inter, shared_inter):
    shape = ms.MoeShape("layer", 0, hidden, experts, top_k, inter, shared_inter, layer_seed, 0)
    return ms.make_layer(shape, x=np.zeros((0, hidden), np.uint16))


def weights_of(shape: ms.MoeShape) -> ms.LayerInputs:
    """Expert and router weights of a shape's layer (no tokens); cached per layer."""
    return _weights(shape.layer_seed, shape.hidden, shape.experts, shape.top_k, shape.inter,
                    shape.shared_inter)


def layer_with_tokens(shape: ms.MoeShape, n_tokens: int | None = None,
                      bias=None) -> ms.LayerInputs:
    """Weights of the shape's layer plus a guarded token draw of n_tokens rows.

    The router bias is the shape's own (the fitted Zipf bias for skewed
    layers) unless ``bias`` is given.
    """
    base = weights_of(shape)
    n = shape.tokens if n_tokens is None else n_tokens
    b = ms.router_bias(shape) if bias is None else np.asarray(bias, np.float32)
    sh = shape.with_tokens(n)
    x = ms.tokens(sh, n)
    if n:
        x = ms.guard_margins(sh, x, margin_fn(sh, base.router_w, b))
    return ms.LayerInputs(sh, x, base.router_w, b, base.experts, base.shared)


def oracle(layer: ms.LayerInputs, subset=None):
    return mo.moe_forward(layer.x, layer.router_w, layer.router_b, layer.experts, layer.shared,
                          layer.shape.top_k, token_subset=subset)


def bf16_bits_to_f64(bits):
    return mo.bf16_to_f64(np.asarray(bits).view(np.uint16))


def check_output(out_bits, ref):
    got = bf16_bits_to_f64(out_bits)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    err = got - ref
    max_ref = float(np.abs(ref).max()) if ref.size else 0.0
    max_err = float(np.abs(err).max()) if ref.size else 0.0
    frob = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)) if ref.size else 0.0
    assert max_err <= MAX_ERR_REL * max_ref + MAX_ERR_ABS, (max_err, max_ref)
    assert frob <= FROB_REL, frob
    return max_err, frob


def check_routing(gpu: dict, ref: dict, E: int):
    np.testing.assert_array_equal(gpu["ids"], ref["ids"])
    np.testing.assert_array_equal(gpu["offsets"], ref["offsets"])
    np.testing.assert_array_equal(gpu["perm"], ref["perm"])
    np.testing.assert_array_equal(gpu["inv"], ref["inv"])
    np.testing.assert_allclose(gpu["weights"], ref["weights"], rtol=2e-6, atol=1e-7)
    assert gpu["offsets"][-1] == ref["ids"].size


# ---------------------------------------------------- full-size output checks
def covering_tokens(route: dict, tile_rows: int = 256) -> np.ndarray:
    """Tokens whose outputs touch every active expert's segment at both ends.

    For each expert with rows: the token of its first and of its last row,
    and for segments longer than ``tile_rows`` (the row tile of the
    tensor-core experts) the first and last row of every tile. Every routed
    expert's weights, every row tile boundary and (since whole output rows are
    compared) every output channel tile are then checked against the oracle.
    """
    perm, offsets = route["perm"], route["offsets"]
    picks = {0, int(route["ids"].shape[0]) - 1}
    for e in range(offsets.size - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        for r0 in range(a, b, tile_rows):
            r1 = min(b, r0 + tile_rows) - 1
            picks.add(int(perm[r0]))
            picks.add(int(perm[r1]))
    return np.array(sorted(p for p in picks if p >= 0), dtype=np.int64)


def _expert_rows_worker(args):
    """One expert's SwiGLU output for some token rows, in a pool worker.

    The expert's weights are drawn again from the layer's seeds (the same
    generator as the layer under test), then dequantised and applied with the
    oracle's own functions.
    """
    shape, e, x_bits = args
    w13, w2 = mo.expert_dense(ms.expert_weights(shape, e), shape.group)
    return e, mo.swiglu_expert(mo.bf16_to_f64(x_bits), w13, w2)


def oracle_outputs(layer: ms.LayerInputs, route: dict, subset, workers: int = 0) -> np.ndarray:
    """``mo.moe_forward(...)["out"]`` for ``subset``, with the experts spread over
    a pool of spawned processes.

    The per-expert SwiGLU outputs come from the oracle's functions, and they
    are added up in the order ``moe_forward`` uses (the shared expert, then the
    routed experts in ascending index), so the result equals ``moe_forward``'s
    to fp64 rounding (a CPU test checks that). ``route`` is the oracle's routing of
    the whole batch. The weights must be the ones the shape's seeds draw.
    """
    import concurrent.futures as cf
    import multiprocessing as mp
    import os

    shape = layer.shape
    subset = np.asarray(subset, dtype=np.int64)
    xs = layer.x[subset]
    ids = route["ids"][subset]
    wts = route["weights"][subset]
    experts = [int(e) for e in np.unique(ids)]
    jobs = []
    if shape.shared_inter:
        jobs.append((shape, shape.experts, xs))
    for e in experts:
        rows, _ = np.nonzero(ids == e)
        jobs.append((shape, e, xs[rows]))
    n = workers or min(16, os.cpu_count() or 1)
    if n > 1 and len(jobs) > 1:
        # spawned workers (never forked after CUDA is up); a worker that dies
        # raises in the caller instead of stalling the pool
        with cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn")) as pool:
            ys = dict(pool.map(_expert_rows_worker, jobs))
    else:
        ys = dict(map(_expert_rows_worker, jobs))
    out = np.zeros((subset.size, shape.hidden))
    if shape.shared_inter:
        out += ys[shape.experts]
    for e in experts:
        rows, slots = np.nonzero(ids == e)
        out[rows] += wts[rows, slots][:, None] * ys[e]
    return out

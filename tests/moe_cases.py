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

"""CPU pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently of its own
code: hand-built bit patterns, brute force over all subsets, closed forms,
direct Python loops, and invariances of the layer. A plausible slip anywhere
(a dropped term, a wrong sign or index, a transposed operand, bias leaking into
the combine weights, an unstable permute) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest

import moe_synth as ms
from oracle import moe_oracle as mo

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _pack_codes(codes):
    """Pack rows of 4-bit codes (ints 0..15, K multiple of 8) into uint32 words.

    Written with Python integers, independently of the oracle's unpacking.
    """
    codes = np.asarray(codes)
    n, k = codes.shape
    out = np.zeros((n, k // 8), dtype=np.uint32)
    for r in range(n):
        for w in range(k // 8):
            v = 0
            for j in range(8):
                v |= int(codes[r, 8 * w + j]) << (4 * j)
            out[r, w] = v
    return out


def _bf16(x):
    return ms.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ------------------------------------------------------------------ unpacking
def test_int4_golden_patterns():
    path = os.path.join(GOLDEN, "int4_patterns.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 6
    words = np.array([int(r[0], 16) for r in rows], dtype=np.uint32)
    want = np.array([[int(v) for v in r[1:]] for r in rows])
    got = mo.unpack_int4(words[:, None])
    np.testing.assert_array_equal(got, want)


def test_unpack_word_order_along_k():
    # two words per row: the second word holds K elements 8..15
    w = np.array([[0x88888888, 0x76543210]], dtype=np.uint32)
    np.testing.assert_array_equal(mo.unpack_int4(w)[0], [0] * 8 + list(range(-8, 0)))


def test_bf16_exact_values():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x4300, 0xBE80], dtype=np.uint16)
    np.testing.assert_array_equal(mo.bf16_to_f64(bits),
                                  [1.0, -2.0, 1.0078125, 0.0, 128.0, -0.25])


def test_bf16_rounding_of_generator_is_nearest_even():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 (odd) and 1+2^-6 (even): rounds up.
    vals = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20], dtype=np.float32)
    np.testing.assert_array_equal(mo.bf16_to_f64(_bf16(vals)), [1.0, 1 + 2 ** -6, 1 + 2 ** -7])


def test_dequant_scales_follow_groups_and_rows():
    # row 0: q = +1 everywhere, scales (0.5, 2); row 1: q = -3, scales (4, 0.25)
    codes = np.vstack([np.full(256, 9), np.full(256, 5)])
    words = _pack_codes(codes)
    scales = _bf16([[0.5, 2.0], [4.0, 0.25]])
    w = mo.dequant(words, scales)
    np.testing.assert_array_equal(w[0, :128], 0.5)
    np.testing.assert_array_equal(w[0, 128:], 2.0)
    np.testing.assert_array_equal(w[1, :128], -12.0)
    np.testing.assert_array_equal(w[1, 128:], -0.75)


def test_dequant_unit_scale_gives_exact_integers():
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 16, size=(3, 128))
    w = mo.dequant(_pack_codes(codes), _bf16(np.ones((3, 1))))
    np.testing.assert_array_equal(w, codes - 8)


# -------------------------------------------------------------------- routing
def test_topk_matches_brute_force_over_subsets():
    rng = np.random.default_rng(11)
    T, E, k = 60, 8, 2
    logits = rng.standard_normal((T, E))
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32)
    ids, wts, sel = mo.select_topk(logits, bias, k)
    s = 1.0 / (1.0 + np.exp(-logits))
    b = bias.astype(np.float64)
    for t in range(T):
        best = max(itertools.combinations(range(E), k),
                   key=lambda c: sum(s[t, e] + b[e] for e in c))
        assert set(ids[t]) == set(best)
        # descending selection score
        v = [s[t, e] + b[e] for e in ids[t]]
        assert v == sorted(v, reverse=True)
        # unbiased scores renormalised
        want = np.array([s[t, e] for e in ids[t]])
        np.testing.assert_allclose(wts[t], want / want.sum(), rtol=0, atol=1e-15)
        assert abs(wts[t].sum() - 1.0) < 1e-12


def test_bias_selects_but_does_not_weight():
    logits = np.zeros((1, 4))
    bias = np.array([0.0, 0.5, 0.0, 0.25], dtype=np.float32)
    ids, wts, _ = mo.select_topk(logits, bias, 2)
    assert list(ids[0]) == [1, 3]
    np.testing.assert_array_equal(wts[0], [0.5, 0.5])
    # sigmoid(ln 3) = 3/4 and sigmoid(0) = 1/2: weights 3/5 and 2/5
    logits = np.array([[0.0, math.log(3.0), 0.0, 0.0]])
    ids, wts, _ = mo.select_topk(logits, np.zeros(4, np.float32), 2)
    assert list(ids[0]) == [1, 0]
    np.testing.assert_allclose(wts[0], [0.6, 0.4], rtol=0, atol=1e-15)


def test_topk_ties_take_lower_index():
    logits = np.zeros((1, 6))
    ids, _, _ = mo.select_topk(logits, np.zeros(6, np.float32), 3)
    assert list(ids[0]) == [0, 1, 2]


def test_router_logits_are_x_times_wr_transposed():
    x = _bf16([[1.0, 2.0, 0.0], [0.0, -1.0, 3.0]])
    w = np.array([[1.0, 0.0, 0.0], [0.0, 0.5, 0.5], [2.0, 2.0, 2.0], [0.0, 0.0, -1.0]],
                 dtype=np.float32)
    np.testing.assert_array_equal(mo.router_logits(x, w),
                                  [[1.0, 1.0, 6.0, 0.0], [0.0, 1.0, 4.0, -3.0]])


def test_counts_offsets_and_stable_permutation():
    rng = np.random.default_rng(3)
    T, E, k = 40, 8, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets = mo.expert_counts(ids, E)
    perm, inv = mo.stable_permutation(ids, offsets)
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    for e in range(E):
        want = [t for t in range(T) if e in ids[t]]
        assert list(perm[offsets[e]:offsets[e + 1]]) == want
    for t in range(T):
        for j in range(k):
            r = inv[t, j]
            assert perm[r] == t
            assert offsets[ids[t, j]] <= r < offsets[ids[t, j] + 1]
    assert sorted(inv.ravel()) == list(range(T * k))


def test_empty_batch_routes_to_nothing():
    ids = np.zeros((0, 2), dtype=np.int32)
    counts, offsets = mo.expert_counts(ids, 4)
    assert counts.sum() == 0 and list(offsets) == [0] * 5
    perm, inv = mo.stable_permutation(ids, offsets)
    assert perm.size == 0 and inv.shape == (0, 2)


# ---------------------------------------------------------------- expert FFN
def _direct_ffn_loops(x, codes13, s13, codes2, s2, G=128):
    """SwiGLU expert written as Python loops over the integer codes."""
    two_i, H = codes13.shape
    inter = two_i // 2
    h = []
    for i in range(inter):
        g = sum(x[kk] * (int(codes13[i, kk]) - 8) * s13[i, kk // G] for kk in range(H))
        u = sum(x[kk] * (int(codes13[inter + i, kk]) - 8) * s13[inter + i, kk // G]
                for kk in range(H))
        h.append(g / (1.0 + math.exp(-g)) * u)
    return [sum(h[i] * (int(codes2[n, i]) - 8) * s2[n, i // G] for i in range(inter))
            for n in range(codes2.shape[0])]


def test_single_expert_top1_is_dense_swiglu_ffn():
    rng = np.random.default_rng(5)
    H, I = 128, 128
    mk = lambda n, k: rng.integers(0, 16, size=(n, k))
    c13, c2 = mk(2 * I, H), mk(H, I)
    sc13, sc2 = mk(2 * I, H), mk(H, I)
    s13 = _bf16(rng.uniform(0.01, 0.03, (2 * I, 1)))
    s2 = _bf16(rng.uniform(0.01, 0.03, (H, 1)))
    ss13 = _bf16(rng.uniform(0.01, 0.03, (2 * I, 1)))
    ss2 = _bf16(rng.uniform(0.01, 0.03, (H, 1)))
    x = _bf16(rng.standard_normal((2, H)))
    routed = {"w13_q": _pack_codes(c13), "w13_s": s13, "w2_q": _pack_codes(c2), "w2_s": s2}
    shared = {"w13_q": _pack_codes(sc13), "w13_s": ss13, "w2_q": _pack_codes(sc2), "w2_s": ss2}
    rw = rng.standard_normal((1, H)).astype(np.float32)
    res = mo.moe_forward(x, rw, np.zeros(1, np.float32), [routed], shared, k=1)
    np.testing.assert_array_equal(res["ids"], [[0], [0]])
    np.testing.assert_array_equal(res["weights"], [[1.0], [1.0]])
    xf = mo.bf16_to_f64(x)
    f = lambda v: mo.bf16_to_f64(v)
    for t in range(2):
        want = np.add(_direct_ffn_loops(xf[t], c13, f(s13), c2, f(s2)),
                      _direct_ffn_loops(xf[t], sc13, f(ss13), sc2, f(ss2)))
        np.testing.assert_allclose(res["out"][t], want, rtol=1e-12, atol=1e-12)


def test_constant_weights_closed_form():
    # q = c1 and scale sigma in w13: every gate/up channel equals sigma*c1*sum(x);
    # q = c2 and scale tau in w2: every output equals I * tau * c2 * silu(a) * a
    H, I = 256, 128
    c1, c2, sigma, tau = 3, -2, 0.0625, 0.125
    w13 = {"w13_q": _pack_codes(np.full((2 * I, H), c1 + 8)),
           "w13_s": _bf16(np.full((2 * I, H // 128), sigma)),
           "w2_q": _pack_codes(np.full((H, I), c2 + 8)),
           "w2_s": _bf16(np.full((H, I // 128), tau))}
    x = _bf16(np.linspace(-1, 1, H)[None, :] * 0.5 + 0.1)
    xf = mo.bf16_to_f64(x)[0]
    a = sigma * c1 * xf.sum()
    want = I * tau * c2 * (a / (1 + math.exp(-a))) * a
    res = mo.moe_forward(x, np.ones((1, H), np.float32), np.zeros(1, np.float32),
                         [w13], w13, k=1)
    np.testing.assert_allclose(res["out"][0], np.full(H, 2 * want), rtol=1e-13)


# ------------------------------------------------------------ whole-layer laws
@pytest.fixture(scope="module")
def tiny():
    shape = ms.CONFIGS["tiny16"]
    def margin(rows):
        return mo.selection_margin(mo.router_logits(rows, ms.router_weights(shape)),
                                   ms.router_bias(shape), shape.top_k)
    return ms.make_layer(shape, margin_fn=margin)


def _fwd(layer, **kw):
    s = layer.shape
    return mo.moe_forward(kw.get("x", layer.x), layer.router_w, layer.router_b,
                          kw.get("experts", layer.experts), kw.get("shared", layer.shared),
                          s.top_k, token_subset=kw.get("subset"))


def test_tiny_layer_margins_and_weight_sums(tiny):
    r = _fwd(tiny)
    m = mo.selection_margin(r["logits"], tiny.router_b, tiny.shape.top_k)
    assert (m >= 1e-3).all()
    np.testing.assert_allclose(r["weights"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert r["counts"].sum() == tiny.shape.tokens * tiny.shape.top_k
    for row in r["ids"]:
        assert len(set(row)) == len(row)


def test_token_permutation_permutes_outputs(tiny):
    r = _fwd(tiny)
    p = np.random.default_rng(2).permutation(tiny.shape.tokens)
    rp = _fwd(tiny, x=tiny.x[p])
    np.testing.assert_array_equal(rp["ids"], r["ids"][p])
    np.testing.assert_allclose(rp["out"], r["out"][p], rtol=1e-13, atol=1e-15)


def test_zero_routed_scales_leave_shared_expert(tiny):
    zero = [dict(w, w2_s=np.zeros_like(w["w2_s"])) for w in tiny.experts]
    r = _fwd(tiny, experts=zero)
    w13, w2 = mo.expert_dense(tiny.shared)
    shared_only = mo.swiglu_expert(mo.bf16_to_f64(tiny.x), w13, w2)
    np.testing.assert_allclose(r["out"], shared_only, rtol=1e-13, atol=1e-15)


def test_routed_part_is_linear_in_down_scales(tiny):
    base = _fwd(tiny)
    w13, w2 = mo.expert_dense(tiny.shared)
    shared_only = mo.swiglu_expert(mo.bf16_to_f64(tiny.x), w13, w2)
    # doubling a bf16 scale is exact (exponent + 1)
    twice = [dict(w, w2_s=_bf16(2.0 * mo.bf16_to_f64(w["w2_s"]))) for w in tiny.experts]
    r2 = _fwd(tiny, experts=twice)
    np.testing.assert_allclose(r2["out"] - shared_only, 2 * (base["out"] - shared_only),
                               rtol=1e-12, atol=1e-14)


def test_token_subset_matches_full_forward(tiny):
    full = _fwd(tiny)
    sub = [3, 0, 15, 7]
    r = _fwd(tiny, subset=sub)
    np.testing.assert_allclose(r["out"], full["out"][sub], rtol=1e-12, atol=1e-14)


def test_routing_decision_same_in_fp32_on_guarded_inputs(tiny):
    # The pages keep the router in fp32; on inputs whose k-th/(k+1)-th margin
    # is at least 1e-3 an fp32 evaluation must take the same decision.
    r = _fwd(tiny)
    x32 = mo.bf16_to_f64(tiny.x).astype(np.float32)
    logit32 = x32 @ tiny.router_w.T
    s32 = np.float32(1) / (np.float32(1) + np.exp(-logit32))
    sel32 = s32 + tiny.router_b[None, :]
    ids32 = np.argsort(-sel32, axis=1, kind="stable")[:, :tiny.shape.top_k]
    np.testing.assert_array_equal(ids32, r["ids"])


def test_generator_is_deterministic_and_in_range():
    shape = ms.CONFIGS["tiny16"]
    a, b = ms.expert_weights(shape, 3), ms.expert_weights(shape, 3)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
    s = mo.bf16_to_f64(a["w13_s"])
    lo, hi = 0.5 / (8 * 16), 1.5 / (8 * 16)
    assert s.min() >= lo * (1 - 2 ** -8) and s.max() <= hi * (1 + 2 ** -8)
    q = mo.unpack_int4(a["w13_q"])
    assert q.min() == -8 and q.max() == 7
    assert abs(q.mean() + 0.5) < 0.05   # uniform on [-8, 7] has mean -1/2


def test_zipf_bias_gives_zipf_popularity_on_workload_tokens():
    # The stored bias was fitted on a calibration draw; on the workload's own
    # tokens the routed row counts must still follow Zipf(1.1): the rank-r
    # count falls like r^-1.1 over the head, one expert saturates near T rows,
    # and a long tail of experts gets under 10 rows.
    shape = ms.CONFIGS["zipf2048"]
    x = ms.tokens(shape)
    logits = mo.router_logits(x, ms.router_weights(shape))
    ids, _, _ = mo.select_topk(logits, ms.router_bias(shape), shape.top_k)
    counts = np.sort(mo.expert_counts(ids, shape.experts)[0])[::-1].astype(np.float64)
    assert counts[0] >= 0.9 * shape.tokens
    assert (counts < 10).sum() >= 60
    r = np.arange(2, 41)
    slope = np.polyfit(np.log(r), np.log(counts[1:40]), 1)[0]
    assert -1.35 < slope < -0.85, slope


# ------------------------------------------------------------ selection margin
def test_selection_margin_closed_form_with_bias():
    # logits (ln 3, 0, -ln 3, 0) give s = (3/4, 1/2, 1/4, 1/2); with the bias
    # (0, 0.4, 0.6875, 0.125) the selection scores are (0.75, 0.9, 0.9375, 0.625):
    # sorted 0.9375 > 0.9 > 0.75 > 0.625, so k = 1, 2, 3 give the gaps 0.0375,
    # 0.15 and 0.125. Without the bias (s alone: 0.75, 0.5, 0.5, 0.25) they
    # would be 0.25, 0 and 0.25; with k off by one they would be permuted.
    logits = np.array([[math.log(3.0), 0.0, -math.log(3.0), 0.0]])
    bias = np.array([0.0, 0.4, 0.6875, 0.125], dtype=np.float32)
    want = {1: 0.0375, 2: 0.15, 3: 0.125}
    for k, g in want.items():
        got = mo.selection_margin(logits, bias, k)
        assert got.shape == (1,)
        # 0.4 is not exact in fp32 (0.4 + 6e-9)
        assert abs(got[0] - g) < 1e-7, (k, got)


def test_selection_margin_distinct_gaps_locate_k():
    # selection scores whose consecutive gaps are all different: 0.9, 0.8,
    # 0.55, 0.5 (logits 0, so s = 1/2, plus a bias); the k-th/(k+1)-th gap is
    # 0.1 for k = 1, 0.25 for k = 2 and 0.05 for k = 3, so an off-by-one in k
    # or a swapped pair cannot pass
    bias = np.array([0.05, 0.3, 0.4, 0.0], dtype=np.float32)  # sel 0.55 0.8 0.9 0.5
    logits = np.zeros((1, 4))
    want = {1: 0.1, 2: 0.25, 3: 0.05}
    for k, g in want.items():
        np.testing.assert_allclose(mo.selection_margin(logits, bias, k), [g], rtol=0, atol=1e-7)


def test_selection_margin_brute_force_and_topk_boundary():
    # random rows: the margin equals the gap between the k-th and (k+1)-th
    # value of a plain Python sort of sigmoid(logit) + bias, and it is the
    # smallest chosen selection score minus the largest unchosen one
    rng = np.random.default_rng(17)
    T, E, k = 50, 12, 3
    logits = rng.standard_normal((T, E)) * 2
    bias = (rng.standard_normal(E) * 0.2).astype(np.float32)
    m = mo.selection_margin(logits, bias, k)
    ids, _, sel = mo.select_topk(logits, bias, k)
    for t in range(T):
        vals = sorted((1.0 / (1.0 + math.exp(-float(logits[t, e]))) + float(bias[e])
                       for e in range(E)), reverse=True)
        assert abs(m[t] - (vals[k - 1] - vals[k])) < 1e-14
        chosen = [sel[t, e] for e in ids[t]]
        rest = [sel[t, e] for e in range(E) if e not in set(ids[t])]
        assert abs(m[t] - (min(chosen) - max(rest))) < 1e-15
        assert m[t] >= 0.0


def test_selection_margin_zero_on_a_tie():
    # two experts tie for the k-th place: the margin is exactly 0, which the
    # input guard (margin < 1e-3) rejects
    logits = np.array([[1.0, 0.5, 0.5, -1.0]])
    np.testing.assert_array_equal(mo.selection_margin(logits, np.zeros(4, np.float32), 2), [0.0])


# ------------------------------------------------ test helper on the oracle
def test_parallel_oracle_outputs_equal_moe_forward(tiny):
    from tests import moe_cases as mc
    r = _fwd(tiny)
    subset = mc.covering_tokens(r, tile_rows=3)
    assert subset.size >= 4
    # every routed expert with rows appears among the covering tokens
    got_e = set(np.unique(r["ids"][subset]).tolist())
    assert got_e == set(np.nonzero(r["counts"])[0].tolist())
    want = _fwd(tiny, subset=subset)["out"]
    for workers in (1, 2):
        out = mc.oracle_outputs(tiny, r, subset, workers=workers)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-15)

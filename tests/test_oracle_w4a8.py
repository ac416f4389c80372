"""CPU pins of the W4A8-FP8 oracle (oracle/w4a8_oracle.py).

Each test checks the oracle against something fixed outside its own code: the
e4m3 bit layout enumerated here from the format's definition, hand-built ties
and saturation, blocks whose values are exactly representable, the W4A16
oracle on inputs where fp8 loses nothing, and invariances. One test plants the
missing-input-scale mistake of the page's Humming story in a copy of the
oracle and checks that a pin catches it.
"""
import numpy as np
import pytest

import moe_synth as ms
from oracle import moe_oracle as mo
from oracle import w4a8_oracle as w8


def _e4m3_table():
    """Every finite e4m3 value, from the format: sign, 4 exponent bits (bias
    7), 3 mantissa bits; exponent 0 is subnormal (m * 2^-9); exponent 15 with
    mantissa 7 is NaN. Returned with each value's mantissa LSB (for ties)."""
    vals, lsb = [], []
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
        lsb.append(m & 1)
    return np.array(vals), np.array(lsb)


def _nearest_brute(v, table, lsb):
    """Nearest table value, ties to the even mantissa, saturating at the ends."""
    a = min(abs(v), 448.0)
    pos = table[table >= 0]
    plsb = lsb[table >= 0]
    d = np.abs(pos - a)
    best = d.min()
    cand = np.nonzero(d == best)[0]
    if cand.size > 1:
        cand = cand[plsb[cand] == 0]
    return float(np.copysign(pos[cand[0]], v))


def test_e4m3_table_shape():
    t, _ = _e4m3_table()
    assert t.size == 254                       # 256 codes minus the two NaNs
    assert t.max() == 448.0 and np.min(np.abs(t[t != 0])) == 2.0 ** -9


def test_e4m3_round_matches_brute_force():
    t, lsb = _e4m3_table()
    rng = np.random.default_rng(7)
    # log-uniform magnitudes over the whole range plus the grid points and
    # their midpoints (every tie)
    pos = np.unique(t[t >= 0])
    mids = (pos[1:] + pos[:-1]) / 2
    v = np.concatenate([np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 4000)),
                        pos, mids, [0.0, 460.0, 1e6]])
    v = np.concatenate([v, -v])
    got = w8.e4m3_round(v)
    want = np.array([_nearest_brute(x, t, lsb) for x in v])
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("v,want", [
    (1.0, 1.0), (1.0625, 1.0), (1.1875, 1.25), (448.0, 448.0), (449.0, 448.0), (1e9, 448.0),
    (2.0 ** -9, 2.0 ** -9), (2.0 ** -10, 0.0), (3 * 2.0 ** -10, 2.0 ** -8), (240.0, 240.0),
    (-1.1875, -1.25), (0.0, 0.0)])
def test_e4m3_round_hand_values(v, want):
    assert w8.e4m3_round(np.array([v]))[0] == want


def test_int4_weights_are_exact_in_e4m3():
    q = np.arange(-8, 8, dtype=np.float64)
    np.testing.assert_array_equal(w8.e4m3_round(q), q)


def test_block_scale_and_codes_exact_for_representable_blocks():
    t, _ = _e4m3_table()
    rng = np.random.default_rng(3)
    rows, K = 3, 256
    codes = rng.choice(t, size=(rows, K))
    codes[:, 0] = 448.0                        # each block's amax is 448 * 2^k
    codes[:, 128] = -448.0
    k = np.array([[-3, 2], [0, 5], [-7, -1]], dtype=np.float64)
    x = codes * np.repeat(np.exp2(k), 128, axis=1)
    got_c, got_s = w8.quantize_blocks(x)
    np.testing.assert_array_equal(got_s, np.exp2(k))
    np.testing.assert_array_equal(got_c, codes)


def test_all_zero_block_gets_scale_one():
    x = np.zeros((2, 256), dtype=np.float32)
    x[1, 128:] = 1.5
    c, s = w8.quantize_blocks(x)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 0] == 1.0
    assert np.all(c[0] == 0)


def _random_expert_linear(rng, N, K):
    q = rng.integers(-8, 8, size=(N, K))
    s = rng.uniform(0.002, 0.02, size=(N, K // 128)).astype(np.float32)
    s = mo.bf16_to_f64(ms.f32_to_bf16_bits(s))     # bf16 group scales
    return q, s


def _representable_rows(rng, rows, K):
    """Rows whose every 128-block is e4m3 codes times 2^k with amax 448 * 2^k."""
    t, _ = _e4m3_table()
    c = rng.choice(t, size=(rows, K))
    c[:, ::128] = 448.0
    k = rng.integers(-10, 3, size=(rows, K // 128)).astype(np.float64)
    return c * np.repeat(np.exp2(k), 128, axis=1)


def test_linear_equals_dense_product_when_fp8_is_exact():
    rng = np.random.default_rng(11)
    N, K, rows = 48, 384, 5
    q, s = _random_expert_linear(rng, N, K)
    x = _representable_rows(rng, rows, K)
    c, xs = w8.quantize_blocks(x)
    dense_w = q * np.repeat(s, 128, axis=1)         # the W4A16 weights, exactly
    np.testing.assert_allclose(w8.w4a8_linear(c, xs, q, s), x @ dense_w.T, rtol=1e-12, atol=1e-12)


def test_planted_missing_input_scale_is_caught():
    """The page's Humming bug: the per-128 input scales never reach the
    accumulator. Planted in a copy of the linear, the exactness pin fails."""
    rng = np.random.default_rng(12)
    N, K, rows = 16, 256, 4
    q, s = _random_expert_linear(rng, N, K)
    x = _representable_rows(rng, rows, K)
    c, xs = w8.quantize_blocks(x)

    def linear_missing_input_scale(codes, scales, q_w, s_w, block=128):
        return w8.w4a8_linear(codes, np.ones_like(scales), q_w, s_w, block)

    want = x @ (q * np.repeat(s, 128, axis=1)).T
    bad = linear_missing_input_scale(c, xs, q, s)
    assert not np.allclose(bad, want, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(w8.w4a8_linear(c, xs, q, s), want, rtol=1e-12, atol=1e-12)


def test_linear_scales_with_powers_of_two():
    rng = np.random.default_rng(13)
    N, K, rows = 8, 256, 3
    q, s = _random_expert_linear(rng, N, K)
    x = rng.normal(size=(rows, K)).astype(np.float32)
    c1, s1 = w8.quantize_blocks(x)
    c2, s2 = w8.quantize_blocks(x * np.float32(8.0))
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(w8.w4a8_linear(c2, s2, q, s), 8.0 * w8.w4a8_linear(c1, s1, q, s))


def test_layer_close_to_w4a16_layer():
    """fp8 activations move the tiny layer's output by a few percent of the
    W4A16 oracle's (3 mantissa bits per activation), and routing is the same."""
    shape = ms.CONFIGS["tiny16"]
    layer = ms.make_layer(shape)
    experts, shared = layer.experts, layer.shared
    a16 = mo.moe_forward(layer.x, layer.router_w, layer.router_b, experts, shared, shape.top_k)
    a8 = w8.moe_forward_w4a8(layer.x, layer.router_w, layer.router_b, experts, shared, shape.top_k)
    np.testing.assert_array_equal(a8["ids"], a16["ids"])
    rel = np.linalg.norm(a8["out"] - a16["out"]) / np.linalg.norm(a16["out"])
    assert 1e-4 < rel < 0.08


# ---------------------------------------------------------------------------
# The expert and the layer against an independent brute-force composition:
# its own nibble unpacking and bf16 decoding, the nearest-e4m3 search over the
# enumerated code table (above), per-block scales from the fp32 amax, and the
# per-block scaled dot products summed in fp64.

def _bf16_value(bits):
    b = (np.asarray(bits, dtype=np.uint32) * np.uint32(65536)).astype(np.uint32)
    return b.view(np.float32).astype(np.float64)


def _unpack_brute(words):
    w = np.asarray(words, dtype=np.int64)
    cols = [((w // (16 ** j)) % 16) - 8 for j in range(8)]     # code j at bits 4j..4j+3
    return np.stack(cols, axis=-1).reshape(w.shape[0], -1)


def _nearest_table(v, table, lsb):
    """Vectorised brute force: nearest e4m3 value, ties to the even mantissa,
    saturating at +-448."""
    a = np.minimum(np.abs(v), 448.0)
    pos = table[table >= 0]
    plsb = lsb[table >= 0]
    d = np.abs(pos[None, :] - a[:, None])
    best = d.min(axis=1, keepdims=True)
    tie = (d == best)
    # among the tied grid points prefer the even mantissa, else the only one
    pick = np.where(tie & (plsb[None, :] == 0), 1, 0) * 2 + tie.astype(int)
    return np.copysign(pos[np.argmax(pick, axis=1)], v)


def _quant_brute(rows32, table, lsb):
    rows32 = np.asarray(rows32, dtype=np.float32)
    R, K = rows32.shape
    codes = np.zeros((R, K))
    scales = np.zeros((R, K // 128))
    for r in range(R):
        for g in range(K // 128):
            blk = rows32[r, 128 * g:128 * (g + 1)]
            amax = np.float32(np.max(np.abs(blk)))
            sc = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
            scales[r, g] = float(sc)
            codes[r, 128 * g:128 * (g + 1)] = _nearest_table((blk / sc).astype(np.float64), table, lsb)
    return codes, scales


def _linear_brute(codes, scales, q, s_w):
    R, K = codes.shape
    N = q.shape[0]
    y = np.zeros((R, N))
    for g in range(K // 128):
        part = codes[:, 128 * g:128 * (g + 1)] @ q[:, 128 * g:128 * (g + 1)].T.astype(np.float64)
        y += part * scales[:, g:g + 1] * s_w[None, :, g]
    return y


def _expert_brute(x_rows, wts, table, lsb):
    q13 = _unpack_brute(wts["w13_q"])
    s13 = _bf16_value(wts["w13_s"])
    q2 = _unpack_brute(wts["w2_q"])
    s2 = _bf16_value(wts["w2_s"])
    inter = q13.shape[0] // 2
    xc, xs = _quant_brute(x_rows, table, lsb)
    gu = _linear_brute(xc, xs, q13, s13)
    g, u = gu[:, :inter], gu[:, inter:]
    h = g / (1.0 + np.exp(-g)) * u
    hc, hs = _quant_brute(h.astype(np.float32), table, lsb)
    return _linear_brute(hc, hs, q2, s2)


def test_expert_equals_brute_force_composition():
    table, lsb = _e4m3_table()
    shape = ms.CONFIGS["tiny16"]
    layer = ms.make_layer(shape)
    x = _bf16_value(layer.x[:6])
    for wts in (layer.experts[3], layer.shared):
        want = _expert_brute(x, wts, table, lsb)
        got = w8.swiglu_expert_w4a8(x, wts)
        np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12 * np.abs(want).max())


def test_expert_brute_force_sees_the_h_quantisation():
    """The brute-force expert without the fp8 step on h differs from the
    oracle's expert (the composition pin would catch a dropped h quantisation)."""
    table, lsb = _e4m3_table()
    shape = ms.CONFIGS["tiny16"]
    layer = ms.make_layer(shape)
    x = _bf16_value(layer.x[:4])
    wts = layer.experts[1]
    q13, s13 = _unpack_brute(wts["w13_q"]), _bf16_value(wts["w13_s"])
    q2, s2 = _unpack_brute(wts["w2_q"]), _bf16_value(wts["w2_s"])
    xc, xs = _quant_brute(x, table, lsb)
    gu = _linear_brute(xc, xs, q13, s13)
    inter = q13.shape[0] // 2
    h = gu[:, :inter] / (1.0 + np.exp(-gu[:, :inter])) * gu[:, inter:]
    no_hq = h @ (q2 * np.repeat(s2, 128, axis=1)).T
    got = w8.swiglu_expert_w4a8(x, wts)
    assert not np.allclose(got, no_hq, rtol=1e-6, atol=1e-9)


def test_layer_equals_brute_force_composition():
    """moe_forward_w4a8 on the tiny layer: routing from the W4A16 oracle (pinned
    by its own tests), every (token, slot) expert and the shared expert by the
    brute force above, combined in slot order."""
    table, lsb = _e4m3_table()
    shape = ms.CONFIGS["tiny16"]
    layer = ms.make_layer(shape)
    got = w8.moe_forward_w4a8(layer.x, layer.router_w, layer.router_b, layer.experts,
                              layer.shared, shape.top_k)
    r = mo.route(layer.x, layer.router_w, layer.router_b, shape.experts, shape.top_k)
    x = _bf16_value(layer.x)
    want = np.zeros_like(x)
    for t in range(x.shape[0]):
        row = x[t:t + 1]
        acc = _expert_brute(row, layer.shared, table, lsb)[0]
        for j in range(shape.top_k):
            e = int(r["ids"][t, j])
            acc = acc + r["weights"][t, j] * _expert_brute(row, layer.experts[e], table, lsb)[0]
        want[t] = acc
    np.testing.assert_array_equal(got["ids"], r["ids"])
    np.testing.assert_allclose(got["out"], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())

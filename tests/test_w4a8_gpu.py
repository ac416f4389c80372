"""GPU parity of the W4A8-FP8 building blocks (include/moe_w4a8.h) against
the W4A8 oracle (oracle/w4a8_oracle.py), through the C ABI:

- the per-(row, 128-block) e4m3 quantisation: codes and scales identical to
  the oracle's (the same fp32 amax, fp32 division, nearest-even rounding and
  saturation), including all-zero blocks, saturating and subnormal values;
- the block-scaled INT4 x e4m3 linear: equal to the oracle's fp64 sum of
  per-block scaled partials, within fp32 accumulation inside a block;
- both composed into one expert (quantise x, gate/up, SwiGLU, quantise h,
  down) against the oracle's expert.
"""
import numpy as np
import pytest
import torch

import moe_synth as ms
import w4a16_routed_expert_router_gb300 as moe
from oracle import moe_oracle as mo
from oracle import w4a8_oracle as w8

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _e4m3_values():
    """Value of every e4m3 byte (OCP E4M3FN), from the format's definition."""
    v = np.zeros(256)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            v[code] = np.nan
            continue
        x = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        v[code] = -x if s else x
    return v


E4M3 = _e4m3_values()


def _quantize_gpu(x32):
    rows, K = x32.shape
    x = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(DEV)
    codes = torch.empty((rows, K), dtype=torch.uint8, device=DEV)
    scales = torch.empty((rows, K // 128), dtype=torch.float32, device=DEV)
    moe.moe_w4a8_quantize_blocks(x, codes, scales)
    torch.cuda.synchronize()
    return codes, scales


def _linear_gpu(codes, scales, q_words, s_bits):
    rows = codes.shape[0]
    N = q_words.shape[0]
    wq = torch.from_numpy(q_words.view(np.int32)).to(DEV)
    ws = torch.from_numpy(s_bits.view(np.int16)).to(DEV)
    y = torch.empty((rows, N), dtype=torch.float32, device=DEV)
    moe.moe_w4a8_linear(codes, scales, wq, ws, y)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def _rand_rows(rng, rows, K):
    x = rng.normal(size=(rows, K)).astype(np.float32)
    if rows > 2:
        x[1, :128] = 0.0                                     # all-zero block: scale 1
        x[2, 5] = 3.0e4                                      # one large value: the rest go subnormal
    return x


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.lib()


@pytest.mark.parametrize("rows,K", [(1, 128), (7, 256), (33, 1024), (64, 4096)])
def test_quantize_equals_oracle(rows, K):
    rng = np.random.default_rng(rows * 1000 + K)
    x = _rand_rows(rng, rows, K)
    codes, scales = _quantize_gpu(x)
    want_c, want_s = w8.quantize_blocks(x)
    got_c = E4M3[codes.cpu().numpy()]
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), want_s)
    np.testing.assert_array_equal(got_c, want_c)


def test_quantize_saturates_and_rounds_ties_to_even():
    # one block whose amax is 448 (scale exactly 1): the other values land on
    # e4m3 grid midpoints and beyond
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0] = 448.0
    mids = np.array([1.0625, 1.1875, 17.0, 19.0, 240.0, 2.0 ** -10, 3 * 2.0 ** -10, -1.1875],
                    dtype=np.float32)
    x[0, 1:1 + mids.size] = mids
    codes, scales = _quantize_gpu(x)
    assert float(scales.cpu().numpy()[0, 0]) == 1.0
    np.testing.assert_array_equal(E4M3[codes.cpu().numpy()], w8.quantize_blocks(x)[0])


def _weights(rng, N, K):
    q = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s = rng.uniform(0.002, 0.02, size=(N, K // 128)).astype(np.float32)
    s_bits = ms.f32_to_bf16_bits(s)
    return q, moe.moe_w4a16_pack_int4(q), s_bits


@pytest.mark.parametrize("rows,K,N", [(1, 128, 16), (5, 256, 48), (19, 1024, 128), (16, 4096, 512)])
def test_linear_equals_oracle(rows, K, N):
    rng = np.random.default_rng(rows + K + N)
    q, words, s_bits = _weights(rng, N, K)
    x = _rand_rows(rng, rows, K)
    codes, scales = _quantize_gpu(x)
    c64 = E4M3[codes.cpu().numpy()]
    xs64 = scales.cpu().numpy().astype(np.float64)
    want = w8.w4a8_linear(c64, xs64, q, mo.bf16_to_f64(s_bits))
    got = _linear_gpu(codes, scales, words, s_bits)
    err = np.abs(got - want)
    assert err.max() <= 1e-4 * np.abs(want).max() + 1e-7
    assert np.linalg.norm(got - want) <= 2e-5 * np.linalg.norm(want)


def test_linear_applies_the_input_scales():
    """Scaling one row's input by 2^k scales that row's output by 2^k (its
    codes are unchanged, only the block scales move) and no other row's."""
    rng = np.random.default_rng(5)
    q, words, s_bits = _weights(rng, 32, 256)
    x = _rand_rows(rng, 8, 256)
    x2 = x.copy()
    x2[3] *= np.float32(64.0)
    y1 = _linear_gpu(*_quantize_gpu(x), words, s_bits)
    y2 = _linear_gpu(*_quantize_gpu(x2), words, s_bits)
    np.testing.assert_array_equal(y2[3], 64.0 * y1[3])
    np.testing.assert_array_equal(np.delete(y2, 3, axis=0), np.delete(y1, 3, axis=0))


def test_blocks_compose_to_the_oracle_expert():
    shape = ms.CONFIGS["tiny16"]
    layer = ms.make_layer(shape)
    wts = layer.experts[2]
    x = mo.bf16_to_f64(layer.x[:11])
    inter = shape.inter
    codes, scales = _quantize_gpu(x.astype(np.float32))
    wq13 = torch.from_numpy(wts["w13_q"].view(np.int32)).to(DEV)
    ws13 = torch.from_numpy(wts["w13_s"].view(np.int16)).to(DEV)
    gu = torch.empty((x.shape[0], 2 * inter), dtype=torch.float32, device=DEV)
    moe.moe_w4a8_linear(codes, scales, wq13, ws13, gu)
    g, u = gu[:, :inter], gu[:, inter:]
    h = (g / (1.0 + torch.exp(-g)) * u).contiguous()
    hcodes = torch.empty((x.shape[0], inter), dtype=torch.uint8, device=DEV)
    hscales = torch.empty((x.shape[0], inter // 128), dtype=torch.float32, device=DEV)
    moe.moe_w4a8_quantize_blocks(h, hcodes, hscales)
    wq2 = torch.from_numpy(wts["w2_q"].view(np.int32)).to(DEV)
    ws2 = torch.from_numpy(wts["w2_s"].view(np.int16)).to(DEV)
    y = torch.empty((x.shape[0], shape.hidden), dtype=torch.float32, device=DEV)
    moe.moe_w4a8_linear(hcodes, hscales, wq2, ws2, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    want = w8.swiglu_expert_w4a8(x, wts)
    # fp32 on the GPU against fp64: h may sit on the other side of an e4m3
    # rounding boundary for a few elements, so the bound is the layer's
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= 5e-3
    assert np.abs(got - want).max() <= 2e-2 * np.abs(want).max() + 1e-3


# ------------------------------------------------------------ the W4A8 layer
from moe_synth.device import upload_layer, upload_tokens  # noqa: E402
from tests import moe_cases as mc  # noqa: E402


def _layer_w4a8(layer, tensors, max_tokens, bias=None):
    s = layer.shape
    t = dict(tensors)
    if bias is not None:
        t["router_bias"] = torch.from_numpy(np.asarray(bias, np.float32)).to(DEV)
    return moe.MoeLayer(s.hidden, s.experts, s.top_k, s.inter, s.shared_inter, max_tokens, t,
                        flags=moe.MOE_W4A16_FLAG_W4A8)


def _w4a8_ref(layer, subset):
    """The W4A8 oracle's output rows for ``subset``: each token's experts on
    its own row (the fp8 blocks are per row, so this equals the batched
    oracle), weights generated per expert from the shape's seeds."""
    shape = layer.shape
    r = mo.route(layer.x, layer.router_w, layer.router_b, shape.experts, shape.top_k)
    x = mo.bf16_to_f64(layer.x)
    shared = ms.expert_weights(shape, shape.experts) if shape.shared_inter else None
    cache = {}
    out = np.zeros((len(subset), shape.hidden))
    for i, t in enumerate(subset):
        row = x[t:t + 1]
        acc = w8.swiglu_expert_w4a8(row, shared)[0] if shared is not None else np.zeros(shape.hidden)
        for j in range(shape.top_k):
            e = int(r["ids"][t, j])
            if e not in cache:
                cache[e] = ms.expert_weights(shape, e)
            acc = acc + r["weights"][t, j] * w8.swiglu_expert_w4a8(row, cache[e])[0]
        out[i] = acc
    return r, out


@pytest.fixture(scope="module")
def tiny_w4a8():
    shape = ms.CONFIGS["tiny16"]
    return shape, upload_layer(mc.weights_of(shape), DEV)[0]


@pytest.mark.parametrize("T", [1, 5, 16, 65, 200])
def test_w4a8_layer_tiny(tiny_w4a8, T):
    shape, tensors = tiny_w4a8
    layer = mc.layer_with_tokens(shape, T)
    want = w8.moe_forward_w4a8(layer.x, layer.router_w, layer.router_b, layer.experts,
                               layer.shared, shape.top_k)
    obj = _layer_w4a8(layer, tensors, T)
    x = upload_tokens(layer.x, DEV)
    out = obj.forward(x)
    torch.cuda.synchronize()
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    rt = obj.routing(T)
    names = [n for n, _ in moe.moe_w4a16_last_launches(obj.handle)]
    obj.close()
    mc.check_routing(rt, want, shape.experts)
    mc.check_output(out.cpu().numpy(), want["out"])
    assert "w4a8_gate_up_swiglu" in names and "w4a8_down" in names


def test_w4a8_layer_differs_from_w4a16(tiny_w4a8):
    """The flag changes the arithmetic: the W4A8 output is not the W4A16 one."""
    shape, tensors = tiny_w4a8
    layer = mc.layer_with_tokens(shape, 16)
    x = upload_tokens(layer.x, DEV)
    a = _layer_w4a8(layer, tensors, 16)
    o8 = a.forward(x).cpu().numpy()
    a.close()
    t = dict(tensors)
    b = moe.MoeLayer(shape.hidden, shape.experts, shape.top_k, shape.inter, shape.shared_inter, 16, t)
    o16 = b.forward(x).cpu().numpy()
    b.close()
    assert (o8 != o16).mean() > 0.5


@pytest.fixture(scope="module")
def full_w4a8():
    return upload_layer(mc.weights_of(ms.CONFIGS["decode1"]), DEV)[0]


@pytest.mark.parametrize("name,n", [("decode1", 1), ("decode64", 6)])
def test_w4a8_layer_full_size_sampled(full_w4a8, name, n):
    shape = ms.CONFIGS[name]
    tensors = full_w4a8
    layer = mc.layer_with_tokens(shape)
    T = shape.tokens
    obj = _layer_w4a8(layer, tensors, T, bias=layer.router_b)
    out = obj.forward(upload_tokens(layer.x, DEV))
    torch.cuda.synchronize()
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    rt = obj.routing(T)
    obj.close()
    subset = np.linspace(0, T - 1, n).astype(np.int64)
    r, want = _w4a8_ref(layer, subset)
    mc.check_routing(rt, r, shape.experts)
    mc.check_output(out.cpu().numpy()[subset], want)

"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every output. The full-size V4-Flash-shaped workloads
compare routing for every token; outputs for every token at 1 and 64 tokens,
and at 2048 and 8192 tokens for a covering set: the tokens of the first and
last row of every active expert's segment (and of every 256-row tile of a
longer one), so that every routed expert's weights, every row-tile boundary
and every output channel are checked.
"""
import numpy as np
import pytest

import moe_synth as ms
from moe_synth.device import upload_layer, upload_tokens
from tests import moe_cases as mc

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(1800)]

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import w4a16_routed_expert_router_gb300 as moe  # noqa: E402
from w4a16_routed_expert_router_gb300 import _build  # noqa: E402

_build.build()
DEV = "cuda:0"


def _layer_obj(layer, tensors, max_tokens, flags=0, bias=None):
    s = layer.shape
    t = dict(tensors)
    if bias is not None:
        t["router_bias"] = torch.from_numpy(np.asarray(bias, np.float32)).to(DEV)
    return moe.MoeLayer(s.hidden, s.experts, s.top_k, s.inter, s.shared_inter, max_tokens, t,
                        flags=flags)


def _run(obj, x_bits):
    x = upload_tokens(x_bits, DEV)
    out = obj.forward(x)
    torch.cuda.synchronize()
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    return out.cpu().numpy(), obj.routing(x_bits.shape[0])


# ------------------------------------------------------------------ tiny layer
@pytest.fixture(scope="module")
def tiny():
    shape = ms.CONFIGS["tiny16"]
    base = mc.weights_of(shape)
    tensors = upload_layer(base, DEV)[0]
    return shape, tensors


@pytest.mark.parametrize("T", [16, 1, 2, 3, 7, 8, 9, 15, 17, 31, 33, 63, 64, 65, 100, 129, 200])
def test_tiny_layer_parity(tiny, T):
    shape, tensors = tiny
    layer = mc.layer_with_tokens(shape, T)
    ref = mc.oracle(layer)
    obj = _layer_obj(layer, tensors, max_tokens=256)
    out, rt = _run(obj, layer.x)
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    obj.close()


# hidden 384 (3 K-groups: a partial stage, the plain 2-D weight box), routed
# intermediate 128 (plain box) against a shared intermediate of 256 (swizzled
# box), group scales read without TMA; above 64 tokens the GEMV engine (the
# tensor-core path needs hidden % 256 == 0)
@pytest.fixture(scope="module")
def odd():
    shape = ms.MoeShape("odd384", 16, 384, 8, 2, 128, 256, 1006, 1006)
    tensors = upload_layer(mc.weights_of(shape), DEV)[0]
    return shape, tensors


@pytest.mark.parametrize("T", [1, 5, 16, 64, 65, 130])
def test_odd_shape_parity(odd, T):
    shape, tensors = odd
    layer = mc.layer_with_tokens(shape, T)
    ref = mc.oracle(layer)
    obj = _layer_obj(layer, tensors, max_tokens=256)
    out, rt = _run(obj, layer.x)
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    obj.close()


# hidden and intermediate 1024 (every K a multiple of 1024: the decode
# kernel's wide 32 KB stages) with 8 experts, top-2: at 64 tokens each expert
# holds about 16 rows, so most stages carry a full pass of 8 activation rows
# and the activation pool can hold only a few of them at once; ragged passes
# at the other sizes. Above 64 tokens the tensor-core path.
@pytest.fixture(scope="module")
def wide():
    shape = ms.MoeShape("wide1024", 16, 1024, 8, 2, 1024, 1024, 1008, 1008)
    tensors = upload_layer(mc.weights_of(shape), DEV)[0]
    return shape, tensors


@pytest.mark.parametrize("T", [1, 3, 8, 17, 40, 64, 96])
def test_wide_stage_parity(wide, T):
    shape, tensors = wide
    layer = mc.layer_with_tokens(shape, T)
    ref = mc.oracle(layer)
    obj = _layer_obj(layer, tensors, max_tokens=256)
    out, rt = _run(obj, layer.x)
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    obj.close()


# a layer without a shared expert (shared_inter = 0): the decode kernel, the
# tensor-core path and the GEMV engine
@pytest.fixture(scope="module")
def noshared():
    shape = ms.MoeShape("noshared", 16, 256, 8, 2, 128, 0, 1007, 1007)
    tensors = upload_layer(mc.weights_of(shape), DEV)[0]
    return shape, tensors


@pytest.mark.parametrize("flags,T", [(0, 1), (0, 16), (0, 64), (0, 65), (0, 200),
                                     (moe.MOE_W4A16_FLAG_FORCE_GEMV, 100)])
def test_no_shared_expert_parity(noshared, flags, T):
    shape, tensors = noshared
    layer = mc.layer_with_tokens(shape, T)
    ref = mc.oracle(layer)
    obj = _layer_obj(layer, tensors, max_tokens=256, flags=flags)
    out, rt = _run(obj, layer.x)
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    obj.close()


@pytest.mark.parametrize("flags,T", [
    (moe.MOE_W4A16_FLAG_FORCE_TC, 1), (moe.MOE_W4A16_FLAG_FORCE_TC, 16),
    (moe.MOE_W4A16_FLAG_FORCE_TC, 64), (moe.MOE_W4A16_FLAG_FORCE_TC, 300),
    (moe.MOE_W4A16_FLAG_FORCE_GEMV, 65), (moe.MOE_W4A16_FLAG_FORCE_GEMV, 200)])
def test_tiny_layer_parity_forced_path(tiny, flags, T):
    shape, tensors = tiny
    layer = mc.layer_with_tokens(shape, T)
    ref = mc.oracle(layer)
    obj = _layer_obj(layer, tensors, max_tokens=512, flags=flags)
    out, rt = _run(obj, layer.x)
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    names = [n for n, _ in moe.moe_w4a16_last_launches(obj.handle)]
    if flags == moe.MOE_W4A16_FLAG_FORCE_TC:
        assert "tc_gate_up_swiglu" in names and "tc_down" in names
    else:
        assert "gemv_gate_up_swiglu" in names or "decode_fused" in names
    obj.close()


def test_tiny_default_path_above_64_tokens_is_tensor_core(tiny):
    shape, tensors = tiny
    layer = mc.layer_with_tokens(shape, 65)
    obj = _layer_obj(layer, tensors, 128)
    _run(obj, layer.x)
    names = [n for n, _ in moe.moe_w4a16_last_launches(obj.handle)]
    assert names[-3:] == ["tc_gate_up_swiglu", "tc_down", "combine"]
    obj.close()


def test_tiny_hot_expert_spans_several_row_tiles(tiny):
    # 600 rows of one expert: three 256-row tiles, the last one ragged (88 rows)
    shape, tensors = tiny
    bias = np.zeros(shape.experts, np.float32)
    bias[5] = 4.0
    layer = mc.layer_with_tokens(shape, 600, bias=bias)
    ref = mc.oracle(layer)
    assert (ref["ids"][:, 0] == 5).all()
    obj = _layer_obj(layer, tensors, 600, bias=bias)
    out, rt = _run(obj, layer.x)
    assert rt["offsets"][6] - rt["offsets"][5] == 600
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    obj.close()


def test_tiny_one_expert_takes_every_token(tiny):
    shape, tensors = tiny
    bias = np.zeros(shape.experts, np.float32)
    bias[3] = 4.0
    layer = mc.layer_with_tokens(shape, 40, bias=bias)
    ref = mc.oracle(layer)
    assert (ref["ids"][:, 0] == 3).all()
    obj = _layer_obj(layer, tensors, 64, bias=bias)
    out, rt = _run(obj, layer.x)
    assert rt["offsets"][4] - rt["offsets"][3] == 40
    mc.check_routing(rt, ref, shape.experts)
    mc.check_output(out, ref["out"])
    obj.close()


def test_tiny_empty_batch_and_limits(tiny):
    shape, tensors = tiny
    layer = mc.layer_with_tokens(shape, 4)
    obj = _layer_obj(layer, tensors, 8)
    x = torch.zeros((0, shape.hidden), dtype=torch.int16, device=DEV)
    out = obj.forward(x)
    assert out.shape == (0, shape.hidden)
    assert moe.moe_w4a16_last_launches(obj.handle) == []
    big = torch.zeros((9, shape.hidden), dtype=torch.int16, device=DEV)
    with pytest.raises(moe.MoeError) as ei:
        obj.forward(big)
    assert ei.value.status == moe.MOE_W4A16_ERR_TOO_MANY_TOKENS
    # misaligned activation pointer
    raw = torch.zeros((4 * shape.hidden + 8,), dtype=torch.int16, device=DEV)
    out = torch.empty((4, shape.hidden), dtype=torch.int16, device=DEV)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_w4a16_forward(obj.handle, raw.data_ptr() + 2, 4, obj.weights, out.data_ptr(), 0)
    assert ei.value.status == moe.MOE_W4A16_ERR_MISALIGNED
    # aliasing input and output
    xx = upload_tokens(layer.x, DEV)
    with pytest.raises(moe.MoeError):
        moe.moe_w4a16_forward(obj.handle, xx.data_ptr(), 4, obj.weights, xx.data_ptr(), 0)
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    obj.close()


def test_tiny_deterministic_and_batch_invariant(tiny):
    shape, tensors = tiny
    layer = mc.layer_with_tokens(shape, 48)
    obj = _layer_obj(layer, tensors, 64)
    a, _ = _run(obj, layer.x)
    b, _ = _run(obj, layer.x)
    np.testing.assert_array_equal(a, b)
    c, _ = _run(obj, layer.x[:5])
    np.testing.assert_array_equal(c, a[:5])
    # tiny batches score with more warps; the logits' summation order is fixed
    c, _ = _run(obj, layer.x[:3])
    np.testing.assert_array_equal(c, a[:3])
    obj.close()


def test_tiny_forward_host_matches_device(tiny):
    shape, tensors = tiny
    layer = mc.layer_with_tokens(shape, 16)
    obj = _layer_obj(layer, tensors, 16)
    a, _ = _run(obj, layer.x)
    xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
    oh = torch.empty((16, shape.hidden), dtype=torch.int16).pin_memory()
    obj.forward_host(xh, oh)
    np.testing.assert_array_equal(oh.numpy(), a)
    # pinned buffers replay a recorded graph: new contents of the same buffer,
    # then a different token count (a new recording), then pageable buffers
    other = mc.layer_with_tokens(shape, 16, bias=None).x[::-1].copy()
    b, _ = _run(obj, other)
    xh.copy_(torch.from_numpy(other.view(np.int16)))
    obj.forward_host(xh, oh)
    np.testing.assert_array_equal(oh.numpy(), b)
    oh5 = torch.empty((5, shape.hidden), dtype=torch.int16).pin_memory()
    obj.forward_host(xh[:5], oh5)
    np.testing.assert_array_equal(oh5.numpy(), b[:5])
    ohp = torch.empty((16, shape.hidden), dtype=torch.int16)
    obj.forward_host(torch.from_numpy(other.view(np.int16)), ohp)
    np.testing.assert_array_equal(ohp.numpy(), b)
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    obj.close()


# ------------------------------------------------------------ full-size layer
@pytest.fixture(scope="module")
def full():
    shape = ms.CONFIGS["decode1"]
    base = mc.weights_of(shape)
    tensors = upload_layer(base, DEV)[0]
    return tensors


# oracle references of the full-size cases, shared by the tests of one module
_REFS = {}


def _full_case(full, name, sample, flags=0):
    """Run one full-size workload; routing is compared for every token,
    outputs for the tokens ``sample(route, T)`` picks."""
    shape = ms.CONFIGS[name]
    T = shape.tokens
    key = (name, sample)
    if key not in _REFS:
        layer = mc.layer_with_tokens(shape)
        route = mc.oracle(layer, subset=[])
        subset = sample(route, T)
        _REFS[key] = (layer, route, subset, mc.oracle_outputs(layer, route, subset))
    layer, route, subset, ref = _REFS[key]
    obj = _layer_obj(layer, full, T, flags=flags, bias=layer.router_b)
    out, rt = _run(obj, layer.x)
    mc.check_routing(rt, route, shape.experts)
    mc.check_output(out[subset], ref)
    names = [n for n, _ in moe.moe_w4a16_last_launches(obj.handle)]
    obj.close()
    return rt, names, subset


def _covering(route, T):
    return mc.covering_tokens(route)


def test_decode1_full_layer(full):
    rt, names, _ = _full_case(full, "decode1", lambda r, T: np.arange(T))
    assert names == ["decode_fused"]


def test_decode64_every_token(full):
    _, names, _ = _full_case(full, "decode64", lambda r, T: np.arange(T))
    assert names == ["decode_fused"]


def test_zipf2048_outputs_cover_every_active_expert(full):
    rt, names, subset = _full_case(full, "zipf2048", _covering)
    counts = np.diff(rt["offsets"])
    assert counts.max() >= 1800 and (counts < 10).sum() >= 60
    assert names[-3:] == ["tc_gate_up_swiglu", "tc_down", "combine"]
    assert subset.size >= 200


def test_zipf2048_gemv_path_covers_every_active_expert(full):
    _, names, _ = _full_case(full, "zipf2048", _covering, flags=moe.MOE_W4A16_FLAG_FORCE_GEMV)
    assert "gemv_down" in names


def test_prefill8192_outputs_cover_every_active_expert(full):
    rt, names, subset = _full_case(full, "prefill8192", _covering)
    assert (np.diff(rt["offsets"]) > 0).all()
    assert names[-3:] == ["tc_gate_up_swiglu", "tc_down", "combine"]
    assert subset.size >= 256


@pytest.mark.parametrize("name,flags,kernel", [
    ("zipf2048", 0, "tc_gate_up_swiglu"),
    ("zipf2048", "gemv", "gemv_down"),
    ("decode64", 0, "decode_fused"),
])
def test_repeated_forwards_are_bit_identical(full, name, flags, kernel):
    # Every kernel with a TMA-filled stage ring read through generic loads
    # (tensor-core dequantisers, GEMV and decode consumers) must release a
    # stage only after a proxy fence; a missing one shows up as a few K blocks
    # read from the next fill, differing from run to run. Zipf routing puts
    # ~90 experts with under 10 rows next to a 2048-row expert: tiny and full
    # N-tiles in the same persistent schedule. Every forward of the same input
    # must give the same bits.
    shape = ms.CONFIGS[name]
    layer = mc.layer_with_tokens(shape)
    f = moe.MOE_W4A16_FLAG_FORCE_GEMV if flags == "gemv" else flags
    obj = _layer_obj(layer, full, shape.tokens, flags=f, bias=layer.router_b)
    x = upload_tokens(layer.x, DEV)
    first = obj.forward(x)
    torch.cuda.synchronize()
    first = first.cpu().numpy()
    assert kernel in [n for n, _ in moe.moe_w4a16_last_launches(obj.handle)]
    for _ in range(40):
        again = obj.forward(x)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(again.cpu().numpy(), first)
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    obj.close()

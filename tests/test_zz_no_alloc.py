"""The no-allocation forward (moe_w4a16_forward_noalloc) against the regular one.

Callers that cannot allocate device memory -- code running inside CUDA-graph
stream capture, plugins confined to a framework's memory pool -- use the
entry point that runs on the library's own fixed scratch array. These tests
call it through the C ABI twice in a row (the array keeps the previous call's
contents) and compare it with moe_w4a16_forward on the same inputs, within
the layer's output tolerance. The file sorts last so that a run stopping at
its first failure has already run every other test.
"""
import numpy as np
import pytest

import moe_synth as ms
from moe_synth.device import upload_layer, upload_tokens
from tests import moe_cases as mc

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import w4a16_routed_expert_router_gb300 as moe  # noqa: E402
from w4a16_routed_expert_router_gb300 import _build  # noqa: E402

_build.build()
DEV = "cuda:0"


def _close(a_bits, b_bits):
    a = mc.bf16_bits_to_f64(a_bits)
    b = mc.bf16_bits_to_f64(b_bits)
    err = np.abs(a - b)
    assert err.max() <= mc.MAX_ERR_REL * np.abs(b).max() + mc.MAX_ERR_ABS
    assert np.linalg.norm(a - b) <= mc.FROB_REL * np.linalg.norm(b)


def _compare(shape, T, bias=None):
    layer = mc.layer_with_tokens(shape, T, bias=bias)
    tensors = upload_layer(mc.weights_of(shape), DEV)[0]
    tensors["router_bias"] = torch.from_numpy(layer.router_b).to(DEV)
    obj = moe.MoeLayer(shape.hidden, shape.experts, shape.top_k, shape.inter,
                       shape.shared_inter, max(T, 1), tensors)
    x = upload_tokens(layer.x, DEV)
    ref = obj.forward(x)
    torch.cuda.synchronize()
    assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
    ref = ref.cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full((T, shape.hidden), -1, dtype=torch.int16, device=DEV)
        moe.moe_w4a16_forward_noalloc(obj.cfg, x.data_ptr(), T, obj.weights, out.data_ptr(),
                                      stream)
        assert moe.moe_w4a16_noalloc_check_errors(stream) == 0
        _close(out.cpu().numpy(), ref)
    oracle = mc.oracle(layer)
    mc.check_output(out.cpu().numpy(), oracle["out"])
    obj.close()


def test_noalloc_matches_forward_on_tiny_layer_twice():
    _compare(ms.CONFIGS["tiny16"], 16)


def test_noalloc_matches_forward_on_full_layer_one_token_twice():
    _compare(ms.CONFIGS["decode1"], 1)


def test_noalloc_rejects_more_tokens_than_its_scratch_holds():
    shape = ms.CONFIGS["tiny16"]
    cfg = moe.make_config(shape.hidden, shape.experts, shape.top_k, shape.inter,
                          shape.shared_inter, 64)
    x = torch.zeros((moe.MOE_W4A16_NOALLOC_MAX_TOKENS + 1, shape.hidden), dtype=torch.int16,
                    device=DEV)
    out = torch.empty_like(x)
    w = moe.moe_w4a16_weights(*([x.data_ptr()] * 10))
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_w4a16_forward_noalloc(cfg, x.data_ptr(), x.shape[0], w, out.data_ptr(), 0)
    assert ei.value.status == moe.MOE_W4A16_ERR_TOO_MANY_TOKENS

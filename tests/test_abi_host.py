"""Host-side checks of the C ABI: the library builds, loads and exports every
declared symbol, and invalid arguments are rejected before any device work.
No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import w4a16_routed_expert_router_gb300 as moe
from oracle import moe_oracle as mo
from w4a16_routed_expert_router_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "moe_w4a16.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return moe.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(moe_w4a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert _declared() == sorted(moe.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


HEADER_W4A8 = os.path.join(os.path.dirname(HEADER), "moe_w4a8.h")


def test_w4a8_header_declares_the_binding_names(L):
    names = sorted(set(re.findall(r"\b(moe_w4a8_[a-z0-9_]+)\s*\(", open(HEADER_W4A8).read())))
    assert names == sorted(moe.EXPORTS_W4A8)
    for name in names:
        assert hasattr(L, name), name


def test_w4a8_calls_reject_bad_sizes_before_any_launch(L):
    # K not a multiple of 128, N not a multiple of 16, negative rows: refused
    # on the host with MOE_W4A8_INVALID_ARG (-1); rows == 0 is a no-op
    assert L.moe_w4a8_quantize_blocks(None, 4, 100, None, None, None) == -1
    assert L.moe_w4a8_quantize_blocks(None, -1, 128, None, None, None) == -1
    assert L.moe_w4a8_quantize_blocks(None, 0, 128, None, None, None) == 0
    assert L.moe_w4a8_linear(None, None, 4, 128, None, None, 20, None, None) == -1
    assert L.moe_w4a8_linear(None, None, 4, 96, None, None, 16, None, None) == -1
    assert L.moe_w4a8_linear(None, None, 0, 128, None, None, 16, None, None) == 0
    assert L.moe_w4a8_linear(None, None, 4, 128, None, None, 16, None, None) == -1  # null pointers


def _header_constants():
    """Every MOE_W4A16_* value the header defines (#define or enum member)."""
    text = open(HEADER).read()
    vals = {}
    for name, v in re.findall(r"#define\s+(MOE_W4A16_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", text):
        vals[name] = int(v, 0)
    for name, v in re.findall(r"\b(MOE_W4A16_[A-Z0-9_]+)\s*=\s*(-?\d+)", text):
        vals[name] = int(v)
    return vals


def test_binding_constants_match_the_header():
    vals = _header_constants()
    assert "MOE_W4A16_ERR_NO_DEVICE" in vals and "MOE_W4A16_DEVERR_LAYOUT" in vals
    for name, v in vals.items():
        assert getattr(moe, name, None) == v, name


def test_status_strings(L):
    assert moe.moe_w4a16_status_string(0) == "ok"
    assert "max_tokens" in moe.moe_w4a16_status_string(moe.MOE_W4A16_ERR_TOO_MANY_TOKENS)
    assert moe.moe_w4a16_status_string(-99) == "unknown status"


def _cfg(**kw):
    base = dict(hidden=4096, num_experts=256, top_k=6, inter=2048, shared_inter=2048,
                max_tokens=64, flags=0)
    base.update(kw)
    return moe.make_config(**base)


def test_workspace_bytes_of_a_valid_config(L):
    n = moe.moe_w4a16_workspace_bytes(_cfg())
    # at least: logits, activations copy, h, y for 64 tokens
    T, k, H, I, E = 64, 6, 4096, 2048, 256
    rows = T * k + T
    assert n >= T * E * 4 + T * H * 2 + rows * I * 2 + rows * H * 4


@pytest.mark.parametrize("kw, status", [
    (dict(hidden=4000), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(hidden=0), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(inter=100), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(shared_inter=-128), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(num_experts=0), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(num_experts=257), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(top_k=0), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(top_k=9), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(num_experts=4, top_k=5), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(max_tokens=0), moe.MOE_W4A16_ERR_INVALID_ARG),
    (dict(flags=0x100), moe.MOE_W4A16_ERR_INVALID_ARG),
    (dict(flags=moe.MOE_W4A16_FLAG_FORCE_GEMV | moe.MOE_W4A16_FLAG_FORCE_TC),
     moe.MOE_W4A16_ERR_INVALID_ARG),
    # W4A8 experts: not with a FORCE flag; fp32 h lives in y, so h <= hidden
    (dict(flags=moe.MOE_W4A16_FLAG_W4A8 | moe.MOE_W4A16_FLAG_FORCE_TC), moe.MOE_W4A16_ERR_INVALID_ARG),
    (dict(flags=moe.MOE_W4A16_FLAG_W4A8 | moe.MOE_W4A16_FLAG_FORCE_GEMV), moe.MOE_W4A16_ERR_INVALID_ARG),
    (dict(flags=moe.MOE_W4A16_FLAG_W4A8, hidden=1024, inter=2048), moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
    (dict(flags=moe.MOE_W4A16_FLAG_W4A8, hidden=1024, inter=512, shared_inter=2048),
     moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE),
])
def test_invalid_configs_are_rejected(L, kw, status):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_w4a16_workspace_bytes(_cfg(**kw))
    assert ei.value.status == status
    h = ctypes.c_void_p()
    assert L.moe_w4a16_create(ctypes.byref(_cfg(**kw)), 0, ctypes.byref(h)) == status
    assert not h.value


def test_w4a8_flag_is_a_valid_config(L):
    assert moe.moe_w4a16_workspace_bytes(_cfg(flags=moe.MOE_W4A16_FLAG_W4A8)) == \
        moe.moe_w4a16_workspace_bytes(_cfg())          # no extra workspace


def test_noalloc_refuses_the_w4a8_flag_before_any_device_work(L):
    c = _cfg(flags=moe.MOE_W4A16_FLAG_W4A8, max_tokens=16)
    assert L.moe_w4a16_forward_noalloc(ctypes.byref(c), None, 1, None, None, None) == \
        moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE


def test_group_size_must_be_128(L):
    c = _cfg()
    c.group_size = 64
    n = ctypes.c_size_t()
    assert L.moe_w4a16_workspace_bytes(ctypes.byref(c), ctypes.byref(n)) == \
        moe.MOE_W4A16_ERR_UNSUPPORTED_SHAPE


def test_null_handle_and_out_pointers(L):
    assert L.moe_w4a16_create(ctypes.byref(_cfg()), 0, None) == moe.MOE_W4A16_ERR_INVALID_ARG
    w = moe.moe_w4a16_weights()
    assert L.moe_w4a16_forward(None, None, 1, ctypes.byref(w), None, None) == \
        moe.MOE_W4A16_ERR_INVALID_ARG
    assert L.moe_w4a16_destroy(None) == moe.MOE_W4A16_OK
    assert L.moe_w4a16_get_routing(None, None, None, None, None, None, None) == \
        moe.MOE_W4A16_ERR_INVALID_ARG


def test_create_without_a_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert L.moe_w4a16_create(ctypes.byref(_cfg()), 0, ctypes.byref(h)) == \
        moe.MOE_W4A16_ERR_NO_DEVICE


# ------------------------------------------------------------------ packing
def test_pack_int4_matches_the_documented_patterns():
    # code j of a word holds element 8w + j as u = q + 8
    q = np.array([[-8, -7, -6, -5, -4, -3, -2, -1, 0, 1, 2, 3, 4, 5, 6, 7],
                  [0] * 16], dtype=np.int8)
    words = moe.moe_w4a16_pack_int4(q)
    assert words.dtype == np.uint32 and words.shape == (2, 2)
    assert words[0].tolist() == [0x76543210, 0xFEDCBA98]
    assert words[1].tolist() == [0x88888888, 0x88888888]


def test_pack_int4_inverts_the_oracle_unpack():
    rng = np.random.default_rng(7)
    q = rng.integers(-8, 8, size=(33, 256), dtype=np.int8)
    words = moe.moe_w4a16_pack_int4(q)
    np.testing.assert_array_equal(mo.unpack_int4(words), q.astype(np.int64))


def test_pack_int4_rejects_bad_input_without_writing():
    q = np.zeros((2, 16), dtype=np.int8)
    q[1, 3] = 8
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_w4a16_pack_int4(q)
    assert ei.value.status == moe.MOE_W4A16_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError):
        moe.moe_w4a16_pack_int4(np.zeros((2, 12), dtype=np.int8))

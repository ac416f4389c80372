"""Python binding of the GB300 W4A16 routed-expert MoE layer.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libmoe_w4a16.so`` (built in-tree by ``_build.py``). The functions
carry the names of the C ABI in ``include/moe_w4a16.h``. There is no fallback:
if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_w4a16.so")

MOE_W4A16_OK = 0
MOE_W4A16_ERR_INVALID_ARG = -1
MOE_W4A16_ERR_UNSUPPORTED_SHAPE = -2
MOE_W4A16_ERR_TOO_MANY_TOKENS = -3
MOE_W4A16_ERR_MISALIGNED = -4
MOE_W4A16_ERR_CUDA = -5
MOE_W4A16_ERR_DEVICE = -6
MOE_W4A16_ERR_NO_DEVICE = -7

MOE_W4A16_FLAG_FORCE_GEMV = 0x1
MOE_W4A16_FLAG_FORCE_TC = 0x2
MOE_W4A16_FLAG_PROFILE = 0x4
MOE_W4A16_FLAG_W4A8 = 0x8

# device error flag bits (moe_w4a16_check_device_errors)
MOE_W4A16_DEVERR_TIMEOUT = 0x1
MOE_W4A16_DEVERR_RANGE = 0x2
MOE_W4A16_DEVERR_LAYOUT = 0x4

# every symbol include/moe_w4a16.h declares
EXPORTS = (
    "moe_w4a16_workspace_bytes",
    "moe_w4a16_create",
    "moe_w4a16_destroy",
    "moe_w4a16_forward",
    "moe_w4a16_forward_host",
    "moe_w4a16_get_routing",
    "moe_w4a16_check_device_errors",
    "moe_w4a16_last_launches",
    "moe_w4a16_status_string",
    "moe_w4a16_forward_noalloc",
    "moe_w4a16_noalloc_check_errors",
    "moe_w4a16_pack_int4",
)
# the W4A8-FP8 building blocks (include/moe_w4a8.h)
EXPORTS_W4A8 = (
    "moe_w4a8_quantize_blocks",
    "moe_w4a8_linear",
)
MOE_W4A8_OK = 0
MOE_W4A16_NOALLOC_MAX_TOKENS = 16


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {moe_w4a16_status_string(status)} ({status})")
        self.status = status


class moe_w4a16_config(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("inter", ctypes.c_int32),
        ("shared_inter", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
    ]


class moe_w4a16_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_bias", "w13_q", "w13_s", "w2_q", "w2_s",
        "sh_w13_q", "sh_w13_s", "sh_w2_q", "sh_w2_s")]


_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libmoe_w4a16.so``; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m w4a16_routed_expert_router_gb300._build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
        cfgp = ctypes.POINTER(moe_w4a16_config)
        wp = ctypes.POINTER(moe_w4a16_weights)
        sig = {
            "moe_w4a16_workspace_bytes": ([cfgp, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
            "moe_w4a16_create": ([cfgp, ctypes.c_int, ctypes.POINTER(vp)], ctypes.c_int),
            "moe_w4a16_destroy": ([vp], ctypes.c_int),
            "moe_w4a16_forward": ([vp, vp, i32, wp, vp, vp], ctypes.c_int),
            "moe_w4a16_forward_host": ([vp, vp, i32, wp, vp, vp], ctypes.c_int),
            "moe_w4a16_get_routing": ([vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "moe_w4a16_check_device_errors": ([vp, u32p], ctypes.c_int),
            "moe_w4a16_last_launches": ([vp, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_char_p),
                                         ctypes.POINTER(ctypes.c_float), i32], ctypes.c_int),
            "moe_w4a16_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "moe_w4a16_forward_noalloc": ([cfgp, vp, i32, wp, vp, vp], ctypes.c_int),
            "moe_w4a16_noalloc_check_errors": ([vp, u32p], ctypes.c_int),
            "moe_w4a16_pack_int4": ([vp, ctypes.c_int64, ctypes.c_int64, vp], ctypes.c_int),
            "moe_w4a8_quantize_blocks": ([vp, i32, i32, vp, vp, vp], ctypes.c_int),
            "moe_w4a8_linear": ([vp, vp, i32, i32, vp, vp, i32, vp, vp], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != MOE_W4A16_OK:
        raise MoeError(status, what)


def moe_w4a16_status_string(status: int) -> str:
    return lib().moe_w4a16_status_string(int(status)).decode()


def make_config(hidden, num_experts, top_k, inter, shared_inter, max_tokens,
                flags=0, group_size=128) -> moe_w4a16_config:
    return moe_w4a16_config(hidden, num_experts, top_k, inter, shared_inter, group_size,
                            max_tokens, flags)


def moe_w4a16_workspace_bytes(cfg: moe_w4a16_config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_w4a16_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_w4a16_workspace_bytes")
    return n.value


def moe_w4a16_create(cfg: moe_w4a16_config, device: int = 0) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().moe_w4a16_create(ctypes.byref(cfg), device, ctypes.byref(h)), "moe_w4a16_create")
    return h


def moe_w4a16_destroy(handle) -> None:
    _check(lib().moe_w4a16_destroy(handle), "moe_w4a16_destroy")


def moe_w4a16_forward(handle, x_ptr: int, num_tokens: int, weights: moe_w4a16_weights,
                      out_ptr: int, stream: int = 0) -> None:
    _check(lib().moe_w4a16_forward(handle, x_ptr, num_tokens, ctypes.byref(weights), out_ptr,
                                   stream), "moe_w4a16_forward")


def moe_w4a16_forward_host(handle, x_host_ptr: int, num_tokens: int,
                           weights: moe_w4a16_weights, out_host_ptr: int, stream: int = 0) -> None:
    _check(lib().moe_w4a16_forward_host(handle, x_host_ptr, num_tokens, ctypes.byref(weights),
                                        out_host_ptr, stream), "moe_w4a16_forward_host")


def moe_w4a16_forward_noalloc(cfg: moe_w4a16_config, x_ptr: int, num_tokens: int,
                              weights: moe_w4a16_weights, out_ptr: int, stream: int = 0) -> None:
    """Forward on the library's fixed scratch array: no handle, no allocation."""
    _check(lib().moe_w4a16_forward_noalloc(ctypes.byref(cfg), x_ptr, num_tokens,
                                           ctypes.byref(weights), out_ptr, stream),
           "moe_w4a16_forward_noalloc")


def moe_w4a16_noalloc_check_errors(stream: int = 0) -> int:
    """Device error flags of the last no-allocation forward on this device."""
    v = ctypes.c_uint32(0)
    _check(lib().moe_w4a16_noalloc_check_errors(stream, ctypes.byref(v)),
           "moe_w4a16_noalloc_check_errors")
    return int(v.value)


def moe_w4a16_pack_int4(q):
    """Pack signed 4-bit values (int8 numpy [rows, K], values in [-8, 7]) into
    the uint32 [rows, K/8] layout of the packed weight tensors (host only)."""
    import numpy as np
    q = np.ascontiguousarray(q, dtype=np.int8)
    if q.ndim != 2:
        raise ValueError("q must be 2-D [rows, K]")
    rows, K = q.shape
    out = np.empty((rows, max(K // 8, 0)), dtype=np.uint32)
    _check(lib().moe_w4a16_pack_int4(q.ctypes.data, rows, K, out.ctypes.data),
           "moe_w4a16_pack_int4")
    return out


def moe_w4a8_quantize_blocks(x, codes, scales, stream: int = 0) -> None:
    """fp8 e4m3 codes and fp32 scales of x (fp32 [rows, K] device tensor) per
    row and 128-element block: codes uint8 [rows, K], scales fp32 [rows, K/128]."""
    rows, K = x.shape
    st = lib().moe_w4a8_quantize_blocks(x.data_ptr(), rows, K, codes.data_ptr(),
                                        scales.data_ptr(), stream)
    if st != MOE_W4A8_OK:
        raise RuntimeError(f"moe_w4a8_quantize_blocks failed ({st})")


def moe_w4a8_linear(codes, x_scales, w_q, w_s, y, stream: int = 0) -> None:
    """y[r, n] = sum_g w_s[n, g] x_scales[r, g] sum_{k in g} q[n, k] codes[r, k]
    (device tensors: codes uint8 [rows, K], x_scales fp32 [rows, K/128], w_q
    int32/uint32 [N, K/8], w_s bf16 bits [N, K/128], y fp32 [rows, N])."""
    rows, K = codes.shape
    N = w_q.shape[0]
    st = lib().moe_w4a8_linear(codes.data_ptr(), x_scales.data_ptr(), rows, K, w_q.data_ptr(),
                               w_s.data_ptr(), N, y.data_ptr(), stream)
    if st != MOE_W4A8_OK:
        raise RuntimeError(f"moe_w4a8_linear failed ({st})")


def moe_w4a16_get_routing(handle, ids=0, wts=0, offsets=0, perm=0, inv=0, stream=0) -> None:
    _check(lib().moe_w4a16_get_routing(handle, ids, wts, offsets, perm, inv, stream),
           "moe_w4a16_get_routing")


def moe_w4a16_check_device_errors(handle) -> int:
    """Synchronise and return the device error flag bits (0 when clean)."""
    flags = ctypes.c_uint32(0)
    st = lib().moe_w4a16_check_device_errors(handle, ctypes.byref(flags))
    if st not in (MOE_W4A16_OK, MOE_W4A16_ERR_DEVICE):
        _check(st, "moe_w4a16_check_device_errors")
    return flags.value


def moe_w4a16_last_launches(handle):
    """[(kernel name, ms or -1)] of the last forward (ms needs FLAG_PROFILE)."""
    n = ctypes.c_int32(0)
    cap = 16
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_float * cap)()
    _check(lib().moe_w4a16_last_launches(handle, ctypes.byref(n), names, ms, cap),
           "moe_w4a16_last_launches")
    return [(names[i].decode(), float(ms[i])) for i in range(min(n.value, cap))]


class MoeLayer:
    """A handle plus device-resident weights held as torch tensors.

    torch is used for device memory and streams only; ``forward`` passes raw
    pointers to ``moe_w4a16_forward``.
    """

    def __init__(self, hidden, num_experts, top_k, inter, shared_inter, max_tokens,
                 tensors: dict, flags: int = 0, device: int = 0):
        self.cfg = make_config(hidden, num_experts, top_k, inter, shared_inter, max_tokens, flags)
        self.hidden, self.num_experts, self.top_k = hidden, num_experts, top_k
        self.inter, self.shared_inter, self.max_tokens = inter, shared_inter, max_tokens
        self.device = device
        self.tensors = tensors  # keeps the weights alive
        self.handle = moe_w4a16_create(self.cfg, device)
        self.weights = moe_w4a16_weights(*[
            tensors[n].data_ptr() if tensors.get(n) is not None else None
            for n, _ in moe_w4a16_weights._fields_])

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            moe_w4a16_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x, out=None, stream=None):
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.hidden), dtype=torch.int16, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        moe_w4a16_forward(self.handle, x.data_ptr(), T, self.weights, out.data_ptr(),
                          s.cuda_stream)
        return out

    def forward_host(self, x_host, out_host, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        moe_w4a16_forward_host(self.handle, x_host.data_ptr(), x_host.shape[0], self.weights,
                               out_host.data_ptr(), s.cuda_stream)
        return out_host

    def routing(self, T, stream=None):
        """Routing of the last forward as host numpy arrays."""
        import torch
        dev = torch.device("cuda", self.device)
        k, E = self.top_k, self.num_experts
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        wts = torch.empty((T, k), dtype=torch.float32, device=dev)
        offs = torch.empty((E + 1,), dtype=torch.int32, device=dev)
        perm = torch.empty((T * k,), dtype=torch.int32, device=dev)
        inv = torch.empty((T * k,), dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        moe_w4a16_get_routing(self.handle, ids.data_ptr(), wts.data_ptr(), offs.data_ptr(),
                              perm.data_ptr(), inv.data_ptr(), s.cuda_stream)
        s.synchronize()
        return {"ids": ids.cpu().numpy(), "weights": wts.cpu().numpy(),
                "offsets": offs.cpu().numpy(), "perm": perm.cpu().numpy(),
                "inv": inv.cpu().numpy().reshape(T, k)}

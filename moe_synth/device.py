"""Copy storage-format inputs (numpy) into device tensors (torch) for the CUDA path.

Pure data movement: bf16 bit patterns travel as int16 tensors, packed INT4
words as int32 tensors (bit-identical views of the uint32 words).
"""
from __future__ import annotations

import numpy as np

from . import LayerInputs


def _dev(a: np.ndarray, device):
    import torch
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def upload_layer(layer: LayerInputs, device="cuda:0", copies: int = 1) -> list:
    """Device tensors named like the C ABI's weight struct (one dict per copy).

    ``copies > 1`` makes independent copies of the routed-expert weights (the
    router and shared expert too), used to defeat cache residency in timing.
    """
    import torch
    s = layer.shape
    E, H, I, Is = s.experts, s.hidden, s.inter, s.shared_inter
    out = []
    for _ in range(copies):
        t = {
            "router_w": _dev(layer.router_w, device),
            "router_bias": _dev(layer.router_b, device),
            "w13_q": torch.empty((E, 2 * I, H // 8), dtype=torch.int32, device=device),
            "w13_s": torch.empty((E, 2 * I, H // 128), dtype=torch.int16, device=device),
            "w2_q": torch.empty((E, H, I // 8), dtype=torch.int32, device=device),
            "w2_s": torch.empty((E, H, I // 128), dtype=torch.int16, device=device),
        }
        for e, w in enumerate(layer.experts):
            for key in ("w13_q", "w13_s", "w2_q", "w2_s"):
                t[key][e].copy_(_dev(w[key], "cpu"))
        if Is and layer.shared is not None:
            for key in ("w13_q", "w13_s", "w2_q", "w2_s"):
                t["sh_" + key] = _dev(layer.shared[key], device)
        out.append(t)
    return out


def upload_tokens(x_bits: np.ndarray, device="cuda:0"):
    return _dev(x_bits, device)

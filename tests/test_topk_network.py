"""CPU checks of the warp top-k's in-lane sorting network (csrc/topk.cuh).

The kernel sorts each lane's 8 (key, expert) entries with a fixed list of
compare-exchanges, then takes the lane heads in rounds. The list is read
from the header here, so the test follows the code:
- by the 0-1 principle, a comparator network sorts every input if it sorts
  all 2^8 inputs of zeros and ones; checked exhaustively;
- with the kernel's comparator rule (larger key first, equal keys by the lower
  expert index), the network followed by the k head-taking rounds selects
  exactly what a full stable sort of all the experts selects, on random and
  tie-heavy scores (the routing's tie rule: descending selection key, equal
  keys to the lower expert index).
"""
import itertools
import pathlib
import re

import numpy as np
import pytest

HEADER = pathlib.Path(__file__).resolve().parents[1] / "w4a16_routed_expert_router_gb300" / "csrc" / "topk.cuh"


def _network():
    src = HEADER.read_text()
    body = src[src.index("#define MOE_TOPK_CX"):src.index("#undef MOE_TOPK_CX")]
    pairs = [(int(a), int(b)) for a, b in re.findall(r"MOE_TOPK_CX\((\d+), (\d+)\);", body)]
    per = int(re.search(r"constexpr int kTopkPer = (\d+);", src).group(1))
    return per, pairs


def test_network_shape():
    per, pairs = _network()
    assert per == 8
    assert len(pairs) == 19                   # Batcher's odd-even merge sort of 8
    assert all(0 <= a < b < per for a, b in pairs)


def test_network_sorts_every_zero_one_input():
    per, pairs = _network()
    for bits in itertools.product((0, 1), repeat=per):
        v = list(bits)
        for a, b in pairs:                    # larger first, as in topk_cx
            if v[b] > v[a]:
                v[a], v[b] = v[b], v[a]
        assert v == sorted(bits, reverse=True), bits


def _select_like_kernel(keys, k, pairs, per=8):
    """keys: [E] integer selection keys; expert e lives in lane e % 32 at slot
    e // 32. Sort each lane with the network (larger key, then lower index,
    first), then take k rounds of (max head key, lowest expert among the lanes
    holding it) and pop the winner's head."""
    E = keys.size
    lanes = []
    for lane in range(32):
        ent = [(int(keys[lane + 32 * i]), lane + 32 * i) if lane + 32 * i < E else (-1, 1 << 30)
               for i in range(per)]
        for a, b in pairs:
            ka, ia = ent[a]
            kb, ib = ent[b]
            if kb > ka or (kb == ka and ib < ia):
                ent[a], ent[b] = ent[b], ent[a]
        lanes.append(ent)
    out = []
    for _ in range(k):
        m = max(ent[0][0] for ent in lanes)
        win = min(ent[0][1] for ent in lanes if ent[0][0] == m)
        out.append(win)
        ent = lanes[win % 32]
        lanes[win % 32] = ent[1:] + [(-1, 1 << 30)]
    return out


@pytest.mark.parametrize("E,k", [(256, 6), (256, 8), (200, 6), (64, 2)])
def test_selection_matches_stable_sort(E, k):
    _, pairs = _network()
    rng = np.random.default_rng(E * 10 + k)
    for trial in range(60):
        if trial % 3 == 0:
            keys = rng.integers(0, 1 << 30, size=E)
        elif trial % 3 == 1:
            keys = rng.integers(0, 5, size=E)     # many equal keys
        else:
            keys = rng.integers(0, 2, size=E)     # almost all equal
        want = sorted(range(E), key=lambda e: (-int(keys[e]), e))[:k]
        assert _select_like_kernel(keys, k, pairs) == want

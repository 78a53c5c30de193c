"""The roofline numerator: bench.phase_bytes against a count of the bytes each buffer must move,
taken token by token and destination by destination on small workloads (no GPU)."""
import types

import numpy as np
import pytest

import bench
from combine_ep_dispatch_02_gb300 import workloads as wlmod


def _counted(wl):
    """Bytes dispatch and combine must move, counted per buffer over the routed (token, dest) pairs."""
    H, b, k, sd, W, E = wl.H, wl.elem_bytes, wl.k, wl.sd, wl.W, wl.E
    has_w = wl.weights is not None
    d = c = 0
    pairs = 0
    for s in range(W):
        for t in range(int(wl.n_tok[s])):
            dests = {int(e) // E for e in wl.indices[s, t]}
            # dispatch: the source rows are read once ...
            src = H * b + 4 * k + (4 * k if has_w else 0) + 4 * sd
            d += src
            # ... and each destination receives the rows plus one reverse-map entry
            d += len(dests) * (src + 4)
            # combine: one expert-output row (16-bit) and weight row per destination are read,
            # one output row and weight row written, and the forward map row of min(W, k) read
            c += len(dests) * (2 * H + (4 * k if has_w else 0))
            c += 2 * H + (4 * k if has_w else 0) + 4 * min(W, k)
            pairs += len(dests)
    return d, c, pairs


@pytest.mark.parametrize("kw", [
    dict(W=4, E=8, k=6, H=64, M=20, n_tok=[20, 3, 0, 17]),
    dict(W=3, E=2, k=4, H=128, dtype="fp8", sd=2, M=9, n_tok=[9, 9, 1]),
    dict(W=8, E=1, k=8, H=16, M=5, n_tok=[5, 0, 1, 2, 3, 4, 5, 5], with_weights=False),
    dict(W=1, E=4, k=2, H=32, dtype="fp16", M=7, n_tok=[7]),
])
def test_phase_bytes_match_a_per_buffer_count(kw):
    wl = wlmod.custom_workload(seed=3, **kw)
    d, c, P = _counted(wl)
    got = bench.phase_bytes(wl, P)
    assert got["dispatch"] == d
    assert got["combine"] == c
    assert got["pair"] == d + c
    # the scatter is dispatch without the reverse-map entries; the route reads index rows and
    # writes the reverse map
    assert got["scatter"] == d - 4 * P
    assert got["route"] == wl.N * 4 * wl.k + 4 * P


def test_phase_bytes_deepseek_v3_full_size():
    """W=8, 32 experts per rank, top-8, hidden 7168 BF16, 4096 tokens per rank with weights:
    N = 32768 tokens and P = 173981 (token, destination) pairs, the values the bench reports."""
    wl = types.SimpleNamespace(N=32768, H=7168, elem_bytes=2, k=8, sd=0, W=8, weights=True)
    got = bench.phase_bytes(wl, 173981)
    assert got["dispatch"] == 32768 * (14336 + 64) + 173981 * (14336 + 64 + 4) == 2977881524
    assert got["combine"] == (173981 + 32768) * (14336 + 32) + 32768 * 4 * 8 == 2971618208
    assert got["scatter"] == 2977185600
    assert got["route"] == 32768 * 32 + 173981 * 4 == 1744500

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


def test_profile_case_kernel_bytes_agree_with_the_bench():
    """The profiling driver's per-kernel algorithmic bytes are the bench's (route, scatter and
    combine at the full DeepSeek-V3 size), so a recorded traffic ratio scales consistently."""
    from combine_ep_dispatch_02_gb300 import profile_case
    wl = types.SimpleNamespace(N=32768, H=7168, elem_bytes=2, k=8, sd=0, W=8, weights=True)
    got = bench.phase_bytes(wl, 173981)
    for phase in ("route", "scatter", "combine"):
        assert profile_case.kernel_bytes(phase, 32768, 173981, 8, 7168, 8) == got[phase], phase


def test_profile_case_grouped_bytes_agree_with_the_bench():
    """The grouped phases' per-kernel bytes: the inverse's are the bench's ungroup bytes, and
    the fused copy's are the bench's fused-dispatch bytes less the reverse map's 4 bytes per
    received row (the fused call's routing writes those)."""
    from combine_ep_dispatch_02_gb300 import profile_case
    wl = types.SimpleNamespace(N=1024, H=7168, k=8, W=4)
    rows, entries = 3689, 8192
    got = bench.grouped_bytes(wl, rows, entries)
    assert profile_case.kernel_bytes("ungroup", wl.N, rows, wl.W, wl.H, wl.k, entries) == got["ungroup"]
    assert profile_case.kernel_bytes("fused_copy", wl.N, rows, wl.W, wl.H, wl.k, entries) == got["fused"] - 4 * rows
    assert got["ungroup"] == 8192 * 14336 + 3689 * (14336 + 32) == 170444064


def test_recorded_traffic_scales_and_expires(tmp_path, monkeypatch):
    """A capture entered by profile_case.record gives bench.recorded_traffic its DRAM bytes per
    algorithmic byte, applied to the full launch; a code digest that no longer matches voids it."""
    from combine_ep_dispatch_02_gb300 import profile_case
    path = tmp_path / "dram_traffic.json"
    monkeypatch.setattr(profile_case, "TRAFFIC_FILE", str(path))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    csv_path = tmp_path / "ncu.csv"
    hdr = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",' \
          '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
    rows = []
    for i, (r, w) in enumerate([(100.0, 300.0), (110.0, 290.0)]):
        for name, v in (("dram__bytes_read.sum", r), ("dram__bytes_write.sum", w)):
            rows.append(f'"{i}","1","python3","h","ep_combine_kernel","1","7","(192, 1, 1)","(304, 1, 1)",'
                        f'"0","10.3","Command line profiler metrics","{name}","Mbyte","{v}"\n')
    csv_path.write_text("==PROF== noise\n" + hdr + "".join(rows))
    line = {"tokens_per_rank": 1024, "tokens": 8192, "token_dest_pairs": 43601,
            "kernel_algorithmic_bytes": 500_000_000}
    rec = profile_case.record("combine", line, str(csv_path), "ncu ... (test)")
    assert rec["dram_bytes_per_launch"] == 400_000_000 and rec["captured_launches"] == 2
    assert rec["traffic_over_algorithmic"] == 0.8
    traffic, note = bench.recorded_traffic("combine", 2_000_000_000)
    assert traffic == 1_600_000_000 and "0.8000" in note
    monkeypatch.setattr(bench, "kernel_digest", lambda k: "0" * 64)
    assert bench.recorded_traffic("combine", 2_000_000_000)[0] is None

"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Bar: dispatch counts, reverse map and every received row (payload, indices, weights, scales)
bit-exact; combine outputs bit-exact under the fixed ascending-rank FP32 order (NaN compared as
NaN); combined FP32 weights bit-exact.
"""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_02_gb300 as ep
import gpu_path
import harness
import oracle
from combine_ep_dispatch_02_gb300 import workloads as wlmod

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA GPU")
    from combine_ep_dispatch_02_gb300 import build
    build.build()
    oracle.build()


def _oracle(wl):
    return oracle.run_workload(wl, harness.expert_np)


def _check(wl, variant="auto"):
    disp, _, o_out, o_w = _oracle(wl)
    gpu = gpu_path.run(wl, DEV, variant)
    gpu_path.compare(wl, gpu, disp, o_out, o_w)
    return gpu, disp


# ---------------------------------------------------------------- the five workloads

def test_tiny_full():
    _check(wlmod.make_workload("tiny"))


@pytest.mark.parametrize("variant", ["auto", "whole_row", "tiled_512", "tiled_1024"])
def test_small_full_scalar_expert(variant):
    _check(wlmod.make_workload("small"), variant)


# the workload's sweep, plus 31 and 63: one slot short of a 32-slot batch, in each batch
@pytest.mark.parametrize("k", sorted(set(wlmod.TOPK_SWEEP) | {31, 63}))
def test_topk_sweep_fp16(k):
    _check(wlmod.make_workload("topk", k=k))


def test_dsv3_reduced_ragged_tiles():
    # 300 tokens per rank: 2400 tokens = 9 full routing tiles of 256 and a ragged tail
    _check(wlmod.make_workload("dsv3", max_tok=300))


def test_fp8_reduced():
    _check(wlmod.make_workload("fp8", max_tok=512))


def test_fp8_full_ragged():
    _check(wlmod.make_workload("fp8"))


def test_dsv3_full():
    """The DeepSeek-V3-shaped workload at full size, in the launch configuration the benchmark
    times (AUTO variant), every row and every output compared."""
    _check(wlmod.make_workload("dsv3"))


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("case", [
    dict(W=1, E=8, k=3, H=64, M=40, n_tok=[37]),
    dict(W=32, E=2, k=64, H=16, M=70, n_tok=list(range(0, 64, 2))),
    dict(W=32, E=4, k=5, H=8, M=9, n_tok=[9] * 32),
    dict(W=5, E=3, k=1, H=24, M=300, n_tok=[300, 0, 257, 1, 255]),
    dict(W=3, E=5, k=9, H=520, M=600, n_tok=[600, 513, 0]),
    dict(W=8, E=1, k=8, H=7168, M=64, n_tok=[64, 63, 1, 0, 2, 33, 64, 5]),
    dict(W=4, E=64, k=33, H=2048, M=129, n_tok=[129, 128, 127, 1]),
], ids=lambda c: f"W{c['W']}k{c['k']}H{c['H']}")
def test_edge_shapes(case):
    for dtype in ("bf16", "fp16"):
        _check(wlmod.custom_workload(dtype=dtype, seed=3, **case))


def test_fp8_with_odd_scale_dim():
    _check(wlmod.custom_workload(W=4, E=4, k=4, H=256, dtype="fp8", sd=3, M=50, n_tok=[50, 7, 0, 31]))


def test_empty_dispatch():
    wl = wlmod.custom_workload(W=4, E=4, k=2, H=64, M=16, n_tok=[0, 0, 0, 0])
    gpu = gpu_path.run(wl, DEV)
    assert gpu["status"] == 0
    assert not gpu["recv_count"].any()


def test_zipf_hot_rank():
    wl = wlmod.custom_workload(W=8, E=4, k=4, H=256, M=1000, n_tok=[1000] * 8, routing="zipf")
    _check(wl)


def test_invalid_ids_set_status_and_are_skipped():
    wl = wlmod.custom_workload(W=3, E=2, k=3, H=64, M=300, n_tok=[300, 200, 100], seed=4)
    wl.indices[0, 5, 1] = -1
    wl.indices[1, 199, 0] = 6
    disp, _, o_out, o_w = _oracle(wl)
    assert disp["status"] == oracle.ERR_INDEX
    gpu = gpu_path.run(wl, DEV)
    assert gpu["status"] == ep.EP_ERR_INDEX
    gpu["status"] = 0
    gpu_path.compare(wl, gpu, disp, o_out, o_w)


def test_no_weights():
    wl = wlmod.custom_workload(W=4, E=8, k=4, H=128, M=100, n_tok=[100, 50, 3, 99],
                               with_weights=False)
    _check(wl)


# ---------------------------------------------------------------- lifecycle

def _setup(wl):
    plan = gpu_path.make_plan(wl, DEV)
    return plan, gpu_path.to_device(wl, DEV)


def test_double_combine_is_bit_identical():
    wl = wlmod.make_workload("small", max_tok=64)
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    eo = harness.expert_torch(wl, d.recv_x, d.recv_idx, d.recv_w, d.recv_scales, d.recv_count)
    o1, w1 = plan.combine(eo, d.recv_w, d.epoch)
    o2, w2 = plan.combine(eo, d.recv_w, d.epoch)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(w1, w2)
    plan.close()


def test_handle_interleave_and_reset():
    wl_a = wlmod.custom_workload(W=4, E=4, k=3, H=64, M=80, n_tok=[80, 10, 40, 79], seed=1)
    wl_b = wlmod.custom_workload(W=4, E=4, k=3, H=64, M=80, n_tok=[5, 80, 0, 33], seed=2)
    plan = gpu_path.make_plan(wl_a, DEV)
    xa, wa, _, ia = gpu_path.to_device(wl_a, DEV)
    xb, wb, _, ib = gpu_path.to_device(wl_b, DEV)
    da = plan.dispatch(xa, wa, None, ia, wl_a.n_tok)
    db = plan.dispatch(xb, wb, None, ib, wl_b.n_tok)
    with pytest.raises(ep.EpError) as e:
        plan.combine(da.recv_x, da.recv_w, da.epoch)
    assert e.value.code == ep.EP_ERR_STATE
    out_b, _ = plan.combine(db.recv_x, db.recv_w, db.epoch)
    _, _, o_out_b, _ = oracle.run_workload(wl_b)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_path.raw(out_b), o_out_b)
    # re-dispatch A, combine A
    da = plan.dispatch(xa, wa, None, ia, wl_a.n_tok)
    out_a, _ = plan.combine(da.recv_x, da.recv_w, da.epoch)
    _, _, o_out_a, _ = oracle.run_workload(wl_a)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_path.raw(out_a), o_out_a)
    plan.reset()
    with pytest.raises(ep.EpError) as e:
        plan.combine(da.recv_x, da.recv_w, da.epoch)
    assert e.value.code == ep.EP_ERR_STATE
    assert plan.status() == 0
    plan.close()


def test_host_errors_before_launch():
    wl = wlmod.custom_workload(W=2, E=4, k=2, H=64, M=16, n_tok=[16, 16])
    plan, (x, w, sc, idx) = _setup(wl)
    with pytest.raises(ep.EpError) as e:
        plan.dispatch(x, w, None, idx, [17, 0])
    assert e.value.code == ep.EP_ERR_CAPACITY
    with pytest.raises(ep.EpError) as e:
        plan.dispatch(x, w, None, idx, [-1, 0])
    assert e.value.code == ep.EP_ERR_ARG
    with pytest.raises(ep.EpError) as e:   # scales on a plan without scale_dim
        plan.dispatch(x, w, torch.zeros(4, device=DEV), idx, [1, 1])
    assert e.value.code == ep.EP_ERR_ARG
    with pytest.raises(ep.EpError) as e:   # misaligned x (full size, 2 bytes past a 16-byte boundary)
        xs = torch.empty(x.numel() + 8, dtype=x.dtype, device=DEV)[1:1 + x.numel()].view(x.shape)
        plan.dispatch(xs, w, None, idx, [1, 1])
    assert e.value.code == ep.EP_ERR_ARG and "aligned" in str(e.value)
    with pytest.raises(ep.EpError) as e:   # combine before any dispatch
        plan.combine(torch.zeros((2, 32, 64), dtype=torch.bfloat16, device=DEV), None, 1)
    assert e.value.code == ep.EP_ERR_STATE
    # the binding checks buffer sizes and element widths against the plan before any launch
    with pytest.raises(ep.EpError) as e:   # x one element short
        plan.dispatch(x.view(-1)[1:], w, None, idx, [1, 1])
    assert e.value.code == ep.EP_ERR_ARG and "x holds" in str(e.value)
    with pytest.raises(ep.EpError) as e:   # int64 indices
        plan.dispatch(x, w, None, idx.long(), [1, 1])
    assert e.value.code == ep.EP_ERR_ARG and "indices" in str(e.value)
    with pytest.raises(ep.EpError) as e:   # expert_out of [W][M][H] instead of [W][W*M][H]
        plan.combine(x, None, 1)
    assert e.value.code == ep.EP_ERR_ARG and "expert_out" in str(e.value)
    d = plan.dispatch(x, w, None, idx, wl.n_tok)
    with pytest.raises(ep.EpError) as e:   # out_w without weights
        plan.combine(d.recv_x, None, d.epoch, out_w=torch.zeros((2, 16, 2), device=DEV))
    assert e.value.code == ep.EP_ERR_ARG
    with pytest.raises(ep.EpError) as e:   # scatter without route
        plan.dispatch_scatter(x, w, None, idx)
    assert e.value.code == ep.EP_ERR_STATE
    assert plan.status() == 0
    plan.close()


def test_route_plus_scatter_equals_dispatch():
    wl = wlmod.make_workload("dsv3", max_tok=200)
    disp, _, o_out, o_w = _oracle(wl)
    plan, (x, w, sc, idx) = _setup(wl)
    gpu_path.poison(plan, DEV)
    d = plan.dispatch_route(idx, wl.n_tok)
    plan.dispatch_scatter(x, w, sc, idx)
    out, out_w = plan.combine(d.recv_x, d.recv_w, d.epoch)
    torch.cuda.synchronize()
    res = {"recv_count": d.recv_count.cpu().numpy(), "recv_x": gpu_path.raw(d.recv_x),
           "recv_idx": gpu_path.raw(d.recv_idx), "recv_w": gpu_path.raw(d.recv_w),
           "recv_scales": None, "src_pos": gpu_path.raw(d.src_token_pos),
           "out": gpu_path.raw(out), "out_w": gpu_path.raw(out_w), "status": plan.status()}
    gpu_path.compare(wl, res, disp, o_out, o_w)
    plan.close()


def test_many_calls_reuse_scan_flags():
    """Sixty dispatches on one plan with changing token counts: every call's scan words carry
    a fresh stamp, so no call reads a stale prefix."""
    wl = wlmod.make_workload("dsv3", max_tok=160)
    plan, (x, w, sc, idx) = _setup(wl)
    rng = np.random.default_rng(0)
    ref = {}
    for i in range(60):
        n_tok = rng.integers(0, wl.M + 1, size=wl.W).astype(np.int32)
        if i % 7 == 0:
            n_tok[:] = wl.M
        d = plan.dispatch(x, w, sc, idx, n_tok)
        key = tuple(n_tok.tolist())
        if i % 10 == 0 or key not in ref:
            sub = wlmod.Workload(**{**wl.__dict__, "n_tok": n_tok})
            o = oracle.dispatch(sub.W, sub.E, sub.k, sub.H, sub.elem_bytes, sub.sd, sub.M, sub.x,
                                sub.weights, sub.scales, sub.indices, sub.n_tok)
            ref[key] = o
        o = ref[key]
        cnt = d.recv_count.cpu().numpy()
        assert np.array_equal(cnt, o["recv_count"]), i
        for r in range(wl.W):
            n = int(cnt[r])
            assert np.array_equal(d.src_token_pos[r, :n].cpu().numpy(), o["src_pos"][r, :n]), (i, r)
    assert plan.status() == 0
    plan.close()


def _with_n_tok(wl, n_tok):
    return wlmod.Workload(**{**wl.__dict__, "n_tok": np.asarray(n_tok, dtype=np.int32)})


def test_small_calls_on_a_large_plan():
    """A plan sized for 2048 tokens per rank (64 routing tiles, 16 grouping chunks per rank)
    serving calls of 0 to 16384 tokens: the routing grid follows each call (a CTA per 256 of its
    tokens, at least one), and its ticket and stamp generation reset on the device, so calls of
    any size interleave on one plan.  Each call is compared with the oracle, and a small call
    captured in a CUDA graph replays correctly between eager calls of other sizes."""
    base = wlmod.custom_workload(W=8, E=32, k=8, H=256, M=2048, n_tok=[2048] * 8, seed=31,
                                 routing="zipf")
    plan, (x, w, sc, idx) = _setup(base)
    sizes = [[8] * 8, [0] * 8, [2048] * 8, [1, 0, 0, 0, 0, 0, 0, 2], [300] * 8, [2048] + [0] * 7,
             [256, 257, 255, 0, 1, 512, 2047, 3], [5] * 8]
    for n_tok in sizes:
        wl = _with_n_tok(base, n_tok)
        disp, _, o_out, o_w = _oracle(wl)
        gpu_path.compare(wl, gpu_path.run(wl, DEV, plan=plan, do_poison=False), disp, o_out, o_w)
    # a graph of an 8-token-per-rank dispatch + combine, replayed between eager calls
    small = _with_n_tok(base, [8] * 8)
    disp, _, o_out, o_w = _oracle(small)
    out = torch.zeros((base.W, base.M, base.H), dtype=torch.bfloat16, device=DEV)
    out_w = torch.zeros((base.W, base.M, base.k), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d = plan.dispatch(x, w, sc, idx, small.n_tok, stream=s)
        plan.combine(d.recv_x, d.recv_w, d.epoch, out=out, out_w=out_w, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        d = plan.dispatch(x, w, sc, idx, small.n_tok, stream=cs)
        plan.combine(d.recv_x, d.recv_w, d.epoch, out=out, out_w=out_w, stream=cs)
    for n_tok in ([2048] * 8, [3] * 8, [700] * 8):
        wl = _with_n_tok(base, n_tok)
        d_e = plan.dispatch(x, w, sc, idx, wl.n_tok)
        o = oracle.dispatch(wl.W, wl.E, wl.k, wl.H, wl.elem_bytes, wl.sd, wl.M, wl.x, wl.weights,
                            wl.scales, wl.indices, wl.n_tok)
        assert np.array_equal(d_e.recv_count.cpu().numpy(), o["recv_count"])
        out.zero_()
        out_w.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(gpu_path.raw(out), o_out)
        assert np.array_equal(out_w.cpu().numpy().view(np.uint32), o_w.view(np.uint32))
    assert plan.status() == 0
    plan.close()


def test_grouped_small_call_on_a_two_pass_plan():
    """Plans whose capacity would take the two-pass grouping scan (16 chunks per rank): a call
    of 2000 tokens groups with the one-pass scan (no rank can hold more than two chunks of
    rows), one of 6000 with the two-pass scan at the call's 6-chunk stride."""
    base = wlmod.custom_workload(W=8, E=4, k=4, H=64, M=2048, n_tok=[2048] * 8, seed=32)
    for n_tok in ([250] * 8, [750] * 8):
        wl = _with_n_tok(base, n_tok)
        _check_grouped(wl)
        _check_grouped(wl, fused=True)


def test_single_tile_calls():
    """Calls around one routing tile (0, 1, 255, 256 and 257 tokens, and the full 800) through
    ep_dispatch and through ep_dispatch_route + ep_dispatch_scatter give the oracle's rows; small
    and large calls, eager and replayed from a CUDA graph, interleave on one plan; an invalid
    expert id in a small call is skipped and reported."""
    base = wlmod.custom_workload(W=4, E=8, k=6, H=264, M=200, n_tok=[200] * 4, seed=51, routing="zipf")
    plan, (x, w, sc, idx) = _setup(base)
    for n_tok in ([0, 0, 0, 0], [0, 1, 0, 0], [64, 64, 63, 64], [64, 64, 64, 64], [64, 65, 64, 64],
                  [200, 200, 200, 200], [1, 0, 0, 2]):
        wl = _with_n_tok(base, n_tok)
        disp, _, o_out, o_w = _oracle(wl)
        gpu_path.compare(wl, gpu_path.run(wl, DEV, plan=plan, do_poison=False), disp, o_out, o_w)
        d = plan.dispatch_route(idx, wl.n_tok)                 # the two phases called apart: same rows
        plan.dispatch_scatter(x, w, sc, idx)
        torch.cuda.synchronize()
        cnt = d.recv_count.cpu().numpy()
        assert np.array_equal(cnt, disp["recv_count"])
        for r in range(wl.W):
            n = int(cnt[r])
            assert np.array_equal(d.src_token_pos[r, :n].cpu().numpy(), disp["src_pos"][r, :n])
            assert np.array_equal(gpu_path.raw(d.recv_x)[r, :n], disp["recv_x"][r, :n])
    # a 40-token call captured in a graph, replayed between multi-tile calls
    small = _with_n_tok(base, [10, 10, 10, 10])
    disp, _, o_out, o_w = _oracle(small)
    out = torch.zeros((base.W, base.M, base.H), dtype=torch.bfloat16, device=DEV)
    out_w = torch.zeros((base.W, base.M, base.k), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d = plan.dispatch(x, w, sc, idx, small.n_tok, stream=s)
        plan.combine(d.recv_x, d.recv_w, d.epoch, out=out, out_w=out_w, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        d = plan.dispatch(x, w, sc, idx, small.n_tok, stream=cs)
        plan.combine(d.recv_x, d.recv_w, d.epoch, out=out, out_w=out_w, stream=cs)
    for n_tok in ([200] * 4, [3, 0, 0, 0], [150] * 4):
        plan.dispatch(x, w, sc, idx, n_tok)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(gpu_path.raw(out), o_out)
        assert np.array_equal(out_w.cpu().numpy().view(np.uint32), o_w.view(np.uint32))
    assert plan.status() == 0
    # an invalid id in a small call: skipped on the device and reported
    bad = wlmod.Workload(**{**small.__dict__, "indices": small.indices.copy()})
    bad.indices[1, 2, 0] = base.W * base.E + 5
    ib = torch.from_numpy(bad.indices).to(DEV)
    plan.dispatch(x, w, sc, ib, bad.n_tok)
    assert plan.status() == ep.EP_ERR_INDEX
    plan.close()


def test_grouped_fused_routing_tile_boundaries():
    """The grouped dispatch numbers the lists in its routing kernel: source boundaries on tile
    edges (256 and 512 tokens, an empty source, the end at exactly three tiles), a single token,
    and an empty call, each against the oracle, grouped and inverted."""
    for n_tok in ([256, 256, 0, 256], [0, 0, 1, 0], [0, 0, 0, 0], [255, 1, 257, 0]):
        wl = wlmod.custom_workload(W=4, E=16, k=5, H=64, M=300, n_tok=n_tok, seed=41)
        _check_grouped(wl, fused=True, repeats=2)


def test_cuda_graph_replay_matches_eager():
    """Dispatch + combine captured once in a CUDA graph and replayed: the per-call stamps live
    on the device (a generation count), so replays stay correct and bit-identical to eager calls."""
    wl = wlmod.make_workload("small", max_tok=96)
    disp, _, o_out, o_w = _oracle(wl)
    plan, (x, w, sc, idx) = _setup(wl)
    out = torch.zeros((wl.W, wl.M, wl.H), dtype=torch.bfloat16, device=DEV)
    out_w = torch.zeros((wl.W, wl.M, wl.k), dtype=torch.float32, device=DEV)
    # warm up eagerly on a side stream (graph capture requires a non-default stream)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d = plan.dispatch(x, w, sc, idx, wl.n_tok, stream=s)
        eo = harness.expert_torch(wl, d.recv_x, d.recv_idx, d.recv_w, d.recv_scales, d.recv_count)
        plan.combine(eo, d.recv_w, d.epoch, out=out, out_w=out_w, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = gpu_path.raw(out).copy()
    assert np.array_equal(eager, o_out)
    eo_buf = torch.empty((wl.W, wl.W * wl.M, wl.H), dtype=torch.int16, device=DEV)
    counts = d.recv_count.cpu().tolist()
    c = torch.from_numpy(wl.expert_scale).to(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        d = plan.dispatch(x, w, sc, idx, wl.n_tok, stream=cs)
        # the scalar expert, with the counts known from the eager run (static shapes)
        for r in range(wl.W):
            n = counts[r]
            X = d.recv_x[r, :n].to(torch.float32)
            IDX = d.recv_idx[r, :n].long()
            acc = torch.zeros((n, wl.H), dtype=torch.float32, device=DEV)
            for j in range(wl.k):
                m = torch.div(IDX[:, j], wl.E, rounding_mode="floor") == r
                term = torch.mul(torch.mul(d.recv_w[r, :n, j], c[IDX[:, j]])[:, None], X)
                acc = torch.where(m[:, None], torch.add(acc, term), acc)
            eo_buf[r, :n] = acc.to(torch.bfloat16).view(torch.int16)
        plan.combine(eo_buf, d.recv_w, d.epoch, out=out, out_w=out_w, stream=cs)
    for _ in range(3):
        out.zero_()
        out_w.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(gpu_path.raw(out), eager)
        assert np.array_equal(out_w.cpu().numpy().view(np.uint32), o_w.view(np.uint32))
    assert plan.status() == 0
    plan.close()


def test_scatter_work_queue_reuse_and_graph_replay():
    """Dispatches with more than four rounds of work units per warp (2400 tokens cut into
    512-element slices), so the scatter draws its last units from the plan's work queue.  They
    run three times in a row on one plan and are replayed three times from a CUDA graph, with
    the receive rows poisoned before each: a queue left short of zero would skip units."""
    wl = wlmod.make_workload("dsv3", max_tok=300)
    disp, _, o_out, o_w = _oracle(wl)
    plan = gpu_path.make_plan(wl, DEV, "tiled_512")
    for _ in range(3):
        gpu_path.compare(wl, gpu_path.run(wl, DEV, "tiled_512", plan=plan), disp, o_out, o_w)
    x, w, sc, idx = gpu_path.to_device(wl, DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.dispatch(x, w, sc, idx, wl.n_tok, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d = plan.dispatch(x, w, sc, idx, wl.n_tok, stream=torch.cuda.current_stream())
    for _ in range(3):
        d.recv_x.view(torch.uint8).fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        rx = gpu_path.raw(d.recv_x)
        for r in range(wl.W):
            n = int(disp["recv_count"][r])
            assert np.array_equal(rx[r, :n], disp["recv_x"][r, :n]), f"rank {r}"
    assert plan.status() == 0
    plan.close()

    # the quantising scatters share the queue
    dq = oracle.dispatch_quantized(wl)
    q, qs = oracle.quantize_e4m3_blockwise(wl.x)
    wq = gpu_path.quantised_view(wl, q, qs)
    eo = harness.expert_np(wq, dq)
    qo, qw = oracle.combine(wl.W, wl.k, wl.H, False, wl.M, wl.n_tok, dq["slot_of"], eo, dq["recv_w"])
    plan = gpu_path.make_plan(wl, DEV, "tiled_512", "bf16_fp8")
    for _ in range(2):
        gpu_path.compare(wq, gpu_path.run(wl, DEV, plan=plan, quantise=True), dq, qo, qw)
    plan.close()
    _check_mxfp4_dispatch(wl, "tiled_512", repeats=2)


def test_mid_size_sliced_rows_with_work_queue():
    """1024 tokens per rank of the DeepSeek-V3 shape: the AUTO variant cuts rows into 1024-element
    slices (fewer than four whole rows per resident warp) and the scatters draw their last slices
    from the work queue; BF16, FP8 and MX FP4 dispatch and the combine against the oracle."""
    wl = wlmod.make_workload("dsv3", max_tok=1024)
    _check(wl)
    _check_quantised(wl)
    _check_mxfp4_dispatch(wl)


# ---------------------------------------------------------------- quantising FP8 dispatch

def _check_quantised(wl, variant="auto"):
    disp = oracle.dispatch_quantized(wl)
    q, sc = oracle.quantize_e4m3_blockwise(wl.x)
    wq = gpu_path.quantised_view(wl, q, sc)
    eo = harness.expert_np(wq, disp)
    o_out, o_w = oracle.combine(wl.W, wl.k, wl.H, False, wl.M, wl.n_tok, disp["slot_of"], eo,
                                disp["recv_w"])
    gpu = gpu_path.run(wl, DEV, variant, quantise=True)
    gpu_path.compare(wq, gpu, disp, o_out, o_w)


def test_quantised_dispatch_dsv3_reduced():
    _check_quantised(wlmod.make_workload("dsv3", max_tok=300))


@pytest.mark.parametrize("variant", ["tiled_512", "tiled_1024", "whole_row"])
def test_quantised_dispatch_small_variants(variant):
    _check_quantised(wlmod.make_workload("small", max_tok=64), variant)


def test_quantised_dispatch_dsv3_full():
    _check_quantised(wlmod.make_workload("dsv3"))


def test_quantised_dispatch_edge_values():
    wl = wlmod.custom_workload(W=4, E=4, k=3, H=384, M=40, n_tok=[40, 0, 17, 33], seed=9)
    xf = (wl.x.astype(np.uint32) << 16).view(np.float32).copy()
    xf[0, 0] = 0.0                                   # all-zero rows and blocks
    xf[0, 1, 128:256] = 0.0
    xf[2, 3] *= np.float32(1e-30)                    # values the scale must lift out of underflow
    xf[2, 4, :128] = np.float32(3e38)                # huge values
    xf[3, 5, 7] = -0.0
    wl.x[:] = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    _check_quantised(wl)


def _e4m3_boundaries():
    """The positive e4m3fn rounding boundaries below 448: midpoints of consecutive codes, and
    half the smallest subnormal."""
    vals = sorted({float(v) for v in torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float()})
    return [(a + b) / 2 for a, b in zip(vals, vals[1:])]


def test_quantised_dispatch_at_e4m3_boundaries():
    # blocks whose quotient x / scale sits exactly on, or one BF16 step around, an e4m3 rounding
    # boundary, at scales that are and are not powers of two: the quantiser's bracketing must
    # hand these to the exact division and still match the oracle's FP32 division
    mids = np.array(_e4m3_boundaries(), dtype=np.float64)          # 126 boundaries
    cs = [1.0, 1.5, 0.75, 3.0, 2.0 ** -5 * 1.25, 2.0 ** 7 * 1.125, 1.0 / 3.0, 2.0 ** -20 * 1.75]
    rows = []
    for c in cs:
        for nudge in (0, 1, -1):
            r = np.empty(128, dtype=np.float32)
            r[0] = 448.0 * c
            r[1:127] = mids * c
            r[127] = -mids[63] * c
            b = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy()
            b[1:] = b[1:] + np.int16(nudge) * np.sign(b[1:]).astype(np.int16)   # one BF16 step
            rows.append(b.view(np.uint16))
            rows.append((b.view(np.uint16) ^ np.uint16(0x8000)))             # negated row
    rows = np.stack(rows)
    W, M = 2, (len(rows) + 1) // 2
    wl = wlmod.custom_workload(W=W, E=2, k=2, H=128, M=M, n_tok=[M, len(rows) - M], seed=5)
    wl.x[:] = 0
    wl.x.reshape(-1, 128)[:len(rows)] = rows
    _check_quantised(wl)


def _quantiser_class_blocks():
    """128-element BF16 blocks covering the FP8 quantiser's inputs class by class.

    A block's scale depends only on its maximum m, and the code of x depends only on x and m.
    Scaling both by a power of two leaves the code unchanged while no intermediate under- or
    overflows, so every significand of m (7 fraction bits) at a few exponents, with every BF16 x
    of either sign whose exponent lies within 24 of m's, covers the normal range; anything
    smaller quantises to +-0.  The exponents span subnormal maxima, the scale 2^-60 below which
    the quantiser divides (m near 2^-51), ordinary values and the BF16 maximum.  Each block
    holds m once, at a position that moves from block to block, and 127 values of magnitude
    <= m."""
    blocks = []
    frac = np.arange(128, dtype=np.uint32)
    for e_m in (0, 1, 58, 75, 76, 77, 100, 127, 140, 200, 254):
        for f_m in range(128):
            if e_m == 0 and f_m == 0:
                continue
            m_bits = (e_m << 7) | f_m
            e = np.arange(max(0, e_m - 24), e_m + 1, dtype=np.uint32)
            xs = ((e[:, None] << 7) | frac[None, :]).ravel()
            xs = xs[xs <= m_bits]
            xs = np.concatenate([xs, xs | 0x8000]).astype(np.uint16)
            nb = -(-len(xs) // 127)
            pad = np.zeros(nb * 127, dtype=np.uint16)
            pad[:len(xs)] = xs
            for chunk in pad.reshape(nb, 127):
                i = len(blocks)
                blocks.append(np.insert(chunk, i % 128, np.uint16(m_bits ^ (0x8000 if i & 1 else 0))))
    return np.stack(blocks).astype(np.uint16)


def test_fp8_quantisers_over_every_input_class():
    """Both FP8 quantisers (inside the quantising dispatch, and on received expert rows for the
    FP8 wire) against the oracle's division, code for code, on _quantiser_class_blocks()."""
    H = 7168
    blocks = _quantiser_class_blocks()
    M = -(-len(blocks) * 128 // H)
    rows = np.zeros((M * H // 128, 128), dtype=np.uint16)
    rows[:len(blocks)] = blocks
    rows = rows.reshape(1, M, H)

    wl = wlmod.custom_workload(W=1, E=1, k=1, H=H, M=M, n_tok=[M], seed=11)
    wl.x[:] = rows
    _check_quantised(wl)

    q, sc = oracle.quantize_e4m3_blockwise(rows)
    plan = ep.Plan(1, 1, 1, H, "bf16", 0, M, device=DEV)
    x, w, _, idx = gpu_path.to_device(wl, DEV)
    d = plan.dispatch(x, w, None, idx, [M])
    eo = torch.from_numpy(rows.view(np.int16)).to(DEV).view(torch.bfloat16)
    qg, scg = plan.quantize_received(eo, d.epoch)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert np.array_equal(gpu_path.raw(qg)[0, :M], q[0])
    assert np.array_equal(scg.cpu().numpy()[0, :M].view(np.uint32), sc[0].view(np.uint32))
    plan.close()


# ---------------------------------------------------------------- quantising MX FP4 dispatch

def _check_mxfp4_dispatch(wl, variant="auto", repeats=1):
    """Dispatch through the MX FP4 dtype: codes, scale bytes, index / weight rows, reverse map
    and counts against the oracle (its MX quantiser, then its byte-exact dispatch), bit for bit;
    then the combine of the dequantised rows (an exact dequantising expert on both sides).
    repeats > 1 dispatches again on the same plan, receive rows poisoned before each call."""
    disp = oracle.dispatch_quantized_mxfp4(wl)
    eo = harness.mxfp4_dequant_np(disp["recv_x"], disp["recv_scales"].view(np.uint8))
    o_out, o_w = oracle.combine(wl.W, wl.k, wl.H, False, wl.M, wl.n_tok, disp["slot_of"], eo,
                                disp["recv_w"])
    plan = gpu_path.make_plan(wl, DEV, variant, "bf16_mxfp4")
    x, w, _, idx = gpu_path.to_device(wl, DEV)
    wq = wlmod.Workload(**{**wl.__dict__, "sd": wl.H // 128})   # scale rows are compared
    for _ in range(repeats):
        gpu_path.poison(plan, DEV)
        d = plan.dispatch(x, w, None, idx, wl.n_tok)
        assert d.recv_x.shape == (wl.W, wl.W * wl.M, wl.H // 2)
        assert d.recv_scales.shape == (wl.W, wl.W * wl.M, wl.H // 32)
        eo_g = harness.mxfp4_dequant_torch(d.recv_x, d.recv_scales)
        out, out_w = plan.combine(eo_g, d.recv_w, d.epoch)
        torch.cuda.synchronize()
        gpu = {"recv_count": d.recv_count.cpu().numpy(), "recv_x": gpu_path.raw(d.recv_x),
               "recv_idx": gpu_path.raw(d.recv_idx), "recv_w": gpu_path.raw(d.recv_w),
               "recv_scales": gpu_path.raw(d.recv_scales), "src_pos": gpu_path.raw(d.src_token_pos),
               "out": gpu_path.raw(out), "out_w": gpu_path.raw(out_w), "status": plan.status()}
        gpu_path.compare(wq, gpu, disp, o_out, o_w)
    plan.close()


def test_mxfp4_dispatch_dsv3_reduced():
    _check_mxfp4_dispatch(wlmod.make_workload("dsv3", max_tok=300))


@pytest.mark.parametrize("variant", ["tiled_512", "tiled_1024", "whole_row"])
def test_mxfp4_dispatch_small_variants(variant):
    _check_mxfp4_dispatch(wlmod.make_workload("small", max_tok=64), variant)


def test_mxfp4_dispatch_dsv3_full():
    _check_mxfp4_dispatch(wlmod.make_workload("dsv3"))


def test_mxfp4_dispatch_edge_values():
    wl = wlmod.custom_workload(W=4, E=4, k=3, H=384, M=40, n_tok=[40, 0, 17, 33], seed=9)
    xf = (wl.x.astype(np.uint32) << 16).view(np.float32).copy()
    xf[0, 0] = 0.0                                   # all-zero rows and blocks (scale code 127)
    xf[0, 1, 32:64] = 0.0
    xf[2, 3] *= np.float32(1e-38)                    # BF16 subnormal blocks: scale code clamps to 0
    xf[2, 4, :32] = np.float32(3e38)                 # near the BF16 maximum: code 252
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0], np.float32) * np.float32(4.0)
    xf[3, 5, 64:96] = np.tile(np.concatenate([ties, -ties]), 2)   # exact e2m1 ties, amax 28
    xf[3, 5, 7] = -0.0
    wl.x[:] = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    _check_mxfp4_dispatch(wl)


def test_mxfp4_plan_grouped_view_moves_code_bytes():
    wl = wlmod.make_workload("small", max_tok=32)
    disp = oracle.dispatch_quantized_mxfp4(wl)
    g = oracle.group_by_expert(wl.W, wl.E, wl.k, wl.H // 2, 1, wl.M, disp)
    plan = gpu_path.make_plan(wl, DEV, "auto", "bf16_mxfp4")
    x, w, _, idx = gpu_path.to_device(wl, DEV)
    d = plan.dispatch(x, w, None, idx, wl.n_tok)
    px, cnt, info, layout = plan.group_by_expert(d.epoch)
    torch.cuda.synchronize()
    assert plan.status() == 0
    cnt, px, info = cnt.cpu().numpy(), px.cpu().numpy(), info.cpu().numpy()
    assert px.shape == (wl.W, wl.E, wl.W * wl.M, wl.H // 2)
    assert np.array_equal(cnt, g["packed_count"])
    assert np.array_equal(layout.cpu().numpy(), g["layout_range"])
    for r in range(wl.W):
        for e in range(wl.E):
            n = int(cnt[r, e])
            assert np.array_equal(info[r, e, :n], g["packed_src_info"][r, e, :n]), (r, e)
            assert np.array_equal(px[r, e, :n], g["packed_x"][r, e, :n]), (r, e)
    with pytest.raises(ep.EpError):
        plan.dispatch_grouped(x, w, None, idx, wl.n_tok)    # quantising dtypes are not fused
    plan.close()


# ---------------------------------------------------------------- combine over an FP8 wire

def _check_fp8_wire(wl, variant="auto"):
    disp, eo, _, _ = oracle.run_workload(wl, harness.expert_np)
    q, sc = oracle.quantize_e4m3_blockwise(eo)
    o_out, o_w = oracle.combine_fp8(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], q, sc,
                                    disp["recv_w"])
    plan, (x, w, scales, idx) = _setup(wl)
    plan.set_variant(variant)
    d = plan.dispatch(x, w, scales, idx, wl.n_tok)
    eo_g = harness.expert_torch(wl, d.recv_x, d.recv_idx, d.recv_w, d.recv_scales, d.recv_count)
    qg, scg = plan.quantize_received(eo_g, d.epoch)
    out, out_w = plan.combine_fp8(qg, scg, d.recv_w, d.epoch)
    torch.cuda.synchronize()
    assert plan.status() == 0
    qg, scg = gpu_path.raw(qg), scg.cpu().numpy()
    cnt = d.recv_count.cpu().numpy()
    for r in range(wl.W):
        n = int(cnt[r])
        assert np.array_equal(qg[r, :n], q[r, :n]), f"rank {r}: codes"
        assert np.array_equal(scg[r, :n].view(np.uint32), sc[r, :n].view(np.uint32)), f"rank {r}: scales"
    out = gpu_path.raw(out)
    for s in range(wl.W):
        n = int(wl.n_tok[s])
        assert gpu_path.nan_aware_equal_bf16(out[s, :n], o_out[s, :n]), f"source rank {s}"
        if o_w is not None:
            assert np.array_equal(out_w[s, :n].cpu().numpy().view(np.uint32), o_w[s, :n].view(np.uint32))
    plan.close()


def test_wire_combines_with_16_byte_aligned_out():
    """The wire combines store an output piece as one 32-byte vector when `out` is 32-byte
    aligned, and as two 16-byte vectors when it is only 16-byte aligned (the ABI's requirement):
    both give the oracle's bits."""
    wl = wlmod.make_workload("dsv3", max_tok=96)
    disp, _, _, _ = _oracle(wl)
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    n_out = wl.W * wl.M * wl.H
    for fmt in ("fp8", "fp4"):
        if fmt == "fp8":
            q, scl = plan.quantize_received(d.recv_x, d.epoch)
            oq, osc = oracle.quantize_e4m3_blockwise(disp["recv_x"])
            o_out, _ = oracle.combine_fp8(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], oq, osc)
            comb = plan.combine_fp8
        else:
            q, scl = plan.quantize_received_fp4(d.recv_x, d.epoch)
            oq, osc = oracle.quantize_mxfp4(disp["recv_x"])
            o_out, _ = oracle.combine_fp4(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], oq, osc)
            comb = plan.combine_fp4
        buf = torch.zeros(n_out + 16, dtype=torch.bfloat16, device=DEV)
        for off in (0, 8):                             # 32-byte aligned, then 16 bytes past it
            out = buf[off:off + n_out].view(wl.W, wl.M, wl.H)
            assert out.data_ptr() % 32 == (0 if off == 0 else 16)
            out.zero_()
            comb(q, scl, None, d.epoch, out=out)
            torch.cuda.synchronize()
            got = gpu_path.raw(out)
            for s_ in range(wl.W):
                n = int(wl.n_tok[s_])
                assert gpu_path.nan_aware_equal_bf16(got[s_, :n], o_out[s_, :n]), (fmt, off, s_)
    assert plan.status() == 0
    plan.close()


def test_fp8_wire_dsv3_reduced():
    _check_fp8_wire(wlmod.make_workload("dsv3", max_tok=300))


@pytest.mark.parametrize("variant", ["auto", "tiled_512", "whole_row"])
def test_fp8_wire_small_scalar_expert(variant):
    _check_fp8_wire(wlmod.make_workload("small", max_tok=64), variant)


def test_fp8_wire_fp8_payload():
    _check_fp8_wire(wlmod.make_workload("fp8", max_tok=256))


def test_fp8_wire_wide_fan_in():
    # min(W, k) = 16 > 8: rows fold in ascending batches of 8
    _check_fp8_wire(wlmod.custom_workload(W=16, E=2, k=32, H=256, M=40, n_tok=[40] * 8 + [3] * 8, seed=6))


def test_fp8_wire_dsv3_full():
    _check_fp8_wire(wlmod.make_workload("dsv3"))


def test_fp8_wire_rejects_fp16_plans_and_stale_epochs():
    wl = wlmod.make_workload("topk", k=8, max_tok=16)
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    with pytest.raises(ep.EpError) as e:
        plan.quantize_received(d.recv_x, d.epoch)
    assert e.value.code == ep.EP_ERR_ARG
    plan.close()
    wl = wlmod.make_workload("dsv3", max_tok=16)
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    q, s = plan.quantize_received(d.recv_x, d.epoch)
    plan.reset()
    with pytest.raises(ep.EpError) as e:
        plan.combine_fp8(q, s, None, d.epoch)
    assert e.value.code == ep.EP_ERR_STATE
    plan.close()


# ---------------------------------------------------------------- combine over an MX FP4 wire

def _check_fp4_wire(wl, variant="auto", edit_expert_out=None):
    """quantize_received_fp4 codes + scales and combine_fp4 outputs against the oracle, bit-exact.
    edit_expert_out(eo_np) may overwrite the received expert rows (in place) before quantising."""
    disp, eo, _, _ = oracle.run_workload(wl, harness.expert_np)
    plan, (x, w, scales, idx) = _setup(wl)
    plan.set_variant(variant)
    d = plan.dispatch(x, w, scales, idx, wl.n_tok)
    eo_g = harness.expert_torch(wl, d.recv_x, d.recv_idx, d.recv_w, d.recv_scales, d.recv_count)
    if edit_expert_out is not None:
        eo = eo.copy()
        edit_expert_out(eo)
        eo_g = torch.from_numpy(eo.view(np.int16)).to(DEV).view(torch.bfloat16)
    q, sc = oracle.quantize_mxfp4(eo)
    o_out, o_w = oracle.combine_fp4(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], q, sc,
                                    disp["recv_w"])
    qg, scg = plan.quantize_received_fp4(eo_g, d.epoch)
    out, out_w = plan.combine_fp4(qg, scg, d.recv_w, d.epoch)
    torch.cuda.synchronize()
    assert plan.status() == 0
    qg, scg = qg.cpu().numpy(), scg.cpu().numpy()
    cnt = d.recv_count.cpu().numpy()
    for r in range(wl.W):
        n = int(cnt[r])
        assert np.array_equal(scg[r, :n], sc[r, :n]), f"rank {r}: e8m0 scales"
        assert np.array_equal(qg[r, :n], q[r, :n]), f"rank {r}: e2m1 codes"
    out = gpu_path.raw(out)
    for s in range(wl.W):
        n = int(wl.n_tok[s])
        assert gpu_path.nan_aware_equal_bf16(out[s, :n], o_out[s, :n]), f"source rank {s}"
        if o_w is not None:
            assert np.array_equal(out_w[s, :n].cpu().numpy().view(np.uint32), o_w[s, :n].view(np.uint32))
    plan.close()


def test_fp4_wire_dsv3_reduced():
    _check_fp4_wire(wlmod.make_workload("dsv3", max_tok=300))


@pytest.mark.parametrize("variant", ["auto", "tiled_512", "whole_row"])
def test_fp4_wire_small_scalar_expert(variant):
    _check_fp4_wire(wlmod.make_workload("small", max_tok=64), variant)


def test_fp4_wire_fp8_payload():
    _check_fp4_wire(wlmod.make_workload("fp8", max_tok=256))


def test_fp4_wire_wide_fan_in():
    # min(W, k) = 16 > 8: rows fold in ascending batches of 8
    _check_fp4_wire(wlmod.custom_workload(W=16, E=2, k=32, H=256, M=40, n_tok=[40] * 8 + [3] * 8, seed=6))


def test_fp4_wire_ragged_blocks():
    # H = 96: three 32-element blocks per row, fewer than a warp's lanes; H = 1056: 33 blocks,
    # one past a warp's worth
    _check_fp4_wire(wlmod.custom_workload(W=4, E=3, k=4, H=96, M=37, n_tok=[37, 5, 0, 20], seed=11))
    _check_fp4_wire(wlmod.custom_workload(W=4, E=3, k=4, H=1056, M=37, n_tok=[37, 5, 0, 20], seed=12))
    # hidden % 128 == 0 takes the shared-memory pipeline: 12 blocks (one partial step) and 36
    # blocks (a full step of 32 and a partial one)
    _check_fp4_wire(wlmod.custom_workload(W=4, E=3, k=4, H=384, M=37, n_tok=[37, 5, 0, 20], seed=13))
    _check_fp4_wire(wlmod.custom_workload(W=4, E=3, k=4, H=1152, M=37, n_tok=[37, 5, 0, 20], seed=14))


def test_fp4_wire_edge_values():
    wl = wlmod.make_workload("small", max_tok=48)

    def edit(eo):
        f = eo.view(np.uint16).astype(np.uint32) << 16
        xf = f.view(np.float32).reshape(eo.shape).copy()
        H = xf.shape[-1]
        # every received row of rank 0 and 1 gets crafted blocks
        xf[0, :, :32] = 0.0                                           # all-zero block: scale code 127
        xf[0, :, 32:64] = np.float32(2.0) ** -130                     # subnormal BF16 block: code clamps to 0
        ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0], np.float32)
        xf[0, :, 64:96] = np.tile(np.concatenate([ties, -ties]), 2) * np.float32(4.0)   # amax 28: e = 2
        xf[1, :, :32] = np.float32(3e38)                              # near BF16 max: code 252
        xf[1, :, 32:64] = -np.float32(1e-3)
        xf[1, :, 64] = -0.0
        xf[1, :, 96:128] = np.linspace(-6.5, 6.5, 32, dtype=np.float32) * np.float32(2.0) ** -20
        if H > 160:
            xf[1, :, 128:160] = np.float32(2.0) ** -126 * np.float32(3.0)   # normal/subnormal edge
        if H >= 128:
            # rounding ties at the scale codes either side of the f16-scale window (113..142)
            for i, code in enumerate((112, 113, 142, 143)):
                xf[2, :, 32 * i:32 * i + 32] = np.tile(np.concatenate([ties, -ties]), 2) * np.float32(2.0) ** (code - 127)
        eo[:] = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    _check_fp4_wire(wl, edit_expert_out=edit)


def test_fp4_wire_dsv3_full():
    _check_fp4_wire(wlmod.make_workload("dsv3"))


def test_fp4_wire_rejects_bad_plans():
    wl = wlmod.make_workload("topk", k=8, max_tok=16)          # FP16 payload
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    with pytest.raises(ep.EpError) as e:
        plan.quantize_received_fp4(d.recv_x, d.epoch)
    assert e.value.code == ep.EP_ERR_ARG
    plan.close()
    wl = wlmod.custom_workload(W=2, E=2, k=2, H=48, M=8, n_tok=[8, 8], seed=3)   # 48 % 32 != 0
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    with pytest.raises(ep.EpError) as e:
        plan.quantize_received_fp4(d.recv_x, d.epoch)
    assert e.value.code == ep.EP_ERR_ARG
    plan.close()
    wl = wlmod.make_workload("dsv3", max_tok=16)
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    q, s = plan.quantize_received_fp4(d.recv_x, d.epoch)
    plan.reset()
    with pytest.raises(ep.EpError) as e:
        plan.combine_fp4(q, s, None, d.epoch)
    assert e.value.code == ep.EP_ERR_STATE
    plan.close()


# ---------------------------------------------------------------- expert-grouped layout

def _check_grouped(wl, seed=0, fused=False, repeats=1):
    """repeats > 1 groups again on the same plan into a packed buffer filled with 0xFF bytes, so
    rows a call fails to write show."""
    disp = oracle.dispatch(wl.W, wl.E, wl.k, wl.H, wl.elem_bytes, wl.sd, wl.M, wl.x, wl.weights,
                           wl.scales, wl.indices, wl.n_tok)
    g = oracle.group_by_expert(wl.W, wl.E, wl.k, wl.H, wl.elem_bytes, wl.M, disp)
    fp16 = wl.dtype == "fp16"
    rng = np.random.default_rng(seed)
    yf = torch.from_numpy(rng.standard_normal(g["packed_x"].shape[:3] + (wl.H,)).astype(np.float32))
    y = (yf.to(torch.float16) if fp16 else yf.to(torch.bfloat16)).view(torch.int16).numpy().view(np.uint16)
    o_out = oracle.ungroup_by_expert(wl.W, wl.E, wl.H, fp16, wl.M, disp["recv_count"], g, y)

    plan, (x, w, sc, idx) = _setup(wl)
    for rep in range(repeats):
        _check_grouped_once(wl, plan, x, w, sc, idx, disp, g, y, o_out, fused, rep > 0)
    plan.close()


def _check_grouped_once(wl, plan, x, w, sc, idx, disp, g, y, o_out, fused, poisoned):
    px = None
    if poisoned:
        px = torch.empty((wl.W, wl.E, wl.W * wl.M, plan.row_elems), dtype=plan.payload_torch_dtype, device=DEV)
        px.view(torch.uint8).fill_(0xFF)
    if fused:
        d, px, cnt, info, layout = plan.dispatch_grouped(x, w, sc, idx, wl.n_tok, packed_x=px)
    else:
        d = plan.dispatch(x, w, sc, idx, wl.n_tok)
        px, cnt, info, layout = plan.group_by_expert(d.epoch, packed_x=px)
    out = plan.ungroup_by_expert(torch.from_numpy(y.view(np.int16)).to(DEV), d.epoch)
    torch.cuda.synchronize()
    assert plan.status() == 0
    # the receive metadata is exactly the plain dispatch's (fused: payload rows are not written)
    dc = d.recv_count.cpu().numpy()
    assert np.array_equal(dc, disp["recv_count"])
    for r in range(wl.W):
        n = int(dc[r])
        assert np.array_equal(d.src_token_pos[r, :n].cpu().numpy(), disp["src_pos"][r, :n])
        assert np.array_equal(d.recv_idx[r, :n].cpu().numpy(), disp["recv_idx"][r, :n])
        if wl.weights is not None:
            assert np.array_equal(d.recv_w[r, :n].cpu().numpy(), disp["recv_w"][r, :n])
        if wl.sd:
            assert np.array_equal(d.recv_scales[r, :n].cpu().numpy(), disp["recv_scales"][r, :n])
    cnt = cnt.cpu().numpy()
    assert np.array_equal(cnt, g["packed_count"])
    assert np.array_equal(layout.cpu().numpy(), g["layout_range"])
    px, info = gpu_path.raw(px), info.cpu().numpy()
    for r in range(wl.W):
        for e in range(wl.E):
            n = int(cnt[r, e])
            assert np.array_equal(info[r, e, :n], g["packed_src_info"][r, e, :n]), (r, e)
            assert np.array_equal(px[r, e, :n], g["packed_x"][r, e, :n]), (r, e)
    out = gpu_path.raw(out)
    for r in range(wl.W):
        n = int(disp["recv_count"][r])
        assert np.array_equal(out[r, :n], o_out[r, :n]), r


@pytest.mark.parametrize("case", [
    dict(W=4, E=8, k=6, H=512, M=100, n_tok=[100, 37, 0, 64], dtype="bf16"),
    dict(W=8, E=4, k=8, H=256, M=40, n_tok=[40, 1, 2, 3, 40, 0, 39, 17], dtype="fp16"),
    dict(W=4, E=4, k=3, H=256, M=50, n_tok=[50, 7, 0, 31], dtype="fp8", sd=2),
    dict(W=2, E=32, k=33, H=128, M=70, n_tok=[70, 33], dtype="bf16"),
], ids=lambda c: f"W{c['W']}E{c['E']}k{c['k']}{c['dtype']}")
def test_grouped_layout(case):
    _check_grouped(wlmod.custom_workload(seed=5, **case))
    _check_grouped(wlmod.custom_workload(seed=5, **case), fused=True)


def test_grouped_layout_work_queue():
    """About 54 000 received rows, more than four rounds per warp of the grouped copy, so its
    last rows come from the plan's grouping queue; grouped twice on one plan, the second time
    into a poisoned buffer, and through the fused dispatch twice."""
    wl = wlmod.custom_workload(W=8, E=4, k=4, H=64, M=2048, n_tok=[2048] * 8, seed=12)
    _check_grouped(wl, repeats=2)
    _check_grouped(wl, fused=True, repeats=2)
    # rows of 4096 elements cut into 1024-element slices (fewer than four rows per warp), more than
    # four rounds of slices: the fused dispatch draws its last slices from the queue
    wl = wlmod.custom_workload(W=8, E=4, k=4, H=4096, M=1024, n_tok=[1024] * 8, seed=13)
    _check_grouped(wl, fused=True, repeats=2)


def _chunk_edge_workload(k):
    """Receive capacity 4 * 1100 rows, five 1024-row chunks, so grouping scans in two passes.
    Rank 0 receives all 3300 tokens (a ragged last chunk, up to three local experts a row),
    rank 1 exactly 2048 (two full chunks; sources 2 and 3 send it nothing; its expert 2 gets
    no row), rank 2 1025 (source 0 sends it nothing, source 2 has no tokens) and rank 3
    nothing.  Some rows name the same expert twice."""
    W, E, M = 4, 3, 1100
    wl = wlmod.custom_workload(W=W, E=E, k=k, H=64, M=M, n_tok=[M, M, 0, M], seed=21)
    g = 0
    for s in (0, 1, 3):
        for t in range(M):
            row = [g % 3]                                        # rank 0
            if g < 2048:
                row.append(E + (g // 7) % 2)                     # rank 1, experts 0 and 1
            elif g < 2048 + 1025:
                row.append(2 * E + g % 3)                        # rank 2
            else:
                row.append((g + 1) % 3)                          # rank 0 again
            row.append(row[0] if g % 5 == 0 else (g + 2) % 3)    # a repeat, or rank 0
            wl.indices[s, t] = [row[j % 3] for j in range(k)]
            g += 1
    return wl


@pytest.mark.parametrize("k", [3, 8])
def test_grouped_layout_chunked_scan(k):
    """The two-pass grouping scan at its chunk edges: empty ranks and sources, a rank whose
    rows end exactly on a chunk boundary and one a row past it, repeated ids; the one-row
    index loop (top-k 3) and the 16-byte-vector one (top-k 8)."""
    wl = _chunk_edge_workload(k)
    disp = oracle.dispatch(wl.W, wl.E, wl.k, wl.H, wl.elem_bytes, wl.sd, wl.M, wl.x, wl.weights,
                           wl.scales, wl.indices, wl.n_tok)
    assert list(disp["recv_count"]) == [3300, 2048, 1025, 0]
    _check_grouped(wl, repeats=2)
    _check_grouped(wl, fused=True, repeats=2)


def test_grouped_layout_chunk_strides():
    """More chunks than the scan grid's chunk stride: 512 lists take every fourth chunk of the
    12 (about 5 with rows), and 2500 lists one CTA per list for every chunk."""
    wl = wlmod.custom_workload(W=8, E=64, k=4, H=16, M=1536, n_tok=[1536] * 8, seed=22)
    _check_grouped(wl, repeats=2)
    _check_grouped(wl, fused=True)
    wl = wlmod.custom_workload(W=2, E=1250, k=2, H=8, M=1536, n_tok=[1536, 1500], seed=23)
    _check_grouped(wl)
    _check_grouped(wl, fused=True)


def test_grouped_layout_wide_rows():
    # hidden 2304 (288 16-byte vectors: nine full warp steps of 32 vectors) in BF16 and FP16,
    # grouped, fused and inverted
    for dt in ("bf16", "fp16"):
        wl = wlmod.custom_workload(W=4, E=8, k=6, H=2304, M=40, n_tok=[40, 17, 0, 33], dtype=dt, seed=8)
        _check_grouped(wl)
        _check_grouped(wl, fused=True)


def test_grouped_layout_duplicate_ids_and_small_workload():
    wl = wlmod.custom_workload(W=4, E=8, k=4, H=256, M=30, n_tok=[30, 30, 5, 9], seed=2)
    wl.indices[0, 3, 2] = wl.indices[0, 3, 0]       # the same expert twice in one top-k row
    wl.indices[1, 7, 3] = wl.indices[1, 7, 1]
    _check_grouped(wl)
    _check_grouped(wl, fused=True)
    _check_grouped(wlmod.make_workload("small", max_tok=24), seed=1)
    _check_grouped(wlmod.make_workload("small", max_tok=24), seed=1, fused=True)


@pytest.mark.parametrize("k", [4, 16])
def test_route_compiled_row_widths(k):
    _check(wlmod.custom_workload(W=8, E=8, k=k, H=256, M=300, n_tok=[300, 299, 0, 1, 256, 257, 2, 300], seed=k))


def test_route_with_indices_only_4_byte_aligned():
    """k % 4 == 0 but the index array starts 4 bytes past a 16-byte boundary: the routing kernel
    must fall back to scalar loads and route exactly as with an aligned array."""
    wl = wlmod.make_workload("dsv3", max_tok=200)
    plan, (x, w, sc, idx) = _setup(wl)
    d = plan.dispatch_route(idx, wl.n_tok)
    torch.cuda.synchronize()
    ref_cnt = d.recv_count.cpu().numpy().copy()
    ref_pos = d.src_token_pos.cpu().numpy().copy()
    buf = torch.empty(idx.numel() + 4, dtype=torch.int32, device=DEV)
    shifted = buf[1:1 + idx.numel()].view(idx.shape)
    shifted.copy_(idx)
    assert shifted.data_ptr() % 16 == 4
    d = plan.dispatch_route(shifted, wl.n_tok)
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert np.array_equal(d.recv_count.cpu().numpy(), ref_cnt)
    for r in range(wl.W):
        n = int(ref_cnt[r])
        assert np.array_equal(d.src_token_pos[r, :n].cpu().numpy(), ref_pos[r, :n])
    plan.close()


def test_many_tiles_long_lookback():
    """W = 32 ranks, 16384 tokens per rank: 2048 routing tiles whose lookback windows cover 8
    predecessors per step, with tiny rows so the oracle stays fast."""
    wl = wlmod.custom_workload(W=32, E=2, k=4, H=8, M=16384, n_tok=[16384] * 31 + [1000], seed=12,
                               with_weights=False)
    _check(wl)


def test_cuda_graph_replay_quantising_dispatch_and_fp8_wire():
    """The quantising dispatch, the wire quantiser and the FP8 combine captured in one CUDA graph
    and replayed give the eager results bit for bit."""
    wl = wlmod.make_workload("dsv3", max_tok=64)
    plan = gpu_path.make_plan(wl, DEV, plan_dtype="bf16_fp8")
    x, w, _, idx = gpu_path.to_device(wl, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = plan.dispatch(x, w, None, idx, wl.n_tok, stream=s)
        y = torch.empty((wl.W, wl.W * wl.M, wl.H), dtype=torch.bfloat16, device=DEV)
        counts = d.recv_count.cpu().tolist()
    torch.cuda.synchronize()
    # dequantising identity expert outside the graph's timed part: a fixed buffer
    eo = harness.expert_torch(gpu_path.quantised_view(wl), d.recv_x, d.recv_idx, d.recv_w,
                              d.recv_scales, d.recv_count)
    y.view(torch.int16).copy_(eo.view(torch.int16))
    q, sc = plan.quantize_received(y, d.epoch)
    out, out_w = plan.combine_fp8(q, sc, d.recv_w, d.epoch)
    torch.cuda.synchronize()
    eager = (gpu_path.raw(d.recv_x).copy(), gpu_path.raw(out).copy())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        d = plan.dispatch(x, w, None, idx, wl.n_tok, stream=s)
        plan.quantize_received(y, d.epoch, q=q.view(torch.uint8), scales=sc, stream=s)
        plan.combine_fp8(q, sc, d.recv_w, d.epoch, out=out, out_w=out_w, stream=s)
    for _ in range(3):
        out.zero_()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(gpu_path.raw(d.recv_x), eager[0])
        assert np.array_equal(gpu_path.raw(out), eager[1])
        assert d.recv_count.cpu().tolist() == counts
    assert plan.status() == 0
    plan.close()

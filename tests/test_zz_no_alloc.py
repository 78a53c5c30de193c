"""The allocation-free routing entry point, ep_route_noalloc, against the plan-based one.

ep_route_noalloc exists for callers that must not call cudaMalloc -- a serving runtime whose own
pool allocator already owns nearly all of HBM, or a plug-in whose host forbids allocation on the
hot path -- and so cannot create an ep_plan.  Whatever memory it is given, it must route exactly
as ep_dispatch_route does: the same receive counts, the same reverse map, and a forward map that
points back at each token; and all three must equal the oracle's, bit for bit.  Its scratch is one static array shared by every call, so two calls
in a row with different shapes check that each call starts from clean scan words.

This file is collected last on purpose (it adds no coverage the others depend on).
"""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_02_gb300 as ep
import oracle
from combine_ep_dispatch_02_gb300 import workloads as wlmod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA GPU")
    from combine_ep_dispatch_02_gb300 import build
    build.build()


def _with_plan(wl, dev):
    """Routing through the existing entry point (ep_dispatch_route on a plan)."""
    plan = ep.Plan(wl.W, wl.E, wl.k, wl.H, wl.dtype, wl.sd, wl.M, device=dev)
    d = plan.dispatch_route(torch.from_numpy(wl.indices).to(dev), wl.n_tok)
    torch.cuda.synchronize()
    counts = d.recv_count.cpu().numpy().copy()
    pos = d.src_token_pos.cpu().numpy().copy()
    assert plan.status() == 0
    plan.close()
    return counts, pos


def _without_alloc(wl, dev):
    W, M, F = wl.W, wl.M, min(wl.W, wl.k)
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.from_numpy(wl.indices).to(dev)
    pos = torch.full((W, W * M), -7, **i32)
    cnt = torch.full((W,), -7, **i32)
    fwd = torch.full((W, M, F), -7, **i32)
    status = torch.full((1,), 123, **i32)
    ep.route_noalloc(W, wl.E, wl.k, M, idx, wl.n_tok, pos, cnt, fwd, status)
    torch.cuda.synchronize()
    return cnt.cpu().numpy(), pos.cpu().numpy(), fwd.cpu().numpy(), int(status.item())


def _oracle_routing(wl):
    """The oracle's dispatch of the same routing (the payload does not affect routing, so a
    hidden of 8 zero elements stands in for the workload's rows)."""
    x = np.zeros((wl.W, wl.M, 8), dtype=np.uint16)
    d = oracle.dispatch(wl.W, wl.E, wl.k, 8, 2, 0, wl.M, x, None, None, wl.indices, wl.n_tok)
    return d["recv_count"], d["src_pos"], d["slot_of"]


def _check_same_routing(wl, dev):
    ref_cnt, ref_pos = _with_plan(wl, dev)
    cnt, pos, fwd, status = _without_alloc(wl, dev)
    o_cnt, o_pos, o_slot = _oracle_routing(wl)
    assert status == ep.EP_OK
    assert np.array_equal(cnt, ref_cnt)
    assert np.array_equal(cnt, o_cnt)                          # bit-exact against the oracle
    for r in range(wl.W):
        n = int(cnt[r])
        assert np.array_equal(pos[r, :n], ref_pos[r, :n]), f"rank {r}"
        assert np.array_equal(pos[r, :n], o_pos[r, :n]), f"rank {r} against the oracle"
    rows = wl.W * wl.M
    for s in range(wl.W):
        n = int(wl.n_tok[s])
        f = fwd[s, :n]                                        # [n][F]
        valid = f >= 0
        nvalid = valid.sum(axis=1)
        # entries are packed first, then -1
        assert np.array_equal(valid, np.arange(f.shape[1])[None, :] < nvalid[:, None])
        ranks = np.where(valid, f // rows, -1)
        want = [sorted({int(e) // wl.E for e in wl.indices[s, t]}) for t in range(n)]
        for t in range(n):
            assert ranks[t, :nvalid[t]].tolist() == want[t], (s, t)
        r_idx, slot = np.divmod(f[valid], rows)
        tok = np.repeat(np.arange(n), nvalid)
        assert np.array_equal(pos[r_idx, slot], s * rows + tok)
        # the forward map's rows are the oracle's slots, rank by rank
        assert np.array_equal(slot, o_slot[s, tok, r_idx])


def test_noalloc_routing_matches_plan_routing_two_calls_in_a_row():
    dev = torch.device("cuda", 0)
    # first call: the DeepSeek-V3 shape at 300 tokens per rank (several tiles, ragged tail)
    _check_same_routing(wlmod.make_workload("dsv3", max_tok=300), dev)
    # second call, another shape: W=4, top-33, two 32-slot batches per token
    _check_same_routing(wlmod.make_workload("topk", k=33), dev)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda", 0)
    W, M = 32, 8192          # 1 + 32 * 1024 scan words > 16384
    i32 = dict(dtype=torch.int32, device=dev)
    with pytest.raises(ep.EpError) as e:     # full-size buffers (40 MB), so only the shape is wrong
        ep.route_noalloc(W, 2, 4, M, torch.zeros((W, M, 4), **i32), [0] * W,
                         torch.zeros((W, W * M), **i32), torch.zeros(W, **i32), torch.zeros((W, M, 4), **i32),
                         torch.zeros(1, **i32))
    assert e.value.code == ep.EP_ERR_ARG
    assert "static scratch" in str(e.value)

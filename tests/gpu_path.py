"""Runs a workload through the CUDA library (C ABI via the binding) and returns host copies.

Shared by the GPU parity tests; the expert between dispatch and combine is the harness's
(tests/harness.py), applied on the GPU to the GPU's own receive rows."""
import numpy as np
import torch

import combine_ep_dispatch_02_gb300 as ep
import harness


def to_device(wl, dev):
    x = torch.from_numpy(wl.x.view(np.int16) if wl.elem_bytes == 2 else wl.x).to(dev)
    idx = torch.from_numpy(wl.indices).to(dev)
    w = torch.from_numpy(wl.weights).to(dev) if wl.weights is not None else None
    sc = torch.from_numpy(wl.scales).to(dev) if wl.sd else None
    return x, w, sc, idx


def make_plan(wl, dev, variant="auto", plan_dtype=None):
    plan = ep.Plan(wl.W, wl.E, wl.k, wl.H, plan_dtype or wl.dtype, 0 if plan_dtype else wl.sd,
                   wl.M, device=dev)
    plan.set_variant(variant)
    return plan


def poison(plan, dev):
    """Fill the plan's receive buffers with 0xFF bytes so rows the kernels fail to write show."""
    d = plan.dispatch_route(torch.zeros((plan.W, plan.M, plan.k), dtype=torch.int32, device=dev),
                            [0] * plan.W)
    for t in (d.recv_x, d.recv_idx, d.recv_w, d.recv_scales, d.src_token_pos):
        if t is not None:
            t.view(torch.uint8).fill_(0xFF)
    plan.reset()


def quantised_view(wl, q=None, scales=None):
    """The workload as the receiving side sees it after a quantising dispatch: FP8 rows and one
    FP32 scale per 128 elements (q / scales: the oracle's codes, when they are needed)."""
    from combine_ep_dispatch_02_gb300 import workloads as wlmod
    return wlmod.Workload(**{**wl.__dict__, "dtype": "fp8", "sd": wl.H // 128,
                             "x": wl.x if q is None else q, "scales": scales})


def raw(t):
    if t is None:
        return None
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


def run(wl, dev, variant="auto", plan=None, do_poison=True, quantise=False):
    """quantise=True: a BF16 workload through the quantising dtype; the expert then sees FP8
    rows with one scale per 128 elements (dequantising identity)."""
    own = plan is None
    if own:
        plan = make_plan(wl, dev, variant, "bf16_fp8" if quantise else None)
    if do_poison:
        poison(plan, dev)
    x, w, sc, idx = to_device(wl, dev)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    wl_e = quantised_view(wl) if quantise else wl
    eo = harness.expert_torch(wl_e, d.recv_x, d.recv_idx, d.recv_w, d.recv_scales, d.recv_count)
    out, out_w = plan.combine(eo, d.recv_w, d.epoch)
    torch.cuda.synchronize()
    res = {
        "recv_count": d.recv_count.cpu().numpy(),
        "recv_x": raw(d.recv_x), "recv_idx": raw(d.recv_idx), "recv_w": raw(d.recv_w),
        "recv_scales": raw(d.recv_scales), "src_pos": raw(d.src_token_pos),
        "out": raw(out), "out_w": raw(out_w), "status": plan.status(), "epoch": d.epoch,
    }
    if own:
        plan.close()
    return res


def nan_aware_equal_bf16(a, b):
    """Bitwise equality of 16-bit float arrays, any NaN equal to any NaN."""
    a = a.view(np.uint16)
    b = b.view(np.uint16)
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return np.array_equal(nan_a, nan_b) and np.array_equal(a[~nan_a], b[~nan_b])


def compare(wl, gpu, orc, o_out, o_w):
    """Assert GPU results equal the oracle's: counts, every received row (payload, indices,
    weights, scales, reverse map) bit for bit, and combine outputs bit for bit."""
    assert gpu["status"] == 0, gpu["status"]
    assert np.array_equal(gpu["recv_count"], orc["recv_count"]), (gpu["recv_count"], orc["recv_count"])
    for r in range(wl.W):
        n = int(orc["recv_count"][r])
        g_pos = gpu["src_pos"][r, :n]
        o_pos = orc["src_pos"][r, :n]
        # compare through src_token_pos: the multiset of (source position, row content) must
        # agree; the routing kernel's scan also fixes the order, so the rows line up one to one
        gi = np.argsort(g_pos, kind="stable")
        oi = np.argsort(o_pos, kind="stable")
        assert np.array_equal(g_pos[gi], o_pos[oi]), f"rank {r}: reverse map differs"
        assert np.array_equal(g_pos, o_pos), f"rank {r}: row order differs from (src rank, token) order"
        assert np.array_equal(gpu["recv_x"][r, :n], orc["recv_x"][r, :n]), f"rank {r}: payload"
        assert np.array_equal(gpu["recv_idx"][r, :n], orc["recv_idx"][r, :n]), f"rank {r}: indices"
        if wl.weights is not None:
            assert np.array_equal(gpu["recv_w"][r, :n].view(np.uint32),
                                  orc["recv_w"][r, :n].view(np.uint32)), f"rank {r}: weights"
        if wl.sd:
            assert np.array_equal(gpu["recv_scales"][r, :n].view(np.uint32),
                                  orc["recv_scales"][r, :n].view(np.uint32)), f"rank {r}: scales"
    for s in range(wl.W):
        n = int(wl.n_tok[s])
        assert nan_aware_equal_bf16(gpu["out"][s, :n], o_out[s, :n]), f"source rank {s}: combine"
        assert not gpu["out"][s, n:].any(), f"source rank {s}: rows past n_tok were written"
        if o_w is not None:
            assert np.array_equal(gpu["out_w"][s, :n].view(np.uint32), o_w[s, :n].view(np.uint32)), \
                f"source rank {s}: combined weights"

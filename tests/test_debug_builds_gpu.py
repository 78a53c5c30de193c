"""The two debug builds of libep.so on the GPU: EP_PROBE (per-phase device timestamps) and
EP_CHECKS (indices the kernels derive from device data are bounds-checked, and a failed check is
recorded as EP_ERR_DEVICE_BOUNDS instead of becoming an out-of-bounds access).

Both builds must give the oracle's results bit for bit.  The checks are exercised with one
corrupted input whose unchecked accesses would still stay inside the buffers (a receive count
one row past rank 0's capacity: its extra row is rank 1's first), so the test cannot fault a GPU
whether or not the check works.
"""
import os

import numpy as np
import pytest
import torch

import combine_ep_dispatch_02_gb300 as ep
import gpu_path
import harness
import oracle
from combine_ep_dispatch_02_gb300 import build
from combine_ep_dispatch_02_gb300 import workloads as wlmod

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
VARIANTS = os.path.join(build.PKG, "_build", "variants")


def _variant(define):
    d = os.path.join(VARIANTS, define.lower())
    return build.build(defines=[define], lib_path=os.path.join(d, f"libep_{define.lower()}.so"), build_dir=d)


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA GPU")
    build.build()
    oracle.build()
    return {"probe": ep.load_library(_variant("EP_PROBE")), "checks": ep.load_library(_variant("EP_CHECKS")),
            "default": ep.load_library()}


@pytest.fixture
def use_lib(monkeypatch, libs):
    def use(name):
        monkeypatch.setattr(ep, "_lib", libs[name])
    return use


def test_probe_build_records_each_phase_in_stream_order(use_lib):
    wl = wlmod.make_workload("dsv3", max_tok=200)
    disp, _, o_out, o_w = oracle.run_workload(wl, harness.expert_np)
    use_lib("probe")
    plan = gpu_path.make_plan(wl, DEV)
    plan.probe()                                           # clear what plan setup recorded
    gpu = gpu_path.run(wl, DEV, plan=plan, do_poison=False)
    gpu_path.compare(wl, gpu, disp, o_out, o_w)            # probes change no result
    t = plan.probe()
    for ph in ("route", "scatter", "combine"):
        assert t[ph] is not None and 0 < t[ph][0] <= t[ph][1], (ph, t[ph])
    # one stream: each phase starts after the previous one ended
    assert t["route"][1] <= t["scatter"][0] and t["scatter"][1] <= t["combine"][0], t
    for ph in ("quantise", "wire_combine", "group_scan", "group_copy", "ungroup"):
        assert t[ph] is None, (ph, t[ph])
    # reading reset the words; a grouped dispatch records routing and the grouped copy
    assert all(v is None for v in plan.probe().values())
    x, w, sc, idx = gpu_path.to_device(wl, DEV)
    plan.dispatch_grouped(x, w, sc, idx, wl.n_tok)
    t = plan.probe()
    assert t["route"] is not None and t["group_copy"] is not None and t["route"][1] <= t["group_copy"][0]
    assert plan.status() == 0
    plan.close()


def test_default_build_has_no_probes(use_lib):
    wl = wlmod.make_workload("tiny")
    use_lib("default")
    plan = gpu_path.make_plan(wl, DEV)
    with pytest.raises(ep.EpError) as e:
        plan.probe()
    assert e.value.code == ep.EP_ERR_STATE
    plan.close()


def test_checks_build_matches_oracle(use_lib):
    use_lib("checks")
    for wl in (wlmod.make_workload("dsv3", max_tok=300), wlmod.make_workload("topk", k=33),
               wlmod.make_workload("fp8", max_tok=128)):
        disp, _, o_out, o_w = oracle.run_workload(wl, harness.expert_np)
        gpu_path.compare(wl, gpu_path.run(wl, DEV), disp, o_out, o_w)


def test_checks_build_reports_a_receive_count_past_capacity(use_lib):
    """Rank 0's receive count set to its capacity + 1 before the inverse of the grouped view: the
    checked kernel skips rank 0's rows and records EP_ERR_DEVICE_BOUNDS; the plan then works
    again once the count is a real one."""
    use_lib("checks")
    wl = wlmod.custom_workload(W=4, E=8, k=4, H=64, M=40, n_tok=[40, 12, 0, 33], seed=3)
    plan = gpu_path.make_plan(wl, DEV)
    x, w, sc, idx = gpu_path.to_device(wl, DEV)
    d = plan.dispatch(x, w, sc, idx, wl.n_tok)
    px, cnt, info, lay = plan.group_by_expert(d.epoch)
    y = torch.zeros((wl.W, wl.E, wl.W * wl.M, wl.H), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    good = int(d.recv_count[0].item())
    d.recv_count[0] = wl.W * wl.M + 1
    plan.ungroup_by_expert(y, d.epoch)
    assert plan.status() == ep.EP_ERR_DEVICE_BOUNDS
    assert plan.status() == 0                              # reading cleared it
    d.recv_count[0] = good
    plan.ungroup_by_expert(y, d.epoch)
    assert plan.status() == 0
    plan.close()

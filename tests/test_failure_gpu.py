"""Failure detection on the GPU without a fault: an expired wait reports a status.

A test-only build of the library (EP_TEST_WITHHOLD_TILE0, short EP_SPIN_LIMIT) makes routing tile
0 never publish its scan words -- a flag nothing sets.  Every later tile's bounded lookback must
then give up, record EP_ERR_DEVICE_TIMEOUT in the plan's status word, and finish; the kernel
returns, the host reads the status, and the context stays usable for the normal library."""
import os

import numpy as np
import pytest
import torch

import combine_ep_dispatch_02_gb300 as ep
from combine_ep_dispatch_02_gb300 import build, workloads as wlmod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def withheld_lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA GPU")
    build.build()
    d = str(tmp_path_factory.mktemp("withheld"))
    path = build.build(force=True, defines=["EP_TEST_WITHHOLD_TILE0=1", "EP_SPIN_LIMIT=2048"],
                       lib_path=os.path.join(d, "libep.so"), build_dir=d)
    return ep.load_library(path)


def test_expired_wait_reports_timeout_and_context_survives(withheld_lib):
    dev = torch.device("cuda", 0)
    wl = wlmod.make_workload("dsv3", max_tok=256)        # 2048 tokens: 8 routing tiles
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev)
    idx = torch.from_numpy(wl.indices).to(dev)
    normal = ep.load_library()
    try:
        ep._lib = withheld_lib
        plan = ep.Plan(wl.W, wl.E, wl.k, wl.H, "bf16", 0, wl.M, device=dev)
        plan.dispatch(x, None, None, idx, wl.n_tok)
        torch.cuda.synchronize()
        assert plan.status() == ep.EP_ERR_DEVICE_TIMEOUT
        assert plan.status() == ep.EP_OK              # reading clears the word
        plan.close()
    finally:
        ep._lib = normal
    # the context still works: the normal library routes the same tokens without error
    plan = ep.Plan(wl.W, wl.E, wl.k, wl.H, "bf16", 0, wl.M, device=dev)
    d = plan.dispatch(x, None, None, idx, wl.n_tok)
    torch.cuda.synchronize()
    assert plan.status() == ep.EP_OK
    assert int(d.recv_count.sum()) > 0
    plan.close()

"""GPU parity on seeded random shapes: the CUDA path against the oracle, bit for bit, on shapes
drawn across the ABI's ranges rather than picked by hand.

Each case draws W (1..32), experts per rank, top-k (up to 64 and W*E), hidden, dtype (BF16, FP16, FP8
with its block scales as caller scales), the work split, the routing (uniform or Zipf) and ragged token counts with
empty ranks; it runs dispatch and combine through the C ABI and compares counts, reverse map,
every received row and the combined outputs with the oracle.  Shapes whose hidden is a multiple
of 128 also run the quantising dispatches and the combine wires; shapes whose grouped view stays
under 256 MB also run it through the fused dispatch.  Fan-in above 8 (W > 8 and k > 8)
reaches the wide folds.
"""
import numpy as np
import pytest
import torch

import gpu_path
import harness
import oracle
import test_parity_gpu as parity
from combine_ep_dispatch_02_gb300 import workloads as wlmod

pytestmark = pytest.mark.gpu

VARIANTS = ("auto", "whole_row", "tiled_512", "tiled_1024")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA GPU")
    from combine_ep_dispatch_02_gb300 import build
    build.build()
    oracle.build()


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    W = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 32]))
    E = int(rng.integers(1, 9))
    k = int(rng.integers(1, min(64, W * E) + 1))
    dtype = str(rng.choice(["bf16", "fp16", "fp8"]))
    sd = 0
    H = int(rng.choice([128, 256, 384, 1024, 2176])) if rng.random() < 0.5 else 16 * int(rng.integers(1, 90))
    if dtype == "fp8":                  # FP8 rows are quantised per 128-element block by the generator,
        H = 128 * max(1, H // 128)      # their scale rows are the block scales (the harness dequantises)
        sd = H // 128
    M = int(rng.integers(1, 160))
    n_tok = rng.integers(0, M + 1, size=W)
    n_tok[rng.random(W) < 0.2] = 0
    if rng.random() < 0.3:
        n_tok[rng.integers(0, W)] = M
    routing = "zipf" if rng.random() < 0.4 else "uniform"
    variant = str(rng.choice(VARIANTS))
    return dict(W=W, E=E, k=k, H=H, dtype=dtype, sd=sd, M=M, n_tok=[int(v) for v in n_tok], routing=routing), variant


@pytest.mark.parametrize("seed", range(48))
def test_random_shape_dispatch_combine(seed):
    case, variant = _draw(seed)
    wl = wlmod.custom_workload(seed=seed, **case)
    disp, _, o_out, o_w = oracle.run_workload(wl, harness.expert_np)
    gpu = gpu_path.run(wl, parity.DEV, variant)
    gpu_path.compare(wl, gpu, disp, o_out, o_w)


@pytest.mark.parametrize("seed", range(48))
def test_random_shape_next_rows(seed):
    """The quantising dispatches and both combine wires (hidden a multiple of 128, BF16), and the
    grouped view through the fused dispatch (any payload dtype, where the view stays under 256 MB)."""
    case, variant = _draw(seed)
    if case["dtype"] == "bf16" and case["H"] % 128 == 0:
        bf = dict(case, sd=0)
        wl = wlmod.custom_workload(seed=seed, **bf)
        parity._check_quantised(wl, variant)
        parity._check_mxfp4_dispatch(wl, variant)
        parity._check_fp8_wire(wl, variant)
        parity._check_fp4_wire(wl, variant)
    W, E, M, H = case["W"], case["E"], case["M"], case["H"]
    if W * E * W * M * H * 2 <= 256 << 20:      # the grouped view (and its host copy) stays small
        wl = wlmod.custom_workload(seed=seed, **case)
        parity._check_grouped(wl, seed=seed, fused=True)

"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: IEEE conversions of numpy and
torch, brute-force enumeration on tiny inputs written directly in Python, closed forms that
follow from the pages' definitions, and hand-worked values (tests/golden).  Passages pinned:
MORI-EP gfx1201 PR, "How the gfx1201 kernels work" (Dispatch: one receive row per token per
destination rank, shared hidden payload, reverse mapping; Combine: FP32 sum, BF16/FP16
conversion, weights summed separately, routing weights not applied) and the MORI-EP guide,
"Operator API" (output shapes, src_token_pos encoding).
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from combine_ep_dispatch_02_gb300 import workloads as wlmod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- conversions

def _edge_f32():
    v = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e30, -1e30, 3.3895314e38,
         3.4028235e38, np.inf, -np.inf, 2.0 ** -14, 2.0 ** -15, 2.0 ** -24, 2.0 ** -25,
         1.5 * 2.0 ** -25, 2.0 ** -26, 2.0 ** -126, 2.0 ** -149, 1.0 + 2.0 ** -8,
         1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -8 + 2.0 ** -23]
    return np.array(v + [-a for a in v], dtype=np.float32)


def _random_f32(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32)


def test_bf16_rne_matches_torch_cast():
    a = np.concatenate([_edge_f32(), _random_f32(200000, 1),
                        np.random.default_rng(2).standard_normal(100000).astype(np.float32)])
    mine = oracle.bf16_from_f32(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(a)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7F80) == 0x7F80) and np.all((mine[nan] & 0x7F) != 0)


def test_f16_rne_matches_numpy_cast():
    # numpy's float32 -> float16 cast is IEEE round-to-nearest-even, subnormals included
    a = np.concatenate([_edge_f32(), _random_f32(200000, 3),
                        (np.random.default_rng(4).standard_normal(100000) * 1e-5).astype(np.float32),
                        (np.random.default_rng(5).standard_normal(100000) * 3e4).astype(np.float32)])
    mine = oracle.f16_from_f32(a)
    with np.errstate(over="ignore"):
        ref = a.astype(np.float16).view(np.uint16)
    nan = np.isnan(a)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7C00) == 0x7C00) and np.all((mine[nan] & 0x3FF) != 0)


def test_f32_from_f16_exact_all_codes():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.f32_from_f16(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(mine[nan]))


# ---------------------------------------------------------------- dispatch invariants

def _brute_pairs(wl):
    """(s, t, r) for every token and every DISTINCT valid destination rank, by enumeration."""
    pairs = []
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            ranks = set()
            for e in wl.indices[s, t]:
                if 0 <= int(e) < wl.W * wl.E:
                    ranks.add(int(e) // wl.E)
            pairs += [(s, t, r) for r in sorted(ranks)]
    return pairs


def _check_dispatch(wl, disp):
    W, M = wl.W, wl.M
    rows = W * M
    pairs = _brute_pairs(wl)
    # counts: brute-force tally of tokens per destination rank
    tally = np.zeros(W, dtype=np.int64)
    for (_, _, r) in pairs:
        tally[r] += 1
    assert np.array_equal(disp["recv_count"], tally)
    # every (token, destination) pair appears exactly once, found by inverting src_pos
    got = []
    for r in range(W):
        for i in range(int(disp["recv_count"][r])):
            s, t = divmod(int(disp["src_pos"][r, i]), rows)
            got.append((s, t, r))
            # round trip: every byte of the row is the named source token's
            assert np.array_equal(disp["recv_x"][r, i], wl.x[s, t])
            assert np.array_equal(disp["recv_idx"][r, i], wl.indices[s, t])
            if wl.weights is not None:
                assert np.array_equal(disp["recv_w"][r, i].view(np.uint32), wl.weights[s, t].view(np.uint32))
            if wl.sd:
                assert np.array_equal(disp["recv_scales"][r, i].view(np.uint32), wl.scales[s, t].view(np.uint32))
            # the forward map points back at this row
            assert disp["slot_of"][s, t, r] == i
    assert sorted(got) == sorted(pairs)
    assert len(set(got)) == len(got)
    # rows are handed out in (source rank, token) order on each destination rank
    for r in range(W):
        n = int(disp["recv_count"][r])
        assert np.all(np.diff(disp["src_pos"][r, :n].astype(np.int64)) > 0)
    # slot_of is -1 exactly where the token was not sent
    sent = {(s, t, r) for (s, t, r) in pairs}
    for s in range(W):
        for t in range(int(wl.n_tok[s])):
            for r in range(W):
                assert (disp["slot_of"][s, t, r] >= 0) == ((s, t, r) in sent)


def _run(wl):
    return oracle.dispatch(wl.W, wl.E, wl.k, wl.H, wl.elem_bytes, wl.sd, wl.M, wl.x, wl.weights,
                           wl.scales, wl.indices, wl.n_tok)


CASES = [
    dict(W=2, E=4, k=2, H=64, M=16, n_tok=[16, 9]),
    dict(W=3, E=2, k=4, H=32, M=8, n_tok=[0, 8, 5]),
    dict(W=5, E=3, k=7, H=16, M=12, n_tok=[12, 1, 0, 7, 11]),
    dict(W=1, E=6, k=3, H=40, M=10, n_tok=[10]),
    dict(W=4, E=8, k=1, H=24, M=9, n_tok=[9, 9, 2, 4]),
    dict(W=4, E=16, k=33, H=8, M=6, n_tok=[6, 3, 6, 1]),
    dict(W=8, E=2, k=6, H=16, M=5, n_tok=[5, 0, 4, 5, 1, 2, 3, 5], sd=3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"W{c['W']}E{c['E']}k{c['k']}")
def test_dispatch_invariants(case):
    wl = wlmod.custom_workload(dtype="bf16", seed=7, **case)
    disp = _run(wl)
    assert disp["status"] == 0
    _check_dispatch(wl, disp)


def test_dispatch_fp8_payload_and_scales():
    wl = wlmod.make_workload("fp8", max_tok=24)
    disp = _run(wl)
    _check_dispatch(wl, disp)


def test_brute_force_every_subset():
    """W in {1,2,3}, E in {1,2}, every k-subset of the W*E experts as one token."""
    for W in (1, 2, 3):
        for E in (1, 2):
            n_exp = W * E
            for k in range(1, n_exp + 1):
                subsets = list(itertools.combinations(range(n_exp), k))
                M = -(-len(subsets) // W)
                n_tok = np.zeros(W, dtype=np.int32)
                idx = np.full((W, M, k), -1, dtype=np.int32)
                for i, sub in enumerate(subsets):
                    s, t = i % W, i // W
                    idx[s, t] = sub[::-1] if i % 2 else sub
                    n_tok[s] = max(n_tok[s], t + 1)
                rng = np.random.default_rng(W * 100 + E * 10 + k)
                x = torch.from_numpy(rng.standard_normal((W, M, 8)).astype(np.float32)) \
                    .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                wl = wlmod.Workload("brute", W, E, k, 8, "bf16", 0, M, n_tok, x, idx, None, None,
                                    "identity")
                disp = _run(wl)
                _check_dispatch(wl, disp)
                # combine with the identity expert: |D| * x, exactly representable before rounding
                out, _ = oracle.combine(W, k, 8, False, M, n_tok, disp["slot_of"], disp["recv_x"])
                for i, sub in enumerate(subsets):
                    s, t = i % W, i // W
                    nd = len({e // E for e in sub})
                    xf = (x[s, t].astype(np.uint32) << 16).view(np.float32)
                    exp = torch.from_numpy(xf * np.float32(nd)).to(torch.bfloat16).view(torch.int16) \
                        .numpy().view(np.uint16)
                    assert np.array_equal(out[s, t], exp), (W, E, k, sub)


def test_invalid_expert_ids_route_nowhere():
    wl = wlmod.custom_workload(W=3, E=2, k=3, H=16, M=4, n_tok=[4, 4, 4], seed=3)
    wl.indices[0, 1, 0] = -5
    wl.indices[2, 3, 2] = 6          # == W*E: out of range
    disp = _run(wl)
    assert disp["status"] == oracle.ERR_INDEX
    _check_dispatch(wl, disp)        # brute force skips the same ids


def test_capacity_rejected():
    wl = wlmod.custom_workload(W=2, E=2, k=2, H=8, M=4, n_tok=[4, 4], seed=1)
    with pytest.raises(ValueError):
        oracle.dispatch(2, 2, 2, 8, 2, 0, 4, wl.x, wl.weights, None, wl.indices,
                        np.array([5, 0], dtype=np.int32))


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_identity_combine_closed_form(dtype):
    """Identity expert: out = RNE(|D(s,t)| * x).  x has 8 (BF16) or 11 (FP16) significant bits,
    so every partial sum j*x is exact in FP32 and the FP32 sum equals |D| * x before rounding."""
    wl = wlmod.custom_workload(W=8, E=4, k=8, H=96, M=40, n_tok=[40, 17, 0, 40, 3, 40, 25, 1],
                               dtype=dtype, seed=11)
    disp = _run(wl)
    out, out_w = oracle.combine(wl.W, wl.k, wl.H, dtype == "fp16", wl.M, wl.n_tok, disp["slot_of"],
                                disp["recv_x"], disp["recv_w"])
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            nd = len({int(e) // wl.E for e in wl.indices[s, t]})
            if dtype == "bf16":
                xf = (wl.x[s, t].astype(np.uint32) << 16).view(np.float32)
                exp = torch.from_numpy(xf * np.float32(nd)).to(torch.bfloat16).view(torch.int16).numpy()
            else:
                xf = wl.x[s, t].view(np.float16).astype(np.float32)
                exp = (xf * np.float32(nd)).astype(np.float16).view(np.int16)
            assert np.array_equal(out[s, t].view(np.int16), exp)
    # rows past n_tok stay untouched (zero)
    assert not out[2].any() and not out[7, 1:].any()


def test_combine_order_golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "combine_order.txt")):
        if line.strip() and not line.startswith("#"):
            rows.append([int(v, 16) for v in line.split()])
    W, H, M = 4, 24, 1
    for vals in rows:
        slot_of = np.zeros((W, M, W), dtype=np.int32)       # the token's row is slot 0 on every rank
        eo = np.zeros((W, W * M, H), dtype=np.uint16)
        for r in range(W):
            eo[r, 0, :] = vals[r]
        out, _ = oracle.combine(W, 4, H, False, M, np.array([1, 0, 0, 0], np.int32), slot_of, eo)
        assert np.all(out[0, 0] == vals[4]), [hex(v) for v in vals]


def test_combine_weights_dyadic_closed_form():
    """Weights with few significant bits add exactly: out_w[s,t,j] = |D| * w[s,t,j]."""
    wl = wlmod.custom_workload(W=4, E=8, k=6, H=16, M=20, n_tok=[20, 20, 7, 13], seed=5)
    rng = np.random.default_rng(9)
    wl.weights[:] = rng.integers(-64, 64, size=wl.weights.shape).astype(np.float32) / np.float32(256)
    disp = _run(wl)
    _, out_w = oracle.combine(wl.W, wl.k, wl.H, False, wl.M, wl.n_tok, disp["slot_of"],
                              disp["recv_x"], disp["recv_w"])
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            nd = len({int(e) // wl.E for e in wl.indices[s, t]})
            assert np.array_equal(out_w[s, t], wl.weights[s, t] * np.float32(nd))


def test_single_destination_returns_expert_row():
    """k = 1, or all of a token's experts on one rank: |D| = 1, so combine returns the expert
    row unchanged (0.0f + v is exact, except that -0 becomes +0)."""
    for k, E in ((1, 8), (4, 16)):
        W, M, H = 4, 16, 40
        wl = wlmod.custom_workload(W=W, E=E, k=k, H=H, M=M, n_tok=[16, 5, 16, 9], seed=k)
        if k > 1:    # force every token's experts into one rank
            for s in range(W):
                for t in range(int(wl.n_tok[s])):
                    r = (s + t) % W
                    wl.indices[s, t] = r * E + np.arange(k)
        disp = _run(wl)
        rng = np.random.default_rng(1)
        eo = torch.from_numpy(rng.standard_normal((W, W * M, H)).astype(np.float32)) \
            .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        out, _ = oracle.combine(W, k, H, False, M, wl.n_tok, disp["slot_of"], eo)
        for s in range(W):
            for t in range(int(wl.n_tok[s])):
                r = int(wl.indices[s, t, 0]) // E
                exp = eo[r, disp["slot_of"][s, t, r]].copy()
                exp[exp == 0x8000] = 0
                assert np.array_equal(out[s, t], exp)


def test_single_rank_is_a_permuted_copy():
    """W = 1: every token has exactly one row, in order; identity combine returns x."""
    wl = wlmod.custom_workload(W=1, E=8, k=3, H=64, M=50, n_tok=[37], seed=2)
    disp = _run(wl)
    assert disp["recv_count"][0] == 37
    assert np.array_equal(disp["recv_x"][0, :37], wl.x[0, :37])
    assert np.array_equal(disp["src_pos"][0, :37], np.arange(37))
    out, _ = oracle.combine(1, 3, 64, False, 50, wl.n_tok, disp["slot_of"], disp["recv_x"])
    assert np.array_equal(out[0, :37], wl.x[0, :37])


def test_scalar_expert_pipeline_close_to_dense_formula():
    """Sanity (not a parity criterion): with the per-expert scalar expert, the combined output is
    sum_j w_j c_j x within a few BF16 ulps."""
    import harness
    wl = wlmod.make_workload("small", max_tok=12)
    disp, eo, out, _ = oracle.run_workload(wl, harness.expert_np)
    c = wl.expert_scale
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            xf = (wl.x[s, t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            coef = sum(float(wl.weights[s, t, j]) * float(c[wl.indices[s, t, j]]) for j in range(wl.k))
            got = (out[s, t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            err = np.abs(got - coef * xf)
            assert np.all(err <= 2.0 ** -6 * np.abs(coef * xf) + 1e-30)


def test_workload_generator_is_seeded():
    a = wlmod.make_workload("tiny")
    b = wlmod.make_workload("tiny")
    assert np.array_equal(a.x, b.x) and np.array_equal(a.indices, b.indices)
    assert np.array_equal(a.weights.view(np.uint32), b.weights.view(np.uint32))
    c = wlmod.make_workload("tiny", seed=1)
    assert not np.array_equal(a.x, c.x)
    # routing draws k distinct experts per token
    for name, kk in (("tiny", None), ("topk", 33), ("fp8", None)):
        wl = wlmod.make_workload(name, k=kk, max_tok=32)
        for s in range(wl.W):
            for t in range(int(wl.n_tok[s])):
                row = wl.indices[s, t]
                assert len(set(row.tolist())) == wl.k and row.min() >= 0 and row.max() < wl.W * wl.E


# ---------------------------------------------------------------- FP8 quantising dispatch (next row F1)

def test_e4m3_rne_matches_torch_cast():
    rng = np.random.default_rng(12)
    a = np.concatenate([
        rng.uniform(-448, 448, 200000).astype(np.float32),
        (rng.standard_normal(100000) * 2.0 ** -7).astype(np.float32),          # subnormal range
        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -6, 2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -10,
                  2.0 ** -11, 7 * 2.0 ** -9, 7.5 * 2.0 ** -9, 1.0625, 1.1875, 240.0, 248.0,
                  440.0, 447.99997], dtype=np.float32),
    ])
    a = np.concatenate([a, -a])
    mine = oracle.e4m3_from_f32(a)
    ref = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)
    # saturation: everything at or beyond 448 (and infinities) gives +-448; NaN stays NaN
    big = np.array([448.0, 449.0, 464.0, 465.0, 1e6, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_from_f32(big) == 0x7E) and np.all(oracle.e4m3_from_f32(-big) == 0xFE)
    assert (oracle.e4m3_from_f32(np.array([np.nan], np.float32))[0] & 0x7F) == 0x7F


def test_e4m3_decode_exact_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.f32_from_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_blockwise_quantiser_properties():
    rng = np.random.default_rng(3)
    rows, H = 64, 512
    xf = rng.standard_normal((rows, H)).astype(np.float32) * np.float32(3.0)
    xf[5, :128] = 0.0                       # an all-zero block: scale 1, codes 0
    xf[6, 128:256] *= np.float32(1e-4)      # tiny values: the scale keeps them representable
    xf[7, 256:384] = -xf[7, 256:384]
    x = _bf16(xf)
    q, sc = oracle.quantize_e4m3_blockwise(x)
    xs = (x.astype(np.uint32) << 16).view(np.float32).reshape(rows, H // 128, 128)
    amax = np.abs(xs).max(axis=2)
    assert sc[5, 0] == 1.0 and not (q[5, :128] & 0x7F).any()
    nz = amax > 0
    # scale = amax / 448 rounded once in FP32
    assert np.array_equal(sc[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    # the block maximum lands on +-448 exactly
    qb = q.reshape(rows, H // 128, 128)
    assert np.all(((qb & 0x7F) == 0x7E).any(axis=2)[nz])
    # every code is within half an e4m3 step of x / scale (relative 2^-4, or 2^-10 absolute
    # in the subnormal range)
    v = xs.astype(np.float64) / sc[:, :, None].astype(np.float64)
    deq = oracle.f32_from_e4m3(q).astype(np.float64).reshape(v.shape)
    assert np.all(np.abs(deq - v) <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))
    # signs survive (a negative value never becomes a positive code)
    assert np.all((xs < 0) <= ((qb & 0x80) != 0))


def test_blockwise_quantiser_scale_one_is_plain_cast():
    """A block whose maximum is 448 has scale 1, so every code is the plain e4m3 cast of x."""
    rng = np.random.default_rng(4)
    xf = rng.uniform(-440, 440, (8, 256)).astype(np.float32)
    xf[:, 0] = 448.0
    xf[:, 128] = -448.0
    x = _bf16(xf)
    q, sc = oracle.quantize_e4m3_blockwise(x)
    assert np.all(sc == 1.0)
    xb = (x.astype(np.uint32) << 16).view(np.float32)
    ref = torch.from_numpy(xb).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def _discriminating_blocks(n_max=300, seed=9):
    """BF16 blocks whose codes tell the IEEE quotient x / scale apart from x * (1 / scale).

    For seeded random block maxima (BF16 normals from 2^-31 to 2^31), every positive BF16 x no
    larger than the maximum is divided by scale = RN(amax / 448) two ways with torch on the CPU:
    the correctly rounded FP32 quotient, and the product with the rounded reciprocal.  Where the
    two land on different sides of an e4m3 rounding boundary, x goes into the block.  Returns
    (blocks [n][128] float32 holding BF16 values, count of such x)."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    allx = (bits << 16).view(np.float32)
    rng = np.random.default_rng(seed)
    blocks, hits = [], 0
    for amax_bits in rng.integers(0x3000, 0x4F00, n_max):
        amax = (np.uint32(amax_bits) << np.uint32(16)).view(np.float32)
        s = torch.tensor(amax, dtype=torch.float32) / torch.tensor(448.0, dtype=torch.float32)
        xs = torch.from_numpy(allx[allx <= amax])
        c_div = (xs / s).to(torch.float8_e4m3fn).view(torch.uint8)
        c_mul = (xs * (torch.tensor(1.0, dtype=torch.float32) / s)).to(torch.float8_e4m3fn).view(torch.uint8)
        sel = xs[c_div != c_mul].numpy()[:63]
        if len(sel) == 0:
            continue
        hits += 2 * len(sel)
        blk = rng.uniform(-1.0, 1.0, 128).astype(np.float32) * amax
        blk[0] = amax
        blk[1:1 + len(sel)] = sel
        blk[64:64 + len(sel)] = -sel
        blocks.append(blk)
    return np.stack(blocks), hits


def test_blockwise_quantiser_codes_are_the_ieee_quotient_cast():
    """Exact pin of the per-element quotient (reading of the guide's fp8_direct_cast): every code
    equals torch's e4m3fn cast of the correctly rounded FP32 quotient x / scale, with scale the
    FP32 quotient amax / 448.  The blocks hold random values and, above all, values whose
    quotient sits so close to an e4m3 rounding boundary that x * RN(1 / scale) rounds to the
    other code, so a reciprocal-multiply quotient fails here."""
    blocks, hits = _discriminating_blocks()
    assert hits >= 100
    x = _bf16(blocks)                       # one 128-element block per row
    q, sc = oracle.quantize_e4m3_blockwise(x)
    xs = torch.from_numpy((x.astype(np.uint32) << 16).view(np.float32)).reshape(x.shape[0], -1, 128)
    amax = xs.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / torch.tensor(448.0), torch.ones_like(amax))
    assert np.array_equal(sc.view(np.uint32), scale.numpy().view(np.uint32))
    ref = (xs / scale[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(x.shape).numpy()
    assert np.array_equal(q, ref)
    # random rows as well, across many binades
    rng = np.random.default_rng(31)
    xf = (rng.standard_normal((32, 512)) * np.exp(rng.uniform(-20, 20, (32, 1)))).astype(np.float32)
    x = _bf16(xf)
    q, sc = oracle.quantize_e4m3_blockwise(x)
    xs = torch.from_numpy((x.astype(np.uint32) << 16).view(np.float32)).reshape(32, 4, 128)
    scale = xs.abs().amax(dim=2) / torch.tensor(448.0)
    ref = (xs / scale[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(32, 512).numpy()
    assert np.array_equal(q, ref)


def test_quantised_dispatch_routes_quantised_rows():
    wl = wlmod.make_workload("dsv3", max_tok=24)
    disp = oracle.dispatch_quantized(wl)
    q, sc = oracle.quantize_e4m3_blockwise(wl.x)
    wq = wlmod.Workload(**{**wl.__dict__, "x": q, "dtype": "fp8", "sd": wl.H // 128, "scales": sc})
    _check_dispatch(wq, disp)


# ---------------------------------------------------------------- FP8 combine wire (next row F2)

def _fp8_wire_case(seed, W=4, E=4, k=3, H=256, M=12, n_tok=(12, 5, 0, 9)):
    wl = wlmod.custom_workload(W=W, E=E, k=k, H=H, M=M, n_tok=list(n_tok), seed=seed)
    disp = _run(wl)
    q, sc = oracle.quantize_e4m3_blockwise(disp["recv_x"])
    return wl, disp, q, sc


def test_fp8_combine_single_row_is_dequantised_row():
    """|D| = 1: out = BF16(float(q) * scale), with torch's e4m3 decode and an FP32 multiply."""
    wl = wlmod.custom_workload(W=3, E=5, k=1, H=256, M=10, n_tok=[10, 4, 7], seed=2)
    disp = _run(wl)
    q, sc = oracle.quantize_e4m3_blockwise(disp["recv_x"])
    out, _ = oracle.combine_fp8(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], q, sc)
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32) * \
        torch.from_numpy(np.repeat(sc, 128, axis=-1))
    ref = deq.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            r = int(wl.indices[s, t, 0]) // wl.E
            assert np.array_equal(out[s, t], ref[r, disp["slot_of"][s, t, r]])


def test_fp8_combine_power_of_two_scales_closed_form():
    """Scales that are powers of two make every product and partial sum exact (codes carry 4
    significant bits): out = BF16(sum over ranks of float(q) * scale), computed in float64."""
    wl, disp, q, sc = _fp8_wire_case(5)
    rng = np.random.default_rng(0)
    sc = (2.0 ** rng.integers(-6, 6, size=sc.shape)).astype(np.float32)
    out, _ = oracle.combine_fp8(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], q, sc)
    deq = oracle.f32_from_e4m3(q).astype(np.float64) * np.repeat(sc, 128, axis=-1)
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            tot = np.zeros(wl.H)
            for r in range(wl.W):
                if disp["slot_of"][s, t, r] >= 0:
                    tot += deq[r, disp["slot_of"][s, t, r]]
            ref = torch.from_numpy(tot.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(out[s, t].view(np.int16), ref)


def test_fp8_combine_close_to_bf16_combine():
    """Sanity (not a parity criterion): the FP8 wire moves each term by at most 2^-4 relative,
    so the FP8 combine stays within that of the BF16 combine of the same rows."""
    wl, disp, q, sc = _fp8_wire_case(8, W=8, E=2, k=6, H=384, M=20, n_tok=[20] * 8)
    out8, _ = oracle.combine_fp8(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], q, sc)
    out16, _ = oracle.combine(wl.W, wl.k, wl.H, False, wl.M, wl.n_tok, disp["slot_of"], disp["recv_x"])
    a = (out8.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = (out16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    amax = np.abs(b).max()
    assert np.all(np.abs(a - b) <= 2.0 ** -4 * np.abs(b) + 2.0 ** -3 * amax * 2.0 ** -7)


# ---------------------------------------------------------------- expert-grouped layout (next row F3)

def _check_grouping_brute_force(wl):
    disp = _run(wl)
    g = oracle.group_by_expert(wl.W, wl.E, wl.k, wl.H, 2, wl.M, disp)
    for r in range(wl.W):
        for e in range(wl.E):
            ge = r * wl.E + e
            lst = [(s, t) for s in range(wl.W) for t in range(int(wl.n_tok[s]))
                   if ge in set(int(v) for v in wl.indices[s, t])]
            n = len(lst)
            assert g["packed_count"][r, e] == n
            assert [int(v) for v in g["packed_src_info"][r, e, :n]] == [t for _, t in lst]
            for slot, (s, t) in enumerate(lst):
                assert np.array_equal(g["packed_x"][r, e, slot], wl.x[s, t])
                i = g["packed_row"][r, e, slot]
                assert disp["src_pos"][r, i] == s * wl.W * wl.M + t
            first = 0
            for s in range(wl.W):
                c = sum(1 for (ss, _) in lst if ss == s)
                assert g["layout_range"][r, e, s] == (first << 32) | c
                first += c


def test_group_by_expert_brute_force():
    for case in ({"W": 3, "E": 4, "k": 3, "H": 16, "M": 10, "n_tok": [10, 0, 7]},
                 {"W": 4, "E": 2, "k": 5, "H": 8, "M": 6, "n_tok": [6, 6, 1, 3]},
                 {"W": 1, "E": 8, "k": 8, "H": 24, "M": 9, "n_tok": [9]}):
        wl = wlmod.custom_workload(seed=4, **case)
        wl.indices[0, 0, 1] = wl.indices[0, 0, 0]          # a duplicate id counts once
        _check_grouping_brute_force(wl)


def test_group_by_expert_brute_force_random_shapes():
    """40 seeded small shapes: 1-6 ranks, 1-5 experts per rank, top-1..6 (at most W*E), empty
    ranks, and repeated ids in about a tenth of the rows."""
    rng = np.random.default_rng(2024)
    for case in range(40):
        W, E, M = int(rng.integers(1, 7)), int(rng.integers(1, 6)), int(rng.integers(1, 13))
        k = min(int(rng.integers(1, 7)), W * E)            # top-k picks distinct experts
        n_tok = [int(v) for v in rng.integers(0, M + 1, size=W)]
        wl = wlmod.custom_workload(W=W, E=E, k=k, H=8, M=M, n_tok=n_tok, seed=100 + case)
        if k > 1:
            dup = rng.random((W, M)) < 0.1
            wl.indices[:, :, 1] = np.where(dup, wl.indices[:, :, 0], wl.indices[:, :, 1])
        _check_grouping_brute_force(wl)


def test_ungroup_identity_closed_form():
    """Expert outputs equal to the grouped rows: each received row comes back as m * x, with m its
    number of distinct local experts (exact before the one rounding)."""
    wl = wlmod.custom_workload(W=4, E=8, k=6, H=32, M=12, n_tok=[12, 3, 0, 11], seed=8)
    disp = _run(wl)
    g = oracle.group_by_expert(wl.W, wl.E, wl.k, wl.H, 2, wl.M, disp)
    out = oracle.ungroup_by_expert(wl.W, wl.E, wl.H, False, wl.M, disp["recv_count"], g, g["packed_x"])
    for r in range(wl.W):
        for i in range(int(disp["recv_count"][r])):
            m = len({int(v) for v in disp["recv_idx"][r, i] if int(v) // wl.E == r})
            xf = (disp["recv_x"][r, i].astype(np.uint32) << 16).view(np.float32)
            exp = torch.from_numpy(xf * np.float32(m)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(out[r, i].view(np.int16), exp)


def test_ungroup_sums_in_ascending_expert_order():
    """Hand-worked values (tests/golden/combine_order.txt, row 2): experts 0..3 contribute
    2^-24, 2^-24, 2^-8, 1; the top-k lists them 3, 2, 1, 0.  Ascending expert order gives
    1 + 2^-7 (0x3F81); top-k order would give 1.0."""
    W, E, k, H, M = 1, 4, 4, 8, 1
    x = np.zeros((W, M, H), dtype=np.uint16)
    idx = np.array([[[3, 2, 1, 0]]], dtype=np.int32)
    wl = wlmod.Workload("order", W, E, k, H, "bf16", 0, M, np.array([1], np.int32), x, idx, None,
                        None, "identity")
    disp = _run(wl)
    g = oracle.group_by_expert(W, E, k, H, 2, M, disp)
    y = np.zeros_like(g["packed_x"])
    for e, v in enumerate((0x3380, 0x3380, 0x3B80, 0x3F80)):
        y[0, e, 0, :] = v
    out = oracle.ungroup_by_expert(W, E, H, False, M, disp["recv_count"], g, y)
    assert np.all(out[0, 0] == 0x3F81)


# ---------------------------------------------------------------- MX FP4 wire (F2, FP4 form)

_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_brute(v):
    """Nearest e2m1 magnitude by enumeration in float64; ties to the even code; saturate at 6."""
    a = min(abs(float(v)), 6.0)
    d = [abs(a - m) for m in _E2M1]
    best = min(range(8), key=lambda c: (d[c], c & 1))
    return best | (8 if np.signbit(v) else 0)


def test_e2m1_rne_brute_force():
    grid = np.concatenate([np.arange(0, 7.01, 0.03125), np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
                                                                 5.99, 6.01, 100.0, 1e-9])])
    vals = np.concatenate([grid, -grid]).astype(np.float32)
    for v in vals:
        assert oracle.e2m1_from_f32(v) == _e2m1_brute(v), v
    for c in range(16):                         # decode then encode is the identity (but -0)
        v = oracle.f32_from_e2m1(c)
        assert oracle.e2m1_from_f32(v) == (c if c != 8 else 8)
        assert abs(v) == _E2M1[c & 7]


def test_mxfp4_quantiser_against_numpy():
    rng = np.random.default_rng(21)
    rows, H = 40, 256
    xf = (rng.standard_normal((rows, H)) * np.exp(rng.uniform(-8, 8, (rows, 1)))).astype(np.float32)
    xf[3, :32] = 0.0                                   # all-zero block: scale code 127
    x = _bf16(xf)
    q, sc = oracle.quantize_mxfp4(x)
    xs = (x.astype(np.uint32) << 16).view(np.float32).reshape(rows, H // 32, 32).astype(np.float64)
    amax = np.abs(xs).max(axis=2)
    exp_code = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2 + 127, 127)
    assert np.array_equal(sc.astype(np.int64), np.clip(exp_code, 0, 254).astype(np.int64))
    scale = 2.0 ** (sc.astype(np.float64) - 127)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(rows, H // 32, 32)
    for r in range(0, rows, 7):
        for b in range(H // 32):
            for i in range(32):
                assert codes[r, b, i] == _e2m1_brute(xs[r, b, i] / scale[r, b]), (r, b, i)


def test_e8m0_decode_every_code():
    """Every scale code c in 0..254 decodes to 2^(c - 127) exactly, including code 0, the FP32
    subnormal 2^-127."""
    for c in range(255):
        v = np.float32(oracle.f32_from_e8m0(c))
        assert v == np.float32(2.0 ** (c - 127)), c
    assert np.float32(oracle.f32_from_e8m0(0)).view(np.uint32) == 0x00400000


def test_mxfp4_quantiser_tiny_blocks_take_scale_code_zero():
    """Blocks whose maximum is a BF16 subnormal give a scale code below 0, clamped to 0 (scale
    2^-127), and their codes are the brute-force e2m1 encoding of x / 2^-127; decoding them
    through the FP4 combine of one row gives BF16(e2m1 value * 2^-127)."""
    xf = np.zeros((2, 64), dtype=np.float32)
    xf[0, :32] = np.float32(2.0 ** -133) * np.arange(-16, 16, dtype=np.float32)   # subnormal BF16
    xf[0, 32:] = np.float32(2.0 ** -126) * np.linspace(-6, 6, 32, dtype=np.float32)
    xf[1, :32] = np.float32(2.0 ** -128)
    xf[1, 32:] = np.float32(-(2.0 ** -127)) * np.float32(3.0)
    x = _bf16(xf)
    q, sc = oracle.quantize_mxfp4(x)
    xs = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(2, 2, 32)
    amax = np.abs(xs).max(axis=2)
    exp_code = np.clip(np.floor(np.log2(amax)) - 2 + 127, 0, 254)
    assert np.array_equal(sc.astype(np.int64), exp_code.astype(np.int64))
    assert (sc == 0).sum() >= 2
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(2, 2, 32)
    scale = 2.0 ** (sc.astype(np.float64) - 127)
    for r in range(2):
        for b in range(2):
            for i in range(32):
                assert codes[r, b, i] == _e2m1_brute(xs[r, b, i] / scale[r, b]), (r, b, i)
    # the combine of a single row dequantises with the code-0 scale
    wl = wlmod.custom_workload(W=1, E=1, k=1, H=64, M=2, n_tok=[2], seed=0)
    slot_of = np.array([[[0]], [[1]]], dtype=np.int32)
    out, _ = oracle.combine_fp4(1, 1, 64, 2, wl.n_tok, slot_of, q[None], sc[None])
    mags = np.array(_E2M1 * 2) * np.where(np.arange(16) >= 8, -1.0, 1.0)
    deq = 0.0 + mags[codes.reshape(2, 64)] * np.repeat(scale.reshape(2, 2), 32, axis=-1)   # the sum starts at +0
    ref = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(out[0].view(np.int16), ref)


def test_fp4_combine_exact_sums():
    """Dequantised terms are exact (2-bit significands times powers of two) and span a small
    exponent range here, so the FP32 sum is exact: out = BF16(float64 sum of the terms)."""
    wl = wlmod.custom_workload(W=4, E=4, k=3, H=64, M=12, n_tok=[12, 5, 0, 9], seed=3)
    disp = _run(wl)
    q, sc = oracle.quantize_mxfp4(disp["recv_x"])
    out, _ = oracle.combine_fp4(wl.W, wl.k, wl.H, wl.M, wl.n_tok, disp["slot_of"], q, sc)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[:-1] + (wl.H,))
    mags = np.array(_E2M1 * 2) * np.where(np.arange(16) >= 8, -1.0, 1.0)
    deq = mags[codes] * np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=-1)
    for s in range(wl.W):
        for t in range(int(wl.n_tok[s])):
            tot = np.zeros(wl.H)
            for r in range(wl.W):
                if disp["slot_of"][s, t, r] >= 0:
                    tot += deq[r, disp["slot_of"][s, t, r]]
            ref = torch.from_numpy(tot.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(out[s, t].view(np.int16), ref)

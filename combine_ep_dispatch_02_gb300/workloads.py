"""Seeded synthetic inputs for MoE expert-parallel Dispatch / Combine.

This module only draws inputs: token rows, top-k expert indices, routing weights,
FP8 block scales and per-rank token counts.  It holds none of the dispatch or
combine arithmetic, so both the CUDA path and the CPU oracle can consume the
same arrays without sharing any code of the method.

The five workloads follow the shapes the MORI-EP pages measure on:

* ``tiny``      W=2, 4 experts/rank, top-2, hidden 256 BF16, 64 tokens/rank, uniform routing
                (the small case a plain CPU oracle finishes instantly).
* ``small``     W=4, 64 experts/rank, top-8, hidden 7168 BF16, 256 tokens/rank, uniform routing,
                expert = per-expert scalar c_e ~ U(0.5, 1.5) (the "<= 256 source tokens" small-batch
                regime of the gfx1201 launch policy, MORI-EP gfx1201 PR, "Wave32 and launch policy").
* ``dsv3``      W=8, 32 experts/rank (256 total), top-8, hidden 7168 BF16, 4096 tokens/rank,
                Zipf(s=1.2) expert popularity, identity expert (the DeepSeek-V3 example of the
                MORI-EP guide, "Configuration").
* ``topk``      W=4, 64 experts/rank, hidden 2048 FP16, 512 tokens/rank, top-k in
                {1, 2, 8, 9, 32, 33, 64} (runtime routing loops over 32-slot batches).
* ``fp8``       W=8, 96 experts/rank (768 total), top-6, hidden 7168 FP8 e4m3 payload with one FP32
                scale per 128 elements (scale_dim 56), ragged per-rank counts in [16, 4096], BF16
                combine output.

Randomness: numpy PCG64 streams, ``SeedSequence(seed).spawn(8)[workload_id]``.  Token values are
drawn in float32 from N(0, 1) and rounded to nearest even into BF16 / FP16 / FP8 by torch's CPU
casts (IEEE conversions; the method never depends on how its inputs were drawn).

Arrays are numpy, laid out exactly as the device expects them:
``x [W][M][H]`` (raw element bits: uint16 for BF16/FP16, uint8 for FP8), ``indices [W][M][k]``
int32, ``weights [W][M][k]`` float32, ``scales [W][M][sd]`` float32, ``n_tok [W]`` int32.
Rows at or past ``n_tok[s]`` are padding: x and weights are zero, indices are -1.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

DTYPES = ("bf16", "fp16", "fp8")
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp8": 1}
FP8_E4M3_MAX = 448.0
FP8_BLOCK = 128

WORKLOAD_IDS = {"tiny": 1, "small": 2, "dsv3": 3, "topk": 4, "fp8": 5}
TOPK_SWEEP = (1, 2, 8, 9, 32, 33, 64)


@dataclasses.dataclass
class Workload:
    name: str
    W: int                      # logical expert-parallel ranks
    E: int                      # experts per rank
    k: int                      # top-k experts per token
    H: int                      # hidden size (elements)
    dtype: str                  # payload dtype: bf16 | fp16 | fp8
    sd: int                     # FP32 scales per token row (0 = none)
    M: int                      # max tokens per rank (capacity)
    n_tok: np.ndarray           # int32 [W]
    x: np.ndarray               # raw bits [W][M][H]
    indices: np.ndarray         # int32 [W][M][k]
    weights: Optional[np.ndarray]   # float32 [W][M][k] or None
    scales: Optional[np.ndarray]    # float32 [W][M][sd] or None
    expert: str                 # identity | scalar (harness-side expert model)
    expert_scale: Optional[np.ndarray] = None   # float32 [W*E] for expert == "scalar"

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def combine_dtype(self) -> str:
        return "fp16" if self.dtype == "fp16" else "bf16"

    @property
    def N(self) -> int:
        return int(self.n_tok.sum())

    def describe(self) -> dict:
        return {"workload": self.name, "W": self.W, "experts_per_rank": self.E, "topk": self.k,
                "hidden": self.H, "dtype": self.dtype, "scale_dim": self.sd,
                "max_tok_per_rank": self.M, "tokens": self.N}


def _rng(workload_id: int, seed: int) -> np.random.Generator:
    child = np.random.SeedSequence(seed).spawn(8)[workload_id]
    return np.random.Generator(np.random.PCG64(child))


def _to_bits(xf: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(xf, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp16":
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def _uniform_routing(rng, n: int, n_experts: int, k: int) -> np.ndarray:
    # first k entries of a uniformly random permutation of all experts, per token
    keys = rng.random((n, n_experts))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _zipf_routing(rng, n: int, n_experts: int, k: int, s: float) -> np.ndarray:
    # expert popularity p_i ~ i^-s over i = 1..n_experts, assigned to experts by a random
    # permutation; each token takes k experts without replacement (Gumbel-top-k on log p).
    p = np.arange(1, n_experts + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    perm = rng.permutation(n_experts)
    logp = np.empty(n_experts)
    logp[perm] = np.log(p)
    out = np.empty((n, k), dtype=np.int32)
    step = 4096
    for a in range(0, n, step):
        b = min(n, a + step)
        g = rng.gumbel(size=(b - a, n_experts))
        out[a:b] = np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :k]
    return out


def _softmax_weights(rng, n: int, k: int) -> np.ndarray:
    z = rng.standard_normal((n, k))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def _fp8_blockwise(rng, n: int, H: int):
    # per-128-element block: scale = amax / 448 (amax 0 -> 1), q = saturating RNE e4m3fn(x / scale)
    xf = rng.standard_normal((n, H), dtype=np.float32)
    blocks = xf.reshape(n, H // FP8_BLOCK, FP8_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(FP8_E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = np.clip(blocks / scale[:, :, None], -FP8_E4M3_MAX, FP8_E4M3_MAX).reshape(n, H)
    q = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), scale


def make_workload(name: str, *, k: Optional[int] = None, max_tok: Optional[int] = None,
                  seed: int = 0, with_weights: bool = True) -> Workload:
    """Build one named workload.

    ``k`` selects the top-k of the ``topk`` sweep (default 8).  ``max_tok`` shrinks the per-rank
    capacity M (token counts are clipped / rescaled to it) so parity tests can run the same
    distributions at sizes a CPU oracle finishes in seconds.
    """
    if name not in WORKLOAD_IDS:
        raise ValueError(f"unknown workload {name!r}; choose from {sorted(WORKLOAD_IDS)}")
    rng = _rng(WORKLOAD_IDS[name], seed)
    expert, expert_scale, sd = "identity", None, 0
    if name == "tiny":
        W, E, kk, H, dt, M = 2, 4, 2, 256, "bf16", 64
    elif name == "small":
        W, E, kk, H, dt, M = 4, 64, 8, 7168, "bf16", 256
        expert = "scalar"
    elif name == "dsv3":
        W, E, kk, H, dt, M = 8, 32, 8, 7168, "bf16", 4096
    elif name == "topk":
        W, E, kk, H, dt, M = 4, 64, (8 if k is None else k), 2048, "fp16", 512
        if kk not in TOPK_SWEEP and k is None:
            raise ValueError(kk)
    else:  # fp8
        W, E, kk, H, dt, M = 8, 96, 6, 7168, "fp8", 4096
        sd = H // FP8_BLOCK
    if k is not None:
        kk = k
    if not 1 <= kk <= W * E:
        raise ValueError(f"top-k {kk} outside 1..{W * E}")

    if name == "fp8":
        n_full = rng.integers(16, M + 1, size=W)
    else:
        n_full = np.full(W, M)
    if max_tok is not None and max_tok < M:
        n_tok = np.maximum(1, (n_full * max_tok) // M) if name == "fp8" else np.full(W, max_tok)
        M = max_tok
    else:
        n_tok = n_full
    n_tok = n_tok.astype(np.int32)
    N = int(n_tok.sum())
    n_exp = W * E

    if name == "dsv3":
        flat_idx = _zipf_routing(rng, N, n_exp, kk, 1.2)
    else:
        flat_idx = _uniform_routing(rng, N, n_exp, kk)
    flat_w = _softmax_weights(rng, N, kk) if with_weights else None

    eb = ELEM_BYTES[dt]
    x = np.zeros((W, M, H), dtype=np.uint8 if eb == 1 else np.uint16)
    indices = np.full((W, M, kk), -1, dtype=np.int32)
    weights = np.zeros((W, M, kk), dtype=np.float32) if with_weights else None
    scales = np.zeros((W, M, sd), dtype=np.float32) if sd else None
    off = 0
    for s in range(W):
        n = int(n_tok[s])
        if dt == "fp8":
            q, sc = _fp8_blockwise(rng, n, H)
            x[s, :n] = q
            scales[s, :n] = sc
        else:
            x[s, :n] = _to_bits(rng.standard_normal((n, H), dtype=np.float32), dt)
        indices[s, :n] = flat_idx[off:off + n]
        if with_weights:
            weights[s, :n] = flat_w[off:off + n]
        off += n
    if expert == "scalar":
        expert_scale = rng.uniform(0.5, 1.5, size=n_exp).astype(np.float32)
    return Workload(name=name, W=W, E=E, k=kk, H=H, dtype=dt, sd=sd, M=M, n_tok=n_tok, x=x,
                    indices=indices, weights=weights, scales=scales, expert=expert,
                    expert_scale=expert_scale)


def custom_workload(*, W: int, E: int, k: int, H: int, dtype: str = "bf16", sd: int = 0,
                    M: int, n_tok, seed: int = 0, routing: str = "uniform",
                    with_weights: bool = True) -> Workload:
    """A workload of arbitrary shape with uniform (or Zipf) routing, for edge-case tests."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, W, E, k, H, M])))
    n_tok = np.asarray(n_tok, dtype=np.int32).reshape(W)
    N = int(n_tok.sum())
    eb = ELEM_BYTES[dtype]
    if routing == "zipf":
        flat_idx = _zipf_routing(rng, N, W * E, k, 1.2)
    else:
        flat_idx = _uniform_routing(rng, N, W * E, k)
    flat_w = _softmax_weights(rng, N, k) if with_weights else None
    x = np.zeros((W, M, H), dtype=np.uint8 if eb == 1 else np.uint16)
    indices = np.full((W, M, k), -1, dtype=np.int32)
    weights = np.zeros((W, M, k), dtype=np.float32) if with_weights else None
    scales = np.zeros((W, M, sd), dtype=np.float32) if sd else None
    off = 0
    for s in range(W):
        n = int(n_tok[s])
        if dtype == "fp8":
            q, sc = _fp8_blockwise(rng, n, H)
            x[s, :n] = q
            if sd:
                scales[s, :n] = (sc if sc.shape[1] == sd
                                 else rng.standard_normal((n, sd)).astype(np.float32))
        else:
            x[s, :n] = _to_bits(rng.standard_normal((n, H), dtype=np.float32), dtype)
            if sd:
                scales[s, :n] = rng.standard_normal((n, sd)).astype(np.float32)
        indices[s, :n] = flat_idx[off:off + n]
        if with_weights:
            weights[s, :n] = flat_w[off:off + n]
        off += n
    return Workload(name="custom", W=W, E=E, k=k, H=H, dtype=dtype, sd=sd, M=M, n_tok=n_tok,
                    x=x, indices=indices, weights=weights, scales=scales, expert="identity")

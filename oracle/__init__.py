"""CPU oracle for MoE expert-parallel Dispatch / Combine (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding) never does.

The arithmetic lives in plain C (``ep_oracle.c``, single-threaded, ``-O2 -ffp-contract=off``);
this module builds it with gcc on first use and marshals numpy arrays through ctypes.
Every function restates the definitions of the MORI-EP pages (gfx1201 PR, "How the gfx1201
kernels work"; MORI-EP guide, "Operator API"), see the C file's header for the readings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB = os.path.join(_HERE, "libep_oracle.so")
_lock = threading.Lock()
_lib = None

ERR_ARG = -1
ERR_INDEX = -6

_p = ctypes.c_void_p


def use_library(path):
    """Point this module at another build of the oracle (the mutation tests compile copies
    with planted mistakes); None restores the default build."""
    global _lib
    with _lock:
        _lib = None
    if path is not None:
        _load(path)


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into libep_oracle.so next to it (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load(path=None):
    global _lib
    with _lock:
        if _lib is None:
            if path is None:
                build()
            lib = ctypes.CDLL(path or _LIB)
            lib.ep_oracle_dispatch.restype = ctypes.c_int
            lib.ep_oracle_dispatch.argtypes = [ctypes.c_int] * 7 + [_p] * 12
            lib.ep_oracle_combine.restype = ctypes.c_int
            lib.ep_oracle_combine.argtypes = [ctypes.c_int] * 5 + [_p] * 6
            lib.ep_oracle_group_by_expert.restype = ctypes.c_int
            lib.ep_oracle_group_by_expert.argtypes = [ctypes.c_int] * 6 + [_p] * 9
            lib.ep_oracle_ungroup_by_expert.restype = ctypes.c_int
            lib.ep_oracle_ungroup_by_expert.argtypes = [ctypes.c_int] * 5 + [_p] * 5
            lib.ep_oracle_quantize_mxfp4.restype = ctypes.c_int
            lib.ep_oracle_quantize_mxfp4.argtypes = [ctypes.c_int64, ctypes.c_int, _p, _p, _p]
            lib.ep_oracle_combine_fp4.restype = ctypes.c_int
            lib.ep_oracle_combine_fp4.argtypes = [ctypes.c_int] * 4 + [_p] * 7
            lib.ep_oracle_e2m1_from_f32.restype = ctypes.c_uint8
            lib.ep_oracle_e2m1_from_f32.argtypes = [ctypes.c_float]
            lib.ep_oracle_f32_from_e2m1.restype = ctypes.c_float
            lib.ep_oracle_f32_from_e2m1.argtypes = [ctypes.c_uint8]
            lib.ep_oracle_f32_from_e8m0.restype = ctypes.c_float
            lib.ep_oracle_f32_from_e8m0.argtypes = [ctypes.c_uint8]
            lib.ep_oracle_combine_fp8.restype = ctypes.c_int
            lib.ep_oracle_combine_fp8.argtypes = [ctypes.c_int] * 4 + [_p] * 7
            lib.ep_oracle_quantize_e4m3_blockwise.restype = ctypes.c_int
            lib.ep_oracle_quantize_e4m3_blockwise.argtypes = [ctypes.c_int64, ctypes.c_int, _p, _p, _p]
            for name in ("ep_oracle_bf16_from_f32_array", "ep_oracle_f16_from_f32_array",
                         "ep_oracle_f32_from_f16_array", "ep_oracle_e4m3_from_f32_array",
                         "ep_oracle_f32_from_e4m3_array"):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = [_p, _p, ctypes.c_int64]
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def dispatch(W, E, k, H, elem_bytes, sd, M, x, weights, scales, indices, n_tok):
    """Dispatch every source token to one receive row per distinct destination rank.

    Returns a dict with ``recv_x [W][W*M][H]`` (raw bits), ``recv_idx``, ``recv_w`` (or None),
    ``recv_scales`` (or None), ``src_pos [W][W*M]``, ``slot_of [W][M][W]`` (row of token (s,t)
    on rank r, -1 if not sent there), ``recv_count [W]`` and ``status`` (0, or -6 when an expert
    id was out of range).  Receive rows at or past ``recv_count[r]`` are zero.
    """
    lib = _load()
    rows = W * M
    x = np.ascontiguousarray(x)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    n_tok = np.ascontiguousarray(n_tok, dtype=np.int32)
    dt = np.uint8 if elem_bytes == 1 else np.uint16
    out = {
        "recv_x": np.zeros((W, rows, H), dtype=dt),
        "recv_idx": np.zeros((W, rows, k), dtype=np.int32),
        "recv_w": np.zeros((W, rows, k), dtype=np.float32) if weights is not None else None,
        "recv_scales": np.zeros((W, rows, sd), dtype=np.float32) if sd else None,
        "src_pos": np.full((W, rows), -1, dtype=np.int32),
        "slot_of": np.full((W, M, W), -1, dtype=np.int32),
        "recv_count": np.zeros(W, dtype=np.int32),
    }
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    sc = None if not sd else np.ascontiguousarray(scales, dtype=np.float32)
    st = lib.ep_oracle_dispatch(W, E, k, H, elem_bytes, sd, M, _ptr(x), _ptr(w), _ptr(sc),
                                _ptr(indices), _ptr(n_tok), _ptr(out["recv_x"]),
                                _ptr(out["recv_idx"]), _ptr(out["recv_w"]),
                                _ptr(out["recv_scales"]), _ptr(out["src_pos"]),
                                _ptr(out["slot_of"]), _ptr(out["recv_count"]))
    if st == ERR_ARG:
        raise ValueError("ep_oracle_dispatch: invalid arguments")
    out["status"] = st
    return out


def combine(W, k, H, out_fp16, M, n_tok, slot_of, expert_out, w_in=None, out=None):
    """Gather each source token's rows back, sum in FP32 in ascending rank order, round to
    nearest even into BF16 (``out_fp16=False``) or FP16.  Returns ``(out [W][M][H] uint16,
    out_w [W][M][k] float32 or None)``; rows past ``n_tok[s]`` are zero (or ``out``'s content)."""
    lib = _load()
    n_tok = np.ascontiguousarray(n_tok, dtype=np.int32)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    expert_out = np.ascontiguousarray(expert_out).view(np.uint16)
    if out is None:
        out = np.zeros((W, M, H), dtype=np.uint16)
    out_w = np.zeros((W, M, k), dtype=np.float32) if w_in is not None else None
    w_in = None if w_in is None else np.ascontiguousarray(w_in, dtype=np.float32)
    st = lib.ep_oracle_combine(W, k, H, 1 if out_fp16 else 0, M, _ptr(n_tok), _ptr(slot_of),
                               _ptr(expert_out), _ptr(w_in), _ptr(out), _ptr(out_w))
    if st != 0:
        raise ValueError("ep_oracle_combine: invalid arguments")
    return out, out_w


def combine_fp8(W, k, H, M, n_tok, slot_of, q, scales, w_in=None):
    """Combine over an FP8 wire: each row's codes are dequantised as float(q) * scale (one FP32
    multiply) and added in ascending rank order in FP32; BF16 RNE output.  Returns (out, out_w)."""
    lib = _load()
    n_tok = np.ascontiguousarray(n_tok, dtype=np.int32)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    q = np.ascontiguousarray(q).view(np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.zeros((W, M, H), dtype=np.uint16)
    out_w = np.zeros((W, M, k), dtype=np.float32) if w_in is not None else None
    w_in = None if w_in is None else np.ascontiguousarray(w_in, dtype=np.float32)
    if lib.ep_oracle_combine_fp8(W, k, H, M, _ptr(n_tok), _ptr(slot_of), _ptr(q), _ptr(scales),
                                 _ptr(w_in), _ptr(out), _ptr(out_w)) != 0:
        raise ValueError("ep_oracle_combine_fp8: invalid arguments")
    return out, out_w


def group_by_expert(W, E, k, H, elem_bytes, M, disp):
    """Expert-grouped view of a dispatch output (see ep_oracle_group_by_expert): returns a dict
    with packed_x [W][E][W*M][H], packed_count [W][E], packed_src_info [W][E][W*M],
    layout_range [W][E][W] (int64) and packed_row [W][E][W*M]."""
    lib = _load()
    rows = W * M
    dt = np.uint8 if elem_bytes == 1 else np.uint16
    out = {"packed_x": np.zeros((W, E, rows, H), dtype=dt),
           "packed_count": np.zeros((W, E), dtype=np.int32),
           "packed_src_info": np.full((W, E, rows), -1, dtype=np.int32),
           "layout_range": np.zeros((W, E, W), dtype=np.int64),
           "packed_row": np.full((W, E, rows), -1, dtype=np.int32)}
    st = lib.ep_oracle_group_by_expert(
        W, E, k, H, elem_bytes, M, _ptr(np.ascontiguousarray(disp["recv_x"])),
        _ptr(np.ascontiguousarray(disp["recv_idx"])), _ptr(np.ascontiguousarray(disp["recv_count"])),
        _ptr(np.ascontiguousarray(disp["src_pos"])), _ptr(out["packed_x"]), _ptr(out["packed_count"]),
        _ptr(out["packed_src_info"]), _ptr(out["layout_range"]), _ptr(out["packed_row"]))
    if st != 0:
        raise ValueError("ep_oracle_group_by_expert: invalid arguments")
    return out


def ungroup_by_expert(W, E, H, out_fp16, M, recv_count, grouped, packed_y):
    """Per received row, the ascending-expert FP32 sum of its local experts' outputs, rounded
    to BF16 / FP16: returns out [W][W*M][H] (uint16 bits; rows past recv_count are zero)."""
    lib = _load()
    out = np.zeros((W, W * M, H), dtype=np.uint16)
    st = lib.ep_oracle_ungroup_by_expert(
        W, E, H, 1 if out_fp16 else 0, M, _ptr(np.ascontiguousarray(recv_count, dtype=np.int32)),
        _ptr(grouped["packed_count"]), _ptr(grouped["packed_row"]),
        _ptr(np.ascontiguousarray(packed_y).view(np.uint16)), _ptr(out))
    if st != 0:
        raise ValueError("ep_oracle_ungroup_by_expert: invalid arguments")
    return out


def e2m1_from_f32(v):
    return int(_load().ep_oracle_e2m1_from_f32(float(v)))


def f32_from_e2m1(c):
    return float(_load().ep_oracle_f32_from_e2m1(int(c)))


def f32_from_e8m0(c):
    return float(_load().ep_oracle_f32_from_e8m0(int(c)))


def quantize_mxfp4(x_bf16):
    """MX FP4 quantisation of BF16 rows [..., H] (H a multiple of 32): returns (q uint8
    [..., H/2] packed nibbles, scales uint8 [..., H/32] e8m0 codes)."""
    x = np.ascontiguousarray(x_bf16).view(np.uint16)
    H = x.shape[-1]
    rows = x.size // H
    q = np.empty(x.shape[:-1] + (H // 2,), dtype=np.uint8)
    sc = np.empty(x.shape[:-1] + (H // 32,), dtype=np.uint8)
    if _load().ep_oracle_quantize_mxfp4(rows, H, _ptr(x), _ptr(q), _ptr(sc)) != 0:
        raise ValueError("quantize_mxfp4: hidden must be a positive multiple of 32")
    return q, sc


def combine_fp4(W, k, H, M, n_tok, slot_of, q, scales, w_in=None):
    """Combine over the MX FP4 wire (see ep_oracle_combine_fp4): returns (out, out_w)."""
    lib = _load()
    n_tok = np.ascontiguousarray(n_tok, dtype=np.int32)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    q = np.ascontiguousarray(q).view(np.uint8)
    scales = np.ascontiguousarray(scales).view(np.uint8)
    out = np.zeros((W, M, H), dtype=np.uint16)
    out_w = np.zeros((W, M, k), dtype=np.float32) if w_in is not None else None
    w_in = None if w_in is None else np.ascontiguousarray(w_in, dtype=np.float32)
    if lib.ep_oracle_combine_fp4(W, k, H, M, _ptr(n_tok), _ptr(slot_of), _ptr(q), _ptr(scales),
                                 _ptr(w_in), _ptr(out), _ptr(out_w)) != 0:
        raise ValueError("ep_oracle_combine_fp4: invalid arguments")
    return out, out_w


def bf16_from_f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    o = np.empty(a.shape, dtype=np.uint16)
    _load().ep_oracle_bf16_from_f32_array(_ptr(a), _ptr(o), a.size)
    return o


def f16_from_f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    o = np.empty(a.shape, dtype=np.uint16)
    _load().ep_oracle_f16_from_f32_array(_ptr(a), _ptr(o), a.size)
    return o


def f32_from_f16(a):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    o = np.empty(a.shape, dtype=np.float32)
    _load().ep_oracle_f32_from_f16_array(_ptr(a), _ptr(o), a.size)
    return o


def e4m3_from_f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    o = np.empty(a.shape, dtype=np.uint8)
    _load().ep_oracle_e4m3_from_f32_array(_ptr(a), _ptr(o), a.size)
    return o


def f32_from_e4m3(a):
    a = np.ascontiguousarray(a, dtype=np.uint8)
    o = np.empty(a.shape, dtype=np.float32)
    _load().ep_oracle_f32_from_e4m3_array(_ptr(a), _ptr(o), a.size)
    return o


def quantize_e4m3_blockwise(x_bf16):
    """Block-wise FP8 quantisation of BF16 rows [..., H] (H a multiple of 128): returns
    (q uint8 [..., H], scales float32 [..., H/128]); see ep_oracle_quantize_e4m3_blockwise."""
    x = np.ascontiguousarray(x_bf16).view(np.uint16)
    H = x.shape[-1]
    rows = x.size // H
    q = np.empty(x.shape, dtype=np.uint8)
    sc = np.empty(x.shape[:-1] + (H // 128,), dtype=np.float32)
    if _load().ep_oracle_quantize_e4m3_blockwise(rows, H, _ptr(x), _ptr(q), _ptr(sc)) != 0:
        raise ValueError("quantize_e4m3_blockwise: hidden must be a positive multiple of 128")
    return q, sc


def dispatch_quantized(wl):
    """Quantising dispatch: every source row is quantised block-wise to FP8 once, then the
    FP8 rows and their scales are dispatched like any FP8 payload."""
    q, sc = quantize_e4m3_blockwise(wl.x)
    return dispatch(wl.W, wl.E, wl.k, wl.H, 1, wl.H // 128, wl.M, q, wl.weights, sc,
                    wl.indices, wl.n_tok)


def dispatch_quantized_mxfp4(wl):
    """Dispatch of BF16 rows quantised to MX FP4 (the pages' FP4 dispatch): every source row is
    quantised once (quantize_mxfp4), then its H/2 code bytes are dispatched as the payload and
    its H/32 scale bytes as the scale row (H/128 four-byte words, copied bit for bit).
    Returns the dispatch dict plus "q" / "sc", the quantised source rows."""
    q, sc = quantize_mxfp4(wl.x)
    sc_words = np.ascontiguousarray(sc).view(np.float32)           # [W][M][H/128] byte carriers
    disp = dispatch(wl.W, wl.E, wl.k, wl.H // 2, 1, wl.H // 128, wl.M, q, wl.weights, sc_words,
                    wl.indices, wl.n_tok)
    disp["q"], disp["sc"] = q, sc
    return disp


def run_workload(wl, expert_out_fn=None):
    """Oracle dispatch -> harness expert -> oracle combine for one workload.

    ``expert_out_fn(wl, disp)`` returns the expert output rows ``[W][W*M][H]`` (16-bit bits);
    None means the identity expert on a 16-bit payload (expert output = receive rows).
    """
    disp = dispatch(wl.W, wl.E, wl.k, wl.H, wl.elem_bytes, wl.sd, wl.M, wl.x, wl.weights,
                    wl.scales, wl.indices, wl.n_tok)
    eo = disp["recv_x"] if expert_out_fn is None else expert_out_fn(wl, disp)
    out, out_w = combine(wl.W, wl.k, wl.H, wl.combine_dtype == "fp16", wl.M, wl.n_tok,
                         disp["slot_of"], eo, disp["recv_w"])
    return disp, eo, out, out_w

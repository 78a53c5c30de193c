"""GB300-native MoE expert-parallel Dispatch / Combine.

A thin Python binding over ``libep.so`` (C ABI in ``include/ep.h``).  Every step of dispatch and
combine runs in the library's CUDA kernels; this module only marshals arguments.  PyTorch
supplies device memory, the current stream and zero-copy tensor views of the plan's buffers.
If ``libep.so`` is missing the binding raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep.so")

EP_BF16, EP_FP16, EP_FP8_E4M3, EP_BF16_TO_FP8_E4M3, EP_BF16_TO_MXFP4 = 0, 1, 2, 3, 4
# "bf16_fp8": BF16 input that dispatch quantises to FP8 e4m3 + one FP32 scale per 128 elements;
# "bf16_mxfp4": BF16 input that dispatch quantises to MX FP4 (e2m1 codes, one e8m0 scale per 32)
DTYPE_CODES = {"bf16": EP_BF16, "fp16": EP_FP16, "fp8": EP_FP8_E4M3, "bf16_fp8": EP_BF16_TO_FP8_E4M3,
               "bf16_mxfp4": EP_BF16_TO_MXFP4}
EP_OK, EP_ERR_ARG, EP_ERR_ALLOC, EP_ERR_CUDA, EP_ERR_STATE = 0, -1, -2, -3, -4
EP_ERR_CAPACITY, EP_ERR_INDEX, EP_ERR_DEVICE_TIMEOUT, EP_ERR_DEVICE_BOUNDS = -5, -6, -7, -8
# phases of ep_probe_read, in the order of its (earliest start, latest end) pairs
PROBE_PHASES = ("route", "scatter", "combine", "quantise", "wire_combine", "group_scan", "group_copy",
                "ungroup")
VARIANTS = {"auto": 0, "whole_row": 1, "tiled_512": 2, "tiled_1024": 3}

# every entry point include/ep.h declares
EXPORTS = ("ep_plan_create", "ep_plan_destroy", "ep_plan_set_variant", "ep_plan_device_bytes",
           "ep_dispatch", "ep_dispatch_route", "ep_dispatch_scatter", "ep_combine", "ep_reset",
           "ep_status", "ep_strerror", "ep_last_error", "ep_route_noalloc",
           "ep_quantize_received", "ep_combine_fp8", "ep_group_by_expert", "ep_ungroup_by_expert",
           "ep_dispatch_grouped", "ep_quantize_received_fp4", "ep_combine_fp4", "ep_probe_read")


class EpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class DispatchOut(ctypes.Structure):
    _fields_ = [("recv_x", ctypes.c_void_p), ("recv_idx", ctypes.c_void_p),
                ("recv_w", ctypes.c_void_p), ("recv_scales", ctypes.c_void_p),
                ("recv_count", ctypes.c_void_p), ("src_token_pos", ctypes.c_void_p),
                ("rows_per_rank", ctypes.c_int64), ("epoch", ctypes.c_uint64)]


_lib = None


def load_library(path: Optional[str] = None):
    """Load libep.so (built by ``build.build()``); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libep.so not found at {p}: build it with "
                           "combine_ep_dispatch_02_gb300.build.build()")
    lib = ctypes.CDLL(p)
    V, I, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    sig = {
        "ep_plan_create": (I, [ctypes.POINTER(V), I, I, I, I, I, I, I]),
        "ep_plan_destroy": (I, [V]),
        "ep_plan_set_variant": (I, [V, I]),
        "ep_plan_device_bytes": (SZ, [I, I, I, I, I, I, I]),
        "ep_dispatch": (I, [V, V, V, V, V, V, V, ctypes.POINTER(DispatchOut)]),
        "ep_dispatch_route": (I, [V, V, V, V, ctypes.POINTER(DispatchOut)]),
        "ep_dispatch_scatter": (I, [V, V, V, V, V, V]),
        "ep_combine": (I, [V, V, V, V, V, U64, V]),
        "ep_reset": (I, [V, V]),
        "ep_status": (I, [V, ctypes.POINTER(I)]),
        "ep_strerror": (ctypes.c_char_p, [I]),
        "ep_last_error": (ctypes.c_char_p, []),
        "ep_route_noalloc": (I, [I, I, I, I, V, V, V, V, V, V, V]),
        "ep_quantize_received": (I, [V, V, V, V, U64, V]),
        "ep_combine_fp8": (I, [V, V, V, V, V, V, U64, V]),
        "ep_group_by_expert": (I, [V, V, V, V, V, U64, V]),
        "ep_ungroup_by_expert": (I, [V, V, V, U64, V]),
        "ep_dispatch_grouped": (I, [V, V, V, V, V, V, V, V, V, V, V, ctypes.POINTER(DispatchOut)]),
        "ep_quantize_received_fp4": (I, [V, V, V, V, U64, V]),
        "ep_combine_fp4": (I, [V, V, V, V, V, V, U64, V]),
        "ep_probe_read": (I, [V, ctypes.POINTER(ctypes.c_uint64), I]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != EP_OK:
        lib = load_library()
        raise EpError(rc, f"{lib.ep_strerror(rc).decode()}: {lib.ep_last_error().decode()}")


def plan_device_bytes(W, experts_per_rank, topk, hidden, dtype, scale_dim, max_tok_per_rank) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype
    return load_library().ep_plan_device_bytes(W, experts_per_rank, topk, hidden, code, scale_dim,
                                               max_tok_per_rank)


def route_noalloc(W: int, experts_per_rank: int, topk: int, max_tok_per_rank: int,
                  indices: torch.Tensor, n_tok: Sequence[int], src_token_pos: torch.Tensor,
                  recv_count: torch.Tensor, fwd_map: torch.Tensor, device_status: torch.Tensor,
                  stream=None) -> None:
    """``ep_route_noalloc``: the routing step into caller-owned tensors, with no device
    allocation by the library (see include/ep.h).  Shapes: indices [W][M][k] int32,
    src_token_pos [W][W*M], recv_count [W], fwd_map [W][M][min(W,k)], device_status [1], all
    int32 on indices' device, where the call runs."""
    arr = np.ascontiguousarray(np.asarray(n_tok, dtype=np.int32).reshape(W))
    M, F = max_tok_per_rank, min(W, topk)
    dev = indices.device
    if dev.type != "cuda":
        raise EpError(EP_ERR_ARG, f"indices is on {dev}, not a CUDA device")
    with torch.cuda.device(dev):
        _check(load_library().ep_route_noalloc(
            W, experts_per_rank, topk, max_tok_per_rank, _buf(indices, 4 * W * M * topk, "indices", 4, dev),
            arr.ctypes.data_as(ctypes.c_void_p),
            _buf(src_token_pos, 4 * W * W * M, "src_token_pos", 4, dev),
            _buf(recv_count, 4 * W, "recv_count", 4, dev), _buf(fwd_map, 4 * W * M * F, "fwd_map", 4, dev),
            _buf(device_status, 4, "device_status", 4, dev), _stream(stream)))


class _DevPtr:
    """Zero-copy __cuda_array_interface__ view of plan-owned device memory."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 2, "strides": None}


def _view(ptr, shape, typestr, device):
    if not ptr:
        return None
    return torch.as_tensor(_DevPtr(ptr, shape, typestr), device=device)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("arguments must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _buf(t: Optional[torch.Tensor], nbytes: int, what: str, itemsize: Optional[int] = None,
         device: Optional[torch.device] = None):
    """_ptr after the host checks the C ABI leaves to its caller: the tensor holds at least the
    nbytes the call reads or writes, has itemsize-byte elements where the ABI fixes the type, and
    lives on the plan's device.  A failed check raises EpError(EP_ERR_ARG) before any launch."""
    if t is None:
        return None
    p = _ptr(t)
    if device is not None and t.device != device:
        raise EpError(EP_ERR_ARG, f"{what} is on {t.device}, the plan on {device}")
    if itemsize is not None and t.element_size() != itemsize:
        raise EpError(EP_ERR_ARG, f"{what} has {t.element_size()}-byte elements, the call takes {itemsize}")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise EpError(EP_ERR_ARG, f"{what} holds {have} bytes, the call needs {nbytes}")
    return p


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclasses.dataclass
class Dispatched:
    """Views of the plan's receive buffers after one dispatch (valid until the next dispatch or
    reset of the plan; the plan must outlive them)."""
    recv_x: torch.Tensor          # [W][W*M][H] payload dtype ([W][W*M][H/2] uint8 for MX FP4)
    recv_idx: torch.Tensor        # [W][W*M][k] int32
    recv_w: Optional[torch.Tensor]       # [W][W*M][k] float32
    recv_scales: Optional[torch.Tensor]  # [W][W*M][sd] float32 ([W][W*M][H/32] uint8 for MX FP4)
    recv_count: torch.Tensor      # [W] int32
    src_token_pos: torch.Tensor   # [W][W*M] int32
    epoch: int


class Plan:
    """One expert-parallel Dispatch/Combine problem shape; owns the receive buffers.

    ``Plan(W, experts_per_rank, topk, hidden, dtype, scale_dim, max_tok_per_rank)`` maps to
    ``ep_plan_create``; dtype is "bf16", "fp16", "fp8" (e4m3 with caller scales), "bf16_fp8"
    (BF16 input quantised by dispatch to e4m3 with one FP32 scale per 128 elements) or
    "bf16_mxfp4" (BF16 input quantised by dispatch to MX FP4: receive rows of H/2 packed e2m1
    bytes and H/32 e8m0 scale bytes)."""

    def __init__(self, W: int, experts_per_rank: int, topk: int, hidden: int, dtype: str = "bf16",
                 scale_dim: int = 0, max_tok_per_rank: int = 1, device=None):
        self._lib = load_library()
        self.W, self.E, self.k, self.H = W, experts_per_rank, topk, hidden
        self.dtype, self.sd, self.M = dtype, scale_dim, max_tok_per_rank
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        self._h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(self._lib.ep_plan_create(ctypes.byref(self._h), W, experts_per_rank, topk, hidden,
                                            DTYPE_CODES[dtype], scale_dim, max_tok_per_rank))
        self.rows = W * max_tok_per_rank
        if dtype in ("bf16_fp8", "bf16_mxfp4"):
            self.sd = hidden // 128
        self.payload_torch_dtype = {"bf16": torch.bfloat16, "fp16": torch.float16,
                                    "fp8": torch.float8_e4m3fn, "bf16_fp8": torch.float8_e4m3fn,
                                    "bf16_mxfp4": torch.uint8}[dtype]
        # elements of payload_torch_dtype per received row (MX FP4 packs two codes per byte)
        self.row_elems = hidden // 2 if dtype == "bf16_mxfp4" else hidden
        self.combine_torch_dtype = torch.float16 if dtype == "fp16" else torch.bfloat16
        self._in_bytes = 1 if dtype == "fp8" else 2            # bytes of one caller x element
        self._row_bytes = {"bf16": 2 * hidden, "fp16": 2 * hidden, "fp8": hidden, "bf16_fp8": hidden,
                           "bf16_mxfp4": hidden // 2}[dtype]   # bytes of one received payload row

    # -- lifetime
    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            _check(self._lib.ep_plan_destroy(self._h))
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def set_variant(self, variant: str):
        _check(self._lib.ep_plan_set_variant(self._h, VARIANTS[variant]))

    # -- calls
    def _arg(self, t, nbytes, what, itemsize=None):
        return _buf(t, nbytes, what, itemsize, self.device)

    def _source_args(self, x, weights, scales, indices):
        """Pointers of dispatch's [W][M][...] inputs, checked against the plan's shape."""
        W, M, k, H = self.W, self.M, self.k, self.H
        sd = 0 if self.dtype in ("bf16_fp8", "bf16_mxfp4") else self.sd
        return (self._arg(x, W * M * H * self._in_bytes, "x", self._in_bytes),
                self._arg(weights, 4 * W * M * k, "weights", 4),
                self._arg(scales, 4 * W * M * sd, "scales", 4),
                self._arg(indices, 4 * W * M * k, "indices", 4))

    def _combine_outs(self, weights, out, out_w):
        """Pointers of a combine's received weights [W][W*M][k] and outputs [W][M][H], [W][M][k]."""
        W, M, k = self.W, self.M, self.k
        return (self._arg(weights, 4 * W * self.rows * k, "weights", 4),
                self._arg(out, 2 * W * M * self.H, "out", 2), self._arg(out_w, 4 * W * M * k, "out_w", 4))

    def _n_tok(self, n_tok: Sequence[int]):
        arr = np.ascontiguousarray(np.asarray(n_tok, dtype=np.int32).reshape(self.W))
        return arr, arr.ctypes.data_as(ctypes.c_void_p)

    def _wrap(self, o: DispatchOut) -> Dispatched:
        W, R, k, H, sd, dev = self.W, self.rows, self.k, self.H, self.sd, self.device
        if self.dtype in ("fp8", "bf16_fp8"):
            rx = _view(o.recv_x, (W, R, H), "|u1", dev).view(torch.float8_e4m3fn)
        elif self.dtype == "bf16_mxfp4":
            rx = _view(o.recv_x, (W, R, H // 2), "|u1", dev)
        else:
            rx = _view(o.recv_x, (W, R, H), "<i2", dev).view(self.payload_torch_dtype)
        if not sd:
            rs = None
        elif self.dtype == "bf16_mxfp4":                 # H/32 e8m0 scale codes per row
            rs = _view(o.recv_scales, (W, R, H // 32), "|u1", dev)
        else:
            rs = _view(o.recv_scales, (W, R, sd), "<f4", dev)
        return Dispatched(recv_x=rx, recv_idx=_view(o.recv_idx, (W, R, k), "<i4", dev),
                          recv_w=_view(o.recv_w, (W, R, k), "<f4", dev),
                          recv_scales=rs,
                          recv_count=_view(o.recv_count, (W,), "<i4", dev),
                          src_token_pos=_view(o.src_token_pos, (W, R), "<i4", dev),
                          epoch=int(o.epoch))

    def dispatch(self, x: torch.Tensor, weights: Optional[torch.Tensor], scales: Optional[torch.Tensor],
                 indices: torch.Tensor, n_tok: Sequence[int], stream=None) -> Dispatched:
        """x [W][M][H], weights [W][M][k] fp32 or None, scales [W][M][sd] fp32 or None,
        indices [W][M][k] int32, n_tok: W host ints."""
        arr, nt = self._n_tok(n_tok)
        o = DispatchOut()
        _check(self._lib.ep_dispatch(self._h, *self._source_args(x, weights, scales, indices),
                                     nt, _stream(stream), ctypes.byref(o)))
        return self._wrap(o)

    def dispatch_route(self, indices: torch.Tensor, n_tok: Sequence[int], stream=None) -> Dispatched:
        arr, nt = self._n_tok(n_tok)
        o = DispatchOut()
        idx = self._arg(indices, 4 * self.W * self.M * self.k, "indices", 4)
        _check(self._lib.ep_dispatch_route(self._h, idx, nt, _stream(stream), ctypes.byref(o)))
        return self._wrap(o)

    def dispatch_scatter(self, x, weights, scales, indices, stream=None):
        _check(self._lib.ep_dispatch_scatter(self._h, *self._source_args(x, weights, scales, indices),
                                             _stream(stream)))

    def combine(self, expert_out: torch.Tensor, weights: Optional[torch.Tensor], epoch: int,
                out: Optional[torch.Tensor] = None, out_w: Optional[torch.Tensor] = None,
                want_weights: bool = True, stream=None):
        """expert_out [W][W*M][H] (BF16, or FP16 for FP16 plans); returns (out [W][M][H],
        out_w [W][M][k] or None)."""
        if out is None:
            out = torch.zeros((self.W, self.M, self.H), dtype=self.combine_torch_dtype,
                              device=self.device)
        if out_w is None and weights is not None and want_weights:
            out_w = torch.zeros((self.W, self.M, self.k), dtype=torch.float32, device=self.device)
        _check(self._lib.ep_combine(self._h, self._arg(expert_out, 2 * self.W * self.rows * self.H, "expert_out", 2),
                                    *self._combine_outs(weights, out, out_w), ctypes.c_uint64(epoch),
                                    _stream(stream)))
        return out, out_w

    def quantize_received(self, expert_out: torch.Tensor, epoch: int, q: Optional[torch.Tensor] = None,
                          scales: Optional[torch.Tensor] = None, stream=None):
        """Quantise the received BF16 expert rows block-wise to e4m3 codes + FP32 scales (the
        FP8 combine wire); returns (q [W][W*M][H] float8_e4m3fn, scales [W][W*M][H/128])."""
        if q is None:
            q = torch.empty((self.W, self.rows, self.H), dtype=torch.uint8, device=self.device)
        if scales is None:
            scales = torch.empty((self.W, self.rows, self.H // 128), dtype=torch.float32, device=self.device)
        n = self.W * self.rows * self.H
        _check(self._lib.ep_quantize_received(self._h, self._arg(expert_out, 2 * n, "expert_out", 2),
                                              self._arg(q, n, "q", 1), self._arg(scales, 4 * (n // 128), "scales", 4),
                                              ctypes.c_uint64(epoch), _stream(stream)))
        return q.view(torch.float8_e4m3fn), scales

    def combine_fp8(self, q: torch.Tensor, scales: torch.Tensor, weights: Optional[torch.Tensor],
                    epoch: int, out: Optional[torch.Tensor] = None, out_w: Optional[torch.Tensor] = None,
                    want_weights: bool = True, stream=None):
        """Combine over the FP8 wire; returns (out [W][M][H] BF16, out_w or None)."""
        if out is None:
            out = torch.zeros((self.W, self.M, self.H), dtype=torch.bfloat16, device=self.device)
        if out_w is None and weights is not None and want_weights:
            out_w = torch.zeros((self.W, self.M, self.k), dtype=torch.float32, device=self.device)
        n = self.W * self.rows * self.H
        _check(self._lib.ep_combine_fp8(self._h, self._arg(q, n, "q", 1), self._arg(scales, 4 * (n // 128), "scales", 4),
                                        *self._combine_outs(weights, out, out_w), ctypes.c_uint64(epoch),
                                        _stream(stream)))
        return out, out_w

    def quantize_received_fp4(self, expert_out: torch.Tensor, epoch: int, q: Optional[torch.Tensor] = None,
                              scales: Optional[torch.Tensor] = None, stream=None):
        """Quantise the received BF16 expert rows to the MX FP4 wire; returns (q [W][W*M][H/2]
        uint8 packed e2m1 pairs, scales [W][W*M][H/32] uint8 e8m0 codes)."""
        if q is None:
            q = torch.empty((self.W, self.rows, self.H // 2), dtype=torch.uint8, device=self.device)
        if scales is None:
            scales = torch.empty((self.W, self.rows, self.H // 32), dtype=torch.uint8, device=self.device)
        n = self.W * self.rows * self.H
        _check(self._lib.ep_quantize_received_fp4(self._h, self._arg(expert_out, 2 * n, "expert_out", 2),
                                                  self._arg(q, n // 2, "q", 1), self._arg(scales, n // 32, "scales", 1),
                                                  ctypes.c_uint64(epoch), _stream(stream)))
        return q, scales

    def combine_fp4(self, q: torch.Tensor, scales: torch.Tensor, weights: Optional[torch.Tensor],
                    epoch: int, out: Optional[torch.Tensor] = None, out_w: Optional[torch.Tensor] = None,
                    want_weights: bool = True, stream=None):
        """Combine over the MX FP4 wire; returns (out [W][M][H] BF16, out_w or None)."""
        if out is None:
            out = torch.zeros((self.W, self.M, self.H), dtype=torch.bfloat16, device=self.device)
        if out_w is None and weights is not None and want_weights:
            out_w = torch.zeros((self.W, self.M, self.k), dtype=torch.float32, device=self.device)
        n = self.W * self.rows * self.H
        _check(self._lib.ep_combine_fp4(self._h, self._arg(q, n // 2, "q", 1), self._arg(scales, n // 32, "scales", 1),
                                        *self._combine_outs(weights, out, out_w), ctypes.c_uint64(epoch),
                                        _stream(stream)))
        return out, out_w

    def group_by_expert(self, epoch: int, packed_x: Optional[torch.Tensor] = None, stream=None):
        """Expert-grouped view of the live dispatch: returns (packed_x [W][E][W*M][H],
        packed_count [W][E], packed_src_info [W][E][W*M], layout_range [W][E][W] int64)."""
        W, E, R, H = self.W, self.E, self.rows, self.H
        if packed_x is None:
            packed_x = torch.empty((W, E, R, self.row_elems), dtype=self.payload_torch_dtype,
                                   device=self.device)
        count = torch.empty((W, E), dtype=torch.int32, device=self.device)
        src_info = torch.empty((W, E, R), dtype=torch.int32, device=self.device)
        layout = torch.empty((W, E, W), dtype=torch.int64, device=self.device)
        _check(self._lib.ep_group_by_expert(self._h, self._arg(packed_x, W * E * R * self._row_bytes, "packed_x"),
                                            _ptr(count), _ptr(src_info), _ptr(layout), ctypes.c_uint64(epoch),
                                            _stream(stream)))
        return packed_x, count, src_info, layout

    def dispatch_grouped(self, x: torch.Tensor, weights: Optional[torch.Tensor],
                         scales: Optional[torch.Tensor], indices: torch.Tensor, n_tok: Sequence[int],
                         packed_x: Optional[torch.Tensor] = None, stream=None):
        """Dispatch straight into the grouped view: returns (Dispatched, packed_x, packed_count,
        packed_src_info, layout_range); the Dispatched views' recv_x holds unspecified data."""
        W, E, R, H = self.W, self.E, self.rows, self.H
        if packed_x is None:
            packed_x = torch.empty((W, E, R, self.row_elems), dtype=self.payload_torch_dtype,
                                   device=self.device)
        count = torch.empty((W, E), dtype=torch.int32, device=self.device)
        src_info = torch.empty((W, E, R), dtype=torch.int32, device=self.device)
        layout = torch.empty((W, E, W), dtype=torch.int64, device=self.device)
        arr, nt = self._n_tok(n_tok)
        o = DispatchOut()
        _check(self._lib.ep_dispatch_grouped(self._h, *self._source_args(x, weights, scales, indices), nt,
                                             self._arg(packed_x, W * E * R * self._row_bytes, "packed_x"),
                                             _ptr(count), _ptr(src_info), _ptr(layout), _stream(stream),
                                             ctypes.byref(o)))
        return self._wrap(o), packed_x, count, src_info, layout

    def ungroup_by_expert(self, packed_y: torch.Tensor, epoch: int, out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
        """Per received row, the ascending-expert sum of its local experts' outputs: the combine
        input [W][W*M][H] (BF16, FP16 for FP16 plans)."""
        if out is None:
            out = torch.empty((self.W, self.rows, self.H), dtype=self.combine_torch_dtype, device=self.device)
        n = self.W * self.rows * self.H
        _check(self._lib.ep_ungroup_by_expert(self._h, self._arg(packed_y, 2 * self.E * n, "packed_y", 2),
                                              self._arg(out, 2 * n, "out", 2), ctypes.c_uint64(epoch),
                                              _stream(stream)))
        return out

    def reset(self, stream=None):
        _check(self._lib.ep_reset(self._h, _stream(stream)))

    def probe(self) -> dict:
        """``ep_probe_read``: per phase, (earliest start, latest end) in ns of the launches since
        the last read, or None for a phase that did not run; raises EpError(EP_ERR_STATE) unless
        the library was built with EP_PROBE."""
        buf = (ctypes.c_uint64 * (2 * len(PROBE_PHASES)))()
        _check(self._lib.ep_probe_read(self._h, buf, len(buf)))
        return {name: (None if buf[2 * i] == 2 ** 64 - 1 else (int(buf[2 * i]), int(buf[2 * i + 1])))
                for i, name in enumerate(PROBE_PHASES)}

    def status(self) -> int:
        v = ctypes.c_int(0)
        _check(self._lib.ep_status(self._h, ctypes.byref(v)))
        return v.value

"""C ABI checks that need no GPU: the library loads, exports every declared entry point, sizes
its device buffers as documented, and rejects invalid shapes and calls on the host."""
import ctypes
import os
import re

import pytest

import combine_ep_dispatch_02_gb300 as ep
from combine_ep_dispatch_02_gb300 import build as epbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    epbuild.build()
    return ep.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ep.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) == set(ep.EXPORTS), declared
    for name in declared:
        assert hasattr(lib, name), name


def _align(v):
    return (v + 255) // 256 * 256


def _scan_bytes(W, E, M):
    # grouping scan counts [W*E][chunks][W] int32, for three or more 1024-row chunks of capacity,
    # up to 64 MiB
    chunks = -(-(W * M) // 1024)
    b = W * E * chunks * W * 4
    return b if chunks >= 3 and b <= 64 << 20 else 0


def _route_group_bytes(W, E, M):
    # the routing kernel's expert columns (fused grouped dispatch): lookback words [tiles][W*E] u64
    # and list prefixes [W+1][W*E] int32, for up to 1024 experts and 64 MiB of words
    tiles = -(-(W * M) // 256)
    if W * E > 1024 or tiles * W * E * 8 > 64 << 20:
        return 0, 0
    return tiles * W * E * 8, (W + 1) * W * E * 4


def _layout_bytes(W, E, k, H, eb, sd, M):
    rows = W * M
    F = min(W, k)
    tiles = -(-rows // 256)
    parts = [W * rows * H * eb, W * rows * k * 4, W * rows * k * 4, W * rows * sd * 4, W * rows * 4,
             rows * F * 4, _scan_bytes(W, E, M), W * 4, W * rows * k * 4, tiles * W * 8,
             *_route_group_bytes(W, E, M), 8, 4]
    return sum(_align(p) for p in parts)


def test_device_bytes_golden(lib):
    # DeepSeek-V3 shape: recv rows 8 * 32768 * 14336 B, index / weight rows 8 MiB each,
    # src_pos and forward map 1 MiB each, grouping scan counts 256 lists * 32 chunks * 8 sources
    # * 4 B, the expert-slot map 8 MiB, 128 tiles * 8 scan words, the expert columns' 128 tiles *
    # 256 words and 9 * 256 list prefixes, the control words
    assert lib.ep_plan_device_bytes(8, 32, 8, 7168, ep.EP_BF16, 0, 4096) == 3785630464 + 262144 + 9216
    # FP8 with 56 scales per row
    assert lib.ep_plan_device_bytes(8, 96, 6, 7168, ep.EP_FP8_E4M3, 56, 4096) == \
        _layout_bytes(8, 96, 6, 7168, 1, 56, 4096)
    for shape in [(2, 4, 2, 256, 0, 0, 64), (4, 64, 64, 2048, 1, 0, 512), (1, 1, 1, 8, 0, 0, 1),
                  (32, 8, 64, 16, 2, 3, 100), (2, 1 << 20, 2, 16, 0, 0, 4096),
                  # grouping scan counts: 2048 rows are two chunks (none), 2049 three; at W=2 and
                  # three chunks, 1398101 experts per rank need 67108848 B (kept) and one more
                  # 67108896 B, past 64 MiB (none)
                  (1, 1, 1, 8, 0, 0, 2048), (1, 1, 1, 8, 0, 0, 2049),
                  (2, 1398101, 2, 8, 0, 0, 1536), (2, 1398102, 2, 8, 0, 0, 1536)]:
        W, E, k, H, dt, sd, M = shape
        eb = 1 if dt == ep.EP_FP8_E4M3 else 2
        assert lib.ep_plan_device_bytes(*shape) == _layout_bytes(W, E, k, H, eb, sd, M), shape
    assert _scan_bytes(1, 1, 2048) == 0 and _scan_bytes(1, 1, 2049) == 12
    assert _scan_bytes(2, 1398101, 1536) == 67108848 and _scan_bytes(2, 1398102, 1536) == 0
    big = lib.ep_plan_device_bytes(2, 1398101, 2, 8, 0, 0, 1536)
    assert big - lib.ep_plan_device_bytes(2, 1398102, 2, 8, 0, 0, 1536) == _align(67108848)


@pytest.mark.parametrize("shape,why", [
    ((0, 4, 2, 256, 0, 0, 64), "W"), ((33, 4, 2, 256, 0, 0, 64), "W"),
    ((2, 0, 2, 256, 0, 0, 64), "experts_per_rank"), ((2, 4, 0, 256, 0, 0, 64), "topk"),
    ((2, 4, 65, 256, 0, 0, 64), "topk"), ((2, 4, 2, 4, 0, 0, 64), "hidden"),
    ((2, 4, 2, 8, 2, 0, 64), "hidden"), ((2, 4, 2, 256, 5, 0, 64), "dtype"),
    ((2, 4, 2, 96, 4, 0, 64), "128"), ((2, 4, 2, 256, 4, 1, 64), "scale_dim"),
    ((2, 4, 2, 256, 0, -1, 64), "scale_dim"), ((2, 4, 2, 256, 0, 0, 0), "max_tok"),
    ((32, 4, 2, 256, 0, 0, 1 << 21), "2^31"),
    # the combine's 16-bit expert outputs [W][W*M][H] reach 64 GiB (W*W*M*H = 2^35)
    ((32, 8, 8, 8192, 0, 0, 4096), "64 GiB"), ((32, 8, 8, 4096, 0, 0, 8192), "64 GiB"),
    ((32, 8, 8, 4096, 1, 0, 8192), "64 GiB"), ((32, 8, 8, 8192, 2, 0, 4096), "64 GiB"),
    ((32, 8, 8, 8192, 3, 0, 4096), "64 GiB"), ((32, 8, 8, 8192, 4, 0, 4096), "64 GiB"),
    ((16, 8, 8, 7168, 0, 0, 18725), "64 GiB"),
])
def test_invalid_shapes_rejected_on_host(lib, shape, why):
    h = ctypes.c_void_p(123)
    rc = lib.ep_plan_create(ctypes.byref(h), *shape)
    assert rc == ep.EP_ERR_ARG
    assert h.value is None
    assert why in lib.ep_last_error().decode()
    assert lib.ep_plan_device_bytes(*shape) == 0


def test_route_group_words_boundary(lib):
    """The routing kernel's expert columns are allocated for up to 1024 experts in all and 64 MiB
    of lookback words, else the grouped dispatch keeps the separate grouping scan."""
    for W, E, M in [(8, 128, 64), (8, 129, 64), (32, 32, 8192), (4, 256, 524288), (4, 256, 524289),
                    (2, 512, 1 << 20), (2, 512, (1 << 20) + 1)]:
        assert lib.ep_plan_device_bytes(W, E, 4, 8, ep.EP_BF16, 0, M) == _layout_bytes(W, E, 4, 8, 2, 0, M)
    assert _route_group_bytes(8, 128, 64)[0] > 0 and _route_group_bytes(8, 129, 64) == (0, 0)
    # 64 MiB of words exactly (8192 tiles * 1024 experts * 8 B) is kept, one tile more is not
    assert _route_group_bytes(4, 256, 524288)[0] == 64 << 20
    assert _route_group_bytes(4, 256, 524289) == (0, 0)


def test_combine_offset_limit_boundary(lib):
    """The largest accepted shapes sit one unit below W*W*M*H = 2^35 (64 GiB of 16-bit expert
    outputs): one vector of hidden, or one token per rank, less than the rejected shapes."""
    for dt in (ep.EP_BF16, ep.EP_FP16, ep.EP_FP8_E4M3, ep.EP_BF16_TO_FP8_E4M3, ep.EP_BF16_TO_MXFP4):
        H = 8192 - 128                       # W*W*M*H = 2^35 - 2^29 at W=32, M=4096
        assert lib.ep_plan_device_bytes(32, 8, 8, H, dt, 0, 4096) > 0, dt
        assert lib.ep_plan_device_bytes(32, 8, 8, 8192, dt, 0, 4096) == 0, dt
    # W=16, H=7168: 2^35 / (256 * 7168) = 18724.57 tokens per rank
    assert lib.ep_plan_device_bytes(16, 8, 8, 7168, ep.EP_BF16, 0, 18724) > 0
    assert lib.ep_plan_device_bytes(16, 8, 8, 7168, ep.EP_BF16, 0, 18725) == 0
    assert 16 * 16 * 18724 * 7168 < 2 ** 35 <= 16 * 16 * 18725 * 7168


def test_null_plan_calls_fail_cleanly(lib):
    o = ep.DispatchOut()
    n = (ctypes.c_int32 * 2)(1, 1)
    assert lib.ep_dispatch(None, None, None, None, None, n, None, ctypes.byref(o)) == ep.EP_ERR_ARG
    assert lib.ep_combine(None, None, None, None, None, 0, None) == ep.EP_ERR_ARG
    assert lib.ep_reset(None, None) == ep.EP_ERR_ARG
    assert lib.ep_plan_set_variant(None, 0) == ep.EP_ERR_ARG
    st = ctypes.c_int(0)
    assert lib.ep_status(None, ctypes.byref(st)) == ep.EP_ERR_ARG
    assert lib.ep_plan_destroy(None) == ep.EP_OK
    for code in range(-8, 1):
        assert lib.ep_strerror(code) and lib.ep_strerror(code) != b"unknown status"
    buf = (ctypes.c_uint64 * 16)()
    assert lib.ep_probe_read(None, buf, 16) == ep.EP_ERR_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        ep.load_library(str(tmp_path / "missing" / "libep.so"))


def test_quantising_dtype_sizes_and_shape_checks(lib):
    # BF16 input quantised to FP8 on the wire: 1-byte payload rows and hidden/128 scales per row
    for sd in (0, 56):
        assert lib.ep_plan_device_bytes(8, 32, 8, 7168, ep.EP_BF16_TO_FP8_E4M3, sd, 4096) == \
            _layout_bytes(8, 32, 8, 7168, 1, 56, 4096)
    h = ctypes.c_void_p()
    assert lib.ep_plan_create(ctypes.byref(h), 8, 32, 8, 7168 + 64, ep.EP_BF16_TO_FP8_E4M3, 0, 16) == ep.EP_ERR_ARG
    assert "128" in lib.ep_last_error().decode()
    assert lib.ep_plan_create(ctypes.byref(h), 8, 32, 8, 7168, ep.EP_BF16_TO_FP8_E4M3, 3, 16) == ep.EP_ERR_ARG
    assert "scale" in lib.ep_last_error().decode()


def test_mxfp4_dtype_sizes(lib):
    # BF16 input quantised to MX FP4: H/2 code bytes per received row, and H/32 scale bytes
    # carried as H/128 four-byte words
    for sd in (0, 56):
        assert lib.ep_plan_device_bytes(8, 32, 8, 7168, ep.EP_BF16_TO_MXFP4, sd, 4096) == \
            _layout_bytes(8, 32, 8, 3584, 1, 56, 4096)
    # DeepSeek-V3 shape: 8 * 32768 rows of 3584 code bytes, scale rows of 224 bytes, and the
    # grouping scan's 256 * 32 * 8 counts
    assert lib.ep_plan_device_bytes(8, 32, 8, 7168, ep.EP_BF16_TO_MXFP4, 0, 4096) == \
        8 * 32768 * 3584 + 3 * (8 << 20) + 8 * 32768 * 224 + 2 * (1 << 20) + 256 * 32 * 8 * 4 + \
        256 + 8192 + 128 * 256 * 8 + 9 * 256 * 4 + 256 + 256

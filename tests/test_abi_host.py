"""Host-side checks of the C ABI (no GPU needed).

The library builds for sm_103a, loads, exports every function declared in
include/adacomp.h, sizes buffers as the header states, and rejects bad arguments
synchronously before any CUDA call is made.
"""
import ctypes
import os
import re

import pytest

import residual_gradient_compression_gb300 as ac
from residual_gradient_compression_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    ac.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "adacomp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(adacomp_\w+)\s*\(", text))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert {"adacomp_init_layer", "adacomp_compress", "adacomp_decode_accumulate", "adacomp_free"} <= names
    for name in names:
        assert hasattr(ac.lib(), name), name


def test_sizes_follow_the_message_format():
    for n, L, w in ((10, 4, 1), (400_000, 500, 2), (1003, 63, 1), (1003, 64, 2), (1, 1, 1)):
        h = ac.adacomp_init_layer(n, L, ac.F32)
        B = -(-n // L)
        assert h.max_msg_bytes == [8 + 2 * B + w * n]
        assert h.compress_ws_bytes > 0 and h.decode_ws_bytes_per_learner > 0
        ac.adacomp_free(h)


def _tiles(n, L):
    """Tiles of a single layer: eight warp slices of floor(509 / L) bins for
    16 <= L <= 509, else about 4096 elements of whole bins (at least one bin)."""
    B = -(-n // L)
    bpt = 8 * (509 // L) if 16 <= L <= 509 else max(1, 4096 // L)
    bpt = min(bpt, 1024, B)
    return -(-B // bpt)


def _pad16(b):
    return -(-b // 16) * 16


@pytest.mark.parametrize("n,L", [(1_000_000, 500), (777_777, 50), (65_537, 16), (10, 509)])
def test_sliced_workspace_layout(n, L):
    """16 <= L_T <= 509: control block, one 2112-byte layer block, then per tile a
    u64 code offset and a u32 code total (each array padded to 16 bytes) and two
    512-byte masks; the deferred fix-up needs no more."""
    T = _tiles(n, L)
    expect = 64 + 2112 + _pad16(8 * T) + _pad16(4 * T) + 1024 * T
    h = ac.adacomp_init_layer(n, L, ac.F32)
    assert h.compress_ws_bytes == expect
    assert ac.adacomp_set_lazy_fixup(h, True) == expect
    # per learner: a u64 code offset and a u32 code sum per tile (the sums padded to 16 B)
    assert h.decode_ws_bytes(3) == ac.DECODE_WS_FIXED + 3 * (8 * T + _pad16(4 * T))
    ac.adacomp_free(h)


@pytest.mark.parametrize("n,L", [(77_777, 7), (100_003, 4), (8191, 8192), (250_000, 8190)])
def test_lookback_workspace_layout(n, L):
    """L_T < 16 and L_T > 8189: control block, layer block, a u64 descriptor and a
    u64 code offset per tile; the deferred fix-up adds a 512-byte mask per tile."""
    T = _tiles(n, L)
    h = ac.adacomp_init_layer(n, L, ac.F32)
    assert h.compress_ws_bytes == 64 + 2112 + 16 * T
    assert ac.adacomp_set_lazy_fixup(h, True) == 64 + 2112 + 16 * T + 512 * T
    ac.adacomp_free(h)


@pytest.mark.parametrize("n,L", [(1_000_000, 5000), (300_007, 510), (40_000, 4096), (4095, 4097), (10, 8189)])
def test_block_sliced_workspace_layout(n, L):
    """510 <= L_T <= 8189: the sliced layout with sixteen 512-slot slices per tile,
    i.e. two 1024-byte masks per tile; the deferred fix-up needs no more."""
    T = _tiles(n, L)
    expect = 64 + 2112 + _pad16(8 * T) + _pad16(4 * T) + 2048 * T
    h = ac.adacomp_init_layer(n, L, ac.F32)
    assert h.compress_ws_bytes == expect
    assert ac.adacomp_set_lazy_fixup(h, True) == expect
    ac.adacomp_free(h)


def test_group_workspace_takes_the_lookback_layout_when_mixed():
    """A group is sliced only when every layer is; one block per layer."""
    ns, Ls = [40_000, 30_000], [50, 500]
    T = sum(_tiles(n, L) for n, L in zip(ns, Ls))
    h = ac.adacomp_init_group(ns, Ls, [ac.F32, ac.F32])
    assert h.compress_ws_bytes == 64 + 2 * 2112 + _pad16(8 * T) + _pad16(4 * T) + 1024 * T
    ns2, Ls2 = ns + [20_000], Ls + [5000]
    T2 = T + _tiles(20_000, 5000)
    h2 = ac.adacomp_init_group(ns2, Ls2, [ac.F32] * 3)
    assert h2.compress_ws_bytes == 64 + 3 * 2112 + 16 * T2
    # all bins of 510 .. 8189: the block-sliced layout
    ns3, Ls3 = [20_000, 50_000], [5000, 600]
    T3 = sum(_tiles(n, L) for n, L in zip(ns3, Ls3))
    h3 = ac.adacomp_init_group(ns3, Ls3, [ac.F32] * 2)
    assert h3.compress_ws_bytes == 64 + 2 * 2112 + _pad16(8 * T3) + _pad16(4 * T3) + 2048 * T3


@pytest.mark.parametrize("n,L,dt", [(0, 4, 0), (-5, 4, 0), (10, 0, 0), (10, 8193, 0), (10, 4, 2)])
def test_init_rejects_bad_arguments(n, L, dt):
    with pytest.raises(ac.AdacompError) as e:
        ac.adacomp_init_layer(n, L, dt)
    assert e.value.status == ac.ERR_INVALID_ARG


def test_group_limits():
    with pytest.raises(ac.AdacompError):
        ac.adacomp_init_group([], [], [])
    with pytest.raises(ac.AdacompError):
        ac.adacomp_init_group([10] * 129, [4] * 129, [0] * 129)
    h = ac.adacomp_init_group([10, 20, 30], [4, 64, 500], [0, 1, 0])
    assert len(h.max_msg_bytes) == 3
    ac.adacomp_free(h)


def _raw_compress(h, residue, dw, msg, cap, ws, wsb):
    return ac.lib().adacomp_compress(h.ptr if h else None, residue, dw, msg, cap, ws, wsb, None)


def test_compress_argument_checks_return_before_launch():
    h = ac.adacomp_init_layer(1000, 50, ac.F32)
    cap, wsb = h.max_msg_bytes[0], h.compress_ws_bytes
    A = 1 << 20  # a 16-byte-aligned stand-in address; no call below reaches the GPU
    assert _raw_compress(None, A, A, A, cap, A, wsb) == ac.ERR_INVALID_ARG
    assert _raw_compress(h, None, A, A, cap, A, wsb) == ac.ERR_INVALID_ARG
    assert _raw_compress(h, A + 4, A, A, cap, A, wsb) == ac.ERR_ALIGNMENT
    assert _raw_compress(h, A, A + 2, A, cap, A, wsb) == ac.ERR_ALIGNMENT
    assert _raw_compress(h, A, A, A + 8, cap, A, wsb) == ac.ERR_ALIGNMENT
    assert _raw_compress(h, A, A, A, cap - 1, A, wsb) == ac.ERR_CAPACITY
    assert _raw_compress(h, A, A, A, cap, A, wsb - 1) == ac.ERR_WORKSPACE
    assert _raw_compress(h, A, A, A, cap, None, wsb) == ac.ERR_INVALID_ARG
    ac.adacomp_free(h)


def test_decode_argument_checks_return_before_launch():
    h = ac.adacomp_init_layer(1000, 50, ac.F32)
    A = 1 << 20
    L = ac.lib()
    one = (ctypes.c_void_p * 1)(A)
    ln = (ctypes.c_uint64 * 1)(h.max_msg_bytes[0])
    wsb = h.decode_ws_bytes(1)
    assert L.adacomp_decode_accumulate(h.ptr, one, ln, 0, A, A, wsb, None) == ac.ERR_INVALID_ARG
    assert L.adacomp_decode_accumulate(h.ptr, one, ln, 257, A, A, 1 << 30, None) == ac.ERR_INVALID_ARG
    assert L.adacomp_decode_accumulate(h.ptr, one, ln, 1, A + 4, A, wsb, None) == ac.ERR_ALIGNMENT
    bad = (ctypes.c_void_p * 1)(A + 2)
    assert L.adacomp_decode_accumulate(h.ptr, bad, ln, 1, A, A, wsb, None) == ac.ERR_ALIGNMENT
    assert L.adacomp_decode_accumulate(h.ptr, one, ln, 1, A, A, wsb - 1, None) == ac.ERR_WORKSPACE
    null = (ctypes.c_void_p * 1)(None)
    assert L.adacomp_decode_accumulate(h.ptr, null, ln, 1, A, A, wsb, None) == ac.ERR_INVALID_ARG
    assert L.adacomp_decode_accumulate(h.ptr, one, None, 1, A, A, wsb, None) == ac.ERR_INVALID_ARG
    ac.adacomp_free(h)


def test_status_strings_and_free_null():
    for s in range(8):
        assert ac.adacomp_status_string(s) not in ("", "unknown status")
    ac.lib().adacomp_free(None)
    assert ac.lib().adacomp_set_timeout_ns(None, 5) == ac.ERR_INVALID_ARG


def test_static_workspace_size_constant_matches_the_header():
    text = open(os.path.join(ROOT, "include", "adacomp.h")).read()
    m = re.search(r"#define ADACOMP_STATIC_WS_BYTES \(\(size_t\)1 << (\d+)\)", text)
    assert m and (1 << int(m.group(1))) == ac.STATIC_WS_BYTES

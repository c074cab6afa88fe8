"""AdaComp CPU oracle — TEST INFRASTRUCTURE ONLY.

ctypes binding over ``adacomp_oracle.c``: a plain single-threaded C restatement of
AdaComp's per-layer compressor (Algorithm 2 as restated in the "AdaComp (Adaptive
Residual Gradient Compression)" entry, Claims > Mechanism
#r629-local-bin-soft-threshold-and-mean-gmax-quantization) and of the K-learner
decoder. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the CUDA product path never does, and the two
share no code.

All arrays are numpy; residue is updated in place like the CUDA entry point does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adacomp_oracle.c")
_LIB = os.path.join(_HERE, "libadacomp_oracle.so")
_lib = None

OK, ERR_ARG, ERR_CAPACITY, ERR_BAD_MESSAGE = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc: -O2, no FMA contraction, no fast-math."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a test's copy)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, i32, u64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        vp = ctypes.c_void_p
        lib.adacomp_oracle_max_msg_bytes.argtypes = [i64, i32]
        lib.adacomp_oracle_max_msg_bytes.restype = i64
        lib.adacomp_oracle_exact_sum_f32.argtypes = [vp, i64]
        lib.adacomp_oracle_exact_sum_f32.restype = ctypes.c_double
        lib.adacomp_oracle_compress.argtypes = [i64, i32, ctypes.c_int, vp, vp, vp, u64,
                                                ctypes.POINTER(u64), vp, vp, vp, ctypes.c_int, ctypes.c_int]
        lib.adacomp_oracle_compress.restype = ctypes.c_int
        lib.adacomp_oracle_decode_accumulate.argtypes = [i64, i32, vp, vp, i32, vp, vp]
        lib.adacomp_oracle_decode_accumulate.restype = ctypes.c_int
        f32 = ctypes.c_float
        lib.adacomp_oracle_decode_sgd.argtypes = [i64, i32, vp, vp, i32, vp, vp, f32, f32, f32]
        lib.adacomp_oracle_decode_adam.argtypes = [i64, i32, vp, vp, i32, vp, vp, vp] + [f32] * 7
        lib.adacomp_oracle_decode_adam.restype = ctypes.c_int
        lib.adacomp_oracle_decode_sgd.restype = ctypes.c_int
        self.lib = lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = Oracle(_LIB).lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_msg_bytes(n: int, bin_len: int, lib=None) -> int:
    return int((lib or _load()).adacomp_oracle_max_msg_bytes(n, bin_len))


def exact_sum_f32(x: np.ndarray, lib=None) -> float:
    """Exact sum of non-negative fp32 values, correctly rounded to fp64."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float((lib or _load()).adacomp_oracle_exact_sum_f32(_ptr(x), x.size))


class CompressResult:
    __slots__ = ("msg", "s", "gmax", "sel")

    def __init__(self, msg, s, gmax, sel):
        self.msg, self.s, self.gmax, self.sel = msg, s, gmax, sel


def compress(residue: np.ndarray, dw: np.ndarray, bin_len: int,
             literal_zero_select: bool = False, lib=None, local_selection: bool = False) -> CompressResult:
    """One step for one layer. ``residue`` (fp32, contiguous) is updated in place.

    ``dw`` is fp32, or uint16 holding bf16 bit patterns. Returns the message bytes,
    s, g_max per bin and the 0/1 selection mask. ``local_selection`` selects the hard
    Local Selection rule (abs(G) >= g_max, no soft-threshold probe) instead of AdaComp's.
    """
    lib = lib or _load()
    assert residue.dtype == np.float32 and residue.flags.c_contiguous
    if dw.dtype == np.float32:
        bf16 = 0
    elif dw.dtype == np.uint16:
        bf16 = 1
    else:
        raise TypeError("dw must be float32 or uint16 (bf16 bits)")
    dw = np.ascontiguousarray(dw)
    n = residue.size
    assert dw.size == n and n >= 1
    cap = max_msg_bytes(n, bin_len, lib)
    if cap < 0:
        raise ValueError("bad n / bin_len")
    nb = -(-n // bin_len)
    msg = np.zeros(cap, dtype=np.uint8)
    gmax = np.zeros(nb, dtype=np.float32)
    sel = np.zeros(n, dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    mlen = ctypes.c_uint64(0)
    rc = lib.adacomp_oracle_compress(n, bin_len, bf16, _ptr(residue), _ptr(dw), _ptr(msg), cap,
                                     ctypes.byref(mlen), _ptr(s), _ptr(gmax), _ptr(sel),
                                     int(literal_zero_select), int(local_selection))
    if rc != OK:
        raise RuntimeError(f"oracle compress failed: {rc}")
    return CompressResult(msg[: mlen.value].copy(), s[0], gmax, sel.astype(bool))


def _msg_arrays(msgs, lens):
    bufs = [np.ascontiguousarray(m, dtype=np.uint8) for m in msgs]
    if lens is None:
        lens = [b.size for b in bufs]
    if len(lens) != len(bufs):
        raise ValueError("one length per message")
    ptrs = (ctypes.c_void_p * len(bufs))(*[b.ctypes.data for b in bufs])
    ln = (ctypes.c_uint64 * len(bufs))(*[int(x) for x in lens])
    return bufs, ptrs, ln


def decode_accumulate(n: int, bin_len: int, msgs, dense: np.ndarray, lib=None, lens=None, bad=None) -> int:
    """Adds every well-formed message's sign*s_k into ``dense`` (fp32, in place), k in order.

    ``lens``: each message's length in bytes (default: the length of its array).
    Returns the oracle status (0 = OK, 3 = at least one message was rejected and
    added nothing). ``bad``: an optional uint8 array of K entries set to 1 for each
    rejected message.
    """
    lib = lib or _load()
    assert dense.dtype == np.float32 and dense.flags.c_contiguous and dense.size == n
    bufs, ptrs, ln = _msg_arrays(msgs, lens)
    bad_ptr = None
    if bad is not None:
        assert bad.dtype == np.uint8 and bad.size == len(bufs)
        bad_ptr = _ptr(bad)
    return int(lib.adacomp_oracle_decode_accumulate(n, bin_len, ptrs, ln, len(bufs), _ptr(dense), bad_ptr))


def decode_sgd(n: int, bin_len: int, msgs, w: np.ndarray, v: np.ndarray, lr: float, mu: float,
               scale: float = 1.0, lib=None, lens=None) -> int:
    """Decodes the messages into a zero gradient and applies one momentum-SGD step to
    ``w`` and ``v`` (fp32, in place); a rejected message adds nothing. Returns the
    oracle status."""
    lib = lib or _load()
    assert w.dtype == np.float32 and v.dtype == np.float32 and w.size == n and v.size == n
    bufs, ptrs, ln = _msg_arrays(msgs, lens)
    return lib.adacomp_oracle_decode_sgd(n, bin_len, ptrs, ln, len(bufs), _ptr(w), _ptr(v), lr, mu, scale)


def decode_adam(n: int, bin_len: int, msgs, w: np.ndarray, m: np.ndarray, v: np.ndarray, lr: float,
                beta1: float, beta2: float, eps: float, bc1: float, bc2: float, scale: float = 1.0, lib=None,
                lens=None) -> int:
    """Decodes the messages into a zero gradient and applies one Adam step to ``w``,
    ``m`` and ``v`` (fp32, in place); bc1 and bc2 are the step's bias corrections
    1 - beta1^t and 1 - beta2^t. A rejected message adds nothing. Returns the
    oracle status."""
    lib = lib or _load()
    for a in (w, m, v):
        assert a.dtype == np.float32 and a.size == n and a.flags.c_contiguous
    bufs, ptrs, ln = _msg_arrays(msgs, lens)
    return lib.adacomp_oracle_decode_adam(n, bin_len, ptrs, ln, len(bufs), _ptr(w), _ptr(m), _ptr(v), lr, beta1,
                                          beta2, eps, bc1, bc2, scale)

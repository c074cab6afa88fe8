"""GB300-native AdaComp: per-layer adaptive residual gradient compression.

A thin ctypes binding over the C ABI of ``libadacomp.so`` (``include/adacomp.h``).
Every function keeps the C name and only marshals arguments: torch tensors become
device pointers, the stream defaults to torch's current stream, and a non-OK status
raises :class:`AdacompError`. All computation runs in the library's CUDA kernels;
there is no CPU fallback, and using the binding without the built library raises.

Method: "AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
#r629-local-bin-soft-threshold-and-mean-gmax-quantization.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

from .build import lib_path as _lib_path

# libadacomp.so, or libadacomp_debug.so when ADACOMP_DEBUG_CHECKS=1 (a debug build)
_LIB_PATH = _lib_path()

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT, \
    ERR_BAD_MESSAGE = range(8)
F32, BF16 = 0, 1
RULE_ADACOMP, RULE_LOCAL_SELECTION = 0, 1
MAX_GROUP = 128
MAX_LEARNERS = 256
DECODE_WS_FIXED = 10240
STATIC_WS_BYTES = 1 << 20  # ADACOMP_STATIC_WS_BYTES: the largest workspace adacomp_compress_static_ws holds

_lib = None


class AdacompError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {adacomp_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded libadacomp.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it with "
                              "residual_gradient_compression_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        vp, sz, i32, i64, u64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                 ctypes.c_int64, ctypes.c_uint64)
        P = ctypes.POINTER
        L.adacomp_init_layer.argtypes = [P(vp), i64, i32, ctypes.c_int, P(sz), P(sz), P(sz)]
        L.adacomp_init_group.argtypes = [P(vp), i32, P(i64), P(i32), P(i32), P(sz), P(sz), P(sz)]
        L.adacomp_compress.argtypes = [vp, vp, vp, vp, sz, vp, sz, vp]
        L.adacomp_compress_group.argtypes = [vp, P(vp), P(vp), P(vp), P(sz), vp, sz, vp]
        L.adacomp_decode_accumulate.argtypes = [vp, P(vp), P(u64), i32, vp, vp, sz, vp]
        L.adacomp_decode_accumulate_group.argtypes = [vp, P(vp), P(u64), i32, P(vp), vp, sz, vp]
        L.adacomp_query.argtypes = [vp, vp, i32, vp, P(u64), P(ctypes.c_float), P(i32)]
        L.adacomp_decode_status.argtypes = [vp, vp, vp, P(i32)]
        L.adacomp_set_timeout_ns.argtypes = [vp, u64]
        L.adacomp_set_timing_events.argtypes = [vp, vp, vp, vp]
        L.adacomp_set_fault_injection.argtypes = [vp, ctypes.c_uint32]
        L.adacomp_set_lazy_fixup.argtypes = [vp, i32, P(sz)]
        L.adacomp_set_selection_rule.argtypes = [vp, i32]
        f32 = ctypes.c_float
        L.adacomp_decode_sgd.argtypes = [vp, P(vp), P(u64), i32, vp, vp, f32, f32, f32, vp, sz, vp]
        L.adacomp_decode_sgd_group.argtypes = [vp, P(vp), P(u64), i32, P(vp), P(vp), f32, f32, f32, vp, sz, vp]
        L.adacomp_decode_adam.argtypes = [vp, P(vp), P(u64), i32, vp, vp, vp] + [f32] * 7 + [vp, sz, vp]
        L.adacomp_decode_adam_group.argtypes = [vp, P(vp), P(u64), i32, P(vp), P(vp), P(vp)] + [f32] * 7 + [vp, sz, vp]
        L.adacomp_materialize.argtypes = [vp, vp, vp, sz, vp]
        L.adacomp_materialize_group.argtypes = [vp, P(vp), vp, sz, vp]
        L.adacomp_free.argtypes = [vp]
        L.adacomp_free.restype = None
        L.adacomp_status_string.argtypes = [ctypes.c_int]
        L.adacomp_status_string.restype = ctypes.c_char_p
        for name in ("adacomp_init_layer", "adacomp_init_group", "adacomp_compress",
                     "adacomp_compress_group", "adacomp_decode_accumulate",
                     "adacomp_decode_accumulate_group", "adacomp_query", "adacomp_decode_status",
                     "adacomp_set_timeout_ns", "adacomp_set_timing_events",
                     "adacomp_set_fault_injection", "adacomp_set_lazy_fixup", "adacomp_set_selection_rule",
                     "adacomp_materialize", "adacomp_decode_sgd", "adacomp_decode_sgd_group",
                     "adacomp_decode_adam", "adacomp_decode_adam_group", "adacomp_materialize_group"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != OK:
        raise AdacompError(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t) -> int:
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensors passed to the library must be contiguous")
        return t.data_ptr()
    return int(t)


class Handle:
    """Host-side handle for one layer or a group of layers (no device memory)."""

    def __init__(self, ptr, num_layers, ns, bin_lens, dtypes, max_msg_bytes, ws, dws):
        self.ptr = ptr
        self.num_layers = num_layers
        self.n = list(ns)
        self.bin_len = list(bin_lens)
        self.dtype = list(dtypes)
        self.max_msg_bytes = list(max_msg_bytes)
        self.compress_ws_bytes = ws
        self.decode_ws_bytes_per_learner = dws

    def decode_ws_bytes(self, K: int) -> int:
        return DECODE_WS_FIXED + K * self.decode_ws_bytes_per_learner

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.adacomp_free(self.ptr)
            self.ptr = None


def adacomp_init_layer(n: int, bin_len: int, dw_dtype: int = F32) -> Handle:
    h = ctypes.c_void_p()
    mm, ws, dws = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().adacomp_init_layer(ctypes.byref(h), n, bin_len, dw_dtype, ctypes.byref(mm),
                                    ctypes.byref(ws), ctypes.byref(dws)), "adacomp_init_layer")
    return Handle(h.value, 1, [n], [bin_len], [dw_dtype], [mm.value], ws.value, dws.value)


def adacomp_init_group(ns: Sequence[int], bin_lens: Sequence[int], dw_dtypes: Sequence[int]) -> Handle:
    L = len(ns)
    h = ctypes.c_void_p()
    mm = (ctypes.c_size_t * L)()
    ws, dws = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().adacomp_init_group(ctypes.byref(h), L, (ctypes.c_int64 * L)(*ns),
                                    (ctypes.c_int32 * L)(*bin_lens), (ctypes.c_int32 * L)(*dw_dtypes),
                                    mm, ctypes.byref(ws), ctypes.byref(dws)), "adacomp_init_group")
    return Handle(h.value, L, ns, bin_lens, dw_dtypes, list(mm), ws.value, dws.value)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def adacomp_compress(h: Handle, residue, dW, msg, ws, stream=None):
    _check(lib().adacomp_compress(h.ptr, _ptr(residue), _ptr(dW), _ptr(msg), _nbytes(msg),
                                  _ptr(ws), _nbytes(ws), _stream(stream)), "adacomp_compress")


def adacomp_compress_group(h: Handle, residues, dWs, msgs, ws, stream=None):
    L = h.num_layers
    VP = ctypes.c_void_p * L
    _check(lib().adacomp_compress_group(
        h.ptr, VP(*[_ptr(r) for r in residues]), VP(*[_ptr(d) for d in dWs]),
        VP(*[_ptr(m) for m in msgs]), (ctypes.c_size_t * L)(*[_nbytes(m) for m in msgs]),
        _ptr(ws), _nbytes(ws), _stream(stream)), "adacomp_compress_group")


def _lengths(msg_bytes, count: int):
    lens = [int(b) for b in msg_bytes]
    if len(lens) != count:
        raise ValueError(f"expected {count} message lengths, got {len(lens)}")
    return (ctypes.c_uint64 * count)(*lens)


def adacomp_decode_accumulate(h: Handle, msgs, msg_bytes, dense, ws, stream=None):
    """msgs: K device buffers; msg_bytes: the K message lengths in bytes."""
    K = len(msgs)
    arr = (ctypes.c_void_p * K)(*[_ptr(m) for m in msgs])
    _check(lib().adacomp_decode_accumulate(h.ptr, arr, _lengths(msg_bytes, K), K, _ptr(dense), _ptr(ws),
                                           _nbytes(ws), _stream(stream)), "adacomp_decode_accumulate")


def adacomp_decode_accumulate_group(h: Handle, msgs, msg_bytes, denses, ws, stream=None):
    """msgs[l][k]: learner k's message for layer l, msg_bytes[l][k] its length;
    denses[l]: layer l's dense buffer."""
    L = h.num_layers
    K = len(msgs[0])
    flat = [_ptr(m) for per_layer in msgs for m in per_layer]
    lens = _lengths([b for per_layer in msg_bytes for b in per_layer], L * K)
    _check(lib().adacomp_decode_accumulate_group(
        h.ptr, (ctypes.c_void_p * (L * K))(*flat), lens, K, (ctypes.c_void_p * L)(*[_ptr(d) for d in denses]),
        _ptr(ws), _nbytes(ws), _stream(stream)), "adacomp_decode_accumulate_group")


def adacomp_query(h: Handle, ws, layer: int = 0, stream=None):
    """(message bytes, s, device status) of the last compress that used ws."""
    mb, s, st = ctypes.c_uint64(), ctypes.c_float(), ctypes.c_int32()
    _check(lib().adacomp_query(h.ptr, _ptr(ws), layer, _stream(stream), ctypes.byref(mb),
                               ctypes.byref(s), ctypes.byref(st)), "adacomp_query")
    return mb.value, s.value, st.value


def adacomp_decode_status(h: Handle, ws, stream=None) -> int:
    st = ctypes.c_int32()
    _check(lib().adacomp_decode_status(h.ptr, _ptr(ws), _stream(stream), ctypes.byref(st)),
           "adacomp_decode_status")
    return st.value


def adacomp_set_timeout_ns(h: Handle, ns: int):
    _check(lib().adacomp_set_timeout_ns(h.ptr, ns), "adacomp_set_timeout_ns")


def adacomp_set_timing_events(h: Handle, before=None, mid=None, after=None):
    """Record caller-owned torch.cuda.Event objects around the two compress kernels."""
    def raw(ev):
        return None if ev is None else ctypes.c_void_p(ev.cuda_event)
    _check(lib().adacomp_set_timing_events(h.ptr, raw(before), raw(mid), raw(after)),
           "adacomp_set_timing_events")


def adacomp_set_fault_injection(h: Handle, skip_tile: int = 0xFFFFFFFF):
    """Test hook: the given tile never publishes, so its successors time out."""
    _check(lib().adacomp_set_fault_injection(h.ptr, skip_tile), "adacomp_set_fault_injection")


def adacomp_decode_sgd(h: Handle, msgs, msg_bytes, weights, momentum, lr: float, mu: float, ws,
                       grad_scale: float = 1.0, stream=None):
    K = len(msgs)
    arr = (ctypes.c_void_p * K)(*[_ptr(m) for m in msgs])
    _check(lib().adacomp_decode_sgd(h.ptr, arr, _lengths(msg_bytes, K), K, _ptr(weights), _ptr(momentum), lr, mu,
                                    grad_scale, _ptr(ws), _nbytes(ws), _stream(stream)), "adacomp_decode_sgd")


def adacomp_decode_sgd_group(h: Handle, msgs, msg_bytes, weights, momentum, lr: float, mu: float, ws,
                             grad_scale: float = 1.0, stream=None):
    """msgs, msg_bytes: per layer a list of K messages and their lengths (layer-major, as
    adacomp_decode_accumulate_group)."""
    L = h.num_layers
    K = len(msgs[0])
    arr = (ctypes.c_void_p * (L * K))(*[_ptr(m) for layer in msgs for m in layer])
    lens = _lengths([b for layer in msg_bytes for b in layer], L * K)
    VP = ctypes.c_void_p * L
    _check(lib().adacomp_decode_sgd_group(h.ptr, arr, lens, K, VP(*[_ptr(w) for w in weights]),
                                          VP(*[_ptr(v) for v in momentum]), lr, mu, grad_scale, _ptr(ws),
                                          _nbytes(ws), _stream(stream)), "adacomp_decode_sgd_group")


def adacomp_decode_adam(h: Handle, msgs, msg_bytes, weights, m, v, lr: float, beta1: float, beta2: float,
                        eps: float, bias_correction1: float, bias_correction2: float, ws, grad_scale: float = 1.0,
                        stream=None):
    K = len(msgs)
    arr = (ctypes.c_void_p * K)(*[_ptr(x) for x in msgs])
    _check(lib().adacomp_decode_adam(h.ptr, arr, _lengths(msg_bytes, K), K, _ptr(weights), _ptr(m), _ptr(v), lr,
                                     beta1, beta2, eps, bias_correction1, bias_correction2, grad_scale, _ptr(ws),
                                     _nbytes(ws), _stream(stream)), "adacomp_decode_adam")


def adacomp_decode_adam_group(h: Handle, msgs, msg_bytes, weights, m, v, lr: float, beta1: float, beta2: float,
                              eps: float, bias_correction1: float, bias_correction2: float, ws,
                              grad_scale: float = 1.0, stream=None):
    """msgs, msg_bytes: per layer a list of K messages and their lengths (layer-major);
    weights, m, v: one buffer per layer."""
    L = h.num_layers
    K = len(msgs[0])
    arr = (ctypes.c_void_p * (L * K))(*[_ptr(x) for layer in msgs for x in layer])
    lens = _lengths([b for layer in msg_bytes for b in layer], L * K)
    VP = ctypes.c_void_p * L
    _check(lib().adacomp_decode_adam_group(h.ptr, arr, lens, K, VP(*[_ptr(x) for x in weights]),
                                           VP(*[_ptr(x) for x in m]), VP(*[_ptr(x) for x in v]), lr, beta1, beta2,
                                           eps, bias_correction1, bias_correction2, grad_scale, _ptr(ws),
                                           _nbytes(ws), _stream(stream)), "adacomp_decode_adam_group")


def adacomp_set_selection_rule(h: Handle, rule: int):
    """RULE_ADACOMP (default) or RULE_LOCAL_SELECTION (abs(G) >= g_max, no probe)."""
    _check(lib().adacomp_set_selection_rule(h.ptr, rule), "adacomp_set_selection_rule")


def adacomp_set_lazy_fixup(h: Handle, enable: bool = True) -> int:
    """Defers the residue fix-up to the next compress call; returns (and records on
    the handle) the compress workspace size the mode needs."""
    ws = ctypes.c_size_t()
    _check(lib().adacomp_set_lazy_fixup(h.ptr, int(bool(enable)), ctypes.byref(ws)), "adacomp_set_lazy_fixup")
    h.compress_ws_bytes = ws.value
    return ws.value


def adacomp_materialize(h: Handle, residue, ws, stream=None):
    _check(lib().adacomp_materialize(h.ptr, _ptr(residue), _ptr(ws), _nbytes(ws), _stream(stream)),
           "adacomp_materialize")


def adacomp_materialize_group(h: Handle, residues, ws, stream=None):
    VP = ctypes.c_void_p * h.num_layers
    _check(lib().adacomp_materialize_group(h.ptr, VP(*[_ptr(r) for r in residues]), _ptr(ws), _nbytes(ws),
                                           _stream(stream)), "adacomp_materialize_group")


def adacomp_free(h: Handle):
    if h.ptr:
        lib().adacomp_free(h.ptr)
        h.ptr = None


def adacomp_status_string(status: int) -> str:
    return lib().adacomp_status_string(status).decode()

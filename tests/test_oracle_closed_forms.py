"""Pins the oracle to closed forms that the method reduces to in special cases.

Source of every formula: "AdaComp (Adaptive Residual Gradient Compression)",
Claims > Mechanism #r629-local-bin-soft-threshold-and-mean-gmax-quantization.

* First step (residue = 0): G = dW and H = 2 dW exactly, so an element is sent iff
  dW != 0 and 2|dW| >= g_max, with g_max the bin's largest |dW|.
* L_T = 1 on exactly representable inputs: g_max = |G|, so an element is sent iff
  G != 0 and |G + dW| >= |G|, i.e. G*dW >= 0 or |dW| >= 2|G|; s = mean |G|.
* One bin (L_T >= N): s = max |G|.
* Decoding one learner's message into zeros gives G_q = sign(G) * s on the sent
  elements and 0 elsewhere.

g_max uses numpy's max, the mean of g_max uses math.fsum (the correctly rounded sum),
and the message is assembled from numpy's nonzero: none of it calls the oracle.
"""
import math

import numpy as np
import pytest

import oracle


def _bins(n, L):
    return -(-n // L)


def _gmax(absval, L):
    n = absval.size
    nb = _bins(n, L)
    pad = np.zeros(nb * L, dtype=np.float64)
    pad[:n] = absval
    return pad.reshape(nb, L).max(axis=1)


def _message(s, sel, neg, n, L):
    nb = _bins(n, L)
    j = np.nonzero(sel)[0]
    b = j // L
    counts = np.bincount(b, minlength=nb).astype("<u2")
    codes = ((j - b * L) << 1) | neg[j].astype(np.int64)
    codes = codes.astype("<u1" if L < 64 else "<u2")
    head = np.array([np.float32(s)], "<f4").tobytes() + np.array([nb], "<u4").tobytes()
    return head + counts.tobytes() + codes.tobytes()


def _bf16_bits_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


CASES = [(1, 1), (7, 3), (100, 1), (1000, 50), (1003, 50), (4096, 63), (4097, 64),
         (5000, 500), (12345, 500), (20000, 5000), (999, 1000)]


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("n,L", CASES)
def test_first_step_closed_form(n, L, bf16):
    rng = np.random.default_rng(n * 7 + L)
    dw32 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    dw32[rng.random(n) < 0.05] = 0.0
    if bf16:
        dw_in = (dw32.view(np.uint32) >> 16).astype(np.uint16)
        dw = _bf16_bits_to_f32(dw_in)
    else:
        dw_in = dw32
        dw = dw32
    residue = np.zeros(n, np.float32)
    r = oracle.compress(residue, dw_in, L)

    a = np.abs(dw.astype(np.float64))
    gm = _gmax(a, L)
    sel = (dw != 0) & (2.0 * a >= np.repeat(gm, L)[:n])
    s = np.float32(math.fsum(gm) / _bins(n, L))
    exp_res = dw.copy()
    exp_res[sel] = np.where(dw[sel] > 0, dw[sel] - s, dw[sel] + s)

    assert np.float32(r.s).view(np.uint32) == s.view(np.uint32)
    assert np.array_equal(r.sel, sel)
    assert np.array_equal(residue.view(np.uint32), exp_res.view(np.uint32))
    assert r.msg.tobytes() == _message(s, sel, dw < 0, n, L)


def test_unit_bins_closed_form():
    rng = np.random.default_rng(11)
    n = 4000
    # multiples of 1/8 in [-2, 2]: every sum below is exact in fp32
    residue = (rng.integers(-16, 17, n) / 8).astype(np.float32)
    dw = (rng.integers(-16, 17, n) / 8).astype(np.float32)
    g = residue.astype(np.float64) + dw
    d = dw.astype(np.float64)
    sel = (g != 0) & ((g * d >= 0) | (np.abs(d) >= 2 * np.abs(g)))
    s = np.float32(math.fsum(np.abs(g)) / n)
    r = oracle.compress(residue, dw, 1)
    assert np.array_equal(r.sel, sel)
    assert np.float32(r.s) == s


@pytest.mark.parametrize("n,L", [(1, 1), (10, 10), (37, 64), (500, 500), (300, 32768)])
def test_single_bin_scale_is_max(n, L):
    rng = np.random.default_rng(n)
    residue = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    dw = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    g = residue + dw
    r = oracle.compress(residue, dw, L)
    assert np.float32(r.s) == np.abs(g).max()


@pytest.mark.parametrize("n,L", [(1000, 50), (5001, 500), (777, 64), (300, 1)])
def test_decode_one_learner_gives_gq(n, L):
    rng = np.random.default_rng(n + L)
    residue = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g = residue + dw
    r = oracle.compress(residue, dw, L)
    gq = np.where(r.sel, np.sign(g) * r.s, 0).astype(np.float32)
    dense = np.zeros(n, np.float32)
    assert oracle.decode_accumulate(n, L, [r.msg], dense) == oracle.OK
    assert np.array_equal(dense, gq)


def test_decode_k_learners_matches_sequential_scatter():
    """K messages summed learner by learner equal numpy's unbuffered fp32 add.at."""
    rng = np.random.default_rng(5)
    n, L, K = 3000, 50, 6
    msgs, gqs = [], []
    for _ in range(K):
        residue = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        g = residue + dw
        r = oracle.compress(residue, dw, L)
        msgs.append(r.msg)
        gqs.append((np.nonzero(r.sel)[0], (np.sign(g[r.sel]) * r.s).astype(np.float32)))
    dense0 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    expect = dense0.copy()
    for idx, val in gqs:
        np.add.at(expect, idx, val)
    dense = dense0.copy()
    assert oracle.decode_accumulate(n, L, msgs, dense) == oracle.OK
    assert np.array_equal(dense, expect)

"""Invariants and brute force that pin the oracle independently of its own code.

Source: "AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
#r629-local-bin-soft-threshold-and-mean-gmax-quantization (residue = G - G_q for sent
elements, residue = G otherwise; |H| >= g_max; G_q = sign(G) * s) and the code widths
of Claims > Application / Curated Limitations.

* unsent elements keep residue = G bit for bit;
* sent elements satisfy G_q + residue = G up to the rounding of one fp32 subtraction
  (|sign*s + r - G| <= ulp(r)/2), exactly when s/2 <= |G| <= 2s (Sterbenz);
* every nonzero bin sends its maximum whenever dW does not oppose G's sign
  (monotone rounding gives |H| >= |G| = g_max there);
* bookkeeping: sum of counts = nnz, counts <= bin length, message bytes
  = 8 + 2B + w*nnz, offsets < bin length and strictly increasing within a bin;
* brute force over every input in a tiny grid, evaluated in exact rational
  arithmetic (fractions), where fp32 is exact.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _parse(msg, n, L):
    nb = -(-n // L)
    s = np.frombuffer(msg[:4].tobytes(), "<f4")[0]
    B = int(np.frombuffer(msg[4:8].tobytes(), "<u4")[0])
    counts = np.frombuffer(msg[8:8 + 2 * nb].tobytes(), "<u2").astype(np.int64)
    codes = np.frombuffer(msg[8 + 2 * nb:].tobytes(), "<u1" if L < 64 else "<u2").astype(np.int64)
    return s, B, counts, codes


def _check_step(res_before, dw_f32, r, res_after, L):
    n = res_before.size
    nb = -(-n // L)
    g = res_before + dw_f32  # fp32 sum, the G of this step
    sel = r.sel
    # unsent: residue = G exactly
    assert np.array_equal(res_after[~sel].view(np.uint32), g[~sel].view(np.uint32))
    # sent: G != 0 and G_q + r = G within half an ulp of r
    assert np.all(g[sel] != 0)
    sig = np.sign(g[sel]).astype(np.float64)
    rr = res_after[sel].astype(np.float64)
    err = np.abs(sig * np.float64(r.s) + rr - g[sel].astype(np.float64))
    half_ulp = np.spacing(np.abs(res_after[sel])).astype(np.float64) / 2
    assert np.all(err <= half_ulp)
    ag = np.abs(g[sel]).astype(np.float64)
    sterbenz = (ag >= np.float64(r.s) / 2) & (ag <= 2 * np.float64(r.s))
    assert np.all(err[sterbenz] == 0)
    # g_max and the max rule
    pad = np.zeros(nb * L, np.float32)
    pad[:n] = np.abs(g)
    gm = pad.reshape(nb, L).max(axis=1)
    assert np.array_equal(r.gmax, gm)
    binof = np.arange(n) // L
    is_max = (np.abs(g) == gm[binof]) & (gm[binof] > 0)
    agree = (dw_f32 == 0) | (np.sign(dw_f32) == np.sign(g))
    assert np.all(sel[is_max & agree])
    # s is the mean of g_max (fsum is the correctly rounded sum)
    assert np.float32(r.s) == np.float32(math.fsum(gm.astype(np.float64)) / nb)
    # message bookkeeping
    s, B, counts, codes = _parse(r.msg, n, L)
    w = 1 if L < 64 else 2
    assert B == nb and s == r.s
    assert counts.sum() == sel.sum() == codes.size
    assert r.msg.size == 8 + 2 * nb + w * sel.sum()
    lens = np.minimum(L, n - np.arange(nb) * L)
    assert np.all(counts <= lens)
    offs = codes >> 1
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    for b in np.nonzero(counts)[0]:
        o = offs[starts[b]:starts[b] + counts[b]]
        assert np.all(o < lens[b]) and np.all(np.diff(o) > 0)
    idx = np.repeat(np.arange(nb) * L, counts) + offs
    assert np.array_equal(idx, np.nonzero(sel)[0])
    assert np.array_equal(codes & 1, (g[idx] < 0).astype(np.int64))


@pytest.mark.parametrize("L", [1, 2, 3, 5, 50, 63, 64, 65, 500, 5000])
@pytest.mark.parametrize("bf16", [False, True])
def test_invariants_over_carried_steps(L, bf16):
    rng = np.random.default_rng(L * 3 + bf16)
    for n in (1, 2, L, L + 1, 3 * L - 1, 7 * L + 13, 997):
        residue = np.zeros(n, np.float32)
        sigma = 10.0 ** rng.uniform(-4, -2)
        for step in range(4):
            dw32 = (rng.standard_t(3, n) * sigma).astype(np.float32)
            dw32[rng.random(n) < 0.1] = 0.0
            if bf16:
                dw_in = (dw32.view(np.uint32) >> 16).astype(np.uint16)
                dwf = (dw_in.astype(np.uint32) << 16).view(np.float32)
            else:
                dw_in, dwf = dw32, dw32
            before = residue.copy()
            r = oracle.compress(residue, dw_in, L)
            _check_step(before, dwf, r, residue, L)


def test_all_zero_layer_sends_nothing():
    n, L = 1000, 50
    residue = np.zeros(n, np.float32)
    r = oracle.compress(residue, np.zeros(n, np.float32), L)
    assert r.s == 0 and not r.sel.any() and r.msg.size == 8 + 2 * 20


GRID5 = [-1.0, -0.5, 0.0, 0.5, 1.0]
GRID7 = [-1.0, -0.5, -0.25, 0.0, 0.25, 0.5, 1.0]


def _brute(res, dw, L):
    """The method in exact rationals; only s needs one fp64 and one fp32 rounding."""
    n = len(res)
    nb = -(-n // L)
    G = [Fraction(a) + Fraction(b) for a, b in zip(res, dw)]
    H = [g + Fraction(b) for g, b in zip(G, dw)]
    gm = [max(abs(x) for x in G[b * L:(b + 1) * L]) for b in range(nb)]
    s = np.float32(float(sum(gm)) / nb)  # the sum of grid values is exact in fp64
    sel = [G[j] != 0 and abs(H[j]) >= gm[j // L] for j in range(n)]
    res_new = []
    for j in range(n):
        if sel[j]:
            res_new.append(np.float32(G[j]) - s if G[j] > 0 else np.float32(G[j]) + s)
        else:
            res_new.append(np.float32(G[j]))
    return s, sel, np.array(res_new, np.float32)


@pytest.mark.parametrize("n,Ls,grid", [(2, (1, 2, 64), GRID7), (3, (1, 2, 3), GRID5)])
def test_brute_force_tiny_grid(n, Ls, grid):
    for L in Ls:
        for vals in itertools.product(grid, repeat=2 * n):
            res = np.array(vals[:n], np.float32)
            dw = np.array(vals[n:], np.float32)
            s, sel, res_new = _brute(vals[:n], vals[n:], L)
            r = oracle.compress(res, dw, L)
            assert r.s == s
            assert r.sel.tolist() == sel, (vals, L)
            assert np.array_equal(res.view(np.uint32), res_new.view(np.uint32))

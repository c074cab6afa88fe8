"""The Local Selection rule of the oracle (the contrast the pages draw).

"AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
#r629-self-adjusting-sparsity-prevents-residual-explosion: hard Local Selection,
without AdaComp's soft threshold, transmits only bin maxima and lets the residue of
everything else grow, while AdaComp's probe abs(residue + 2 dW) >= g_max sends more
elements as residues grow and keeps them bounded. The hand case is in
tests/golden/hand_lt4_n10_local_selection.json.
"""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("L", [1, 7, 50, 500])
def test_local_selection_sends_exactly_the_bin_maxima(L):
    rng = np.random.default_rng(L)
    n = 20_011
    residue = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    dw[rng.random(n) < 0.3] = 0.0
    G = residue + dw  # one fp32 rounding, as the method forms G
    r = oracle.compress(residue.copy(), dw, L, local_selection=True)
    bins = np.arange(n) // L
    gmax = np.zeros(bins[-1] + 1, np.float32)
    np.maximum.at(gmax, bins, np.abs(G))
    expect = (G != 0) & (np.abs(G) == gmax[bins])
    assert np.array_equal(r.sel, expect)
    assert np.array_equal(r.gmax, gmax)
    nonzero_bins = np.unique(bins[G != 0])
    assert np.all(np.bincount(bins[expect], minlength=gmax.size)[nonzero_bins] >= 1)


def test_local_selection_residue_grows_where_adacomp_levels_off():
    """Seeded synthetic run (fresh N(0, 1e-3) gradients, L_T = 500): the largest
    residue under Local Selection keeps growing, AdaComp's levels off below it."""
    n, L = 50_000, 500
    out = {}
    for ls in (False, True):
        rng = np.random.default_rng(5)
        res = np.zeros(n, np.float32)
        peaks = []
        for step in range(80):
            dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
            oracle.compress(res, dw, L, local_selection=ls)
            if step % 20 == 19:
                peaks.append(float(np.abs(res).max()))
        out[ls] = peaks
    ada, ls = out[False], out[True]
    assert ada[3] < 1.10 * ada[1]  # AdaComp: bounded
    assert ls[3] > 1.3 * ls[0]     # Local Selection: still growing
    assert ls[3] > 1.5 * ada[3]


def test_local_selection_residue_grows_where_adacomp_stays_bounded():
    """The contrast the entry draws (Claims > Mechanism
    #r629-self-adjusting-sparsity-prevents-residual-explosion): on a designed input, a
    bin of 64 elements receiving the same positive gradient every step with slightly
    different magnitudes (d (1 + j/128)), AdaComp's soft threshold sends every element
    whose G + dW reaches the bin maximum, so the residues stay within about 1.4 d;
    Local Selection sends only the bin maximum each step, so the other elements keep
    accumulating and the largest residue passes 20 d within 50 steps."""
    L = n = 64
    d = np.float32(1e-3)
    dw = (d * (1 + np.arange(n, dtype=np.float32) / 128)).astype(np.float32)
    peak = {}
    for ls in (False, True):
        r = np.zeros(n, np.float32)
        worst = 0.0
        for _ in range(50):
            oracle.compress(r, dw, L, local_selection=ls)
            worst = max(worst, float(np.abs(r).max()))
        peak[ls] = worst / float(d)
    assert peak[False] <= 2.0, peak
    assert peak[True] >= 20.0, peak

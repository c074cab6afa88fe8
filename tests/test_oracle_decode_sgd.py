"""Pins the oracle's decode fused with a momentum-SGD step.

The learners' codes are summed from zero in learner order (as the plain decoder
does), then v = fl32(fl32(mu v) + fl32(scale g)) and w = fl32(w - fl32(lr v)); the
optimiser is the one the pages' learners use ("AdaComp (Adaptive Residual Gradient
Compression)", Claims > Application
#r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers), the exact rule is a
reading. The hand case is tests/golden/hand_decode_sgd.json.
"""
import numpy as np

import oracle
from _golden import f32_array, hex_bytes, load


def test_hand_case():
    c = load("hand_decode_sgd")
    w = f32_array(c["w_in"])
    v = f32_array(c["v_in"])
    rc = oracle.decode_sgd(c["n"], c["bin_len"], [hex_bytes(c["msg_hex"])], w, v, c["lr"], c["mu"], c["scale"])
    assert rc == oracle.OK
    assert np.array_equal(v, f32_array(c["expect_v"]))
    assert np.array_equal(w, f32_array(c["expect_w"]))


def _msgs(n, L, K, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(K):
        res = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        out.append(oracle.compress(res, dw, L).msg)
    return out


def test_zero_momentum_unit_rate_gives_the_decoded_gradient():
    """mu = 0, lr = 1, scale = 1: v becomes exactly the plain decoder's sum and
    w = fl32(w - g)."""
    n, L = 30_011, 50
    msgs = _msgs(n, L, 3, 1)
    g = np.zeros(n, np.float32)
    assert oracle.decode_accumulate(n, L, msgs, g) == oracle.OK
    rng = np.random.default_rng(2)
    w0 = rng.standard_normal(n).astype(np.float32)
    w, v = w0.copy(), rng.standard_normal(n).astype(np.float32)
    assert oracle.decode_sgd(n, L, msgs, w, v, 1.0, 0.0, 1.0) == oracle.OK
    assert np.array_equal(v.view(np.uint32), g.view(np.uint32))
    assert np.array_equal(w.view(np.uint32), (w0 - g).view(np.uint32))


def test_zero_rate_leaves_weights_and_a_bad_message_adds_nothing():
    n, L = 5_003, 500
    msgs = _msgs(n, L, 2, 3)
    w = np.ones(n, np.float32)
    v = np.zeros(n, np.float32)
    assert oracle.decode_sgd(n, L, msgs, w, v, 0.0, 0.9, 0.5) == oracle.OK
    assert np.all(w == 1.0)
    bad = msgs[1].copy()
    bad[4] ^= 1  # wrong B
    w2, v2 = w.copy(), v.copy()
    assert oracle.decode_sgd(n, L, [msgs[0], bad], w2, v2, 0.1, 0.9, 1.0) == oracle.ERR_BAD_MESSAGE
    # the rejected message adds nothing: the step is the one the good message alone gives
    w3, v3 = w.copy(), v.copy()
    assert oracle.decode_sgd(n, L, [msgs[0]], w3, v3, 0.1, 0.9, 1.0) == oracle.OK
    assert np.array_equal(w2, w3) and np.array_equal(v2, v3)
    assert not np.array_equal(w2, w)

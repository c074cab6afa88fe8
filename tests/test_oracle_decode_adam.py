"""Pins the oracle's decode fused with an Adam step.

The learners' codes are summed from zero in learner order (as the plain decoder
does), then one Adam step with the bias corrections written out
(m, v, mh = m / bc1, vh = v / bc2, w -= lr * mh / (sqrt(vh) + eps)), every
operation an fp32 operation rounded once. Adam is one of the two optimisers the
pages' learners use ("AdaComp (Adaptive Residual Gradient Compression)", Claims >
Application #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers); the
exact rule is a reading. The hand case is tests/golden/hand_decode_adam.json.
"""
import numpy as np

import oracle
from _golden import f32_array, hex_bytes, load


def _hand(c):
    return (f32_array(c["w_in"]), f32_array(c["m_in"]), f32_array(c["v_in"]))


def test_hand_case():
    c = load("hand_decode_adam")
    w, m, v = _hand(c)
    rc = oracle.decode_adam(c["n"], c["bin_len"], [hex_bytes(h) for h in c["msgs_hex"]], w, m, v, c["lr"],
                            c["beta1"], c["beta2"], c["eps"], c["bc1"], c["bc2"], c["scale"])
    assert rc == oracle.OK
    assert np.array_equal(m, f32_array(c["expect_m"]))
    assert np.array_equal(v, f32_array(c["expect_v"]))
    assert np.array_equal(w, f32_array(c["expect_w"]))


def test_zero_betas_give_sign_descent():
    """beta1 = beta2 = 0, no bias correction (bc = 1) and eps = 0 reduce Adam to a
    step of lr against the sign of the gradient: m = g, v = fl32(g^2), and
    sqrt(fl32(g^2)) = |g| exactly in binary round-to-nearest, so w = fl32(w - lr sign(g)).
    With L_T = 1 and a zero residue every nonzero element is sent, so g = s sign(dW)."""
    n, L = 20_011, 1
    rng = np.random.default_rng(4)
    dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    dw[dw == 0] = 1e-3
    msg = oracle.compress(np.zeros(n, np.float32), dw, L).msg
    w0 = rng.standard_normal(n).astype(np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    lr = np.float32(0.01)
    assert oracle.decode_adam(n, L, [msg], w, m, v, lr, 0.0, 0.0, 0.0, 1.0, 1.0) == oracle.OK
    g = np.zeros(n, np.float32)
    assert oracle.decode_accumulate(n, L, [msg], g) == oracle.OK
    assert np.array_equal(m.view(np.uint32), g.view(np.uint32))
    assert np.all(np.abs(g) > 0)
    expect = (w0 - lr * np.sign(dw).astype(np.float32)).astype(np.float32)
    assert np.array_equal(w.view(np.uint32), expect.view(np.uint32))


def _msgs(n, L, K, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(K):
        res = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        out.append(oracle.compress(res, dw, L).msg)
    return out


def test_zero_rate_keeps_weights_and_moments_follow_their_recurrences():
    """lr = 0 leaves w unchanged; with beta1 = 1 the first moment keeps its old value
    and with beta2 = 1 the second moment too (1 - beta = 0 adds nothing)."""
    n, L = 5_003, 500
    msgs = _msgs(n, L, 2, 3)
    rng = np.random.default_rng(5)
    w0 = rng.standard_normal(n).astype(np.float32)
    m0 = rng.standard_normal(n).astype(np.float32)
    v0 = np.abs(rng.standard_normal(n)).astype(np.float32)
    w, m, v = w0.copy(), m0.copy(), v0.copy()
    assert oracle.decode_adam(n, L, msgs, w, m, v, 0.0, 1.0, 1.0, 1e-8, 1.0, 1.0) == oracle.OK
    assert np.array_equal(w, w0) and np.array_equal(m, m0) and np.array_equal(v, v0)


def test_bad_message_adds_nothing():
    n, L = 5_003, 500
    msgs = _msgs(n, L, 2, 6)
    bad = msgs[1].copy()
    bad[4] ^= 1  # wrong B
    rng = np.random.default_rng(7)
    w0 = rng.standard_normal(n).astype(np.float32)
    args = (0.01, 0.9, 0.999, 1e-8, 0.1, 0.001)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    assert oracle.decode_adam(n, L, [msgs[0], bad], w, m, v, *args) == oracle.ERR_BAD_MESSAGE
    w2, m2, v2 = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    assert oracle.decode_adam(n, L, [msgs[0]], w2, m2, v2, *args) == oracle.OK
    assert np.array_equal(w, w2) and np.array_equal(m, m2) and np.array_equal(v, v2)

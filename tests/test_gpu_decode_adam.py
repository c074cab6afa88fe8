"""Decode fused with an Adam step against the oracle (GPU).

The learners' codes are summed from zero in learner order and one Adam step (bias
corrections written out, every operation fp32 and rounded once, correctly rounded
division and square root) is applied while the tile is in shared memory. Adam is
one of the optimisers of "AdaComp (Adaptive Residual Gradient Compression)",
Claims > Application #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers;
the rule is a reading. Weights and both moments must match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from _golden import f32_array, hex_bytes, load
from _gpu import ensure_built, workspace
from test_gpu_decode import _learner_msgs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _state(n, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    w = torch.randn(n, generator=g, device="cuda")
    m = torch.randn(n, generator=g, device="cuda") * 1e-3
    v = torch.rand(n, generator=g, device="cuda") * 1e-6
    return w, m, v


def _host(*ts):
    return [t.cpu().numpy().copy() for t in ts]


def _same(gpu, ref, what):
    assert np.array_equal(gpu.cpu().numpy().view(np.uint32), ref.view(np.uint32)), what


def test_hand_case():
    c = load("hand_decode_adam")
    n, L = c["n"], c["bin_len"]
    h = ac.adacomp_init_layer(n, L, ac.F32)
    msgs, lens = [], []
    for hx in c["msgs_hex"]:
        b = hex_bytes(hx)
        buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
        buf[:b.size] = torch.from_numpy(b.copy()).cuda()
        msgs.append(buf)
        lens.append(b.size)
    w = torch.from_numpy(f32_array(c["w_in"])).cuda()
    m = torch.from_numpy(f32_array(c["m_in"])).cuda()
    v = torch.from_numpy(f32_array(c["v_in"])).cuda()
    ws = workspace(h.decode_ws_bytes(len(msgs)))
    ac.adacomp_decode_adam(h, msgs, lens, w, m, v, c["lr"], c["beta1"], c["beta2"], c["eps"], c["bc1"], c["bc2"], ws,
                           grad_scale=c["scale"])
    assert ac.adacomp_decode_status(h, ws) == ac.OK
    _same(w, f32_array(c["expect_w"]), "w")
    _same(m, f32_array(c["expect_m"]), "m")
    _same(v, f32_array(c["expect_v"]), "v")


ADAM = (1e-3, 0.9, 0.999, 1e-8)


@pytest.mark.parametrize("n,L,K,t", [(10, 4, 1, 1), (100_003, 50, 3, 1), (1_000_001, 500, 16, 7),
                                     (300_007, 5000, 5, 100), (77_777, 7, 4, 3), (200_003, 500, 40, 2)])
def test_decode_adam_matches_oracle(n, L, K, t):
    msgs = _learner_msgs(n, L, K, seed=n + L + 1)
    h = ac.adacomp_init_layer(n, L, ac.F32)
    w, m, v = _state(n, K + t)
    wr, mr, vr = _host(w, m, v)
    lr, b1, b2, eps = ADAM
    bc1 = float(np.float32(1.0 - b1 ** t))
    bc2 = float(np.float32(1.0 - b2 ** t))
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_adam(h, [x for x, _ in msgs], [mb for _, mb in msgs], w, m, v, lr, b1, b2, eps, bc1, bc2, ws,
                           grad_scale=1.0 / K)
    assert ac.adacomp_decode_status(h, ws) == ac.OK
    host = [x[:mb].cpu().numpy() for x, mb in msgs]
    assert oracle.decode_adam(n, L, host, wr, mr, vr, lr, b1, b2, eps, bc1, bc2, 1.0 / K) == oracle.OK
    _same(m, mr, "m")
    _same(v, vr, "v")
    _same(w, wr, "w")


def test_decode_adam_group_and_a_rejected_message():
    """A grouped call over layers of both tile kinds, one of whose messages is
    malformed (wrong B): that message adds nothing, the rest matches the oracle."""
    shapes = [(100_003, 50), (500_001, 500), (33_333, 5000)]
    K = 3
    h = ac.adacomp_init_group([n for n, _ in shapes], [L for _, L in shapes], [ac.F32] * len(shapes))
    per_layer = [_learner_msgs(n, L, K, seed=3 * n) for n, L in shapes]
    bad, bad_len = per_layer[1][2][0].clone(), per_layer[1][2][1]
    bad[4] ^= 1
    per_layer[1][2] = (bad, bad_len)
    states = [_state(n, i) for i, (n, _) in enumerate(shapes)]
    refs = [_host(*st) for st in states]
    lr, b1, b2, eps = ADAM
    bc1, bc2 = float(np.float32(1 - b1 ** 5)), float(np.float32(1 - b2 ** 5))
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_adam_group(h, [[x for x, _ in pl] for pl in per_layer], [[mb for _, mb in pl] for pl in per_layer],
                                 [s[0] for s in states], [s[1] for s in states], [s[2] for s in states], lr, b1, b2,
                                 eps, bc1, bc2, ws)
    assert ac.adacomp_decode_status(h, ws) == ac.ERR_BAD_MESSAGE
    for (n, L), pl, st, (wr, mr, vr) in zip(shapes, per_layer, states, refs):
        host = [x[:mb].cpu().numpy() for x, mb in pl]
        rc = oracle.decode_adam(n, L, host, wr, mr, vr, lr, b1, b2, eps, bc1, bc2)
        assert rc == (oracle.ERR_BAD_MESSAGE if L == 500 else oracle.OK)
        _same(st[0], wr, (n, L))
        _same(st[1], mr, (n, L))
        _same(st[2], vr, (n, L))

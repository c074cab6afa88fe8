"""Decode fused with a momentum-SGD step against the oracle (GPU).

The learners' codes are summed from zero in learner order and one step
v = fl32(fl32(mu v) + fl32(scale g)), w = fl32(w - fl32(lr v)) is applied while the
tile is in shared memory (optimiser of "AdaComp (Adaptive Residual Gradient
Compression)", Claims > Application
#r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers; the rule is a
reading). Weights and momentum must match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from _gpu import ensure_built, workspace
from test_gpu_decode import _learner_msgs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _wv(n, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(n, generator=g, device="cuda"), torch.randn(n, generator=g, device="cuda") * 1e-2


@pytest.mark.parametrize("n,L,K", [(10, 4, 1), (100_003, 50, 3), (1_000_001, 500, 16), (300_007, 5000, 5),
                                   (77_777, 7, 4), (65_537, 64, 2), (200_003, 500, 40)])
def test_decode_sgd_matches_oracle(n, L, K):
    msgs = _learner_msgs(n, L, K, seed=n + L)
    h = ac.adacomp_init_layer(n, L, ac.F32)
    w, v = _wv(n, K)
    w_ref, v_ref = w.cpu().numpy().copy(), v.cpu().numpy().copy()
    lr, mu, scale = 0.01, 0.9, 1.0 / K
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_sgd(h, [m for m, _ in msgs], [mb for _, mb in msgs], w, v, lr, mu, ws, grad_scale=scale)
    assert ac.adacomp_decode_status(h, ws) == ac.OK
    host = [m[:mb].cpu().numpy() for m, mb in msgs]
    assert oracle.decode_sgd(n, L, host, w_ref, v_ref, lr, mu, scale) == oracle.OK
    assert np.array_equal(v.cpu().numpy().view(np.uint32), v_ref.view(np.uint32))
    assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))


def test_decode_sgd_group_matches_per_layer():
    shapes = [(100_003, 50), (4_096, 50), (500_001, 500), (33_333, 5000)]
    K = 3
    h = ac.adacomp_init_group([n for n, _ in shapes], [L for _, L in shapes], [ac.F32] * len(shapes))
    per_layer = [_learner_msgs(n, L, K, seed=7 * n) for n, L in shapes]
    ws_ = [_wv(n, i) for i, (n, _) in enumerate(shapes)]
    refs = [(w.cpu().numpy().copy(), v.cpu().numpy().copy()) for w, v in ws_]
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_sgd_group(h, [[m for m, _ in msgs] for msgs in per_layer],
                                [[mb for _, mb in msgs] for msgs in per_layer], [w for w, _ in ws_],
                                [v for _, v in ws_], 0.05, 0.5, ws, grad_scale=1.0)
    assert ac.adacomp_decode_status(h, ws) == ac.OK
    for (n, L), msgs, (w, v), (w_ref, v_ref) in zip(shapes, per_layer, ws_, refs):
        host = [m[:mb].cpu().numpy() for m, mb in msgs]
        assert oracle.decode_sgd(n, L, host, w_ref, v_ref, 0.05, 0.5, 1.0) == oracle.OK
        assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))
        assert np.array_equal(v.cpu().numpy().view(np.uint32), v_ref.view(np.uint32))


def test_decode_sgd_skips_a_malformed_message():
    n, L = 50_000, 500
    msgs = _learner_msgs(n, L, 2, seed=11)
    bad, mb = msgs[1][0].clone(), msgs[1][1]
    bad[4] = (int(bad[4]) + 1) % 256  # wrong B
    h = ac.adacomp_init_layer(n, L, ac.F32)
    w, v = _wv(n, 5)
    w_ref, v_ref = w.cpu().numpy().copy(), v.cpu().numpy().copy()
    ws = workspace(h.decode_ws_bytes(2))
    ac.adacomp_decode_sgd(h, [msgs[0][0], bad], [msgs[0][1], mb], w, v, 0.1, 0.9, ws)
    assert ac.adacomp_decode_status(h, ws) == ac.ERR_BAD_MESSAGE
    # the good learner alone, as the oracle sees it
    assert oracle.decode_sgd(n, L, [msgs[0][0][:msgs[0][1]].cpu().numpy()], w_ref, v_ref, 0.1, 0.9) == oracle.OK
    assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))
    assert np.array_equal(v.cpu().numpy().view(np.uint32), v_ref.view(np.uint32))

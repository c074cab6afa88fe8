"""The Local Selection rule on the GPU against the oracle's (GPU).

"AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
#r629-self-adjusting-sparsity-prevents-residual-explosion: without the soft
threshold only bin maxima are sent (abs(G) >= g_max). Messages, s and residue must
match the oracle bit for bit over carried steps, on every tile shape.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from _gpu import assert_same_step, dw_host, ensure_built, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _dw(n, step, seed, bf16):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed * 1000 + step)
    dw = torch.randn(n, generator=g, device="cuda") * 1e-3
    dw[torch.rand(n, generator=g, device="cuda") < 0.05] = 0.0
    return dw.to(torch.bfloat16) if bf16 else dw


@pytest.mark.parametrize("lazy", [False, True], ids=["eager", "lazy"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("n,L", [(100_003, 50), (500_001, 500), (50_003, 4), (300_007, 5000), (77_777, 20)])
def test_local_selection_matches_oracle(n, L, bf16, lazy):
    h = ac.adacomp_init_layer(n, L, ac.BF16 if bf16 else ac.F32)
    ac.adacomp_set_selection_rule(h, ac.RULE_LOCAL_SELECTION)
    ws = workspace(ac.adacomp_set_lazy_fixup(h, True) if lazy else h.compress_ws_bytes)
    msg = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device="cuda")
    res = torch.zeros(n, device="cuda")
    ref_res = np.zeros(n, np.float32)
    for step in range(3):
        dw = _dw(n, step, L, bf16)
        ac.adacomp_compress(h, res, dw, msg, ws)
        if lazy:
            ac.adacomp_materialize(h, res, ws)
        mb, s, st = ac.adacomp_query(h, ws)
        assert st == ac.OK
        ref = oracle.compress(ref_res, dw_host(dw), L, local_selection=True)
        assert_same_step(msg[:mb].cpu().numpy(), s, res.cpu().numpy(), ref, ref_res, f"step {step}")


def test_rule_can_be_switched_back():
    n, L = 200_000, 50
    h = ac.adacomp_init_layer(n, L, ac.F32)
    ws = workspace(h.compress_ws_bytes)
    msg = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device="cuda")
    res = torch.zeros(n, device="cuda")
    ref_res = np.zeros(n, np.float32)
    for step, rule in enumerate([ac.RULE_LOCAL_SELECTION, ac.RULE_ADACOMP, ac.RULE_LOCAL_SELECTION]):
        ac.adacomp_set_selection_rule(h, rule)
        dw = _dw(n, step, 9, False)
        ac.adacomp_compress(h, res, dw, msg, ws)
        mb, s, st = ac.adacomp_query(h, ws)
        ref = oracle.compress(ref_res, dw_host(dw), L, local_selection=rule == ac.RULE_LOCAL_SELECTION)
        assert_same_step(msg[:mb].cpu().numpy(), s, res.cpu().numpy(), ref, ref_res, f"step {step}")
    with pytest.raises(ac.AdacompError):
        ac.adacomp_set_selection_rule(h, 2)

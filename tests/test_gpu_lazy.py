"""Deferred (lazy) fix-up against the oracle's eager steps (GPU).

With the fix-up deferred, a compress call leaves sent elements at G and the next
call applies residue = fl32(G - sign(G) s_prev) as it loads them ("AdaComp (Adaptive
Residual Gradient Compression)", Claims > Mechanism
#r629-local-bin-soft-threshold-and-mean-gmax-quantization: residue = G - G_q). The
messages and s of every step, and the residue after adacomp_materialize, must equal
the oracle's eager steps bit for bit.
"""
import numpy as np
import pytest
import torch

import residual_gradient_compression_gb300 as ac
from residual_gradient_compression_gb300 import workloads as wl
from _gpu import assert_same_step, dw_host, ensure_built, oracle_step, workspace

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


def _run(shapes, steps, bf16=False, materialize_at=()):
    """Lazy group over `shapes` [(n, L)]: messages and s checked every step, residue
    checked after each materialise and at the end."""
    h = ac.adacomp_init_group([n for n, _ in shapes], [L for _, L in shapes],
                              [ac.BF16 if bf16 else ac.F32] * len(shapes))
    ws_bytes = ac.adacomp_set_lazy_fixup(h, True)
    ws = workspace(ws_bytes)
    msgs = [torch.zeros(m, dtype=torch.uint8, device="cuda") for m in h.max_msg_bytes]
    res = [torch.zeros(n, device="cuda") for n, _ in shapes]
    ref_res = [np.zeros(n, np.float32) for n, _ in shapes]
    for step in range(steps):
        dws = [_dw(n, step, i + 1, bf16) for i, (n, _) in enumerate(shapes)]
        ac.adacomp_compress_group(h, res, dws, msgs, ws)
        for i, (n, L) in enumerate(shapes):
            mb, s, st = ac.adacomp_query(h, ws, i)
            assert st == ac.OK
            ref = oracle_step(ref_res[i], dw_host(dws[i]), L)
            assert np.float32(s).view(np.uint32) == np.float32(ref.s).view(np.uint32), f"s, layer {i} step {step}"
            assert np.array_equal(msgs[i][:mb].cpu().numpy(), ref.msg), f"message, layer {i} step {step}"
        if step in materialize_at or step == steps - 1:
            ac.adacomp_materialize_group(h, res, ws)
            for i in range(len(shapes)):
                got = res[i].cpu().numpy()
                assert np.array_equal(got.view(np.uint32), ref_res[i].view(np.uint32)), f"residue, layer {i} step {step}"
    return h, ws, res, ref_res


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("n,L", [(1_000_003, 50), (500_001, 500), (300_007, 100), (77_777, 16), (4_001, 63),
                                 (500_001, 5000), (123_457, 1365), (65_000, 8189)])
def test_lazy_single_layer(n, L, bf16):
    _run([(n, L)], steps=4, bf16=bf16, materialize_at=(1,))


def test_lazy_group_mixes_deferred_and_eager_layers():
    # L_T = 4 and 5000 take block-wide tiles and are fixed up eagerly; the rest defer
    _run([(200_000, 50), (50_003, 4), (123_457, 500), (400_000, 5000), (4_096, 50)], steps=3)


def test_block_sliced_group_with_a_materialise_between_steps():
    _run([(400_000, 5000), (123_457, 1365), (77_777, 600)], steps=4, materialize_at=(1,))


def test_resnet50_lazy_full_size():
    lys = wl.layers("resnet50")
    h = ac.adacomp_init_group([l.numel for l in lys], [l.bin_len for l in lys], [ac.F32] * len(lys))
    ws = workspace(ac.adacomp_set_lazy_fixup(h, True))
    msgs = [torch.zeros(m, dtype=torch.uint8, device="cuda") for m in h.max_msg_bytes]
    res = [torch.zeros(l.numel, device="cuda") for l in lys]
    ref_res = [np.zeros(l.numel, np.float32) for l in lys]
    for step in range(3):
        dws = [wl.gen_dw("resnet50", i, l, step) for i, l in enumerate(lys)]
        ac.adacomp_compress_group(h, res, dws, msgs, ws)
        torch.cuda.synchronize()
        for i, l in enumerate(lys):
            mb, s, st = ac.adacomp_query(h, ws, i)
            ref = oracle_step(ref_res[i], dw_host(dws[i]), l.bin_len)
            assert st == ac.OK and np.array_equal(msgs[i][:mb].cpu().numpy(), ref.msg), f"{l.name} step {step}"
    ac.adacomp_materialize_group(h, res, ws)
    for i, l in enumerate(lys):
        assert np.array_equal(res[i].cpu().numpy().view(np.uint32), ref_res[i].view(np.uint32)), l.name


def test_switch_back_to_eager_after_materialize():
    n, L = 250_000, 50
    h, ws, res, ref_res = _run([(n, L)], steps=2)
    ac.adacomp_set_lazy_fixup(h, False)  # the workspace stays large enough
    msg = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device="cuda")
    for step in range(2, 4):
        dw = _dw(n, step, 1, False)
        ac.adacomp_compress(h, res[0], dw, msg, ws)
        mb, s, st = ac.adacomp_query(h, ws)
        ref = oracle_step(ref_res[0], dw_host(dw), L)
        assert_same_step(msg[:mb].cpu().numpy(), s, res[0].cpu().numpy(), ref, ref_res[0], f"step {step}")


def test_materialize_twice_changes_nothing():
    h, ws, res, ref_res = _run([(100_003, 50)], steps=2)
    before = res[0].clone()
    ac.adacomp_materialize(h, res[0], ws)
    assert torch.equal(before.view(torch.int32), res[0].view(torch.int32))


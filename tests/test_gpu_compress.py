"""CUDA compress path vs the oracle, element by element (GPU).

Method: "AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
#r629-local-bin-soft-threshold-and-mean-gmax-quantization. The bar is bit-exact:
messages (which fix masks, indices and per-bin counts), s and residue. The readings
make this reachable: s is the exact sum of the bin maxima rounded once to fp64, so
it does not depend on the order tiles finish in, and every other value comes from
single IEEE fp32 additions, which both sides perform alike.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from residual_gradient_compression_gb300 import workloads as wl
from _golden import case_inputs, compress_cases, f32_array, fval, hex_bytes
from _gpu import GpuLayer, assert_same_step, dtype_code, dw_host, ensure_built, oracle_step, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


GOLDEN = [c for c in compress_cases() if not c.get("literal_zero_select")]


@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
def test_hand_cases(case):
    residue, dw = case_inputs(case)
    res_t = torch.from_numpy(residue.copy()).cuda()
    if dw.dtype == np.uint16:
        dw_t = torch.from_numpy(dw.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        dw_t = torch.from_numpy(dw).cuda()
    layer = GpuLayer(residue.size, case["bin_len"], dtype_code(dw_t))
    if case.get("local_selection"):
        ac.adacomp_set_selection_rule(layer.h, ac.RULE_LOCAL_SELECTION)
    msg, s = layer.step(res_t, dw_t)
    exp = case["expect"]
    assert msg.tobytes() == hex_bytes(exp["msg_hex"]).tobytes()
    assert s.view(np.uint32) == np.float32(fval(exp["s"])).view(np.uint32)
    assert np.array_equal(res_t.cpu().numpy().view(np.uint32), f32_array(exp["residue"]).view(np.uint32))


def _dw(n, step, seed, bf16, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + step)
    dw = torch.randn(n, generator=g, device=device) * 1e-3
    dw[torch.rand(n, generator=g, device=device) < 0.05] = 0.0
    if n > 3000:
        dw[n // 3: n // 3 + 1500] = 0.0  # all-zero bins
    return dw.to(torch.bfloat16) if bf16 else dw


SHAPES = [(1, 1), (2, 2), (7, 3), (10, 4), (1000, 1), (5000, 2), (123457, 7), (99999, 6),
          (100003, 50), (200000, 63), (65537, 64), (1000001, 500), (300000, 5000),
          (250000, 8192), (40000, 4096), (4095, 4097), (8191, 8192),
          # more warp-slice shapes: 31, 16, 25 and 5 bins per warp
          (77777, 16), (90001, 30), (33333, 20), (1000003, 100),
          # block-sliced tiles: 8 bins of 510 (the shortest), 3 bins of 1365 (tiles off the
          # 16-byte grid), one bin of 4094, 6000 and 8189 (the longest: 16 slices with the
          # alignment slots), ragged ends
          (300007, 510), (123457, 1365), (99999, 4094), (50001, 6000), (65000, 8189), (2000003, 2048)]


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("n,L", SHAPES)
def test_random_layers_multistep(n, L, bf16):
    layer = GpuLayer(n, L, ac.BF16 if bf16 else ac.F32)
    res_t = torch.zeros(n, device="cuda")
    res_np = np.zeros(n, np.float32)
    for step in range(3):
        dw_t = _dw(n, step, n + L, bf16)
        msg, s = layer.step(res_t, dw_t)
        ref = oracle_step(res_np, dw_host(dw_t), L)
        assert_same_step(msg, s, res_t.cpu().numpy(), ref, res_np, f"n={n} L={L} step={step}")


def test_fc400k_ten_steps():
    """500x800 FC layer, L_T = 500, fresh N(0, 1e-3) dW each of 10 steps, residue from 0."""
    (ly,) = wl.layers("fc400k")
    layer = GpuLayer(ly.numel, ly.bin_len, ac.F32)
    res_t = torch.zeros(ly.numel, device="cuda")
    res_np = np.zeros(ly.numel, np.float32)
    for step in range(10):
        dw_t = wl.gen_dw("fc400k", 0, ly, step)
        msg, s = layer.step(res_t, dw_t)
        ref = oracle_step(res_np, dw_host(dw_t), ly.bin_len)
        assert_same_step(msg, s, res_t.cpu().numpy(), ref, res_np, f"step {step}")


def _group_run(config, steps, layers=None, bin_len=None):
    lys = layers or wl.layers(config, bin_len)
    h = ac.adacomp_init_group([l.numel for l in lys], [l.bin_len for l in lys],
                              [ac.BF16 if l.dw_dtype == "bf16" else ac.F32 for l in lys])
    msgs = [torch.zeros(m, dtype=torch.uint8, device="cuda") for m in h.max_msg_bytes]
    ws = workspace(h.compress_ws_bytes)
    res = [torch.zeros(l.numel, device="cuda") for l in lys]
    res_np = [np.zeros(l.numel, np.float32) for l in lys]
    all_names = [l.name for l in wl.layers(config, bin_len)]
    for step in range(steps):
        dws = [wl.gen_dw(config, all_names.index(l.name), l, step) for l in lys]
        ac.adacomp_compress_group(h, res, dws, msgs, ws)
        torch.cuda.synchronize()
        for i, l in enumerate(lys):
            mb, s, st = ac.adacomp_query(h, ws, i)
            assert st == ac.OK
            ref = oracle_step(res_np[i], dw_host(dws[i]), l.bin_len)
            assert_same_step(msgs[i][:mb].cpu().numpy(), s, res[i].cpu().numpy(), ref, res_np[i],
                             f"{config} layer {l.name} step {step}")


def test_resnet50_group_full_size():
    """All 54 ResNet-50 tensors (25.5M elements) in one grouped launch, 3 carried steps."""
    _group_run("resnet50", 3)


def test_lstm_fc_group_full_size():
    """4 LSTM + 6 FC tensors (134M elements), Student-t dW, 90% zero FC rows, 2 steps."""
    _group_run("lstm_fc", 2)


@pytest.mark.parametrize("bin_len", [50, 500, 5000])
def test_gpt1p3b_sampled_tensors(bin_len):
    """bf16 dW: the 103M-element embedding plus every tensor of one decoder block."""
    lys = [l for l in wl.layers("gpt1p3b", bin_len) if l.name == "wte" or l.name.startswith("h7.")]
    _group_run("gpt1p3b", 2, layers=lys, bin_len=bin_len)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_block_sliced_group_of_mixed_bin_lengths(bf16):
    """One launch over layers whose bins are all 510..8189 but of different lengths:
    the CTA is as wide as the widest tile (16 warps for L_T = 8189), so layers with
    fewer slices per tile leave warps idle; every layer must still match the oracle."""
    shapes = [(400_000, 5000), (123_457, 1365), (77_777, 600), (65_000, 8189), (3_000, 510)]
    h = ac.adacomp_init_group([n for n, _ in shapes], [L for _, L in shapes], [ac.BF16 if bf16 else ac.F32] * len(shapes))
    msgs = [torch.zeros(m, dtype=torch.uint8, device="cuda") for m in h.max_msg_bytes]
    ws = workspace(h.compress_ws_bytes)
    res = [torch.zeros(n, device="cuda") for n, _ in shapes]
    res_np = [np.zeros(n, np.float32) for n, _ in shapes]
    for step in range(3):
        dws = [_dw(n, step, 7 * i + 1, bf16) for i, (n, _) in enumerate(shapes)]
        ac.adacomp_compress_group(h, res, dws, msgs, ws)
        torch.cuda.synchronize()
        for i, (n, L) in enumerate(shapes):
            mb, s, st = ac.adacomp_query(h, ws, i)
            assert st == ac.OK
            ref = oracle_step(res_np[i], dw_host(dws[i]), L)
            assert_same_step(msgs[i][:mb].cpu().numpy(), s, res[i].cpu().numpy(), ref, res_np[i],
                             f"layer {i} L={L} step {step}")


def test_all_zero_layer():
    n, L = 10000, 50
    layer = GpuLayer(n, L, ac.F32)
    res_t = torch.zeros(n, device="cuda")
    msg, s = layer.step(res_t, torch.zeros(n, device="cuda"))
    ref = oracle_step(np.zeros(n, np.float32), np.zeros(n, np.float32), L)
    assert_same_step(msg, s, res_t.cpu().numpy(), ref, np.zeros(n, np.float32))
    assert s == 0 and msg.size == 8 + 2 * 200


def test_deterministic_and_workspace_left_clean():
    n, L = 2_000_003, 500
    dw = _dw(n, 0, 77, False)
    r0 = (torch.randn(n, device="cuda") * 1e-3)
    outs = []
    layer = GpuLayer(n, L, ac.F32)
    tiles = -(-((n + L - 1) // L) // 8)  # eight one-bin warp slices per tile
    hdr, lws = 64, 2112
    for _ in range(3):
        r = r0.clone()
        msg, s = layer.step(r, dw)
        outs.append((msg.tobytes(), s, r.cpu().numpy().tobytes()))
        ws = layer.ws.cpu().numpy()
        # the control block (no deferred corrections pending), the layer's exact-sum
        # buckets and counters, and the per-tile code totals are zero again
        assert not ws[:hdr].any()
        assert not ws[hdr:hdr + 2048 + 16].any()
        tot0 = hdr + lws + 8 * tiles
        assert not ws[tot0:tot0 + 4 * tiles].any()
    assert outs[0] == outs[1] == outs[2]


def test_checkpoint_resume_is_bit_identical(tmp_path):
    n, L = 500_000, 50
    dws = [_dw(n, s, 5, False) for s in range(10)]
    a = GpuLayer(n, L, ac.F32)
    ra = torch.zeros(n, device="cuda")
    for s in range(10):
        msg_a, _ = a.step(ra, dws[s])
    b = GpuLayer(n, L, ac.F32)
    rb = torch.zeros(n, device="cuda")
    for s in range(5):
        b.step(rb, dws[s])
    torch.save(rb.cpu(), tmp_path / "residue.pt")
    del b
    c = GpuLayer(n, L, ac.F32)
    rc = torch.load(tmp_path / "residue.pt").cuda()
    for s in range(5, 10):
        msg_c, _ = c.step(rc, dws[s])
    assert np.array_equal(ra.cpu().numpy().view(np.uint32), rc.cpu().numpy().view(np.uint32))
    assert msg_a.tobytes() == msg_c.tobytes()


@pytest.mark.parametrize("L", [7, 500, 5000], ids=["lookback", "warp-sliced", "block-sliced"])
def test_wait_times_out_with_a_status(L):
    """A tile whose data is never requested (warp- and block-sliced paths) or whose
    look-back descriptor is never published: the bounded waits end, the layer reports
    ADACOMP_ERR_TIMEOUT, and the context stays usable for a normal call afterwards."""
    n = 400_000
    layer = GpuLayer(n, L, ac.F32)
    ac.adacomp_set_timeout_ns(layer.h, 20_000_000)  # 20 ms
    ac.adacomp_set_fault_injection(layer.h, 3)      # tile 3 never publishes
    res_t = torch.zeros(n, device="cuda")
    dw = _dw(n, 0, 9, False)
    ac.adacomp_compress(layer.h, res_t, dw, layer.msg, layer.ws)
    mb, s, st = ac.adacomp_query(layer.h, layer.ws)
    assert st == ac.ERR_TIMEOUT
    # recover: switch the injection off, zero the workspace, run again, match the oracle
    ac.adacomp_set_fault_injection(layer.h)
    layer.ws.zero_()
    res_t.zero_()
    msg, s = layer.step(res_t, dw)
    ref_res = np.zeros(n, np.float32)
    ref = oracle_step(ref_res, dw_host(dw), L)
    assert_same_step(msg, s, res_t.cpu().numpy(), ref, ref_res)

"""CUDA decode-and-accumulate vs the oracle (GPU).

The pages only say that the learners' quantised gradients are combined in
data-parallel training ("AdaComp (Adaptive Residual Gradient Compression)",
abstract and summary paragraph); the library reads this as a plain fp32 sum in
learner order. The bar is bit-exact against the oracle's decoder on the same
message bytes.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from residual_gradient_compression_gb300 import workloads as wl
from _gpu import GpuLayer, dw_host, ensure_built, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _learner_msgs(n, L, K, seed, bf16=False):
    """K learners' messages from the CUDA compressor (itself checked against the
    oracle elsewhere), each with a few steps of carried residue behind it."""
    msgs = []
    layer = GpuLayer(n, L, ac.BF16 if bf16 else ac.F32)
    for k in range(K):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 1000 * k)
        res = torch.randn(n, generator=g, device="cuda") * 1e-3
        dw = torch.randn(n, generator=g, device="cuda") * 1e-3
        if bf16:
            dw = dw.to(torch.bfloat16)
        ac.adacomp_compress(layer.h, res, dw, layer.msg, layer.ws)
        mb, _, st = ac.adacomp_query(layer.h, layer.ws)
        assert st == ac.OK
        buf = torch.zeros(((mb + 15) // 16) * 16, dtype=torch.uint8, device="cuda")
        buf[:mb] = layer.msg[:mb]
        msgs.append((buf, mb))
    return msgs


def _gpu_decode(h, msgs, dense0):
    """msgs: (device buffer, message length) pairs."""
    dense = dense0.clone()
    ws = workspace(h.decode_ws_bytes(len(msgs)))
    ac.adacomp_decode_accumulate(h, [m for m, _ in msgs], [mb for _, mb in msgs], dense, ws)
    return dense.cpu().numpy(), ac.adacomp_decode_status(h, ws)


@pytest.mark.parametrize("n,L,K", [(10, 4, 1), (1, 1, 2), (100_003, 50, 1), (100_003, 50, 3),
                                   (1_000_001, 500, 16), (300_007, 5000, 5), (77_777, 7, 4),
                                   (65_537, 64, 2), (200_003, 500, 40), (123_457, 1000, 3)])
def test_decode_matches_oracle(n, L, K):
    msgs = _learner_msgs(n, L, K, seed=n + L)
    h = ac.adacomp_init_layer(n, L, ac.F32)
    dense0 = torch.randn(n, device="cuda") * 1e-3
    got, st = _gpu_decode(h, msgs, dense0)
    assert st == ac.OK
    ref = dense0.cpu().numpy()
    assert oracle.decode_accumulate(n, L, [m[:mb].cpu().numpy() for m, mb in msgs], ref) == oracle.OK
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_decode_group_matches_per_layer():
    lys = wl.layers("resnet50")[:12]
    K = 3
    h = ac.adacomp_init_group([l.numel for l in lys], [l.bin_len for l in lys], [ac.F32] * len(lys))
    per_layer = [_learner_msgs(l.numel, l.bin_len, K, seed=i) for i, l in enumerate(lys)]
    dense = [torch.zeros(l.numel, device="cuda") for l in lys]
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_accumulate_group(h, [[m for m, _ in pl] for pl in per_layer],
                                       [[mb for _, mb in pl] for pl in per_layer], dense, ws)
    assert ac.adacomp_decode_status(h, ws) == ac.OK
    for l, pl, d in zip(lys, per_layer, dense):
        ref = np.zeros(l.numel, np.float32)
        oracle.decode_accumulate(l.numel, l.bin_len, [m[:mb].cpu().numpy() for m, mb in pl], ref)
        assert np.array_equal(d.cpu().numpy().view(np.uint32), ref.view(np.uint32)), l.name


def _sparse_learner_msgs(n, L, K, seed, keep=0.01):
    """K learners' first-step messages (zero residue) for a dW that is zero except
    for a `keep` fraction of its elements, so that few elements are sent."""
    msgs = []
    layer = GpuLayer(n, L, ac.F32)
    for k in range(K):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 1000 * k)
        dw = torch.randn(n, generator=g, device="cuda") * 1e-3
        dw *= (torch.rand(n, generator=g, device="cuda") < keep).float()
        res = torch.zeros(n, device="cuda")
        ac.adacomp_compress(layer.h, res, dw, layer.msg, layer.ws)
        mb, _, st = ac.adacomp_query(layer.h, layer.ws)
        assert st == ac.OK
        buf = torch.zeros(((mb + 15) // 16) * 16, dtype=torch.uint8, device="cuda")
        buf[:mb] = layer.msg[:mb]
        msgs.append((buf, mb))
    return msgs


def test_decode_group_mixes_streamed_and_in_place_layers():
    """One grouped decode over layers of every kind: warp-sliced (L_T = 50, 500) and
    block-tiled (L_T = 7, 1000) bins, each either streamed through shared memory or,
    when all learners together sent fewer than n/16 codes, summed in place. The
    inputs are checked to cover all four combinations; every layer must match the
    oracle's learner-order sum bit for bit."""
    K = 3
    spec = [(200_003, 50, False), (300_001, 500, True), (50_001, 7, False), (123_457, 1000, True),
            (40_000, 500, False)]
    per_layer = [(_sparse_learner_msgs if sparse else _learner_msgs)(n, L, K, seed=7 * i + 1)
                 for i, (n, L, sparse) in enumerate(spec)]
    kinds = set()
    for (n, L, _), pl in zip(spec, per_layer):
        B = -(-n // L)
        w = 1 if L < 64 else 2
        codes = sum((mb - 8 - 2 * B) // w for _, mb in pl)
        kinds.add((16 <= L <= 509, 16 * codes < n))
    assert kinds == {(True, True), (True, False), (False, True), (False, False)}, kinds
    h = ac.adacomp_init_group([n for n, _, _ in spec], [L for _, L, _ in spec], [ac.F32] * len(spec))
    dense0 = [torch.randn(n, device="cuda") * 1e-3 for n, _, _ in spec]
    dense = [d.clone() for d in dense0]
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_accumulate_group(h, [[m for m, _ in pl] for pl in per_layer],
                                       [[mb for _, mb in pl] for pl in per_layer], dense, ws)
    assert ac.adacomp_decode_status(h, ws) == ac.OK
    for (n, L, _), pl, d0, d in zip(spec, per_layer, dense0, dense):
        ref = d0.cpu().numpy()
        assert oracle.decode_accumulate(n, L, [m[:mb].cpu().numpy() for m, mb in pl], ref) == oracle.OK
        assert np.array_equal(d.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (n, L)


def test_decode_group_mixes_long_and_short_bins():
    """A grouped decode whose layers have bins of 1024 elements or more (L_T = 2048,
    5000: one check task per tile, the lanes over each bin's codes) beside shorter ones
    (L_T = 50, 500: 128-bin tasks over contiguous code runs), so the general check
    kernel takes both branches in one launch; one learner's message of the L_T = 5000
    layer carries a duplicated offset and is rejected alone. Every layer matches the
    oracle's learner-order sum bit for bit."""
    K = 3
    spec = [(200_003, 50, False), (123_457, 5000, False), (80_000, 2048, True), (60_001, 500, False)]
    per_layer = [(_sparse_learner_msgs if sparse else _learner_msgs)(n, L, K, seed=11 * i + 5)
                 for i, (n, L, sparse) in enumerate(spec)]
    # learner 1 of the L_T = 5000 layer: its second code repeats its first
    n5, L5 = spec[1][0], spec[1][1]
    m, mb = per_layer[1][1]
    bad_np, bad_len = _malformed(m[:mb].cpu().numpy(), n5, L5, "duplicate")
    big = torch.zeros(bad_np.size + (1 << 16), dtype=torch.uint8, device="cuda")
    big[:bad_np.size] = torch.from_numpy(bad_np).cuda()
    per_layer[1][1] = (big, bad_len)
    h = ac.adacomp_init_group([n for n, _, _ in spec], [L for _, L, _ in spec], [ac.F32] * len(spec))
    dense0 = [torch.randn(n, device="cuda") * 1e-3 for n, _, _ in spec]
    dense = [d.clone() for d in dense0]
    ws = workspace(h.decode_ws_bytes(K))
    ac.adacomp_decode_accumulate_group(h, [[m for m, _ in pl] for pl in per_layer],
                                       [[mb for _, mb in pl] for pl in per_layer], dense, ws)
    assert ac.adacomp_decode_status(h, ws) == ac.ERR_BAD_MESSAGE
    for i, ((n, L, _), pl, d0, d) in enumerate(zip(spec, per_layer, dense0, dense)):
        ref = d0.cpu().numpy()
        flags = np.zeros(K, np.uint8)
        st = oracle.decode_accumulate(n, L, [m[:mb].cpu().numpy() for m, mb in pl], ref, bad=flags)
        assert list(flags) == ([0, 1, 0] if i == 1 else [0, 0, 0]), (L, list(flags))
        assert st == (oracle.ERR_BAD_MESSAGE if i == 1 else oracle.OK)
        assert np.array_equal(d.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (n, L)


def test_flat100m_sixteen_learners_full_size():
    """The aggregation workload at full size: a flat layer of 10^8 elements at
    L_T = 500, 16 learners each compressing its own N(0, 1e-3) dW (the launch
    configuration the benchmark times), then one decode of all 16 messages. Two of
    the messages are checked against the oracle's compressor byte for byte; the
    decoded gradient against the oracle's decoder of all 16, bit for bit."""
    (ly,) = wl.layers("flat100m")
    n, L, K = ly.numel, ly.bin_len, 16
    layer = GpuLayer(n, L, ac.F32)
    msgs, lens, host_msgs = [], [], []
    for k in range(K):
        res = torch.zeros(n, device="cuda")
        dw = wl.gen_dw("flat100m", 0, ly, 0, learner=k)
        ac.adacomp_compress(layer.h, res, dw, layer.msg, layer.ws)
        mb, s, st = ac.adacomp_query(layer.h, layer.ws)
        assert st == ac.OK
        got = layer.msg[:mb].cpu().numpy()
        if k in (0, K - 1):
            ref = oracle.compress(np.zeros(n, np.float32), dw_host(dw), L)
            assert np.array_equal(got, ref.msg), f"learner {k} message"
        msgs.append(layer.msg[:((mb + 15) // 16) * 16].clone())
        lens.append(mb)
        host_msgs.append(got)
        del dw, res
    dense = torch.zeros(n, device="cuda")
    ws = workspace(layer.h.decode_ws_bytes(K))
    ac.adacomp_decode_accumulate(layer.h, msgs, lens, dense, ws)
    assert ac.adacomp_decode_status(layer.h, ws) == ac.OK
    ref_dense = np.zeros(n, np.float32)
    assert oracle.decode_accumulate(n, L, host_msgs, ref_dense) == oracle.OK
    assert np.array_equal(dense.cpu().numpy().view(np.uint32), ref_dense.view(np.uint32))


def _counts(msg, n, L):
    B = -(-n // L)
    return 8 + 2 * B, np.frombuffer(msg[8:8 + 2 * B].tobytes(), dtype="<u2").astype(np.int64)


def _malformed(good, n, L, kind):
    """A malformed copy of the message bytes `good` (numpy uint8) and the length it claims."""
    w = 1 if L < 64 else 2
    base, counts = _counts(good, n, L)
    bad = good.copy()
    if kind == "wrong_b":
        bad[4] ^= 1
        return bad, bad.size
    if kind == "short":  # too short to hold its counts
        return bad[:8 + counts.size], 8 + counts.size
    if kind == "truncated":
        return bad[:-w], bad.size - w
    if kind == "long":
        return np.concatenate([bad, np.zeros(w, np.uint8)]), bad.size + w
    if kind == "count_too_big":  # a count above its bin's length, the length agreeing with it
        c = min(L, n) + 3
        extra = c - int(counts[0])
        bad[8:10] = np.frombuffer(np.uint16(c).tobytes(), np.uint8)
        return np.concatenate([bad, np.zeros(w * extra, np.uint8)]), bad.size + w * extra
    b = int(np.nonzero(counts >= 2)[0][0])  # a bin with two codes or more
    i = base + w * int(counts[:b].sum())    # its first code
    if kind == "duplicate":                 # its second code repeats the first
        bad[i + w:i + 2 * w] = bad[i:i + w]
        return bad, bad.size
    if kind == "descending":                # its first two codes swapped
        bad[i:i + w] = good[i + w:i + 2 * w]
        bad[i + w:i + 2 * w] = good[i:i + w]
        return bad, bad.size
    if kind == "inflated_count":            # one more code counted and sent: its last code again
        bad[8 + 2 * b:10 + 2 * b] = np.frombuffer(np.uint16(counts[b] + 1).tobytes(), np.uint8)
        j = i + w * (int(counts[b]) - 1)
        bad = np.concatenate([bad[:j + w], bad[j:j + w], bad[j + w:]])
        return bad, bad.size
    raise ValueError(kind)


KINDS = ("wrong_b", "short", "truncated", "long", "count_too_big", "duplicate", "descending", "inflated_count")


@pytest.mark.parametrize("L", [7, 50, 500, 5000])
@pytest.mark.parametrize("kind", KINDS)
def test_malformed_message_adds_nothing(L, kind):
    """Each malformed message sits at the start of a larger zeroed allocation, so no
    read can leave the allocation even before a check, and is decoded with the
    length it claims beside a good message: the call reports ADACOMP_ERR_BAD_MESSAGE,
    the malformed message adds nothing, the good one is added bit for bit as the
    oracle adds it, and the oracle rejects the same message."""
    n = 60_000
    (g0, mb0), (g1, mb1) = _learner_msgs(n, L, 2, seed=3 + L)
    good = g0[:mb0].cpu().numpy()
    bad_np, bad_len = _malformed(g1[:mb1].cpu().numpy(), n, L, kind)
    big = torch.zeros(bad_np.size + (1 << 16), dtype=torch.uint8, device="cuda")
    big[:bad_np.size] = torch.from_numpy(bad_np).cuda()
    h = ac.adacomp_init_layer(n, L, ac.F32)
    dense0 = torch.randn(n, device="cuda") * 1e-3
    got, st = _gpu_decode(h, [(g0, mb0), (big, bad_len)], dense0)
    assert st == ac.ERR_BAD_MESSAGE
    expect = dense0.cpu().numpy()
    flags = np.zeros(2, np.uint8)
    assert oracle.decode_accumulate(n, L, [good, bad_np[:bad_len]], expect, bad=flags) == oracle.ERR_BAD_MESSAGE
    assert list(flags) == [0, 1]
    assert np.array_equal(got.view(np.uint32), expect.view(np.uint32))
    # the same workspace reports OK again on a clean call
    _, st = _gpu_decode(h, [(g0, mb0), (g1, mb1)], dense0)
    assert st == ac.OK


def test_message_length_is_the_one_given():
    """A good message decoded with a length one code too long or too short, or with
    its buffer's length (the buffer holds zeros beyond it), is rejected; with its own
    length it is added."""
    n, L = 40_000, 500
    ((g, mb),) = _learner_msgs(n, L, 1, seed=5)
    h = ac.adacomp_init_layer(n, L, ac.F32)
    big = torch.zeros(mb + 4096, dtype=torch.uint8, device="cuda")
    big[:mb] = g[:mb]
    dense0 = torch.zeros(n, device="cuda")
    for ln, ok in ((mb, True), (mb + 2, False), (mb - 2, False), (big.numel(), False)):
        got, st = _gpu_decode(h, [(big, ln)], dense0)
        assert st == (ac.OK if ok else ac.ERR_BAD_MESSAGE), ln
        assert bool(got.any()) == ok, ln


def test_decode_is_deterministic():
    n, L, K = 2_000_000, 500, 8
    msgs = _learner_msgs(n, L, K, seed=11)
    h = ac.adacomp_init_layer(n, L, ac.F32)
    dense0 = torch.randn(n, device="cuda") * 1e-3
    a, _ = _gpu_decode(h, msgs, dense0)
    b, _ = _gpu_decode(h, msgs, dense0)
    assert a.tobytes() == b.tobytes()

"""adacomp_compress_static_ws, the compress entry point for callers that cannot
allocate device memory, must give exactly what the oracle gives, and what
adacomp_compress gives with a caller-allocated workspace.

Such callers (framework plugins and communication hooks that receive only their
gradient and message buffers, running where the host application's allocator owns
all device memory) get the workspace from a fixed array inside the library instead.
This file runs last so that a failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from _gpu import dw_host, ensure_built, workspace

pytestmark = pytest.mark.gpu


def _entry():
    ensure_built()
    f = ac.lib().adacomp_compress_static_ws
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
    f.restype = ctypes.c_int
    return f


def _parse_result(buf: torch.Tensor):
    raw = buf.cpu().numpy().view(np.uint8)
    s = raw[0:4].view(np.float32)[0]
    status = int(raw[4:8].view(np.uint32)[0])
    nnz = int(raw[8:16].view(np.uint64)[0])
    msg_bytes = int(raw[16:24].view(np.uint64)[0])
    return s, status, nnz, msg_bytes


# warp-sliced tiles (16 <= L_T <= 509) and block tiles with the look-back (L_T < 16,
# whose G is staged in shared memory, and L_T > 509), fp32 and bf16 dW
CASES = [(1_000_003, 500, False), (777_777, 50, True), (100_003, 4, False), (1_000_003, 5000, False),
         (300_007, 700, True)]


@pytest.mark.parametrize("n,L,bf16", CASES)
def test_static_scratch_matches_the_oracle_and_the_workspace_entry_point(n, L, bf16):
    f = _entry()
    h = ac.adacomp_init_layer(n, L, ac.BF16 if bf16 else ac.F32)
    assert h.compress_ws_bytes <= ac.STATIC_WS_BYTES
    stream = torch.cuda.current_stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(n + L)
    r0 = torch.randn(n, generator=g, device="cuda") * 1e-3
    r_ref, r_st = r0.clone(), r0.clone()
    r_host = r0.cpu().numpy().copy()
    msg_ref = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device="cuda")
    msg_st = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device="cuda")
    ws = workspace(h.compress_ws_bytes)
    result = torch.zeros(4, dtype=torch.int64, device="cuda")
    for step in range(2):  # two calls in a row: the second one starts from the first's leftovers
        dw = torch.randn(n, generator=g, device="cuda") * 1e-3
        if bf16:
            dw = dw.to(torch.bfloat16)
        ref = oracle.compress(r_host, dw_host(dw), L)  # r_host carries the oracle's residue
        ac.adacomp_compress(h, r_ref, dw, msg_ref, ws)
        mb_ref, s_ref, st_ref = ac.adacomp_query(h, ws)
        result.fill_(-1)
        st = f(h.ptr, r_st.data_ptr(), dw.data_ptr(), msg_st.data_ptr(), msg_st.numel(),
               result.data_ptr(), stream.cuda_stream)
        assert st == ac.OK, ac.adacomp_status_string(st)
        torch.cuda.synchronize()
        s, status, nnz, mb = _parse_result(result)
        assert status == ac.OK and st_ref == ac.OK
        assert nnz > 0
        # against the oracle: message bytes, s and residue bit for bit
        assert mb == ref.msg.size, f"message length at step {step}"
        assert np.float32(s).view(np.uint32) == np.float32(ref.s).view(np.uint32), f"s at step {step}"
        assert np.array_equal(msg_st[:mb].cpu().numpy(), ref.msg), f"message differs from the oracle at step {step}"
        assert np.array_equal(r_st.cpu().numpy().view(np.uint32), r_host.view(np.uint32)), \
            f"residue differs from the oracle at step {step}"
        # and against the caller-workspace entry point
        assert mb == mb_ref and np.float32(s) == np.float32(s_ref)
        assert torch.equal(msg_st[:mb], msg_ref[:mb]), f"message differs at step {step}"
        assert torch.equal(r_st.view(torch.int32), r_ref.view(torch.int32)), f"residue differs at step {step}"


def test_static_scratch_rejects_layers_that_do_not_fit():
    f = _entry()
    h = ac.adacomp_init_layer(300_000_000, 500, ac.F32)
    assert h.compress_ws_bytes > ac.STATIC_WS_BYTES
    tiny = torch.zeros(16, device="cuda")
    st = f(h.ptr, tiny.data_ptr(), tiny.data_ptr(), tiny.data_ptr(), 16, None,
           torch.cuda.current_stream().cuda_stream)
    assert st == ac.ERR_WORKSPACE


def test_static_scratch_rejects_deferred_fixup_handles():
    """A deferred fix-up keeps state in the workspace between calls, which the fixed
    array cannot hold for the caller."""
    f = _entry()
    h = ac.adacomp_init_layer(10_000, 50, ac.F32)
    ac.adacomp_set_lazy_fixup(h, True)
    r = torch.zeros(10_000, device="cuda")
    msg = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device="cuda")
    st = f(h.ptr, r.data_ptr(), r.data_ptr(), msg.data_ptr(), msg.numel(), None,
           torch.cuda.current_stream().cuda_stream)
    assert st == ac.ERR_INVALID_ARG

"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the
oracle on the same bytes (test helper only)."""
import numpy as np
import torch

import oracle
import residual_gradient_compression_gb300 as ac
from residual_gradient_compression_gb300 import build

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        ac.lib()
        _built = True


def dw_host(dw_t: torch.Tensor) -> np.ndarray:
    """dW on the host as the oracle takes it: fp32, or bf16 bit patterns as uint16."""
    if dw_t.dtype == torch.bfloat16:
        return dw_t.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    return dw_t.cpu().numpy().copy()


def dtype_code(dw_t: torch.Tensor) -> int:
    return ac.BF16 if dw_t.dtype == torch.bfloat16 else ac.F32


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)


class GpuLayer:
    """One layer's handle, message buffer and workspace on the GPU."""

    def __init__(self, n, bin_len, dtype, device="cuda"):
        self.h = ac.adacomp_init_layer(n, bin_len, dtype)
        self.msg = torch.zeros(self.h.max_msg_bytes[0], dtype=torch.uint8, device=device)
        self.ws = workspace(self.h.compress_ws_bytes, device)

    def step(self, residue_t, dw_t):
        ac.adacomp_compress(self.h, residue_t, dw_t, self.msg, self.ws)
        mb, s, st = ac.adacomp_query(self.h, self.ws)
        assert st == ac.OK, ac.adacomp_status_string(st)
        return self.msg[:mb].cpu().numpy(), np.float32(s)


def assert_same_step(gpu_msg, gpu_s, gpu_res, ref, ref_res, where=""):
    assert np.float32(gpu_s).view(np.uint32) == np.float32(ref.s).view(np.uint32), f"s differs {where}"
    assert gpu_msg.size == ref.msg.size, f"message length {gpu_msg.size} != {ref.msg.size} {where}"
    if not np.array_equal(gpu_msg, ref.msg):
        first = int(np.nonzero(gpu_msg != ref.msg)[0][0])
        raise AssertionError(f"message bytes differ first at byte {first} {where}")
    if not np.array_equal(gpu_res.view(np.uint32), ref_res.view(np.uint32)):
        bad = np.nonzero(gpu_res.view(np.uint32) != ref_res.view(np.uint32))[0]
        raise AssertionError(f"residue differs at {bad.size} elements, first {bad[0]} {where}")


def oracle_step(res_np, dw_np, bin_len):
    return oracle.compress(res_np, dw_np, bin_len)

"""Host-side checks of bench.py (no GPU needed): the algorithmic byte counts that
the roofline fractions are computed from, the reference arm's JSON line, and the
profiled-traffic lookup's source check."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _layer(numel, bin_len, dtype="f32"):
    return SimpleNamespace(numel=numel, bin_len=bin_len, dw_dtype=dtype)


def test_stream_bytes_are_residue_dw_residue_and_counts():
    """The streaming kernel must read residue and dW and write residue (12 B per
    element for fp32 dW, 10 B for bf16) and the per-bin counts (2 B per bin)."""
    for dtype, d in (("f32", 4), ("bf16", 2)):
        ly = _layer(1000, 50, dtype)
        stream, _, _ = bench.algorithmic_bytes([ly], [0], 1)
        assert stream == 1000 * (8 + d) + 2 * 20


def test_post_bytes_are_header_codes_and_fix_up():
    """Header (8 B), one code per sent element (1 B below L_T = 64, else 2 B) and a
    read and a write of each sent residue (8 B)."""
    for L, w in ((50, 1), (500, 2)):
        _, post, _ = bench.algorithmic_bytes([_layer(10_000, L)], [123], 1)
        assert post == 8 + w * 123 + 8 * 123


def test_decode_bytes_stream_or_update_in_place():
    """A layer whose learners together sent at least n/16 codes is streamed (8 B per
    element), a sparser one updated in place (8 B per code); the messages are read
    and their counts read once more by the scan."""
    n, L, K = 16_000, 500, 2
    B = n // L
    dense_nnz, sparse_nnz = [600, 400], [300, 200]  # 1000 >= n/16, 500 < n/16
    msg = lambda zs: sum(8 + 2 * B + 2 * z for z in zs)
    _, _, dec = bench.algorithmic_bytes([_layer(n, L)], dense_nnz, K)
    assert dec == 8 * n + msg(dense_nnz) + 2 * B * K
    _, _, dec = bench.algorithmic_bytes([_layer(n, L)], sparse_nnz, K)
    assert dec == 8 * sum(sparse_nnz) + msg(sparse_nnz) + 2 * B * K


def test_learner_major_code_counts():
    """nnz lists learner-major: learner k's count for layer i is nnz[k * layers + i]."""
    lys = [_layer(4000, 50), _layer(8000, 500)]
    nnz = [10, 20, 30, 40]  # learner 0: 10, 20; learner 1: 30, 40
    _, post, _ = bench.algorithmic_bytes(lys, nnz, 2)
    assert post == (8 + 1 * 10 + 80) + (8 + 2 * 20 + 160) + (8 + 1 * 30 + 240) + (8 + 2 * 40 + 320)


def test_profiled_traffic_needs_matching_sources(tmp_path, monkeypatch):
    """A profile summary counts only while the kernel's own sources are unchanged."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"kernel": "slice_kernel", "workload": "w", "source_sha": bench.source_hash("slice_kernel"),
           "dram_bytes_per_launch": 123.0}
    (prof / "slice_kernel_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda kernel=None: rec["source_sha"])
    assert bench.profiled_traffic("slice_kernel", "w", 1000.0) == 123.0
    monkeypatch.setattr(bench, "source_hash", lambda kernel=None: "0" * 16)
    assert bench.profiled_traffic("slice_kernel", "w", 1000.0) is None


def test_profiled_traffic_of_a_smaller_case_is_scaled(tmp_path, monkeypatch):
    """A summary taken on a smaller case scales by the ratio of algorithmic bytes."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"kernel": "block_kernel", "workload": "w", "source_sha": "a" * 16, "dram_bytes_per_launch": 90.0,
           "algorithmic_bytes_per_launch": 100.0, "scale_by_algorithmic_bytes": True}
    (prof / "block_kernel_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda kernel=None: "a" * 16)
    assert bench.profiled_traffic("block_kernel", "w", 1000.0) == 900.0


def test_reference_arm_line():
    """--impl reference times the oracle and prints the contract's keys, with an
    e2e block that moves no bytes between host and device."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "fc400k", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads(out.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "elements/s" and d["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "dtype",
                "data", "config", "cpu_baseline"):
        assert key in d, key
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"

"""Loader for the hand-derived fixtures under tests/golden/ (test helper only)."""
import glob
import json
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def fval(v):
    """A fixture number: a JSON number or a C99 hex-float string (exact)."""
    return float.fromhex(v) if isinstance(v, str) else float(v)


def f32_array(vals):
    out = np.array([fval(v) for v in vals], dtype=np.float64)
    f = out.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), out), "fixture value not exact in fp32"
    return f


def hex_bytes(s):
    return np.frombuffer(bytes.fromhex(s.replace(" ", "")), dtype=np.uint8)


def load(name):
    with open(os.path.join(GOLDEN_DIR, name + ".json")) as fh:
        return json.load(fh)


def compress_cases():
    out = []
    for path in sorted(glob.glob(os.path.join(GOLDEN_DIR, "hand_*.json"))):
        with open(path) as fh:
            case = json.load(fh)
        if "residue" in case:
            out.append(case)
    return out


def case_inputs(case):
    residue = f32_array(case["residue"])
    if case.get("dw_dtype", "f32") == "bf16":
        dw = np.array(case["dw_bits"], dtype=np.uint16)
    else:
        dw = f32_array(case["dw"])
    return residue, dw

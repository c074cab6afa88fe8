"""Pins the oracle to hand-derived worked cases (tests/golden/hand_*.json).

Each fixture is derived by hand from the formulas of "AdaComp (Adaptive Residual
Gradient Compression)", Claims > Mechanism
#r629-local-bin-soft-threshold-and-mean-gmax-quantization, and names the reading it
pins. None of the expected values come from the oracle or the CUDA path.
"""
import numpy as np
import pytest

import oracle
from _golden import compress_cases, case_inputs, f32_array, fval, hex_bytes, load

CASES = compress_cases()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_compress_matches_hand_derivation(case):
    residue, dw = case_inputs(case)
    exp = case["expect"]
    r = oracle.compress(residue, dw, case["bin_len"],
                        literal_zero_select=case.get("literal_zero_select", False),
                        local_selection=case.get("local_selection", False))
    assert r.msg.tobytes() == hex_bytes(exp["msg_hex"]).tobytes()
    assert np.float32(r.s).view(np.uint32) == np.float32(fval(exp["s"])).view(np.uint32)
    assert r.sel.astype(int).tolist() == exp["sel"]
    assert np.array_equal(residue.view(np.uint32), f32_array(exp["residue"]).view(np.uint32))
    if "gmax" in exp:
        assert np.array_equal(r.gmax.view(np.uint32), f32_array(exp["gmax"]).view(np.uint32))
    nb = len(exp["counts"])
    counts = r.msg[8:8 + 2 * nb].view(np.uint16)
    assert counts.tolist() == exp["counts"]
    w = 1 if case["bin_len"] < 64 else 2
    codes = r.msg[8 + 2 * nb:].view(np.uint8 if w == 1 else np.uint16)
    assert codes.tolist() == exp["codes"]


@pytest.mark.parametrize("case", [c for c in CASES if "decode_into_zeros" in c["expect"]],
                         ids=lambda c: c["name"])
def test_decode_single_learner_reproduces_gq(case):
    residue, dw = case_inputs(case)
    r = oracle.compress(residue, dw, case["bin_len"])
    dense = np.zeros(residue.size, np.float32)
    assert oracle.decode_accumulate(residue.size, case["bin_len"], [r.msg], dense) == oracle.OK
    assert np.array_equal(dense, f32_array(case["expect"]["decode_into_zeros"]))


def test_decode_learner_order():
    case = load("hand_decode_learner_order")
    dense = f32_array(case["dense_in"])
    msgs = [hex_bytes(h) for h in case["msgs_hex"]]
    assert oracle.decode_accumulate(case["n"], case["bin_len"], msgs, dense) == oracle.OK
    assert np.array_equal(dense, f32_array(case["expect_dense"]))


def test_decode_rejects_malformed_messages():
    case = load("hand_lt4_n10_partial_bin")
    residue, dw = case_inputs(case)
    good = oracle.compress(residue, dw, 4).msg
    for mutate in ("B", "count", "offset"):
        bad = good.copy()
        if mutate == "B":
            bad[4] = 4                      # header B != ceil(10/4)
        elif mutate == "count":
            bad[8 + 4] = 3                  # bin 2 holds 2 elements, count 3
            bad = np.concatenate([bad, np.zeros(2, np.uint8)])
        else:
            bad[-1] = (2 << 1)              # offset 2 in the 2-element last bin
        dense = np.zeros(10, np.float32)
        assert oracle.decode_accumulate(10, 4, [bad], dense) == oracle.ERR_BAD_MESSAGE
        assert not dense.any()


def test_decode_validation_hand_cases():
    """Every malformed variant of the hand message is rejected and adds nothing; the
    good message beside it is still added (tests/golden/hand_decode_malformed.json)."""
    case = load("hand_decode_malformed")
    n, L = case["n"], case["bin_len"]
    good = hex_bytes(case["good_hex"])
    gq = f32_array(case["good_decode"])
    dense = np.zeros(n, np.float32)
    assert oracle.decode_accumulate(n, L, [good], dense) == oracle.OK
    assert np.array_equal(dense, gq)
    for name, hx in case["bad_hex"].items():
        bad = hex_bytes(hx)
        dense = np.zeros(n, np.float32)
        flags = np.zeros(1, np.uint8)
        assert oracle.decode_accumulate(n, L, [bad], dense, bad=flags) == oracle.ERR_BAD_MESSAGE, name
        assert not dense.any() and flags[0] == 1, name
        dense = np.zeros(n, np.float32)
        flags = np.zeros(2, np.uint8)
        assert oracle.decode_accumulate(n, L, [bad, good], dense, bad=flags) == oracle.ERR_BAD_MESSAGE, name
        assert np.array_equal(dense, gq) and list(flags) == [1, 0], name


def test_decode_length_is_the_one_given():
    """The length that comes with a message decides, not the buffer holding it: the
    good message inside a longer zeroed buffer is accepted with its own length and
    rejected with the buffer's."""
    case = load("hand_decode_malformed")
    good = hex_bytes(case["good_hex"])
    buf = np.zeros(64, np.uint8)
    buf[:good.size] = good
    dense = np.zeros(10, np.float32)
    assert oracle.decode_accumulate(10, 4, [buf], dense, lens=[good.size]) == oracle.OK
    assert np.array_equal(dense, f32_array(case["good_decode"]))
    dense = np.zeros(10, np.float32)
    assert oracle.decode_accumulate(10, 4, [buf], dense, lens=[buf.size]) == oracle.ERR_BAD_MESSAGE
    assert not dense.any()

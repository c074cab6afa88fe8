"""The pins catch plausible mistakes: each mutant of the oracle must fail one of them.

A mutant is a copy of oracle/adacomp_oracle.c with one planted mistake, compiled
into a temporary directory on the CPU. The pins replayed against it are the
hand-derived fixtures, the first-step closed form, the fsum pin of s and the decoder's
message checks; a mutant
that passes them all would mean the pins leave that part of the method unchecked.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from _golden import case_inputs, compress_cases, f32_array, fval, hex_bytes, load

SRC = os.path.join(os.path.dirname(oracle.__file__), "adacomp_oracle.c")

MUTANTS = {
    "strict_threshold": ("fabsf(H[j]) >= gmax[b]", "fabsf(H[j]) > gmax[b]"),
    "h_from_residue_plus_2dw": ("H[j] = G[j] + d;", "H[j] = residue[j] + 2.0f * d;"),
    "sign_from_h": ("(G[j] < 0.0f ? 1u : 0u)", "(H[j] < 0.0f ? 1u : 0u)"),
    "mean_over_full_bins": ("float s = (float)(S / (double)B);",
                            "float s = (float)(S / (double)(n / L > 0 ? n / L : 1));"),
    "left_to_right_fp64_sum": ("double S = adacomp_oracle_exact_sum_f32(gmax, B);",
                               "double S = 0; for (int64_t q = 0; q < B; ++q) S += gmax[q];"),
    "send_zeros": ("int nonzero = G[j] != 0.0f;", "int nonzero = 1;"),
    "width_switch_at_65": ("return L < 64 ? 1 : 2;", "return L <= 64 ? 1 : 2;"),
    "residue_adds_gq": ("if (G[j] > 0.0f) residue[j] = G[j] - s;",
                        "if (G[j] > 0.0f) residue[j] = G[j] + s;"),
    "decode_sign_flipped": ("((code & 1u) ? -s : s)", "((code & 1u) ? s : -s)"),
    "gmax_ignores_partial_bin": ("for (int64_t j = lo; j < hi; ++j)\n            if (fabsf(G[j]) > m)",
                                 "for (int64_t j = lo; j < hi && hi - lo == L; ++j)\n            if (fabsf(G[j]) > m)"),
    "bf16_truncated_to_15_bits": ("(uint32_t)h << 16", "((uint32_t)h << 16) & 0xfffeffffu"),
    "local_selection_keeps_probe": ("if (local_selection) H[j] = G[j];", "if (local_selection) H[j] = H[j];"),
    "sgd_steps_with_old_momentum": ("float delta = lr * v[j];", "float delta = lr * (v[j] - step);"),
    "big_endian_count": ("put_u16(counts + 2 * b, cnt);",
                         "put_u16(counts + 2 * b, ((cnt & 0xff) << 8) | (cnt >> 8));"),
    "duplicate_offsets_accepted": ("if (off >= blen || off <= prev) return 0;",
                                   "if (off >= blen || off < prev) return 0;"),
    "length_unchecked": ("if (len != 8 + 2 * (uint64_t)B + (uint64_t)w * total) return 0;", "(void)total;"),
    "rejected_message_still_added": ("        if (!message_ok(n, L, msgs[k], lens[k])) continue;\n", ""),
    "adam_beta1_swapped": ("float m_keep = beta1 * m[j];\n        float m_add = one_minus_b1 * g;",
                           "float m_keep = one_minus_b1 * m[j];\n        float m_add = beta1 * g;"),
    "adam_no_bias_correction": ("float m_hat = m[j] / bc1;", "float m_hat = m[j];"),
    "adam_eps_inside_sqrt": ("float denom = sqrtf(v_hat) + eps;", "float denom = sqrtf(v_hat + eps);"),
    "adam_v_from_g": ("float g2 = g * g;", "float g2 = g;"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(path), "-lm"])
    return oracle.Oracle(str(so)).lib


def _golden_pins(lib):
    for case in compress_cases():
        residue, dw = case_inputs(case)
        exp = case["expect"]
        r = oracle.compress(residue, dw, case["bin_len"],
                            literal_zero_select=case.get("literal_zero_select", False), lib=lib,
                            local_selection=case.get("local_selection", False))
        assert r.msg.tobytes() == hex_bytes(exp["msg_hex"]).tobytes(), case["name"]
        assert np.float32(r.s) == np.float32(fval(exp["s"])), case["name"]
        assert np.array_equal(residue, f32_array(exp["residue"])), case["name"]
        if "decode_into_zeros" in exp:
            dense = np.zeros(residue.size, np.float32)
            oracle.decode_accumulate(residue.size, case["bin_len"], [r.msg], dense, lib=lib)
            assert np.array_equal(dense, f32_array(exp["decode_into_zeros"])), case["name"]
    case = load("hand_decode_sgd")
    w, v = f32_array(case["w_in"]), f32_array(case["v_in"])
    oracle.decode_sgd(case["n"], case["bin_len"], [hex_bytes(case["msg_hex"])], w, v, case["lr"], case["mu"],
                      case["scale"], lib=lib)
    assert np.array_equal(w, f32_array(case["expect_w"])) and np.array_equal(v, f32_array(case["expect_v"]))
    case = load("hand_decode_adam")
    w, m, v = f32_array(case["w_in"]), f32_array(case["m_in"]), f32_array(case["v_in"])
    oracle.decode_adam(case["n"], case["bin_len"], [hex_bytes(h) for h in case["msgs_hex"]], w, m, v, case["lr"],
                       case["beta1"], case["beta2"], case["eps"], case["bc1"], case["bc2"], case["scale"], lib=lib)
    assert np.array_equal(w, f32_array(case["expect_w"])) and np.array_equal(m, f32_array(case["expect_m"]))
    assert np.array_equal(v, f32_array(case["expect_v"]))
    case = load("hand_decode_learner_order")
    dense = f32_array(case["dense_in"])
    oracle.decode_accumulate(case["n"], case["bin_len"], [hex_bytes(h) for h in case["msgs_hex"]],
                             dense, lib=lib)
    assert np.array_equal(dense, f32_array(case["expect_dense"]))


def _decode_validation_pins(lib):
    case = load("hand_decode_malformed")
    n, L = case["n"], case["bin_len"]
    good = hex_bytes(case["good_hex"])
    gq = f32_array(case["good_decode"])
    for name, hx in case["bad_hex"].items():
        dense = np.zeros(n, np.float32)
        assert oracle.decode_accumulate(n, L, [hex_bytes(hx), good], dense, lib=lib) == oracle.ERR_BAD_MESSAGE, name
        assert np.array_equal(dense, gq), name


def _closed_form_pins(lib):
    rng = np.random.default_rng(3)
    for n, L, bf16 in ((1003, 50, False), (4097, 64, False), (12345, 500, False),
                       (5000, 500, True)):
        dw = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        residue = np.zeros(n, np.float32)
        if bf16:
            bits = (dw.view(np.uint32) >> 16).astype(np.uint16)
            dw = (bits.astype(np.uint32) << 16).view(np.float32)
            r = oracle.compress(residue, bits, L, lib=lib)
        else:
            r = oracle.compress(residue, dw, L, lib=lib)
        nb = -(-n // L)
        pad = np.zeros(nb * L)
        pad[:n] = np.abs(dw)
        gm = pad.reshape(nb, L).max(axis=1)
        sel = (dw != 0) & (2.0 * np.abs(dw) >= np.repeat(gm, L)[:n])
        s = np.float32(math.fsum(gm) / nb)
        assert np.float32(r.s) == s
        assert np.array_equal(r.sel, sel)
        w = 1 if L < 64 else 2
        assert r.msg.size == 8 + 2 * nb + w * sel.sum()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    failures = 0
    for pins in (_golden_pins, _closed_form_pins, _decode_validation_pins):
        try:
            pins(lib)
        except AssertionError:
            failures += 1
    assert failures > 0, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    so = tmp_path / "plain.so"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), SRC, "-lm"])
    lib = oracle.Oracle(str(so)).lib
    _golden_pins(lib)
    _closed_form_pins(lib)
    _decode_validation_pins(lib)

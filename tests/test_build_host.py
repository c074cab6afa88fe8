"""The build's debug variant (no GPU): ADACOMP_DEBUG_CHECKS=1 selects libadacomp_debug.so,
built with -DADACOMP_DEBUG_CHECKS, for the build and the binding alike."""
import os
import subprocess
import sys

from residual_gradient_compression_gb300 import build as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_release_and_debug_builds_are_separate_libraries(monkeypatch):
    monkeypatch.delenv("ADACOMP_DEBUG_CHECKS", raising=False)
    assert b.lib_path() == b.LIB and b.lib_path(True) == b.LIB_DEBUG != b.LIB
    assert "-DADACOMP_DEBUG_CHECKS" not in b.command("x.so")
    monkeypatch.setenv("ADACOMP_DEBUG_CHECKS", "1")
    assert b.lib_path() == b.LIB_DEBUG
    assert "-DADACOMP_DEBUG_CHECKS" in b.command("x.so", debug=True)
    assert all(a in b.command("x.so", debug=True) for a in b.ARCH)


def test_binding_loads_the_selected_library():
    code = ("import residual_gradient_compression_gb300 as ac, os; "
            "print(os.path.basename(ac._LIB_PATH))")
    env = dict(os.environ, ADACOMP_DEBUG_CHECKS="1")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         check=True).stdout.strip()
    assert out == "libadacomp_debug.so"
    env.pop("ADACOMP_DEBUG_CHECKS")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         check=True).stdout.strip()
    assert out == "libadacomp.so"


def test_debug_library_compiles_and_exports_the_abi(tmp_path):
    """The debug variant cross-compiles here (nvcc needs no GPU) and exports every symbol."""
    out = str(tmp_path / "libadacomp_debug_check.so")
    subprocess.check_call(b.command(out, debug=True))
    syms = subprocess.run(["nm", "-D", "--defined-only", out], capture_output=True, text=True, check=True).stdout
    for name in ("adacomp_compress", "adacomp_decode_accumulate", "adacomp_materialize",
                 "adacomp_compress_static_ws"):
        assert f" T {name}" in syms, name

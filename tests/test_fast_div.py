"""The kernel's multiply-high division by launch-fixed divisors (FastDiv, used to
decode key-halves units), checked on the host against integer division: the same
header compiled for the host, run over divisors and dividends across the int range.
No GPU needed (nvcc compiles the host code)."""
import os
import subprocess

from exact_causal_attention_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_fast_division_is_exact(tmp_path):
    exe = str(tmp_path / "fast_div_check")
    subprocess.run([build._nvcc(), "-O2", "-std=c++17", "-I", build.CSRC, "-I", build.INCLUDE,
                    "-o", exe, os.path.join(HERE, "host", "fast_div_check.cu")], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "0 mismatches" in out.stdout

"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle source (a dropped term, a
wrong sign or index, a transposed operand, a flipped mask, a wrong decoder
constant), builds it on the CPU and runs the pin suite against the copy: the
suite has to fail.  The real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_ref.cpp")
SOFTMAX_SRC = os.path.join(ROOT, "oracle", "softmax_ref.cpp")

ATTN = "attn_ref.cpp"
SOFTMAX = "softmax_ref.cpp"
PIN_FILES = [os.path.join(ROOT, "tests", "test_oracle.py"), os.path.join(ROOT, "tests", "test_oracle_softmax.py")]

MUTANTS = {
    "scale_dropped": (ATTN, "s[j] = p.scale * dot;", "s[j] = dot;"),
    "key_transposed": (ATTN, "for (long d = 0; d < p.D; ++d) dot += qi[d] * kj[d];",
                       "for (long d = 0; d < p.D; ++d) dot += qi[d] * kb[(d * p.N + j) % (p.N * p.D)];"),
    "exp_sign_flipped": (ATTN, "for (long j = 0; j <= last; ++j) l += std::exp(s[j] - m);",
                         "for (long j = 0; j <= last; ++j) l += std::exp(m - s[j]);"),
    "mask_strict": (ATTN, "const long last = p.causal ? i : p.N - 1;\n  score_row(p, bh, i, last, s);\n  double m",
                    "const long last = p.causal ? i - 1 : p.N - 1;\n  score_row(p, bh, i, last, s);\n  double m"),
    "no_normalisation": (ATTN, "const double w = std::exp(s[j] - m) / l;", "const double w = std::exp(s[j] - m);"),
    "lse_without_max": (ATTN, "  *lse = m + std::log(l);\n}\n\n// Online", "  *lse = std::log(l);\n}\n\n// Online"),
    "value_row_index": (ATTN, "const double w = std::exp(s[j] - m) / l;\n    const double* vj = vb + j * p.D;",
                        "const double w = std::exp(s[j] - m) / l;\n    const double* vj = vb + i * p.D;"),
    "no_max_subtraction": (ATTN, "const double w = std::exp(s[j] - m) / l;", "const double w = std::exp(s[j]) / l;"),
    "online_no_rescale": (ATTN, "for (long d = 0; d < p.D; ++d) acc[d] *= alpha;", ""),
    "online_beta_dropped": (ATTN, "l = alpha * l + beta * l_tile;", "l = alpha * l + l_tile;"),
    "fp16_exponent_bias": (ATTN, "exponent - 25);", "exponent - 24);"),
    "bf16_hidden_bit": (ATTN, "static_cast<double>(128 + mantissa)", "static_cast<double>(mantissa)"),
    "head_map_modulo": (ATTN, "return b * p.Hkv + h / (p.H / p.Hkv);", "return b * p.Hkv + h % p.Hkv;"),
    "head_map_batch": (ATTN, "return b * p.Hkv + h / (p.H / p.Hkv);", "return b * p.H + h / (p.H / p.Hkv);"),
    "softmax_no_max": (SOFTMAX, "for (long j = 0; j < N; ++j) d += std::exp(x[j] - m);\n  for (long j = 0; j < N; ++j) y[j] = std::exp(x[j] - m) / d;",
                       "for (long j = 0; j < N; ++j) d += std::exp(x[j]);\n  for (long j = 0; j < N; ++j) y[j] = std::exp(x[j]) / d;"),
    "softmax_no_division": (SOFTMAX, "for (long j = 0; j < N; ++j) y[j] = std::exp(x[j] - m) / d;",
                            "for (long j = 0; j < N; ++j) y[j] = std::exp(x[j] - m);"),
    "softmax_recurrence_no_rescale": (SOFTMAX, "s.d * std::exp(s.m - m_new)", "s.d"),
    "softmax_merge_no_rescale": (SOFTMAX, "return State{m, a.d * std::exp(a.m - m) + b.d * std::exp(b.m - m)};",
                                 "return State{m, a.d + b.d};"),
    "softmax_merge_no_empty_guard": (SOFTMAX, "  if (b.d == 0.0) return a;\n  if (a.d == 0.0) return b;\n", ""),
    "softmax_row_stride": (SOFTMAX, "row_two_pass(x + r * N, y + r * N, N);", "row_two_pass(x + r, y + r * N, N);"),
}


def _build_and_run(name, fname, old, new, workdir):
    srcs = {}
    for f in (ATTN, SOFTMAX):
        srcs[f] = open(os.path.join(ROOT, "oracle", f)).read()
    assert old == "" or srcs[fname].count(old) == 1, f"{name}: pattern must occur exactly once"
    srcs[fname] = srcs[fname].replace(old, new)
    paths = []
    for f, text in srcs.items():
        path = os.path.join(workdir, f"{name}_{f}")
        with open(path, "w") as fh:
            fh.write(text)
        paths.append(path)
    lib = os.path.join(workdir, f"lib{name}.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", lib, *paths], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    return name, r.returncode


def test_unmodified_copy_passes_through_the_same_harness():
    workdir = tempfile.mkdtemp(prefix="oracle_control_")
    try:
        assert _build_and_run("control", ATTN, "", "", workdir)[1] == 0
    finally:
        shutil.rmtree(workdir, ignore_errors=True)


def test_every_planted_mistake_fails_a_pin():
    workdir = tempfile.mkdtemp(prefix="oracle_mutants_")
    try:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            results = list(ex.map(lambda kv: _build_and_run(kv[0], *kv[1], workdir), MUTANTS.items()))
    finally:
        shutil.rmtree(workdir, ignore_errors=True)
    survivors = [name for name, rc in results if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"

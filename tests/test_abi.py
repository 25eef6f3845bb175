"""The C ABI without a GPU: the library loads, exports every function that
include/attn.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import exact_causal_attention_gb300 as eca
from exact_causal_attention_gb300 import build

HEADER = os.path.join(build.INCLUDE, "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return eca.load_library()


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    assert "attn_fwd" in names and "attn_fwd_bf16" in names
    assert set(names) == set(eca.SIGNATURES), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_anatomy_build_exports_the_same_symbols(lib):
    """The measurement variant (stamps compiled in) exports every declared function too;
    in the normal build its read-out call refuses."""
    lib2 = ctypes.CDLL(eca.ANATOMY_LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib2, name), name


def test_anatomy_read_refused_in_the_normal_build(lib):
    buf = (ctypes.c_ulonglong * 3200)()
    assert lib.attn_anatomy_read(buf, 3200, 0) == -1


def test_version_and_status_strings(lib):
    assert lib.attn_version() >= 100
    for code, name in eca.STATUS.items():
        text = lib.attn_status_string(code).decode()
        assert text and text != "unknown status", name
    assert lib.attn_status_string(12345).decode() == "unknown status"


# Fake, never-dereferenced addresses: every case below must be refused by the
# host-side checks, which run before the library touches CUDA.
A = 0x10000000
SZ = 1 << 24


def call(lib, fn="attn_fwd", q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=None, B=1, H=1, N=16, D=64,
         causal=1, scale=0.125):
    return getattr(lib, fn)(q, k, v, o, lse, B, H, N, D, causal, scale, None)


@pytest.mark.parametrize("fn", ["attn_fwd", "attn_fwd_bf16"])
def test_argument_errors_without_gpu(lib, fn):
    assert call(lib, fn, q=None) == -1
    assert call(lib, fn, o=None) == -1
    assert call(lib, fn, B=0) == -1
    assert call(lib, fn, H=-3) == -1
    assert call(lib, fn, N=0) == -1
    assert call(lib, fn, D=96) == -3
    assert call(lib, fn, D=256) == -3
    assert call(lib, fn, scale=0.0) == -1
    assert call(lib, fn, scale=-0.5) == -1
    assert call(lib, fn, scale=float("inf")) == -1
    assert call(lib, fn, scale=float("nan")) == -1
    assert call(lib, fn, q=A + 2) == -2
    assert call(lib, fn, o=A + 3 * SZ + 8) == -2
    assert call(lib, fn, lse=A + 4 * SZ + 2) == -2
    # o overlapping an input
    assert call(lib, fn, o=A + 16) == -1
    # grid / tensor-map limits
    assert call(lib, fn, B=1 << 16, H=1 << 16) == -1


def test_selftest_rejects_bad_timeouts(lib):
    assert lib.attn_watchdog_selftest(0, None) == -1
    assert lib.attn_watchdog_selftest(10_000_001, None) == -1


def test_binding_rejects_cpu_tensors():
    import torch

    x = torch.zeros(1, 1, 4, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        eca.attn_fwd(x, x, x)
    # attn_fwd_into's quick check declines what it cannot pass and the full checks raise
    lse = torch.zeros(1, 1, 4)
    with pytest.raises(TypeError):
        eca.attn_fwd_into(x, x, x, torch.empty_like(x), lse)
    with pytest.raises((TypeError, ValueError)):
        eca.attn_fwd_into(x[0], x[0], x[0], torch.empty_like(x[0]), None)


def test_splitkv_workspace_size_without_gpu(lib):
    ws = lib.attn_splitkv_workspace_bytes
    # [splits, BH, N, D] fp32 outputs + [splits, BH, N] fp32 lse, each rounded up to 256 bytes
    assert ws(1, 2, 256, 64, 2) == 2 * 2 * 256 * 64 * 4 + 2 * 2 * 256 * 4
    assert ws(1, 1, 1, 128, 4) == 512 + 256  # one key tile: one segment; 512 B of o, 4 B of lse -> 256
    assert ws(1, 1, 1000, 64, 64) == 8 * 1000 * 64 * 4 + ((8 * 1000 * 4 + 255) // 256) * 256  # 8 key tiles
    assert ws(0, 1, 256, 64, 2) == 0 and ws(1, 1, 256, 96, 2) == 0 and ws(1, 1, 256, 64, 0) == 0
    assert ws(1, 1, 256, 64, 65) == 0
    # the longest sequence an int holds: 2^24 key tiles (tile counts taken without overflow)
    n = 2 ** 31 - 1
    assert ws(1, 1, n, 64, 2) == 2 * n * 64 * 4 + ((2 * n * 4 + 255) // 256) * 256


@pytest.mark.parametrize("fn", ["attn_fwd_splitkv", "attn_fwd_splitkv_bf16"])
def test_splitkv_argument_errors_without_gpu(lib, fn):
    f = getattr(lib, fn)
    W = A + 8 * SZ

    def c(splits=2, ws=W, wsb=1 << 30, **kw):
        a = dict(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=None, B=1, H=1, N=512, D=64, causal=1,
                 scale=0.125)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"], a["causal"],
                 a["scale"], splits, ws, wsb, None)

    assert c(splits=0) == -1
    assert c(splits=65) == -1
    assert c(ws=None) == -1
    assert c(ws=W + 16) == -2
    assert c(wsb=100) == -1
    assert c(ws=A) == -1  # workspace overlapping q
    assert c(D=96) == -3


def test_noalloc_argument_errors_without_gpu(lib):
    """attn_fwd_splitkv_noalloc refuses bad split counts, the usual argument errors and
    a split whose partials need more than its fixed 64 MiB scratch, all before any CUDA
    call (the addresses here are never dereferenced)."""
    f = lib.attn_fwd_splitkv_noalloc

    def c(splits=2, **kw):
        a = dict(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=None, B=1, H=1, N=512, D=64, causal=1,
                 scale=0.125)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"], a["causal"],
                 a["scale"], splits, None)

    assert c(splits=0) == -1
    assert c(splits=65) == -1
    assert c(q=None) == -1
    assert c(D=96) == -3
    assert c(q=A + 2) == -2
    assert c(o=A + 16) == -1
    # 4 segments of B*H*N*D fp32 partials: 4 * 8 * 8192 * 128 * 4 B = 128 MiB > 64 MiB
    big = 8 * 8192 * 128 * 2
    assert c(splits=4, q=A, k=A + big, v=A + 2 * big, o=A + 3 * big, H=8, N=8192, D=128) == -8


def test_splitkv_adjacent_workspace_is_not_overlap(lib):
    # q, k, v, o of 1*1*512*64*2 = 64 KiB each; a workspace starting right after o is legal.
    io = 512 * 64 * 2
    q, k, v, o = A, A + io, A + 2 * io, A + 3 * io
    ws = A + 4 * io
    need = lib.attn_splitkv_workspace_bytes(1, 1, 512, 64, 2)
    rc = lib.attn_fwd_splitkv(q, k, v, o, None, 1, 1, 512, 64, 1, 0.125, 2, ws, need, None)
    assert rc not in (-1, -2, -3)  # passes the argument checks (then needs a GPU)
    rc = lib.attn_fwd_splitkv(q, k, v, o, None, 1, 1, 512, 64, 1, 0.125, 2, o, need, None)
    assert rc == -1  # workspace on top of o


@pytest.mark.parametrize("fn", ["attn_fwd_gqa", "attn_fwd_gqa_bf16"])
def test_gqa_argument_errors_without_gpu(lib, fn):
    f = getattr(lib, fn)
    args = lambda H, Hkv, D=64: (A, A + SZ, A + 2 * SZ, A + 3 * SZ, None, 1, H, Hkv, 256, D, 1, 0.125, None)
    assert f(*args(8, 3)) == -1  # 3 does not divide 8
    assert f(*args(8, 0)) == -1
    assert f(*args(8, 16)) == -1
    assert f(*args(8, 2, 96)) == -3


def test_row_softmax_argument_errors_without_gpu(lib):
    f = lib.attn_row_softmax_f32
    assert f(None, A, 4, 8, None) == -1
    assert f(A, A + SZ, 0, 8, None) == -1
    assert f(A, A + SZ, 4, 0, None) == -1
    assert f(A + 1, A + SZ, 4, 8, None) == -2
    assert f(A, A + 16, 4, 8, None) == -1  # y overlaps x without being x


def g_rows_limit(lib, C, BT, LN):
    """attn_paged_append on a cache of 2^31 token rows (checked before any CUDA call)."""
    return lib.attn_paged_append(A, C, BT, LN, 2, 2, 128, 64, 4, 1 << 24, None)


def test_paged_argument_errors_without_gpu(lib):
    f = lib.attn_decode_paged
    Q, C, BT, LN, O, W = A, A + SZ, A + 2 * SZ, A + 3 * SZ, A + 4 * SZ, A + 6 * SZ

    def c(B=2, Hq=8, Hkv=2, D=128, T=16, mp=4, np_=8, scale=0.1, splits=1, ws=None, wsb=0, q=Q, bt=BT):
        return f(q, C, bt, LN, O, None, B, Hq, Hkv, D, T, mp, np_, scale, splits, ws, wsb, None)

    assert c(Hkv=3) == -1
    assert c(D=96) == -3
    assert c(T=12) == -1
    assert c(splits=0) == -1
    assert c(splits=65) == -1
    assert c(splits=2, mp=16) == -1  # a real split (16 pages = 4 tiles) needs a workspace
    assert c(splits=2, mp=16, ws=W + 8, wsb=1 << 20) == -2
    assert c(scale=-1.0) == -1
    assert c(q=Q + 2) == -2
    assert c(bt=BT + 2) == -2
    assert c(T=64, np_=1 << 24) == -1  # 2^31 token rows: past 32-bit tensor coordinates
    assert g_rows_limit(lib, C, BT, LN) == -1
    assert lib.attn_decode_workspace_bytes(2, 8, 128, 1) == 0
    assert lib.attn_decode_workspace_bytes(2, 8, 128, 4) == 4 * 2 * 8 * 128 * 4 + 256
    g = lib.attn_paged_append
    assert g(None, C, BT, LN, 2, 2, 128, 16, 4, 8, None) == -1
    assert g(A + 8, C, BT, LN, 2, 2, 128, 16, 4, 8, None) == -2
    assert g(A, C, BT, LN, 2, 2, 128, 24, 4, 8, None) == -1


def test_header_compiles_as_c_and_links_every_entry_point(lib, tmp_path):
    """A plain C11 program (tests/host/c_abi_check.c) includes include/attn.h, takes the
    address of every declared entry point from the built library and calls those that
    need no GPU."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    so_dir = os.path.dirname(build.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "host", "c_abi_check.c")
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", build.INCLUDE, "-o", exe, src,
                    "-L", so_dir, "-l:" + os.path.basename(build.LIB_PATH), f"-Wl,-rpath,{so_dir}"], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    names = declared_functions()
    assert f"entry points {len(names)}," in out.stdout, (out.stdout, names)


@pytest.mark.parametrize("probe", ["launch_cost_probe", "ingress_probe"])
def test_measurement_probes_compile(tmp_path, probe):
    """The probes `bench.py --launch-cost` and `--ingress` build and run on the GPU machine
    compile for sm_103a here (no GPU needed to compile)."""
    import subprocess

    src = os.path.join(build.CSRC, probe + ".cu")
    subprocess.run([build._nvcc(), *build.ARCH_FLAGS, "-O2", "-std=c++17", "-o", str(tmp_path / probe), src],
                   check=True)

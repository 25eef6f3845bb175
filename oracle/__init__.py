"""FP64 CPU oracle for exact scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``, never by the product package.  It shares no
code with the CUDA path (no headers, helpers or constants); both sides only read
the same seeded inputs.

The arithmetic lives in ``attn_ref.cpp`` (two-pass definition and the online
recurrence of "CUDA FlashAttention：从在线 Softmax 到长序列 IO 极限", sections 1, 3
and 4).  ``pyref`` holds a pure-Python ``math.fsum`` restatement for tiny shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "attn_ref.cpp"), os.path.join(_HERE, "softmax_ref.cpp")]
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_TWO_PASS = 0
MODE_ONLINE = 1
DTYPE_CODES = {"fp16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle shared library with the host C++ compiler."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(f) for f in _SRCS)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", tmp, *_SRCS]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test that plants a mistake in a copy of the oracle points this at the copy.
            override = os.environ.get("ORACLE_LIB_OVERRIDE")
            lib = ctypes.CDLL(override if override else build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_decode.argtypes = [ctypes.c_void_p, dp, ctypes.c_long, ctypes.c_int, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                            ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_long, ctypes.c_int]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                             ctypes.POINTER(ctypes.c_long), ctypes.c_long, dp, dp,
                                             ctypes.c_int]
            lib.oracle_attn_rows.restype = ctypes.c_int
            lib.oracle_softmax.argtypes = [dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_long,
                                           ctypes.c_int]
            lib.oracle_softmax.restype = ctypes.c_int
            _lib = lib
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def decode(bits: np.ndarray, dtype: str, nthreads: int = 0) -> np.ndarray:
    """Exact value of each fp16 / bf16 bit pattern (uint16 array) as float64."""
    bits = np.ascontiguousarray(bits).view(np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = _load().oracle_decode(bits.ctypes.data, _dptr(out), bits.size, DTYPE_CODES[dtype], nthreads)
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape:
        raise ValueError("q is [B, H, N, D]; k and v share one [B, Hkv, N, D] shape")
    B, H, N, D = q.shape
    if k.shape[0] != B or k.shape[2:] != (N, D) or k.shape[1] < 1 or H % k.shape[1] != 0:
        raise ValueError("k, v must be [B, Hkv, N, D] with Hkv dividing H")
    return B, H, k.shape[1], N, D


def attention(q, k, v, causal: bool, scale: float, mode: str = "two_pass", tile: int = 128,
              nthreads: int = 0):
    """O [B,H,N,D] and lse [B,H,N] in float64.  q is [B,H,N,D]; k, v are [B,Hkv,N,D] with Hkv
    dividing H (query head h reads key/value head h // (H // Hkv))."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, N, D = _shapes(q, k, v)
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    m = {"two_pass": MODE_TWO_PASS, "online": MODE_ONLINE}[mode]
    rc = _load().oracle_attn_fwd(_dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), B, H, Hkv, N, D,
                                 int(bool(causal)), float(scale), m, int(tile), nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def attention_rows(q, k, v, causal: bool, scale: float, rows, nthreads: int = 0):
    """O and lse of selected rows only; rows is a sequence of (b*H + h, i) pairs."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, N, D = _shapes(q, k, v)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    o = np.empty((r.shape[0], D), dtype=np.float64)
    lse = np.empty((r.shape[0],), dtype=np.float64)
    rc = _load().oracle_attn_rows(_dptr(q), _dptr(k), _dptr(v), B, H, Hkv, N, D, int(bool(causal)),
                                  float(scale), r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                  r.shape[0], _dptr(o), _dptr(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return o, lse


def attention_from_bits(qb, kb, vb, dtype: str, causal: bool, scale: float, nthreads: int = 0,
                        rows=None):
    """Decode fp16/bf16 bit patterns exactly, then run the two-pass oracle (all rows or `rows`)."""
    q, k, v = (decode(x, dtype, nthreads) for x in (qb, kb, vb))
    if rows is None:
        return attention(q, k, v, causal, scale, nthreads=nthreads)
    return attention_rows(q, k, v, causal, scale, rows, nthreads=nthreads)


def softmax(x, mode: str = "two_pass", tile: int = 64, nthreads: int = 0) -> np.ndarray:
    """Row softmax of a float64-convertible [M, N] matrix, in float64 (``softmax_ref.cpp``)."""
    x = _f64(x)
    if x.ndim != 2:
        raise ValueError("x must be [M, N]")
    y = np.empty_like(x)
    m = {"two_pass": MODE_TWO_PASS, "online": MODE_ONLINE}[mode]
    rc = _load().oracle_softmax(_dptr(x), _dptr(y), x.shape[0], x.shape[1], m, int(tile), nthreads)
    if rc != 0:
        raise ValueError("oracle_softmax rejected its arguments")
    return y


# ------------------------------------------------------------- paged KV cache

def gather_paged(cache, block_table, lengths, page_size: int):
    """Logical K and V of each request from a paged cache (page "CUDA KV Cache：分页存储
    与长上下文 Decode 极致优化", section 2): cache is [P, 2, T, Hkv, D]; token t of
    request b sits on physical page block_table[b, t // T] at offset t % T.
    Returns a list of (k, v), each [Hkv, lengths[b], D] float64."""
    cache = np.asarray(cache)
    out = []
    for b, L in enumerate(np.asarray(lengths).tolist()):
        t = np.arange(L)
        pages = np.asarray(block_table)[b, t // page_size]
        offs = t % page_size
        k = cache[pages, 0, offs].astype(np.float64)  # [L, Hkv, D]
        v = cache[pages, 1, offs].astype(np.float64)
        out.append((np.ascontiguousarray(k.transpose(1, 0, 2)), np.ascontiguousarray(v.transpose(1, 0, 2))))
    return out


def decode_paged(q, cache, block_table, lengths, page_size: int, scale: float, nthreads: int = 0):
    """One decode query per request against its whole paged context: O [B, Hq, D] and
    lse [B, Hq] in float64.  The query attends every one of its lengths[b] tokens, which
    is the last row of the causal attention over the logical sequence; a request with no
    token gets O = 0 and lse = -inf."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    o = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    for b, (k, v) in enumerate(gather_paged(cache, block_table, lengths, page_size)):
        L = k.shape[1]
        if L == 0:
            continue
        qq = np.zeros((1, Hq, L, D))
        qq[0, :, L - 1] = q[b]
        ob, lb = attention_rows(qq, k[None], v[None], True, scale, [(h, L - 1) for h in range(Hq)],
                                nthreads=nthreads)
        o[b], lse[b] = ob, lb
    return o, lse

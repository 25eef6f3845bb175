"""Exact causal / non-causal attention forward on sm_103a (GB300).

Thin ctypes binding over the C ABI in ``include/attn.h``: it checks and marshals
torch tensors into pointers and sizes and calls the library; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the
shared library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["attn_fwd", "attn_fwd_into", "attn_fwd_gqa", "attn_fwd_splitkv", "splitkv_workspace_bytes",
           "splitkv_default_splits", "row_softmax", "decode_paged", "paged_append", "load_library", "device_status", "watchdog_selftest", "AttnError",
           "STATUS"]

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libeca_attn.so")
# The same library with the attention kernel's per-CTA milestone stamps compiled in.
ANATOMY_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libeca_attn_anatomy.so")
_lock = threading.Lock()
_lib = None

STATUS = {
    0: "ATTN_OK",
    -1: "ATTN_ERR_INVALID_ARG",
    -2: "ATTN_ERR_UNALIGNED",
    -3: "ATTN_ERR_UNSUPPORTED_D",
    -4: "ATTN_ERR_ARCH",
    -5: "ATTN_ERR_LAUNCH",
    -6: "ATTN_ERR_TIMEOUT",
    -7: "ATTN_ERR_CUDA",
    -8: "ATTN_ERR_SCRATCH_LIMIT",
    -9: "ATTN_ERR_BAD_INDEX",
}

# Every exported symbol of include/attn.h with its ctypes signature.
_VP, _I, _F, _U, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _VP]),
    "attn_fwd_bf16": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _VP]),
    "attn_fwd_gqa": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "attn_fwd_gqa_bf16": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "attn_fwd_splitkv": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _VP, _SZ, _VP]),
    "attn_fwd_splitkv_bf16": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _VP, _SZ, _VP]),
    "attn_fwd_splitkv_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _VP]),
    "attn_splitkv_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_splitkv_default_splits": (_I, [_I, _I, _I, _I]),
    "attn_row_softmax_f32": (_I, [_VP, _VP, ctypes.c_longlong, _I, _VP]),
    "attn_decode_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _F, _I, _VP, _SZ, _VP]),
    "attn_decode_paged_bf16": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _F, _I, _VP, _SZ,
                                    _VP]),
    "attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "attn_decode_default_splits": (_I, [_I, _I, _I, _I, _I]),
    "attn_paged_append": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP]),
    "attn_device_status": (_I, [_VP]),
    "attn_watchdog_selftest": (_I, [_U, _VP]),
    "attn_anatomy_read": (_I, [ctypes.POINTER(ctypes.c_ulonglong), _SZ, _I]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_version": (_I, []),
}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_status_text(status)})")


def _status_text(status: int) -> str:
    try:
        return load_library().attn_status_string(status).decode()
    except Exception:  # library missing while formatting an error
        return "?"


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load the CUDA library (built by ``exact_causal_attention_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"CUDA library not built: {p} is missing "
                                   "(run python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_qkv(q, k, v):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, D]")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("q, k, v must all be float16 or all bfloat16")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")


_raw_stream_fn = None


def _raw_stream(device_index: int, stream) -> int:
    """cudaStream_t of ``stream``, or of torch's current stream on the device, as an int.
    torch's raw-stream query skips building a Stream object, which costs microseconds."""
    global _raw_stream_fn
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if _raw_stream_fn is None:
        import torch

        fn = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream_fn = fn if fn is not None else (lambda i: torch.cuda.current_stream(i).cuda_stream)
    return _raw_stream_fn(device_index)


def _fwd_fast(q, k, v, o, lse, causal, scale, stream) -> bool:
    """The common call, checked with few attribute reads: q, k, v, o contiguous CUDA
    tensors of one shape, 16-bit type and device (the current one), lse None or
    contiguous fp32 [B, H, N] there.  Returns False, having launched nothing, for
    anything else, which the checked path then reports."""
    import torch

    try:
        shape = q.shape
        dt = q.dtype
        dev = q.get_device()
        if (len(shape) != 4 or dev < 0 or dt not in (torch.float16, torch.bfloat16)
                or k.shape != shape or v.shape != shape or o.shape != shape
                or k.dtype != dt or v.dtype != dt or o.dtype != dt
                or k.get_device() != dev or v.get_device() != dev or o.get_device() != dev
                or not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous() and o.is_contiguous())):
            return False
        if lse is not None and (lse.dtype != torch.float32 or lse.shape != shape[:3] or lse.get_device() != dev
                                or not lse.is_contiguous()):
            return False
        if torch._C._cuda_getDevice() != dev:
            return False
    except (AttributeError, TypeError):
        return False
    B, H, N, D = shape
    lib = load_library()
    fn = lib.attn_fwd_bf16 if dt == torch.bfloat16 else lib.attn_fwd
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr() if lse is not None else None,
            B, H, N, D, 1 if causal else 0, 1.0 / math.sqrt(D) if scale is None else float(scale),
            _raw_stream(dev, stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd")
    return True


def attn_fwd_into(q, k, v, o, lse, causal: bool = True, scale: float | None = None, stream=None) -> None:
    """Write O into ``o`` ([B,H,N,D], q's dtype) and the natural-log LSE into ``lse``
    ([B,H,N] float32, or None) on ``stream`` (default: torch's current stream)."""
    import torch

    if _fwd_fast(q, k, v, o, lse, causal, scale, stream):
        return
    _check_qkv(q, k, v)
    B, H, N, D = q.shape
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or o.device != q.device:
        raise ValueError("o must be a contiguous tensor shaped and typed like q")
    if lse is not None and (lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous()
                            or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lib = load_library()
    fn = lib.attn_fwd_bf16 if q.dtype == torch.bfloat16 else lib.attn_fwd
    with torch.cuda.device(q.device):
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                lse.data_ptr() if lse is not None else None, B, H, N, D, int(bool(causal)),
                float(scale), _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd")


def attn_fwd(q, k, v, causal: bool = True, scale: float | None = None, return_lse: bool = True,
             stream=None):
    """O = softmax(scale * q k^T + mask) v (and the row LSE) for [B, H, N, D] CUDA tensors."""
    import torch

    _check_qkv(q, k, v)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if return_lse else None
    attn_fwd_into(q, k, v, o, lse, causal=causal, scale=scale, stream=stream)
    return (o, lse) if return_lse else o


def attn_fwd_gqa(q, k, v, causal: bool = True, scale: float | None = None, o=None, lse=None, stream=None):
    """Grouped-head attention: q [B,H,N,D], k and v [B,Hkv,N,D] with Hkv dividing H; query head h
    reads key/value head h // (H // Hkv).  Returns (o, lse)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
    B, H, N, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or tuple(k.shape[2:]) != (N, D):
        raise ValueError("k, v must be [B, Hkv, N, D] matching q's B, N, D")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("q, k, v must all be float16 or all bfloat16")
    Hkv = k.shape[1]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lib = load_library()
    fn = lib.attn_fwd_gqa_bf16 if q.dtype == torch.bfloat16 else lib.attn_fwd_gqa
    with torch.cuda.device(q.device):
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, N, D,
                int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_gqa")
    return o, lse


def splitkv_workspace_bytes(B: int, H: int, N: int, D: int, kv_splits: int) -> int:
    """Workspace bytes attn_fwd_splitkv needs (0 for invalid sizes)."""
    return int(load_library().attn_splitkv_workspace_bytes(B, H, N, D, kv_splits))


def splitkv_default_splits(B: int, H: int, N: int, D: int) -> int:
    rc = load_library().attn_splitkv_default_splits(B, H, N, D)
    if rc < 0:
        raise AttnError(rc, "attn_splitkv_default_splits")
    return rc


def attn_fwd_splitkv(q, k, v, o=None, lse=None, kv_splits: int | None = None, workspace=None,
                     causal: bool = True, scale: float | None = None, stream=None):
    """attn_fwd with the key tiles split into kv_splits segments merged by a second
    kernel.  The fp32 workspace comes from the caller (a uint8 CUDA tensor) or is
    allocated here with torch.  Returns (o, lse)."""
    import torch

    _check_qkv(q, k, v)
    B, H, N, D = q.shape
    if kv_splits is None:
        with torch.cuda.device(q.device):
            kv_splits = splitkv_default_splits(B, H, N, D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = splitkv_workspace_bytes(B, H, N, D, kv_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1) + 256, dtype=torch.uint8, device=q.device)
        off = (-workspace.data_ptr()) % 256
        workspace = workspace[off:off + max(need, 1)]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lib = load_library()
    fn = lib.attn_fwd_splitkv_bf16 if q.dtype == torch.bfloat16 else lib.attn_fwd_splitkv
    with torch.cuda.device(q.device):
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                lse.data_ptr() if lse is not None else None, B, H, N, D, int(bool(causal)), float(scale),
                int(kv_splits), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_splitkv")
    return o, lse


def row_softmax(x, out=None, stream=None):
    """Row softmax of a contiguous 2-D float32 CUDA tensor (online (m, d) kernel)."""
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dim() != 2 or x.dtype != torch.float32:
        raise TypeError("x must be a 2-D float32 CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if out is None:
        out = torch.empty_like(x)
    M, N = x.shape
    with torch.cuda.device(x.device):
        rc = load_library().attn_row_softmax_f32(x.data_ptr(), out.data_ptr(), M, N, _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_row_softmax_f32")
    return out


def decode_paged(q, cache, block_table, lengths, scale: float | None = None, kv_splits: int | None = None,
                 out=None, lse=None, workspace=None, stream=None):
    """One decode step over a paged cache: q [B,Hq,D], cache [P,2,T,Hkv,D] (16-bit),
    block_table [B,max_pages] int32, lengths [B] int32 (all CUDA).  Returns (out, lse)."""
    import torch

    B, Hq, D = q.shape
    P, two, T, Hkv, D2 = cache.shape
    if two != 2 or D2 != D or q.dtype != cache.dtype or q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("cache must be [P, 2, T, Hkv, D] in q's dtype")
    if block_table.dtype != torch.int32 or lengths.dtype != torch.int32 or block_table.shape[0] != B:
        raise ValueError("block_table [B, max_pages] and lengths [B] must be int32")
    for t in (q, cache, block_table, lengths):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    max_pages = block_table.shape[1]
    lib = load_library()
    with torch.cuda.device(q.device):
        if kv_splits is None:
            kv_splits = lib.attn_decode_default_splits(B, Hq, Hkv, T, max_pages)
            if kv_splits < 0:
                raise AttnError(kv_splits, "attn_decode_default_splits")
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        need = int(lib.attn_decode_workspace_bytes(B, Hq, D, kv_splits))
        if workspace is None and need > 0:
            raw = torch.empty(need + 256, dtype=torch.uint8, device=q.device)
            off = (-raw.data_ptr()) % 256
            workspace = raw[off:off + need]
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        fn = lib.attn_decode_paged_bf16 if q.dtype == torch.bfloat16 else lib.attn_decode_paged
        rc = fn(q.data_ptr(), cache.data_ptr(), block_table.data_ptr(), lengths.data_ptr(), out.data_ptr(),
                lse.data_ptr() if lse is not None else None, B, Hq, Hkv, D, T, max_pages, P, float(scale),
                int(kv_splits), workspace.data_ptr() if workspace is not None else None,
                (workspace.numel() if workspace is not None else 0), _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_decode_paged")
    return out, lse


def paged_append(new_kv, cache, block_table, lengths, stream=None) -> None:
    """Write new_kv [B, 2, Hkv, D] at position lengths[b] - 1 of every request's pages."""
    import torch

    B, two, Hkv, D = new_kv.shape
    P, _, T, _, _ = cache.shape
    with torch.cuda.device(cache.device):
        rc = load_library().attn_paged_append(new_kv.data_ptr(), cache.data_ptr(), block_table.data_ptr(),
                                              lengths.data_ptr(), B, Hkv, D, T, block_table.shape[1], P,
                                              _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_paged_append")


def device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word (0 = ok)."""
    return load_library().attn_device_status(_stream_handle(stream))


def watchdog_selftest(timeout_us: int, stream=None) -> None:
    rc = load_library().attn_watchdog_selftest(int(timeout_us), _stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_watchdog_selftest")

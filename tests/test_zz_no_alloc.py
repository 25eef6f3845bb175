"""The allocation-free split entry point, attn_fwd_splitkv_noalloc.

It serves callers that may not allocate device memory themselves (their memory
belongs to a host framework's pool, or an allocation call is too costly on their
path): the partial results go to the library's fixed per-device scratch array
instead of a caller workspace.  Each check calls it through the C ABI and
compares with attn_fwd_splitkv, the entry point that takes a caller workspace,
and with the FP64 oracle, on two calls in a row with different data, so stale
scratch contents from the first call would show up in the second.  This file is
collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from exact_causal_attention_gb300 import inputs

from helpers import compare, oracle_full

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, lse, causal, scale, splits):
    B, H, N, D = q.shape
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        B, H, N, D, int(causal), float(scale), int(splits),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_split_matches_workspace_split_on_two_calls(cuda_lib):
    eca = cuda_lib
    lib = eca.load_library()
    B, H, N, D, splits = 1, 4, 2304, 128, 4
    scale = 1.0 / math.sqrt(D)
    for call, seed in enumerate((71, 72)):
        hq, hk, hv = inputs.make_qkv(B, H, N, D, "fp16", seed=seed, qk_std=1.5)
        q, k, v = hq.cuda(), hk.cuda(), hv.cuda()
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, q, k, v, o, lse, True, scale, splits) == 0, f"call {call}"
        ref_o, ref_lse = eca.attn_fwd_splitkv(q, k, v, kv_splits=splits, causal=True, scale=scale)
        torch.cuda.synchronize()
        assert eca.device_status() == 0
        og, rg = o.double().cpu().numpy(), ref_o.double().cpu().numpy()
        lg, rl = lse.double().cpu().numpy(), ref_lse.double().cpu().numpy()
        assert np.isfinite(og).all() and np.isfinite(lg).all(), f"call {call}: unwritten output"
        # the tolerances of the parity tests (O 4e-3 max / 5e-4 mean, lse 1e-4)
        assert np.abs(og - rg).max() <= 4e-3 and np.abs(og - rg).mean() <= 5e-4, f"call {call}"
        assert np.abs(lg - rl).max() <= 1e-4, f"call {call}"
        # and on its own against the FP64 oracle, at the stated tolerances
        ro, rlo = oracle_full(hq, hk, hv, "fp16", True, scale)
        compare(og, lg, ro, rlo, "fp16", name=f"noalloc_split{splits}_b{B}_h{H}_n{N}_d{D}_fp16_causal_call{call}")


def test_noalloc_rejects_a_split_larger_than_its_scratch(cuda_lib):
    lib = cuda_lib.load_library()
    B, H, N, D, splits = 1, 8, 8192, 128, 4  # needs 4 * 8 * 8192 * 128 * 4 B = 128 MiB > 64 MiB
    assert cuda_lib.splitkv_workspace_bytes(B, H, N, D, splits) > 64 << 20
    x = torch.zeros(B, H, N, D, dtype=torch.float16, device="cuda")
    o = torch.empty_like(x)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, x, x.clone(), x.clone(), o, lse, True, 0.088, splits) == -8
    assert lib.attn_status_string(-8).decode() != "unknown status"

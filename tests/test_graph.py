"""attn_fwd captured in a CUDA graph: the calls only enqueue work on the caller's
stream and allocate nothing, so a captured sequence replays with the same results
as eager calls (bit for bit: same kernels, same unit order).  Covers the three ways
the kernel forms its work units: key halves (short sequences), pairs of query tiles,
and units handed out from a device counter (K and V over 64 MiB), whose counters must
come back to zero after every replay."""
import numpy as np
import pytest
import torch

from exact_causal_attention_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,D", [(1, 32, 512, 128), (1, 32, 2048, 128), (1, 40, 8192, 128), (2, 6, 1000, 64)])
def test_captured_calls_replay_like_eager_calls(cuda_lib, B, H, N, D):
    eca = cuda_lib
    q, k, v = (x.cuda() for x in inputs.make_qkv(B, H, N, D, "fp16", seed=600 + N))
    o_ref = torch.empty_like(q)
    l_ref = torch.empty(B, H, N, device="cuda")
    eca.attn_fwd_into(q, k, v, o_ref, l_ref, causal=True)
    torch.cuda.synchronize()
    assert eca.device_status() == 0

    s = torch.cuda.Stream()
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):  # back-to-back calls inside one graph
            eca.attn_fwd_into(q, k, v, o, lse, causal=True, stream=s)
    for _ in range(3):
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert eca.device_status() == 0
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    # eager calls after the replays still agree (counters back at zero)
    o2 = torch.empty_like(q)
    eca.attn_fwd_into(q, k, v, o2, None, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, o_ref)
    assert np.isfinite(o.float().cpu().numpy()).all()

"""Launch-level behaviour of attn_fwd.

Captured in a CUDA graph: the calls only enqueue work on the caller's stream and
allocate nothing, so a captured sequence replays with the same results as eager
calls (bit for bit: same kernels, same unit order).  Covers the three ways the
kernel forms its work units: key halves (short sequences), pairs of query tiles,
and units handed out from a device counter (K and V over 64 MiB), whose counters
must come back to zero after every replay.  Also: more concurrent counter launches
than counter slots, and the tensor-map cache across shape changes."""
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


def test_more_concurrent_counter_launches_than_slots(cuda_lib):
    """Launches that take their units from a device counter (K and V over 64 MiB) use one
    of 64 counter slots per device, in turn.  66 such launches on 66 streams, none waiting
    for another, must all give the eager result: the 65th and 66th reuse the first two
    slots only after those launches have finished (the library orders them on the GPU)."""
    eca = cuda_lib
    B, H, N, D = 1, 40, 8192, 128  # K + V = 160 MiB
    q, k, v = (x.cuda() for x in inputs.make_qkv(B, H, N, D, "fp16", seed=616))
    o_ref = torch.empty_like(q)
    eca.attn_fwd_into(q, k, v, o_ref, None, causal=True)
    torch.cuda.synchronize()
    outs = [torch.full_like(q, float("nan")) for _ in range(66)]
    streams = [torch.cuda.Stream() for _ in range(66)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for o, s in zip(outs, streams):
        eca.attn_fwd_into(q, k, v, o, None, causal=True, stream=s)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    for i, o in enumerate(outs):
        assert torch.equal(o, o_ref), f"launch {i}"


def test_tensor_map_cache_follows_shape_changes(cuda_lib):
    """The library caches tensor maps by address and shape: calls that reuse the same
    buffers with other lengths, head counts and types must each be encoded anew."""
    from helpers import compare, oracle_full, p_rounding_term

    eca = cuda_lib
    D = 64
    buf = [torch.zeros(2 * 4 * 1024 * D, dtype=torch.float16, device="cuda") for _ in range(4)]
    for (B, H, N, dtype) in [(1, 4, 1024, "fp16"), (2, 2, 700, "fp16"), (1, 4, 1024, "fp16"), (1, 8, 333, "bf16")]:
        hq, hk, hv = inputs.make_qkv(B, H, N, D, dtype, seed=B * 100 + H + N)
        n = B * H * N * D
        t = inputs.TORCH_DTYPES[dtype]
        q, k, v, o = (b.view(torch.int16)[:n].view(t).view(B, H, N, D) for b in buf)
        q.copy_(hq.cuda())
        k.copy_(hk.cuda())
        v.copy_(hv.cuda())
        o.fill_(float("nan"))
        lse = torch.full((B, H, N), float("nan"), device="cuda")
        eca.attn_fwd_into(q, k, v, o, lse, causal=True)
        torch.cuda.synchronize()
        ro, rl = oracle_full(hq, hk, hv, dtype, True, 1.0 / D ** 0.5)
        compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, dtype,
                p_rounding_term(hq, hk, hv, dtype, True, 1.0 / D ** 0.5))


def test_stream_order_launch_gives_the_same_results(cuda_lib, tmp_path):
    """The library launches with programmatic dependent launch by default; ECA_PDL=0
    launches in plain stream order.  Both orders must give bit-identical results for
    back-to-back calls of every unit mode, the key split, and an append followed by a
    split decode (a second process, since the switch is read once per process)."""
    import os
    import subprocess
    import sys

    eca = cuda_lib
    shapes = [(1, 32, 512, 128), (1, 40, 8192, 128), (2, 6, 1000, 64)]
    script = r'''
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import exact_causal_attention_gb300 as eca
from exact_causal_attention_gb300 import inputs
for i, (B, H, N, D) in enumerate(%r):
    q, k, v = (x.cuda() for x in inputs.make_qkv(B, H, N, D, "fp16", seed=700 + N))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    for _ in range(3):
        eca.attn_fwd_into(q, k, v, o, lse, causal=True)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    np.save(sys.argv[2] + f"/o{i}.npy", o.view(torch.int16).cpu().numpy())
    np.save(sys.argv[2] + f"/l{i}.npy", lse.cpu().numpy())
# the key split (attention and merge launches) and the paged append and decode
q, k, v = (x.cuda() for x in inputs.make_qkv(1, 4, 2048, 128, "fp16", seed=731))
o, lse = eca.attn_fwd_splitkv(q, k, v, kv_splits=3, causal=True)
pq, cache, table, lens = inputs.paged_decode_inputs(4, 8, 2, 128, 16, [300, 17, 48, 1], "fp16", seed=732)
new = torch.randn(4, 2, 2, 128, generator=torch.Generator().manual_seed(733), dtype=torch.float64).to(torch.float16)
dc = cache.cuda()
eca.paged_append(new.cuda(), dc, table.cuda(), lens.cuda())
do, dl = eca.decode_paged(pq.cuda(), dc, table.cuda(), lens.cuda(), kv_splits=3)
torch.cuda.synchronize()
assert eca.device_status() == 0
for name, t in (("so", o.view(torch.int16)), ("sl", lse), ("do", do.view(torch.int16)), ("dl", dl)):
    np.save(sys.argv[2] + f"/{name}.npy", t.cpu().numpy())
''' % (shapes,)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, ECA_PDL="0")
    subprocess.run([sys.executable, "-c", script, root, str(tmp_path)], env=env, check=True, timeout=600)
    for i, (B, H, N, D) in enumerate(shapes):
        q, k, v = (x.cuda() for x in inputs.make_qkv(B, H, N, D, "fp16", seed=700 + N))
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, device="cuda")
        for _ in range(3):
            eca.attn_fwd_into(q, k, v, o, lse, causal=True)
        torch.cuda.synchronize()
        assert eca.device_status() == 0
        assert np.array_equal(o.view(torch.int16).cpu().numpy(), np.load(tmp_path / f"o{i}.npy")), (B, H, N, D)
        assert np.array_equal(lse.cpu().numpy(), np.load(tmp_path / f"l{i}.npy")), (B, H, N, D)
    q, k, v = (x.cuda() for x in inputs.make_qkv(1, 4, 2048, 128, "fp16", seed=731))
    so, sl = eca.attn_fwd_splitkv(q, k, v, kv_splits=3, causal=True)
    pq, cache, table, lens = inputs.paged_decode_inputs(4, 8, 2, 128, 16, [300, 17, 48, 1], "fp16", seed=732)
    new = torch.randn(4, 2, 2, 128, generator=torch.Generator().manual_seed(733), dtype=torch.float64).to(torch.float16)
    dc = cache.cuda()
    eca.paged_append(new.cuda(), dc, table.cuda(), lens.cuda())
    do, dl = eca.decode_paged(pq.cuda(), dc, table.cuda(), lens.cuda(), kv_splits=3)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    for name, t in (("so", so.view(torch.int16)), ("sl", sl), ("do", do.view(torch.int16)), ("dl", dl)):
        assert np.array_equal(t.cpu().numpy(), np.load(tmp_path / f"{name}.npy")), name


@pytest.mark.parametrize("B,H,N,D", [(1, 32, 512, 128), (2, 6, 1000, 64), (1, 40, 4096, 128)])
def test_chained_calls_read_the_previous_output(cuda_lib, B, H, N, D):
    """Back-to-back calls on one stream where each call reads the previous call's output
    as its query and writes its own output over the previous call's query, with a copy
    kernel of torch's rewriting the next input after every second call: under
    programmatic launch a call's CTAs may start while the kernel ahead still runs, so
    this checks that nothing is read or written before that kernel has finished.  The
    same chain with a synchronisation after every operation is the reference."""
    eca = cuda_lib
    q0, k, v = (x.cuda() for x in inputs.make_qkv(B, H, N, D, "fp16", seed=900 + N))
    fresh = (q0 * 0.5).contiguous()

    def chain(sync):
        bufs = [q0.clone(), torch.empty_like(q0)]
        outs, src = [], 0
        for i in range(6):
            q, o = bufs[src], bufs[1 - src]
            eca.attn_fwd_into(q, k, v, o, None, causal=True)
            if sync:
                torch.cuda.synchronize()
            outs.append(o.clone())
            if i % 2 == 1:
                o.copy_(fresh)  # the next call's input, rewritten right behind this call
                if sync:
                    torch.cuda.synchronize()
            src = 1 - src
        torch.cuda.synchronize()
        return outs

    ref = chain(True)
    for _ in range(2):
        got = chain(False)
        assert eca.device_status() == 0
        for a, b in zip(ref, got):
            assert torch.equal(a, b)


def test_chained_split_calls_read_the_previous_output(cuda_lib):
    """The same chain through the key split (an attention launch and a merge launch per
    call, both launched programmatically): each call reads the previous call's output."""
    eca = cuda_lib
    B, H, N, D, splits = 1, 4, 2048, 128, 3
    q0, k, v = (x.cuda() for x in inputs.make_qkv(B, H, N, D, "fp16", seed=950))
    need = eca.splitkv_workspace_bytes(B, H, N, D, splits)
    raw = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    off = (-raw.data_ptr()) % 256
    ws = raw[off:off + need]

    def chain(sync):
        bufs = [q0.clone(), torch.empty_like(q0)]
        outs, src = [], 0
        for _ in range(4):
            q, o = bufs[src], bufs[1 - src]
            lse = torch.empty(B, H, N, device="cuda")
            eca.attn_fwd_splitkv(q, k, v, o, lse, kv_splits=splits, workspace=ws, causal=True)
            if sync:
                torch.cuda.synchronize()
            outs.append((o.clone(), lse))
            src = 1 - src
        torch.cuda.synchronize()
        return outs

    ref = chain(True)
    for _ in range(2):
        got = chain(False)
        assert eca.device_status() == 0
        for (a, la), (b, lb) in zip(ref, got):
            assert torch.equal(a, b) and torch.equal(la, lb)

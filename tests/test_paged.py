"""GPU parity of the paged-cache decode and append against the FP64 oracle
("CUDA KV Cache：分页存储与长上下文 Decode 极致优化": address rule of section 2,
grouped heads of section 3.3, append of section 4, split of section 6.4).
Physical pages are a seeded permutation, table entries past a request's pages are
-1, and the cache slots past each length are filled with NaN, so a read of
anything outside the logical sequence shows up as NaN in the output."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from exact_causal_attention_gb300 import inputs

from helpers import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, bf16_ulp

pytestmark = pytest.mark.gpu


def poison_tail(cache, table, lengths, T):
    """NaN in every cache slot that no request's logical sequence covers."""
    used = np.zeros(cache.shape[0] * T, dtype=bool)
    for b, L in enumerate(lengths.tolist()):
        for t in range(L):
            used[int(table[b, t // T]) * T + t % T] = True
    c = cache.clone()
    flat = c.view(cache.shape[0], 2, T, -1)
    for pidx in range(cache.shape[0]):
        for off in range(T):
            if not used[pidx * T + off]:
                flat[pidx, :, off] = float("nan")
    return c


def oracle_decode(q, cache, table, lengths, T, scale, dtype, abs_v=False):
    cb = inputs.bits(cache)
    if abs_v:
        cb = cb & np.uint16(0x7FFF)
    cd = oracle.decode(cb, dtype).reshape(cache.shape)
    qd = oracle.decode(inputs.bits(q), dtype).reshape(q.shape)
    return oracle.decode_paged(qd, np.nan_to_num(cd, nan=0.0), table.numpy(), lengths.numpy(), T, scale)


def run_decode(q, cache, table, lengths, scale, splits):
    import exact_causal_attention_gb300 as eca

    dq, dc, dt, dl = q.cuda(), cache.cuda(), table.cuda(), lengths.cuda()
    out = torch.full_like(dq, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    eca.decode_paged(dq, dc, dt, dl, scale=scale, kv_splits=splits, out=out, lse=lse)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def check(o, lse, ro, rl, dtype, p_term, lengths):
    live = np.asarray(lengths) > 0
    assert np.all(o[~live] == 0.0) and np.all(lse[~live] == -np.inf)
    o, lse, ro, rl = o[live], lse[live], ro[live], rl[live]
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err = np.abs(o - ro)
    assert np.abs(lse - rl).max() <= LSE_MAX_ABS
    if dtype == "fp16":
        assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS
    else:
        assert (err <= O_MAX_ABS + bf16_ulp(ro) + 2.0 ** -8 * p_term[live]).all()


CASES = [
    # B, Hq, Hkv, D, T, lengths, dtype, splits
    (2, 8, 2, 128, 16, [100, 37], "fp16", 1),
    (3, 4, 4, 64, 8, [1, 64, 65], "bf16", 2),
    (2, 32, 8, 128, 16, [1000, 2049], "fp16", None),
    (1, 6, 2, 128, 32, [500], "fp16", 3),
    (2, 16, 1, 64, 64, [0, 300], "fp16", 2),
    (4, 8, 2, 128, 16, [7, 640, 129, 1], "bf16", 5),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,T,lengths,dtype,splits", CASES)
def test_decode_matches_oracle(cuda_lib, B, Hq, Hkv, D, T, lengths, dtype, splits):
    q, cache, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, D, T, lengths, dtype, seed=400 + sum(lengths))
    cache = poison_tail(cache, table, lens, T)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_decode(q, cache, table, lens, scale, splits)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_decode(q, cache, table, lens, T, scale, dtype)
    pt = oracle_decode(q, cache, table, lens, T, scale, dtype, abs_v=True)[0] if dtype == "bf16" else None
    check(o, lse, ro, rl, dtype, pt, lengths)


def test_page_benchmark_geometry(cuda_lib):
    # B=8, Hq=32, Hkv=8, D=128, page size 16 (the page's section 8), context 4096
    w = inputs.PAGED_BENCH
    q, cache, table, lens = inputs.paged_decode_inputs(w.B, w.Hq, w.Hkv, w.D, w.page_size, [4096] * w.B, w.dtype,
                                                       seed=w.seed)
    scale = 1.0 / math.sqrt(w.D)
    for splits in (1, None):
        o, lse = run_decode(q, cache, table, lens, scale, splits)
        ro, rl = oracle_decode(q, cache, table, lens, w.page_size, scale, w.dtype)
        check(o, lse, ro, rl, "fp16", None, [4096] * w.B)


def test_append_then_decode(cuda_lib):
    import exact_causal_attention_gb300 as eca

    B, Hq, Hkv, D, T = 3, 8, 2, 128, 16
    lengths = [17, 48, 1]  # the newest token sits at lengths - 1: mid-page, page end, first slot
    q, cache, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, D, T, lengths, "fp16", seed=77)
    new = torch.randn(B, 2, Hkv, D, generator=torch.Generator().manual_seed(78), dtype=torch.float64).to(torch.float16)
    dc, dt, dl = cache.cuda(), table.cuda(), lens.cuda()
    eca.paged_append(new.cuda(), dc, dt, dl)
    torch.cuda.synchronize()
    assert eca.device_status() == 0
    expect = cache.clone()
    for b, L in enumerate(lengths):
        t = L - 1
        expect[int(table[b, t // T]), :, t % T] = new[b]
    assert torch.equal(dc.cpu(), expect)
    o, lse = run_decode(q, expect, table, lens, 1.0 / math.sqrt(D), 2)
    ro, rl = oracle_decode(q, expect, table, lens, T, 1.0 / math.sqrt(D), "fp16")
    check(o, lse, ro, rl, "fp16", None, lengths)


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_right_behind_append_sees_the_new_token(cuda_lib, splits):
    """The append and the decode are launched back to back on one stream with no
    synchronisation between them (under programmatic launch the decode's CTAs may start
    while the append still runs): the decode must see every appended token.  Repeated
    so that a race would show."""
    import exact_causal_attention_gb300 as eca

    B, Hq, Hkv, D, T = 4, 8, 2, 128, 16
    lengths = [17, 48, 1, 300]
    q, cache, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, D, T, lengths, "fp16", seed=81)
    new = torch.randn(B, 2, Hkv, D, generator=torch.Generator().manual_seed(82), dtype=torch.float64).to(torch.float16)
    expect = cache.clone()
    for b, L in enumerate(lengths):
        t = L - 1
        expect[int(table[b, t // T]), :, t % T] = new[b]
    scale = 1.0 / math.sqrt(D)
    ro, rl = oracle_decode(q, expect, table, lens, T, scale, "fp16")
    dq, dt, dl, dnew = q.cuda(), table.cuda(), lens.cuda(), new.cuda()
    for _ in range(3):
        dc = cache.cuda()
        torch.cuda.synchronize()
        out = torch.full_like(dq, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        ws = None
        if splits > 1:
            need = int(eca.load_library().attn_decode_workspace_bytes(B, Hq, D, splits))
            ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
            off = (-ws.data_ptr()) % 256
            ws = ws[off:off + need]
        eca.paged_append(dnew, dc, dt, dl)
        eca.decode_paged(dq, dc, dt, dl, scale=scale, kv_splits=splits, out=out, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        assert eca.device_status() == 0
        check(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "fp16", None, lengths)


def test_out_of_range_entries_are_rejected_not_read(cuda_lib):
    import exact_causal_attention_gb300 as eca

    B, Hq, Hkv, D, T = 2, 4, 2, 64, 16
    q, cache, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, D, T, [40, 40], "fp16", seed=81)
    bad = table.clone()
    bad[1, 1] = cache.shape[0] + 5  # past the last physical page
    o, lse = run_decode(q, cache, bad, lens, 0.125, 1)
    assert eca.device_status() == -9
    ro, rl = oracle_decode(q, cache, table, lens, T, 0.125, "fp16")
    check(o[:1], lse[:1], ro[:1], rl[:1], "fp16", None, [40])  # the other request is untouched
    assert np.isfinite(o[1]).all()
    long = lens.clone()
    long[0] = table.shape[1] * T + 1  # longer than the table
    run_decode(q, cache, table, long, 0.125, 1)
    assert eca.device_status() == -9
    assert eca.device_status() == 0


@pytest.mark.parametrize("splits", [5, 12])
def test_split_merge_in_kernel_repeats_bit_identically(cuda_lib, splits):
    # The segments of a split are merged by the last one to finish, counted with
    # device counters that return to zero after every launch: repeated launches (the
    # same slot reused after the pool wraps) give identical results, with 5 segments
    # and with 12, and both match the oracle.
    B, Hq, Hkv, D, T = 4, 16, 4, 128, 16
    lengths = [900, 64, 3000, 17]
    q, cache, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, D, T, lengths, "fp16", seed=91)
    scale = 1.0 / math.sqrt(D)
    first = run_decode(q, cache, table, lens, scale, splits)
    for _ in range(10):
        again = run_decode(q, cache, table, lens, scale, splits)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
    ro, rl = oracle_decode(q, cache, table, lens, T, scale, "fp16")
    check(first[0], first[1], ro, rl, "fp16", None, lengths)


def test_split_merge_kernel_for_many_groups(cuda_lib):
    # More (request, K/V head, head chunk) groups than one counter slot holds
    # (520 x 8 = 4160 > 4096): the separate merge kernel runs.  With 64-token pages a
    # tile is one page, so requests of up to 10 pages split 10 ways; shorter ones leave
    # trailing segments empty.
    B, Hq, Hkv, D, T = 520, 8, 8, 64, 64
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(0, 641, size=B)]
    lengths[0] = 640
    q, cache, table, lens = inputs.paged_decode_inputs(B, Hq, Hkv, D, T, lengths, "fp16", seed=92)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_decode(q, cache, table, lens, scale, 10)
    ro, rl = oracle_decode(q, cache, table, lens, T, scale, "fp16")
    check(o, lse, ro, rl, "fp16", None, lengths)

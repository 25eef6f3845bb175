"""GPU parity of the online row softmax (attn_row_softmax_f32) against the FP64
oracle, with the checks of the page "Softmax kernels V1-V9" (lpnh.cn): output
NaN-filled before each call (section 3.4), no NaN or Inf, max-abs error below
1e-6 for fp32 input and output (section 3.2), its inputs (section 3.3: zeros, a
special last element, a constant added to a row, seeded U[-10, 10) rows, odd
lengths such as M = 1025, N = 257)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_causal_attention_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-6


def gpu_softmax(x_cpu, inplace=False, offset=0):
    import exact_causal_attention_gb300 as eca

    M, N = x_cpu.shape
    if offset:
        flat = torch.empty(M * N + offset, dtype=torch.float32, device="cuda")
        x = flat[offset:].view(M, N)
        x.copy_(x_cpu)
    else:
        x = x_cpu.cuda()
    y = x if inplace else torch.full_like(x, float("nan"))
    lib = eca.load_library()
    rc = lib.attn_row_softmax_f32(x.data_ptr(), y.data_ptr(), M, N,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    return y.double().cpu().numpy()


SHAPES = [(1024, 4096), (3, 4096), (5, 3001), (1, 2052), (1025, 257), (3, 1), (5, 2048), (7, 2049), (2, 16384), (2, 16385), (1, 100000),
          (4, 33), (9, 128), (2, 4100), (300, 1000)]


@pytest.mark.parametrize("M,N", SHAPES)
def test_row_softmax_matches_oracle(cuda_lib, M, N):
    x = inputs.uniform_matrix(M, N, seed=M * 7 + N)
    y = gpu_softmax(x)
    ref = oracle.softmax(x.double().numpy())
    assert np.isfinite(y).all()
    assert np.abs(y - ref).max() <= TOL


def test_page_inputs(cuda_lib):
    N = 257
    rows = [np.zeros(N), np.r_[np.zeros(N - 1), 30.0], np.r_[np.zeros(N - 1), -30.0],
            np.linspace(-10, 10, N), np.linspace(-10, 10, N) + 1000.0]
    x = torch.tensor(np.stack(rows), dtype=torch.float32)
    y = gpu_softmax(x)
    ref = oracle.softmax(x.double().numpy())
    assert np.abs(y - ref).max() <= TOL
    assert np.abs(y[3] - y[4]).max() <= TOL  # a constant added to a row changes nothing


def test_in_place_and_unaligned_rows(cuda_lib):
    x = inputs.uniform_matrix(33, 1024, seed=5)
    ref = oracle.softmax(x.double().numpy())
    assert np.abs(gpu_softmax(x, inplace=True) - ref).max() <= TOL
    assert np.abs(gpu_softmax(x, offset=1) - ref).max() <= TOL  # base not 16-byte aligned: scalar path
    x2 = inputs.uniform_matrix(3, 40000, seed=6)
    assert np.abs(gpu_softmax(x2, inplace=True) - oracle.softmax(x2.double().numpy())).max() <= TOL


def test_minus_infinity_and_huge_values(cuda_lib):
    x = inputs.uniform_matrix(4, 3000, seed=8)
    x[0, :1500] = float("-inf")
    x[1, :] = float("-inf")
    x[2] *= 1000.0
    y = gpu_softmax(x)
    ref = oracle.softmax(x.double().numpy())
    assert np.isfinite(y).all()
    assert np.abs(y - ref).max() <= TOL
    assert np.all(y[1] == 0.0) and np.all(y[0, :1500] == 0.0)


def test_argument_errors(cuda_lib):
    lib = cuda_lib.load_library()
    x = torch.zeros(4, 8, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_row_softmax_f32(x.data_ptr(), x.data_ptr(), 0, 8, s) == -1
    assert lib.attn_row_softmax_f32(x.data_ptr(), x.data_ptr(), 4, 0, s) == -1
    assert lib.attn_row_softmax_f32(x.data_ptr(), x.data_ptr() + 4, 4, 8, s) == -1  # partial overlap
    assert lib.attn_row_softmax_f32(x.data_ptr() + 2, x.data_ptr() + 64, 1, 4, s) == -2


@pytest.mark.parametrize("M,N", [(2048, 128), (1024, 4096), (64, 8192), (8, 20000)])
def test_chained_calls_read_the_previous_output(cuda_lib, M, N):
    """The kernels are launched programmatically (each may start while the kernel ahead
    still runs, and waits for it before touching memory).  A chain on one stream where
    each call reads the previous call's output, every third call in place, with a copy
    kernel of torch's rewriting a buffer right behind some calls, must give the same bits
    as the same chain with a synchronisation after every operation.  One shape per
    schedule: warp per row, 128 threads per row, block per row, two passes."""
    import exact_causal_attention_gb300 as eca

    g = torch.Generator().manual_seed(1200 + N)
    x0 = (torch.rand(M, N, generator=g, dtype=torch.float64) * 20 - 10).float().cuda()
    fresh = (x0 * 0.5).contiguous()

    def chain(sync):
        bufs = [x0.clone(), torch.empty_like(x0)]
        outs, src = [], 0
        for i in range(6):
            if i % 3 == 2:
                eca.row_softmax(bufs[src], out=bufs[src])
                dst = src
            else:
                eca.row_softmax(bufs[src], out=bufs[1 - src])
                dst = 1 - src
            if sync:
                torch.cuda.synchronize()
            outs.append(bufs[dst].clone())
            if i == 3:
                bufs[dst].copy_(fresh)  # the next call's input, rewritten right behind this call
                if sync:
                    torch.cuda.synchronize()
            src = dst
        torch.cuda.synchronize()
        return outs

    ref = chain(True)
    for _ in range(2):
        got = chain(False)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)

"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws Q, K, V.  The recipe
stands in for the workloads of "CUDA FlashAttention：从在线 Softmax 到长序列 IO 极限"
(section 1 and the section 8 benchmark: B=1, H=32, D=128, N from 512 to 8192):

* one CPU ``torch.Generator`` seeded with the workload's seed;
* ``torch.randn(B, H, N, D)`` in float64 three times, in the order q, k, v
  (float64 so the draw is the same on x86 and Arm hosts: torch's float32 path
  is vectorised differently per CPU, while an ulp-level difference in a float64
  draw survives the rounding to 16 bits with negligible probability);
* q and k multiplied by ``qk_std`` (3 for the stress case so that scores reach
  tens and the max subtraction matters), v left at N(0, 1);
* round-to-nearest-even to float32, then to fp16 or bf16.

The tensors stay on the CPU; callers move them to the device.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch

TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str
    causal: bool
    seed: int
    qk_std: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 2BHN^2D causal, 4BHN^2D non-causal (section 1 of the page)."""
        f = 2.0 * self.B * self.H * self.N * self.N * self.D
        return f if self.causal else 2.0 * f

    def with_causal(self, causal: bool) -> "Workload":
        return dataclasses.replace(self, causal=causal, name=self.name + ("" if causal else "_noncausal"))


# The five workloads: a small one the oracle finishes in seconds, the page's
# benchmark geometry at N = 512, 2048 (causal and not), 8192, and a bf16 stress
# case whose length is not a multiple of the 128-row tile.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("causal_b1_h2_n256_d64_fp16", 1, 2, 256, 64, "fp16", True, 0),
        Workload("causal_b1_h32_n512_d128_fp16", 1, 32, 512, 128, "fp16", True, 1),
        Workload("causal_b1_h32_n2048_d128_fp16", 1, 32, 2048, 128, "fp16", True, 2),
        Workload("noncausal_b1_h32_n2048_d128_fp16", 1, 32, 2048, 128, "fp16", False, 2),
        Workload("causal_b1_h32_n8192_d128_fp16", 1, 32, 8192, 128, "fp16", True, 3),
        Workload("causal_b4_h32_n1000_d64_bf16", 4, 32, 1000, 64, "bf16", True, 4, qk_std=3.0),
    ]
}

# The sweep of the page's benchmark table (causal fp16, B=1, H=32, D=128).
SWEEP_N = (512, 1024, 2048, 4096, 8192)


def sweep_workload(n: int, seed: int = 1) -> Workload:
    return Workload(f"causal_b1_h32_n{n}_d128_fp16", 1, 32, n, 128, "fp16", True, seed)


def make_qkv(B: int, H: int, N: int, D: int, dtype: str, seed: int, qk_std: float = 1.0):
    """Return CPU tensors (q, k, v) of shape [B, H, N, D] in fp16 or bf16."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn(B, H, N, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, H, N, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, H, N, D, generator=g, dtype=torch.float64)
    if qk_std != 1.0:
        q.mul_(qk_std)
        k.mul_(qk_std)
    t = TORCH_DTYPES[dtype]
    return tuple(x.to(torch.float32).to(t) for x in (q, k, v))


def make_qkv_device(B: int, H: int, N: int, D: int, dtype: str, seed: int, device="cuda"):
    """(q, k, v) of shape [B, H, N, D] in fp16 or bf16, N(0, 1) drawn by torch's generator on
    `device`: for tensors too large to draw on the host.  The same seed gives the same bytes
    for one device type and torch version; a test copies the slices it checks to the host."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    t = TORCH_DTYPES[dtype]
    return tuple(torch.randn(B, H, N, D, generator=g, device=device, dtype=t) for _ in range(3))


def workload_qkv(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.D, w.dtype, w.seed, w.qk_std)


def bits(t: torch.Tensor):
    """The raw 16-bit patterns of a CPU fp16/bf16 tensor as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def sha256(t: torch.Tensor) -> str:
    return hashlib.sha256(bits(t).tobytes()).hexdigest()


def uniform_matrix(M: int, N: int, seed: int, lo: float = -10.0, hi: float = 10.0):
    """A CPU float32 [M, N] matrix of i.i.d. U[lo, hi) draws (float64 draw, one rounding), the
    input recipe of the row-softmax page's section 6.1 (U[-10, 10), seeded)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.rand(M, N, generator=g, dtype=torch.float64)
    return (x * (hi - lo) + lo).to(torch.float32)


# The row-softmax workload of that section (M=1024, N=4096, seed 42) and a larger one for HBM.
SOFTMAX_PAGE_SHAPE = (1024, 4096, 42)
SOFTMAX_HBM_SHAPE = (65536, 4096, 43)


@dataclasses.dataclass(frozen=True)
class PagedWorkload:
    """One decode step over a paged K/V cache (the decode page's section 8 shapes)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    context: int      # tokens per request (every request the same length here)
    dtype: str
    seed: int

    @property
    def kv_bytes(self) -> int:
        """K and V bytes the decode step must read: 2 B L Hkv D s."""
        return 2 * self.B * self.context * self.Hkv * self.D * 2


def paged_decode_inputs(B: int, Hq: int, Hkv: int, D: int, page_size: int, lengths, dtype: str, seed: int,
                        spare_pages: int = 3):
    """CPU tensors for one paged decode step: q [B, Hq, D], cache [P, 2, T, Hkv, D],
    block_table [B, max_pages] int32 (entries past a request's last page are -1),
    lengths [B] int32.  Physical pages are a seeded permutation, so logical order and
    physical order differ; values are N(0, 1) drawn in float64 and rounded once."""
    lengths = [int(x) for x in lengths]
    pages_per = [(L + page_size - 1) // page_size for L in lengths]
    max_pages = max(1, max(pages_per))
    P = sum(pages_per) + spare_pages
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    perm = torch.randperm(P, generator=g)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b, n in enumerate(pages_per):
        table[b, :n] = perm[nxt:nxt + n].to(torch.int32)
        nxt += n
    t = TORCH_DTYPES[dtype]
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float64).to(torch.float32).to(t)
    cache = torch.randn(P, 2, page_size, Hkv, D, generator=g, dtype=torch.float64).to(torch.float32).to(t)
    return q, cache, table, torch.tensor(lengths, dtype=torch.int32)


PAGED_BENCH = PagedWorkload("paged_decode_b8_hq32_hkv8_d128_t16_ctx32768_fp16", 8, 32, 8, 128, 16, 32768,
                            "fp16", 11)
PAGED_CONTEXTS = (1024, 4096, 8192, 16384, 32768)

"""Bounded waits: a kernel whose wait can never complete gives up after its limit,
records ATTN_ERR_TIMEOUT in the device status word and returns normally; the
context stays usable.  No fault, trap or hang is involved."""
import pytest
import torch

from exact_causal_attention_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_times_out_and_context_survives(cuda_lib):
    eca = cuda_lib
    assert eca.device_status() == 0
    eca.watchdog_selftest(20_000)  # 20 ms limit on a barrier nothing arrives on
    assert eca.device_status() == -6
    assert eca.device_status() == 0  # reading clears the word
    q, k, v = (x.cuda() for x in inputs.make_qkv(1, 1, 256, 64, "fp16", seed=1))
    o, lse = eca.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert eca.device_status() == 0

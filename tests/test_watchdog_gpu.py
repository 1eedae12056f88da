"""Failure reporting through the device status word, without faulting the GPU.

Every wait inside the kernels is bounded (2 s of %globaltimer).  A test hook
(FA_TEST_WITHHOLD_K=1, read by fa_fwd at each call) makes CTA 0 of the
forward skip its first K-tile load: nothing is ever copied to that buffer,
so the MMA warps' wait for it, the softmax warps' wait for the first score
tile and the producer's own final wait for its copies all run out.  Each
gives up, records the timeout and falls through to the kernel's exit with no
copy or tensor-core product in flight (the withheld tile was never issued;
the MMA warps issued nothing; every other copy is waited for), so the
context stays usable: the next call is checked against the oracle.

The forward also reports rows whose LSE is not finite (FA_ERR_NONFINITE):
a stabilised row whose repeated maximum is so large that every exponential
underflows ("The modified safe softmax" keeps the rule to rows where the
plain softmax is stable)."""
import numpy as np
import pytest

from conftest import case
from gpu_helpers import dev_bf16, f32, host_f64, o_bound
from oracle import oracle as orc
from precision_flash_attention_attn_gb300.inputs import bf16_bits

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 5
FA_ERR_NONFINITE = 6


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa as fa_mod
    return fa_mod


def _parity(fa, c, mode):
    q, k, v = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v"))
    o, lse = fa.attention_fwd(q, k, v, c.causal, c.scale, mode)
    assert fa.fa_device_status() == 0
    BH = c.B * c.H
    ex = orc.fwd(*(f32(getattr(c, n)).reshape(BH, c.N, c.d) for n in ("q", "k", "v")), c.causal, c.scale, mode)
    og = host_f64(o).reshape(ex["o"].shape)
    assert np.all(np.abs(og - ex["o"]) <= o_bound(ex["o"], mode))


def test_withheld_tile_times_out_and_the_context_survives(fa, monkeypatch):
    import time

    import torch
    c = case("tiny")
    fa.fa_device_status(reset=True)
    q, k, v = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v"))
    monkeypatch.setenv("FA_TEST_WITHHOLD_K", "1")
    t0 = time.time()
    o, lse = fa.attention_fwd(q, k, v, c.causal, c.scale, 0)
    torch.cuda.synchronize()
    waited = time.time() - t0
    monkeypatch.delenv("FA_TEST_WITHHOLD_K")
    assert fa.fa_device_status(reset=True) == FA_ERR_TIMEOUT
    assert 1.5 < waited < 30.0, waited      # the waits ran to their limit, and no further
    assert fa.fa_device_status() == 0       # the reset cleared it
    for mode in (0, 1, 2):
        _parity(fa, c, mode)


def test_backward_after_a_timeout_is_correct(fa, monkeypatch):
    # the backward (its three launches and its scratch) is unaffected by a
    # forward that timed out
    import torch
    from gpu_helpers import GRAD_REL_TOL, rel_fro
    c = case("tiny")
    q, k, v, do = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    monkeypatch.setenv("FA_TEST_WITHHOLD_K", "1")
    fa.attention_fwd(q, k, v, c.causal, c.scale, 0)
    torch.cuda.synchronize()
    monkeypatch.delenv("FA_TEST_WITHHOLD_K")
    assert fa.fa_device_status(reset=True) == FA_ERR_TIMEOUT
    o, lse = fa.attention_fwd(q, k, v, c.causal, c.scale, 0)
    got = fa.attention_bwd(q, k, v, o, lse, do, c.causal, c.scale, 0)
    assert fa.fa_device_status() == 0
    BH = c.B * c.H
    ex = orc.bwd(*(f32(getattr(c, n)).reshape(BH, c.N, c.d) for n in ("q", "k", "v", "do")), c.causal, c.scale)
    for name, g in zip(("dq", "dk", "dv"), got):
        assert rel_fro(host_f64(g).reshape(ex[name].shape), ex[name]) <= GRAD_REL_TOL, name


def test_nonfinite_rows_are_reported(fa):
    # Query and two keys equal to 4 in every component: the repeated maximum
    # is 4*4*64 = 1024, scale 1/8 makes it 128, and the stabilised shift
    # beta*rm with beta = 2 puts every exponential at exp(-128) or below,
    # under the FP32 range: l = 0 and the LSE is -inf.  The baseline row is
    # finite.
    import torch
    B, H, N, d = 1, 1, 128, 64
    rng = np.random.default_rng(3)
    qf = rng.standard_normal((B, H, N, d)).astype(np.float32) * 0.5
    kf = rng.standard_normal((B, H, N, d)).astype(np.float32) * 0.5
    qf[0, 0, 100] = 4.0
    kf[0, 0, 10] = 4.0
    kf[0, 0, 20] = 4.0
    q, k = dev_bf16(bf16_bits(qf)), dev_bf16(bf16_bits(kf))
    v = dev_bf16(bf16_bits(rng.standard_normal((B, H, N, d)).astype(np.float32)))
    fa.fa_device_status(reset=True)
    o, lse = fa.attention_fwd(q, k, v, True, 0.125, 0)
    torch.cuda.synchronize()
    assert fa.fa_device_status(reset=True) == 0
    assert torch.isfinite(lse).all()
    o, lse = fa.attention_fwd(q, k, v, True, 0.125, 1)
    torch.cuda.synchronize()
    assert fa.fa_device_status(reset=True) == FA_ERR_NONFINITE
    bad = (~torch.isfinite(lse)).nonzero().cpu().numpy()
    assert bad.tolist() == [[0, 0, 100]]
    assert fa.fa_device_status() == 0

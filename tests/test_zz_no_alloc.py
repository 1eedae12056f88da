"""The allocation-free backward, fa_bwd_noalloc, through the C ABI.

Some callers cannot allocate device memory while they run: a framework's
caching allocator may already hold nearly all of the GPU's memory, a
latency-critical loop may not afford an allocation call that can block, or a
deployment may forbid allocation after start-up.  fa_bwd_noalloc serves them
with a scratch array compiled into the library.  These tests check that two
calls in a row give the same gradients as fa_bwd (within the backward tests'
tolerance), and that problems too large for the scratch array are refused
before anything runs.

This file is named to be collected last."""
import numpy as np
import pytest

from gpu_helpers import GRAD_REL_TOL, dev_bf16, host_f64, rel_fro
from precision_flash_attention_attn_gb300.inputs import CaseSpec, make_custom


def _fa():
    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa
    return fa


def test_noalloc_rejects_problems_larger_than_the_scratch():
    # host-side check, before any device access: 8 x 16 x 1024 x 64 FP32 alone is 32 MiB
    fa = _fa()
    fake = 1 << 20
    rc = fa.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, 8, 16, 1024, 64, True, 0.125, 0,
                           stream=0, check=False)
    assert rc == 1
    assert "static limit" in fa.fa_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 128, 64, True), (2, 4, 384, 64, True), (1, 2, 200, 128, False)])
def test_noalloc_backward_matches_fa_bwd_twice_in_a_row(B, H, N, d, causal):
    import torch
    fa = _fa()
    c = make_custom(CaseSpec("noalloc", B, H, N, d, causal, 9100 + N + d, plant_frac=0.1, min_plant_row=3))
    q, k, v, do = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    for mode in (0, 1, 2):
        o, lse = fa.attention_fwd(q, k, v, causal, c.scale, mode)
        ref = fa.attention_bwd(q, k, v, o, lse, do, causal, c.scale, mode)
        ref = [host_f64(t) for t in ref]
        floor = 1e-3 * max(np.linalg.norm(r) for r in ref)
        for _call in range(2):
            got = [torch.full_like(q, float("nan")) for _ in range(3)]
            fa.fa_bwd_noalloc(q, k, v, o, lse, do, *got, B, H, N, d, causal, c.scale, mode)
            torch.cuda.synchronize()
            assert fa.fa_device_status() == 0
            for name, g, r in zip(("dq", "dk", "dv"), got, ref):
                err = rel_fro(host_f64(g), r, floor)
                assert err <= GRAD_REL_TOL, (name, mode, _call, err)


@pytest.mark.gpu
def test_noalloc_is_fa_bwd_at_the_gpt2_small_size():
    """The timed path at its full size: fa_bwd_noalloc runs the same kernels as
    fa_bwd (whose gradients the backward tests check against the oracle for
    every head at this size), so dK and dV are bit-identical and dQ differs
    only by the order of the FP32 reduce-adds into its accumulator."""
    import torch
    from conftest import case
    fa = _fa()
    c = case("gpt2s")
    B, H, N, d = c.B, c.H, c.N, c.d
    q, k, v, do = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    for mode in (0, 1, 2):
        o, lse = fa.attention_fwd(q, k, v, c.causal, c.scale, mode)
        ref = fa.attention_bwd(q, k, v, o, lse, do, c.causal, c.scale, mode)
        for _call in range(2):
            got = [torch.full_like(q, float("nan")) for _ in range(3)]
            fa.fa_bwd_noalloc(q, k, v, o, lse, do, *got, B, H, N, d, c.causal, c.scale, mode)
            torch.cuda.synchronize()
            assert fa.fa_device_status() == 0
            assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]), (mode, _call)
            err = rel_fro(host_f64(got[0]), host_f64(ref[0]))
            assert err <= 1e-4, (mode, _call, err)

"""Per-head modes on the CUDA path (section 5, "Head-wise high-precision
substitution": the FP32 output only for the heads implicated in the failure,
here heads 1, 7, 8, 9, 11 and 12 of the page, 0-based 0, 6, 7, 8, 10, 11).

Each head's output, LSE, dK and dV must be bit-identical to those of a
uniform-mode call in that head's mode (the forward and the dK/dV
accumulation are deterministic); dQ (added across CTAs in no fixed order)
must agree to FP32 rounding.  Slices of the other dtype's buffer stay
untouched."""
import numpy as np
import pytest

from conftest import case
from gpu_helpers import dev_bf16

pytestmark = pytest.mark.gpu

FP32_HEADS = (0, 6, 7, 8, 10, 11)


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa as fa_mod
    return fa_mod


@pytest.mark.parametrize("other", [0, 1])
def test_head_modes_match_uniform_calls(fa, other):
    import torch
    c = case("gpt2s")
    B, H, N, d = c.B, c.H, c.N, c.d
    modes = [2 if h in FP32_HEADS else other for h in range(H)]
    q, k, v, do = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    o16 = torch.full((B, H, N, d), float("nan"), device="cuda", dtype=torch.bfloat16)
    o32 = torch.full((B, H, N, d), float("nan"), device="cuda", dtype=torch.float32)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    fa.fa_fwd_heads(q, k, v, o16, o32, lse, B, H, N, d, c.causal, c.scale, modes)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fa.fa_bwd_heads(q, k, v, o16, o32, lse, do, dq, dk, dv, B, H, N, d, c.causal, c.scale, modes)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ref = {}
    for m in sorted(set(modes)):
        o, l = fa.attention_fwd(q, k, v, c.causal, c.scale, m)
        ref[m] = (o, l) + fa.attention_bwd(q, k, v, o, l, do, c.causal, c.scale, m)
    torch.cuda.synchronize()
    for h in range(H):
        m = modes[h]
        o_ref, l_ref, dq_ref, dk_ref, dv_ref = (t[:, h] for t in ref[m])
        got_o, other_o = (o32, o16) if m == 2 else (o16, o32)
        assert torch.equal(got_o[:, h], o_ref), h
        assert torch.isnan(other_o[:, h].float()).all(), h   # the other buffer's slice untouched
        assert torch.equal(lse[:, h], l_ref), h
        assert torch.equal(dk[:, h], dk_ref) and torch.equal(dv[:, h], dv_ref), h
        rel = ((dq[:, h].float() - dq_ref.float()).norm() / dq_ref.float().norm()).item()
        assert rel < 1e-4, (h, rel)


@pytest.mark.parametrize("B,H,N,modes", [(3, 5, 300, [2, 0, 0, 0, 0]), (2, 7, 200, [1, 2, 2, 0, 1, 0, 2]),
                                         (1, 3, 129, [0, 0, 2])])
def test_sparse_head_sets(fa, B, H, N, modes):
    # a launch's item list holds only its own heads: every head of every set
    # size and position must come out as in the uniform call of its mode
    import torch
    from precision_flash_attention_attn_gb300.inputs import CaseSpec, make_custom
    c = make_custom(CaseSpec("heads", B, H, N, 64, True, 9400 + N + H, plant_frac=0.1, min_plant_row=3))
    q, k, v, do = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    o16 = torch.full((B, H, N, 64), float("nan"), device="cuda", dtype=torch.bfloat16)
    o32 = torch.full((B, H, N, 64), float("nan"), device="cuda", dtype=torch.float32)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    fa.fa_fwd_heads(q, k, v, o16, o32, lse, B, H, N, 64, True, c.scale, modes)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fa.fa_bwd_heads(q, k, v, o16, o32, lse, do, dq, dk, dv, B, H, N, 64, True, c.scale, modes)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for m in sorted(set(modes)):
        o, l = fa.attention_fwd(q, k, v, True, c.scale, m)
        gq, gk, gv = fa.attention_bwd(q, k, v, o, l, do, True, c.scale, m)
        torch.cuda.synchronize()
        for h in (h for h in range(H) if modes[h] == m):
            got = o32 if m == 2 else o16
            assert torch.equal(got[:, h], o[:, h]) and torch.equal(lse[:, h], l[:, h]), (m, h)
            assert torch.equal(dk[:, h], gk[:, h]) and torch.equal(dv[:, h], gv[:, h]), (m, h)
            rel = ((dq[:, h].float() - gq[:, h].float()).norm() / gq[:, h].float().norm()).item()
            assert rel < 1e-4, (m, h, rel)

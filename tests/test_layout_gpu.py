"""The [B, N, H, d] layout on the CUDA path: the kernels read and write the
tensors in place (4-D tensor maps), so every output must be bit-identical to
the [B, H, N, d] call on the same values, transposed (dQ, added across CTAs
in no fixed order, to FP32 rounding); the [B, H, N, d] path itself is
checked against the oracle elsewhere."""
import numpy as np
import pytest

from gpu_helpers import dev_bf16
from precision_flash_attention_attn_gb300.inputs import CaseSpec, make_custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa as fa_mod
    return fa_mod


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 200, 64, True), (1, 4, 384, 64, False), (2, 2, 257, 128, True),
                                              (8, 12, 1024, 64, True)])
def test_bnhd_matches_bhnd(fa, B, H, N, d, causal):
    import torch
    c = make_custom(CaseSpec("layout", B, H, N, d, causal, 9300 + N + d, plant_frac=0.1, min_plant_row=3))
    t = {n: dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do")}
    s = {n: x.transpose(1, 2).contiguous() for n, x in t.items()}   # [B, N, H, d]
    for mode in (0, 1, 2):
        for eps in ((None, 1e-3) if mode == 1 else (None,)):
            odt = torch.float32 if mode == 2 else torch.bfloat16
            o_ref = torch.empty((B, H, N, d), device="cuda", dtype=odt)
            l_ref = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
            fa.fa_fwd_ex(t["q"], t["k"], t["v"], o_ref, l_ref, B, H, N, d, causal, c.scale, mode, eps=eps)
            o = torch.empty((B, N, H, d), device="cuda", dtype=odt)
            lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
            fa.fa_fwd_layout(s["q"], s["k"], s["v"], o, lse, B, H, N, d, causal, c.scale, mode, fa.LAYOUT_BNHD,
                             eps=eps)
            torch.cuda.synchronize()
            assert torch.equal(o.transpose(1, 2), o_ref), (mode, eps)
            assert torch.equal(lse, l_ref), (mode, eps)
        g_ref = [torch.empty_like(t["q"]) for _ in range(3)]
        fa.fa_bwd(t["q"], t["k"], t["v"], o_ref, l_ref, t["do"], *g_ref, B, H, N, d, causal, c.scale, mode)
        g = [torch.empty_like(s["q"]) for _ in range(3)]
        fa.fa_bwd_layout(s["q"], s["k"], s["v"], o, lse, s["do"], *g, B, H, N, d, causal, c.scale, mode,
                         fa.LAYOUT_BNHD)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        assert torch.equal(g[1].transpose(1, 2), g_ref[1]) and torch.equal(g[2].transpose(1, 2), g_ref[2]), mode
        rel = ((g[0].transpose(1, 2).float() - g_ref[0].float()).norm() / g_ref[0].float().norm()).item()
        assert rel < 1e-4, (mode, rel)

"""The stabilised softmax with a near-tie tolerance eps > 0 on the CUDA path
("The modified safe softmax": rs = number of keys with scale*(rm - s) <= eps
over the whole row), against the oracle's exact forward, which counts near
ties the same way.

Tie counts must match the oracle bit for bit where the scores are exact in
FP32 (the constructed cases) and on the random workloads' rows; O and the LSE
stay within the usual bounds (the shift is exact in real arithmetic)."""
import numpy as np
import pytest

from conftest import case
from gpu_helpers import LSE_TOL, dev_bf16, f32, host_f64, o_bound
from oracle import oracle as orc
from precision_flash_attention_attn_gb300.inputs import bf16_bits

pytestmark = pytest.mark.gpu

# scores q.k of the constructed row: distances 0, 2^-7, 2^-4, 0, 1, 2^-7, 2.5,
# 0.25 from the maximum 1.5 (every value is BF16-exact, every score exact)
_EPS_A = [1.5, 1.4921875, 1.4375, 1.5, 0.5, 1.4921875, -1.0, 1.25]


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa as fa_mod
    return fa_mod


def _constructed(d=64):
    N = len(_EPS_A)
    q = np.zeros((1, 1, N, d), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, N, d), np.float32)
    k[0, 0, :, 0] = _EPS_A
    v = np.random.default_rng(5).standard_normal((1, 1, N, d)).astype(np.float32)
    return bf16_bits(q), bf16_bits(k), bf16_bits(v)


def _stats(fa, qb, kb, vb, causal, scale, mode, eps, beta=None):
    import torch
    q, k, v = dev_bf16(qb), dev_bf16(kb), dev_bf16(vb)
    B, H, N, d = qb.shape
    o, lse = fa.attention_fwd(q, k, v, causal, scale, mode)
    o = torch.empty_like(o)
    lse = torch.empty_like(lse)
    fa.fa_fwd_ex(q, k, v, o, lse, B, H, N, d, causal, scale, mode, beta=beta, eps=eps)
    tc = torch.empty((B, H, N), device="cuda", dtype=torch.int32)
    pe = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    po = torch.empty((2, B, H, N), device="cuda", dtype=torch.int32)
    fa.fa_tie_stats_ex(q, k, v, o, B, H, N, d, causal, scale, mode, tc, pe, po, beta=beta, eps=eps)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return host_f64(o), host_f64(lse), tc.cpu().numpy().reshape(-1), po.cpu().numpy().reshape(2, -1)


@pytest.mark.parametrize("scale,eps,count", [
    (1.0, 0.005, 2), (1.0, 0.0078125, 4), (1.0, 0.01, 4), (1.0, 0.0625, 5), (1.0, 0.3, 6), (1.0, 3.0, 8),
    (0.5, 0.0038, 2), (0.5, 0.004, 4), (0.5, 0.03, 4), (0.5, 0.032, 5), (0.5, 0.12, 5), (0.5, 0.13, 6),
])
def test_near_tie_counts_by_construction(fa, scale, eps, count):
    qb, kb, vb = _constructed()
    for mode in (0, 1, 2):
        o, lse, tc, _ = _stats(fa, qb, kb, vb, False, scale, mode, eps)
        assert np.all(tc == count), (mode, tc)
        ex = orc.fwd(f32(qb).reshape(1, 8, 64), f32(kb).reshape(1, 8, 64), f32(vb).reshape(1, 8, 64), False,
                     scale, mode, eps=eps)
        assert np.all(ex["ties"].reshape(-1) == count)
        assert np.all(np.abs(o.reshape(8, 64) - ex["o"].reshape(8, 64)) <= o_bound(ex["o"].reshape(8, 64), mode))
        assert np.abs(lse.reshape(-1) - ex["lse"].reshape(-1)).max() <= LSE_TOL


def test_near_tie_counts_causal_prefixes(fa):
    qb, kb, vb = _constructed()
    _, _, tc, _ = _stats(fa, qb, kb, vb, True, 1.0, 1, 0.01)
    assert tc.tolist() == [1, 2, 2, 3, 3, 4, 4, 4]


@pytest.mark.parametrize("eps", [1e-3, 0.05])
def test_tiny_workload(fa, eps):
    # every row: near-tie counts bit-exact against the oracle, O and LSE in
    # bound, and no key with a final weight of 1 on rows with rs > 1 whose
    # scaled maximum is not tiny (the stabilised rule's purpose)
    c = case("tiny")
    BH = c.B * c.H
    qf, kf, vf = (f32(getattr(c, n)).reshape(BH, c.N, c.d) for n in ("q", "k", "v"))
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 1, eps=eps)
    o, lse, tc, po = _stats(fa, c.q, c.k, c.v, c.causal, c.scale, 1, eps)
    np.testing.assert_array_equal(tc, ex["ties"].reshape(-1))
    oe = ex["o"].reshape(-1, c.d)
    assert np.all(np.abs(o.reshape(-1, c.d) - oe) <= o_bound(oe, 1))
    assert np.abs(lse.reshape(-1) - ex["lse"].reshape(-1)).max() <= LSE_TOL
    rm = np.array([(kf[r // c.N, : r % c.N + 1] @ qf[r // c.N, r % c.N]).max() for r in range(BH * c.N)])
    rows = np.flatnonzero((tc > 1) & (np.abs(c.scale * rm) > 2.0 ** -8))
    assert rows.size > 20
    assert np.all(po[1][rows] == 0) and np.all(po[0][rows] == 0)


def test_gpt2s_sampled_rows(fa):
    c = case("gpt2s")
    BH = c.B * c.H
    qf, kf, vf = (f32(getattr(c, n)).reshape(BH, c.N, c.d) for n in ("q", "k", "v"))
    o, lse, tc, _ = _stats(fa, c.q, c.k, c.v, c.causal, c.scale, 1, 1e-3)
    rng = np.random.default_rng(3)
    planted = np.flatnonzero(c.planted.reshape(-1))
    rows = np.unique(np.concatenate([rng.choice(BH * c.N, 512, replace=False), planted[::20]]))
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 1, eps=1e-3, rows=rows)
    np.testing.assert_array_equal(tc[rows], ex["ties"])
    og = o.reshape(-1, c.d)[rows]
    assert np.all(np.abs(og - ex["o"]) <= o_bound(ex["o"], 1))
    assert np.abs(lse.reshape(-1)[rows] - ex["lse"]).max() <= LSE_TOL

"""Tie statistics of the CUDA path against the oracle: tie counts bit-exact,
unit-probability counts against the oracle's BF16 emulation (within the keys
whose FP32 probability sits on the BF16 rounding boundary), and the signed
output error pv_err against the oracle's exact output."""
import numpy as np
import pytest

from conftest import case
from gpu_helpers import dev_bf16, f32
from oracle import oracle as orc
from precision_flash_attention_attn_gb300.inputs import CaseSpec, bf16_bits, make_custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    from precision_flash_attention_attn_gb300 import fa as fa_mod
    return fa_mod


def _arrays(c):
    BH = c.B * c.H
    return [f32(getattr(c, n)).reshape(BH, c.N, c.d) for n in ("q", "k", "v")]


def _stats(fa, c, mode, o=None, beta=None):
    import torch
    q, k, v = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v"))
    if o is None:
        o, _ = fa.attention_fwd(q, k, v, c.causal, c.scale, mode, beta=beta)
    tc, pe, po = fa.tie_stats(q, k, v, o, c.causal, c.scale, mode, beta=beta)
    assert fa.fa_device_status() == 0
    torch.cuda.synchronize()
    return tc.cpu().numpy().reshape(-1), pe.cpu().numpy().reshape(-1).astype(np.float64), po.cpu().numpy().reshape(2, -1)


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "gpt2m", "long", "ties"])
def test_tie_counts_bit_exact(fa, name):
    c = case(name)
    tc, _, _ = _stats(fa, c, 0)
    chk = c.checked.reshape(-1)
    np.testing.assert_array_equal(tc[chk], c.ties.reshape(-1)[chk])
    # and against the oracle's own count on a sample of checked rows
    rows = np.flatnonzero(chk)
    rows = rows[np.random.default_rng(5).choice(rows.size, size=min(2048, rows.size), replace=False)]
    qf, kf, vf = _arrays(c)
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 0, rows=rows)
    np.testing.assert_array_equal(tc[rows], ex["ties"])


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("name", ["tiny", "gpt2s"])
def test_unit_probability_counts_match_emulation(fa, name, mode):
    c = case(name)
    _, _, po = _stats(fa, c, mode)
    qf, kf, vf = _arrays(c)
    BH = c.B * c.H
    rows = np.arange(BH * c.N) if name == "tiny" else \
        np.random.default_rng(6).choice(BH * c.N, size=4096, replace=False)
    em = orc.fwd_emul(qf, kf, vf, c.causal, c.scale, mode, block_n=128, rows=rows)
    amb = em["p_amb"]
    for idx, key in ((0, "p_one0"), (1, "p_one1")):
        diff = np.abs(po[idx][rows] - em[key])
        assert np.all(diff <= amb), (key, int(diff.max()))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_pv_err_matches_oracle(fa, mode):
    import torch
    c = case("tiny")
    qf, kf, vf = _arrays(c)
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 0)
    em = orc.fwd_emul(qf, kf, vf, c.causal, c.scale, mode, block_n=128)
    o_in = em["o"].reshape(c.q.shape)          # an output produced by the oracle
    if mode == 2:
        o_dev = torch.from_numpy(o_in.astype(np.float32)).cuda()
    else:
        o_dev = dev_bf16(bf16_bits(o_in.astype(np.float32)))
    _, pe, _ = _stats(fa, c, mode, o=o_dev)
    want = (o_in.reshape(-1, c.d) - ex["o"].reshape(-1, c.d)).sum(1)
    np.testing.assert_allclose(pe, want, rtol=0, atol=2e-4)


def test_stabilised_mode_has_no_unit_probability_on_tied_rows(fa):
    # invariant: on planted-tie rows the stabilised softmax feeds no Pbar = 1
    # (a single 128-key tile holds every key of the tiny workload), while the
    # baseline feeds at least one per tied key
    c = case("tiny")
    tc0, _, po0 = _stats(fa, c, 0)
    tc1, _, po1 = _stats(fa, c, 1)
    qf, kf, vf = _arrays(c)
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 0)
    smax = (ex["lse"].reshape(-1) * 0)  # shape holder
    rows = np.flatnonzero(c.planted.reshape(-1) & (tc0 > 1))
    # rows whose scaled max is tiny cannot avoid bf16(exp) == 1 (excluded, counted)
    BH = c.B * c.H
    s_max = np.array([max(qf[r // c.N, r % c.N] @ kf[r // c.N, j] for j in range((r % c.N) + 1)) for r in rows])
    keep = rows[np.abs(c.scale * s_max) > 2.0 ** -8]
    assert keep.size > 20
    assert np.all(po1[0][keep] == 0) and np.all(po1[1][keep] == 0)
    assert np.all(po0[0][keep] >= tc0[keep])
    del smax, BH


@pytest.mark.parametrize("beta", [4.0, 8.0])
@pytest.mark.parametrize("name", ["tiny", "gpt2s"])
def test_unit_probability_counts_match_emulation_beta(fa, name, beta):
    # mode 1 with a run-time shift factor: the counts follow the emulation run
    # with the same beta (the product beta * M is formed in FP32 on both sides)
    c = case(name)
    _, _, po = _stats(fa, c, 1, beta=beta)
    qf, kf, vf = _arrays(c)
    BH = c.B * c.H
    rows = np.arange(BH * c.N) if name == "tiny" else \
        np.random.default_rng(7).choice(BH * c.N, size=4096, replace=False)
    em = orc.fwd_emul(qf, kf, vf, c.causal, c.scale, 1, beta=beta, block_n=128, rows=rows)
    amb = em["p_amb"]
    for idx, key in ((0, "p_one0"), (1, "p_one1")):
        diff = np.abs(po[idx][rows] - em[key])
        assert np.all(diff <= amb), (key, int(diff.max()))


def test_stabilised_invariant_with_beta_8(fa):
    # the invariant of the stabilised rule holds for any beta > 1: no Pbar = 1
    # on planted-tie rows whose scaled max is not tiny
    c = case("tiny")
    tc0, _, _ = _stats(fa, c, 0)
    _, _, po = _stats(fa, c, 1, beta=8.0)
    qf, kf, _ = _arrays(c)
    rows = np.flatnonzero(c.planted.reshape(-1) & (tc0 > 1))
    s_max = np.array([max(qf[r // c.N, r % c.N] @ kf[r // c.N, j] for j in range((r % c.N) + 1)) for r in rows])
    keep = rows[np.abs(c.scale * s_max) > 2.0 ** -8]
    assert keep.size > 20
    assert np.all(po[0][keep] == 0) and np.all(po[1][keep] == 0)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_delta_err_matches_oracle(fa, mode):
    # delta_lp - delta_hp = sum_c dO (O - O_hp) ("Cause 2: Biased Rounding Error
    # Leads to Positive (delta_lp - delta_hp)[T]"), for an output O produced by
    # the oracle's emulation, against the oracle's exact output as O_hp
    import torch
    c = case("tiny")
    qf, kf, vf = _arrays(c)
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 0)
    em = orc.fwd_emul(qf, kf, vf, c.causal, c.scale, mode, block_n=128)
    o_in = em["o"].reshape(c.q.shape)
    if mode == 2:
        o_dev = torch.from_numpy(o_in.astype(np.float32)).cuda()
    else:
        o_dev = dev_bf16(bf16_bits(o_in.astype(np.float32)))
    q, k, v, g = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    de = fa.delta_error(q, k, v, o_dev, g, c.causal, c.scale, mode)
    assert fa.fa_device_status() == 0
    gf = f32(c.do).reshape(-1, c.d).astype(np.float64)
    want = (gf * (o_in.reshape(-1, c.d) - ex["o"].reshape(-1, c.d))).sum(1)
    np.testing.assert_allclose(de.cpu().numpy().reshape(-1), want, rtol=0, atol=2e-4 * max(1.0, np.abs(gf).max()))


def test_delta_err_with_unit_gradient_is_pv_err(fa):
    # with dO = 1 the weighted sum is the plain one, term for term
    import torch
    c = case("tiny")
    q, k, v = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v"))
    o, _ = fa.attention_fwd(q, k, v, c.causal, c.scale, 0)
    ones = torch.ones_like(q)
    B, H, N, d = q.shape
    tc = torch.empty((B, H, N), device="cuda", dtype=torch.int32)
    pe = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    de = torch.empty_like(pe)
    fa.fa_tie_stats_ex(q, k, v, o, B, H, N, d, c.causal, c.scale, 0, tc, pe, None, dO=ones, delta_err=de)
    assert fa.fa_device_status() == 0
    assert torch.equal(pe, de)


def test_beta_sweep_runs_on_tiny(fa, capsys):
    # the sweep module end to end: one line per setting; the baseline feeds
    # Pbar = 1 on every tied row, the stabilised settings leave fewer keys
    # with a final weight of exactly 1, and nothing underflows at this scale
    import json
    from precision_flash_attention_attn_gb300 import beta_sweep
    assert beta_sweep.main(["--workload", "tiny", "--betas", "2,8"]) == 0
    lines = [json.loads(ln) for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert [ln["setting"] for ln in lines] == ["baseline", "stabilised beta=2", "stabilised beta=8"]
    assert lines[0]["tied_rows"] > 20 and lines[0]["p_one0_rows"] == 1.0
    for ln in lines[1:]:
        assert ln["p_one1_mean"] < lines[0]["p_one1_mean"]
        assert ln["nonfinite_rows"] == 0
    # the delta error's three parts add up to it (row by row, so in the mean)
    for ln in lines:
        sp = ln["delta_split"]
        total = sp["one"]["mean"] + sp["rest"]["mean"] + sp["out"]["mean"]
        assert abs(total - ln["delta_err"]["mean"]) <= 1e-5, (ln["setting"], total, ln["delta_err"])


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_delta_error_split_matches_oracle(fa, mode):
    # the decomposition of delta_lp - delta_hp (keys with BF16 probability 1,
    # the rest, the output rounding) for an output produced by the oracle's
    # emulation, against the oracle's FP64 decomposition of the same output;
    # the three parts add up to the statistics kernel's delta_err
    import torch
    c = case("tiny")
    qf, kf, vf = _arrays(c)
    gf = f32(c.do).reshape(c.B * c.H, c.N, c.d)
    em = orc.fwd_emul(qf, kf, vf, c.causal, c.scale, mode, block_n=128)
    o_in = em["o"].reshape(c.q.shape)
    if mode == 2:
        o_dev = torch.from_numpy(o_in.astype(np.float32)).cuda()
    else:
        o_dev = dev_bf16(bf16_bits(o_in.astype(np.float32)))
    q, k, v, g = (dev_bf16(getattr(c, n)) for n in ("q", "k", "v", "do"))
    one, rest, out = (t.cpu().numpy().reshape(-1).astype(np.float64)
                      for t in fa.delta_error_split(q, k, v, o_dev, g, c.causal, c.scale, mode))
    de = fa.delta_error(q, k, v, o_dev, g, c.causal, c.scale, mode).cpu().numpy().reshape(-1)
    assert fa.fa_device_status() == 0
    want = orc.delta_split(qf, kf, vf, o_in.reshape(qf.shape).astype(np.float32), gf, c.causal, c.scale, mode)
    tol = 2e-4 * max(1.0, np.abs(gf).max())
    np.testing.assert_allclose(one, want["one"].reshape(-1), rtol=0, atol=tol)
    np.testing.assert_allclose(rest, want["rest"].reshape(-1), rtol=0, atol=tol)
    np.testing.assert_allclose(out, want["out"].reshape(-1), rtol=0, atol=tol)
    np.testing.assert_allclose(one + rest + out, de, rtol=0, atol=tol)
    if mode == 1:
        # no key of a tied row with a non-tiny positive or negative maximum
        # keeps probability 1, so the unit part vanishes there
        tied = np.flatnonzero(c.planted.reshape(-1) & (c.ties.reshape(-1) > 1))
        s_max = np.array([(kf[r // c.N, : r % c.N + 1] @ qf[r // c.N, r % c.N]).max() for r in tied])
        keep = tied[np.abs(c.scale * s_max) > 2.0 ** -8]
        assert keep.size > 20 and np.all(one[keep] == 0.0)

"""Pins of the FP64 CPU oracle against facts that do not come from the oracle.

Every check here ties the oracle to something outside itself: the worked BF16
example printed in "Why Low-Precision Transformer Training Fails: An Analysis
on Flash Attention" (section 3.4.4), closed forms of softmax attention, an
independent library routine (torch float64 scaled-dot-product attention and
autograd), central finite differences, exact rational arithmetic, the
statements of what each line of the stabilised softmax does (section 3.4.5),
and hand-worked BF16 sums.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from conftest import ROOT, case
from oracle import oracle as orc
from precision_flash_attention_attn_gb300.inputs import bf16_bits, bf16_bits_to_f32

GOLDEN = os.path.join(ROOT, "tests", "golden")


def _bits_to_f32(bits: str) -> np.float32:
    return np.array([int(bits, 2)], np.uint32).view(np.float32)[0]


def _f32_bits(x) -> str:
    return format(int(np.array([x], np.float32).view(np.uint32)[0]), "032b")


def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, bits, val = line.split()
            rows[key] = (bits, val)
    return rows


# ---------------------------------------------------------------------------
# BF16 rounding: the pages' worked example, and an independent definition
# ---------------------------------------------------------------------------

def test_bf16_worked_example_bit_exact():
    g = _read_golden("bf16_worked_example.txt")
    a = _bits_to_f32(g["fp32_a"][0])
    b = _bits_to_f32(g["fp32_b"][0])
    assert float(a) == float(g["fp32_a"][1])
    assert float(b) == float(g["fp32_b"][1])
    s = np.float32(a) + np.float32(b)                       # FP32 addition
    assert _f32_bits(s) == g["fp32_sum"][0]
    assert float(s) == pytest.approx(float(g["fp32_sum"][1]), abs=0, rel=1e-15)
    r = orc.bf16_round(np.array([s], np.float32))[0]
    assert _f32_bits(r)[:16] == g["bf16_result"][0] and _f32_bits(r)[16:] == "0" * 16
    assert float(r) == float(g["bf16_result"][1])
    # the error of the rounded sum against the exact sum of the two inputs
    assert float(r) - (float(a) + float(b)) == float(g["error"][1])


def _bf16_round_by_distance(x: np.float32) -> float:
    """Nearest BF16 by exact distance, ties to even mantissa (independent of
    the bit trick used by the oracle)."""
    u = int(np.array([x], np.float32).view(np.uint32)[0])
    lo = u & 0xFFFF0000
    hi = lo + 0x10000
    flo = Fraction(float(np.array([lo], np.uint32).view(np.float32)[0]))
    fhi = Fraction(float(np.array([hi], np.uint32).view(np.float32)[0]))
    fx = Fraction(float(x))
    dlo, dhi = abs(fx - flo), abs(fhi - fx)
    if dlo < dhi:
        return float(flo)
    if dhi < dlo:
        return float(fhi)
    return float(flo) if ((lo >> 16) & 1) == 0 else float(fhi)


def test_bf16_round_matches_exact_nearest_even():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    # add exact halfway cases and values just around them
    base = bf16_bits_to_f32(bf16_bits(rng.standard_normal(500).astype(np.float32)))
    half = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, half, np.nextafter(half, np.float32(np.inf)),
                        np.nextafter(half, np.float32(-np.inf))]).astype(np.float32)
    y = orc.bf16_round(x)
    want = np.array([_bf16_round_by_distance(v) for v in x])
    assert np.array_equal(y.astype(np.float64), want)


# ---------------------------------------------------------------------------
# Forward: closed forms
# ---------------------------------------------------------------------------

def _rand_bf16(rng, shape, sigma=1.0):
    return bf16_bits_to_f32(bf16_bits(rng.standard_normal(shape).astype(np.float32) * sigma))


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_uniform_scores_give_mean_of_visible_values(causal, mode):
    rng = np.random.default_rng(1)
    BH, N, d = 2, 37, 16
    q = np.zeros((BH, N, d), np.float32)
    k = _rand_bf16(rng, (BH, N, d))
    v = _rand_bf16(rng, (BH, N, d))
    f = orc.fwd(q, k, v, causal, 0.25, mode)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(f["o"][:, i], v[:, :n].astype(np.float64).mean(1), rtol=0, atol=1e-13)
        np.testing.assert_allclose(f["lse"][:, i], math.log(n), rtol=0, atol=1e-13)
        # every score is 0, so every visible key ties at the maximum
        assert np.all(f["ties"][:, i] == n)


def test_one_hot_scores_select_a_value_row():
    rng = np.random.default_rng(2)
    BH, N, d = 1, 9, 4
    k = _rand_bf16(rng, (BH, N, d), 0.01)
    v = _rand_bf16(rng, (BH, N, d))
    q = np.zeros((BH, N, d), np.float32)
    jstar = 5
    k[0, jstar] = [16.0, 0, 0, 0]
    q[0, :, 0] = 8.0                       # scaled score gap >= 0.5*(128 - small) > 50
    f = orc.fwd(q, k, v, 0, 0.5, 0)
    np.testing.assert_allclose(f["o"][0], np.broadcast_to(v[0, jstar], (N, d)), atol=1e-20)


@pytest.mark.parametrize("causal", [0, 1])
def test_delta_closed_forms(causal):
    # delta = rowsum(dO o O) (section 3.4.2, "Failure is linked to the
    # computation of delta"), where O is known in closed form: the mean of the
    # visible values when every score is equal, and one value row when a single
    # key dominates
    rng = np.random.default_rng(4)
    BH, N, d = 2, 23, 8
    k = _rand_bf16(rng, (BH, N, d))
    v = _rand_bf16(rng, (BH, N, d))
    g = _rand_bf16(rng, (BH, N, d))
    f = orc.fwd(np.zeros((BH, N, d), np.float32), k, v, causal, 0.5, 0, dout=g)
    for i in range(N):
        n = i + 1 if causal else N
        mean_v = v[:, :n].astype(np.float64).mean(1)
        want = (g[:, i].astype(np.float64) * mean_v).sum(1)
        np.testing.assert_allclose(f["delta"][:, i], want, rtol=0, atol=1e-12)
    q = np.zeros((BH, N, d), np.float32)
    q[:, :, 0] = 8.0
    k2 = _rand_bf16(rng, (BH, N, d), 0.01)
    k2[:, 0] = [16.0] + [0.0] * (d - 1)     # key 0 is visible to every row and dominates
    f = orc.fwd(q, k2, v, causal, 0.5, 0, dout=g)
    want = np.einsum("bnc,bc->bn", g.astype(np.float64), v[:, 0].astype(np.float64))
    np.testing.assert_allclose(f["delta"], want, rtol=0, atol=1e-12)


def test_causal_first_row_is_first_value_row():
    rng = np.random.default_rng(3)
    BH, N, d = 3, 20, 8
    q, k, v = (_rand_bf16(rng, (BH, N, d)) for _ in range(3))
    f = orc.fwd(q, k, v, 1, 0.3, 0)
    np.testing.assert_array_equal(f["o"][:, 0], v[:, 0].astype(np.float64))
    want = 0.3 * np.einsum("bc,bc->b", q[:, 0].astype(np.float64), k[:, 0].astype(np.float64))
    np.testing.assert_allclose(f["lse"][:, 0], want, rtol=0, atol=1e-14)


def test_causal_mask_ignores_future_keys_bit_exact():
    rng = np.random.default_rng(4)
    BH, N, d = 2, 24, 8
    q, k, v = (_rand_bf16(rng, (BH, N, d)) for _ in range(3))
    base = orc.fwd(q, k, v, 1, 0.35, 0)
    i = 11
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1:] = _rand_bf16(rng, (BH, N - i - 1, d), 5.0)
    v2[:, i + 1:] = _rand_bf16(rng, (BH, N - i - 1, d), 5.0)
    pert = orc.fwd(q, k2, v2, 1, 0.35, 0)
    np.testing.assert_array_equal(base["o"][:, : i + 1], pert["o"][:, : i + 1])
    np.testing.assert_array_equal(base["lse"][:, : i + 1], pert["lse"][:, : i + 1])


# ---------------------------------------------------------------------------
# Forward: an independent library routine
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_forward_and_gradients_match_torch_float64(causal):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    BH, N, d = 3, 45, 16
    q, k, v, g = (_rand_bf16(rng, (BH, N, d)) for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    (out * torch.tensor(g, dtype=torch.float64)).sum().backward()
    f = orc.fwd(q, k, v, int(causal), scale, 0)
    np.testing.assert_allclose(f["o"], out.detach().numpy(), rtol=0, atol=1e-12)
    s = torch.einsum("bic,bjc->bij", tq.detach(), tk.detach()) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(f["lse"], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)
    gr = orc.bwd(q, k, v, g, int(causal), scale)
    np.testing.assert_allclose(gr["dq"], tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(gr["dk"], tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(gr["dv"], tv.grad.numpy(), rtol=0, atol=1e-11)


# ---------------------------------------------------------------------------
# Backward: central finite differences of L = sum(dO o O)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [0, 1])
def test_backward_matches_central_differences(causal):
    rng = np.random.default_rng(6)
    BH, N, d = 1, 7, 4
    q, k, v, g = (_rand_bf16(rng, (BH, N, d), 0.5) for _ in range(4))
    scale = 0.5
    h = 2.0 ** -12          # x +- h is exact in FP32 for these BF16 values

    def loss(q_, k_, v_):
        return float((orc.fwd(q_, k_, v_, causal, scale, 0)["o"] * g.astype(np.float64)).sum())

    gr = orc.bwd(q, k, v, g, causal, scale)
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros(arr.shape)
        for idx in np.ndindex(arr.shape):
            xp, xm = arr.copy(), arr.copy()
            xp[idx] += np.float32(h)
            xm[idx] -= np.float32(h)
            assert float(xp[idx]) - float(arr[idx]) == h
            args_p = {"dq": (xp, k, v), "dk": (q, xp, v), "dv": (q, k, xp)}[name]
            args_m = {"dq": (xm, k, v), "dk": (q, xm, v), "dv": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        ana = gr[name].reshape(arr.shape)
        err = np.abs(ana - num).max() / max(np.abs(num).max(), 1e-30)
        assert err <= 1e-6, (name, err)


# ---------------------------------------------------------------------------
# Tie counts: exact rational arithmetic on a planted workload
# ---------------------------------------------------------------------------

def test_tie_counts_match_exact_rationals():
    c = case("tiny")
    q = c.f64("q").reshape(-1, c.N, c.d)
    k = c.f64("k").reshape(-1, c.N, c.d)
    v = c.f64("v").reshape(-1, c.N, c.d)
    f = orc.fwd(q, k, v, c.causal, c.scale, 0)
    BH = q.shape[0]
    for bh in range(BH):
        kf = [[Fraction(x) for x in row] for row in k[bh]]
        for i in range(c.N):
            qi = [Fraction(x) for x in q[bh, i]]
            sc = [sum(a * b for a, b in zip(qi, kf[j])) for j in range(i + 1)]
            mx = max(sc)
            assert f["ties"][bh, i] == sum(1 for s in sc if s == mx)
    # and the generator's own bookkeeping agrees on every checked row
    np.testing.assert_array_equal(f["ties"].reshape(c.ties.shape)[c.checked], c.ties[c.checked])
    assert (f["ties"] > 1).sum() > 0.2 * f["ties"].size


# ---------------------------------------------------------------------------
# Stabilised softmax: shift rule and exactness of the shift
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("beta", [2.0, 8.0])
def test_shift_rule_branches(beta):
    # rm > 0 with repeated maxima: the largest exponent becomes -(beta-1)*rm
    for rm in (0.25, 3.0, 40.0):
        assert rm - orc.row_shift(rm, 2, 1, beta) == pytest.approx(-(beta - 1) * rm, rel=1e-15)
        assert rm - orc.row_shift(rm, 5, 1, beta) < 0
    # rm < 0 with repeated maxima: shift 0, the largest exponent stays rm < 0
    for rm in (-0.25, -7.0):
        assert orc.row_shift(rm, 3, 1, beta) == 0.0
    # a unique maximum, and the baseline / FP32-output modes: plain row max
    for rm in (-3.0, 0.0, 2.5):
        assert orc.row_shift(rm, 1, 1, beta) == rm
        for mode in (0, 2):
            assert orc.row_shift(rm, 4, mode, beta) == rm
    # rm == 0 with repeated maxima: neither strict condition holds
    assert orc.row_shift(0.0, 3, 1, beta) == 0.0


def test_stabilised_shift_is_exact_in_fp64():
    c = case("tiny")
    q = c.f64("q").reshape(-1, c.N, c.d)
    k = c.f64("k").reshape(-1, c.N, c.d)
    v = c.f64("v").reshape(-1, c.N, c.d)
    base = orc.fwd(q, k, v, 1, c.scale, 0)
    for beta in (2.0, 8.0):
        stab = orc.fwd(q, k, v, 1, c.scale, 1, beta=beta)
        np.testing.assert_allclose(stab["o"], base["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(stab["lse"], base["lse"], rtol=0, atol=1e-12)
    # the comparison is not vacuous: many rows take a shifted branch
    assert (base["ties"] > 1).sum() > 50


# ---------------------------------------------------------------------------
# BF16 emulation of the tiled forward
# ---------------------------------------------------------------------------

def _tiny_arrays(**kw):
    c = case("tiny", **kw)
    return c, [c.f64(n).reshape(-1, c.N, c.d) for n in ("q", "k", "v")]


def test_emulation_single_tile_stabilised_has_no_unit_probability():
    c, (q, k, v) = _tiny_arrays()
    ex = orc.fwd(q, k, v, 1, c.scale, 0)
    e0 = orc.fwd_emul(q, k, v, 1, c.scale, 0, block_n=c.N)
    e1 = orc.fwd_emul(q, k, v, 1, c.scale, 1, block_n=c.N)
    tied = ex["ties"] > 1
    # rows excluded by the small-|rm| reading: |alpha * rowmax| <= 2^-8
    s_max = np.array([[max(q[b, i] @ k[b, j] for j in range(i + 1)) for i in range(c.N)]
                      for b in range(q.shape[0])])
    ok = tied & (np.abs(c.scale * s_max) > 2.0 ** -8)
    assert ok.sum() > 50
    # baseline: every tied maximum enters the product as exactly 1.0
    assert np.all(e0["p_one0"][ok] >= ex["ties"][ok])
    assert np.all(e0["p_max"][tied] == 1.0)
    # stabilised: no entry of Pbar equals 1 and none exceeds it
    assert np.all(e1["p_one0"][ok] == 0)
    assert np.all(e1["p_one1"][ok] == 0)
    assert np.all(e1["p_max"][ok] < 1.0)
    # untied rows are unchanged by the stabilised rule
    np.testing.assert_array_equal(e1["o"][~tied], e0["o"][~tied])


@pytest.mark.parametrize("beta", [2.0, 4.0, 8.0])
def test_emulation_largest_probability_follows_beta(beta):
    # "What each line does": on a row with a repeated maximum rm > 0 the largest
    # exponent becomes -(beta-1)*rm, on one with rm < 0 it stays rm (m = 0).  The
    # emulation's largest BF16 Pbar of such a row is that exponential, up to
    # BF16 rounding.
    c, (q, k, v) = _tiny_arrays()
    ex = orc.fwd(q, k, v, 1, c.scale, 0)
    em = orc.fwd_emul(q, k, v, 1, c.scale, 1, beta=beta, block_n=c.N)
    s_max = np.array([[max(q[b, i].astype(np.float64) @ k[b, j].astype(np.float64) for j in range(i + 1))
                       for i in range(c.N)] for b in range(q.shape[0])])
    rmz = c.scale * s_max
    tied = ex["ties"] > 1
    pos, neg = tied & (rmz > 2.0 ** -4), tied & (rmz < -(2.0 ** -4))
    assert pos.sum() > 20 and neg.sum() >= 1
    want = np.where(rmz > 0, np.exp(-(beta - 1.0) * rmz), np.exp(rmz))
    for sel in (pos, neg):
        np.testing.assert_allclose(em["p_max"][sel], want[sel], rtol=2.0 ** -8, atol=0)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("block_n", [16, 128])
def test_emulation_output_is_within_bf16_error_of_exact(mode, block_n):
    c, (q, k, v) = _tiny_arrays()
    ex = orc.fwd(q, k, v, 1, c.scale, 0)
    em = orc.fwd_emul(q, k, v, 1, c.scale, mode, block_n=block_n)
    # Pbar carries a relative error <= 2^-8 from BF16 rounding (2^-9) and the
    # l / Obar mismatch; the output adds half a BF16 ulp in modes 0 and 1.
    vmax = np.abs(v).max()
    bound = 2.0 ** -8 * vmax + (0 if mode == 2 else 2.0 ** -9 * np.abs(ex["o"]).max())
    assert np.abs(em["o"] - ex["o"]).max() <= bound
    np.testing.assert_allclose(em["lse"], ex["lse"], rtol=0, atol=1e-6)


def test_emulation_tiled_ties_across_tiles():
    # With 16-key tiles a running maximum is fed as 1.0 in its own tile before
    # a later tile raises the maximum or supplies its tie partner; the rescale
    # then lowers its weight.  No key keeps a final weight of exactly 1 on a
    # tied row, and the stabilised rule never adds unit entries.
    c, (q, k, v) = _tiny_arrays()
    e0 = orc.fwd_emul(q, k, v, 1, c.scale, 0, block_n=16)
    e1 = orc.fwd_emul(q, k, v, 1, c.scale, 1, block_n=16)
    ex = orc.fwd(q, k, v, 1, c.scale, 0)
    tied = ex["ties"] > 1
    assert np.all(e1["p_one1"][tied] == 0)
    assert np.all(e1["p_one0"] <= e0["p_one0"])
    assert np.all(e0["p_one1"][tied] >= ex["ties"][tied])
    assert (e1["p_one0"][tied] > 0).any()   # the cross-tile case does occur


def test_per_addition_rounding_hand_worked():
    # One query, three identical keys (all tied, Pbar = 1 under the baseline).
    # Per-addition BF16 sums, worked by hand:
    #   -2.40625 + -2.296875 = -4.703125, exactly halfway between the BF16
    #   neighbours -4.6875 and -4.71875 -> even mantissa -> -4.6875;
    #   -4.6875 + -1.0 = -5.6875 (representable).
    q = np.zeros((1, 3, 8), np.float32)
    q[0, :, 0] = 1.0
    k = np.zeros((1, 3, 8), np.float32)
    k[0, :, 0] = 0.5
    v = np.zeros((1, 3, 8), np.float32)
    v[0, :, 0] = [-2.40625, -2.296875, -1.0]
    em = orc.fwd_emul(q, k, v, 0, 1.0, 0, block_n=128)
    ex = orc.fwd(q, k, v, 0, 1.0, 0)
    assert em["o_peradd"][0, 2, 0] == -5.6875 / 3
    assert ex["o"][0, 2, 0] == pytest.approx(-5.703125 / 3, rel=1e-15)
    assert em["p_one0"][0, 2] == 3


# Near-tie tolerance eps > 0 (section 3.4.5, "rs = rowsum(rm - S <= eps)"): one
# query e_0 against keys whose first component is a chosen BF16-exact value,
# so the raw score of key j is exactly A[j] and the distances to the maximum
# 1.5 are known by construction: 0 (twice), 2^-7 (twice), 2^-4, 0.25, 1, 2.5.
_EPS_A = [1.5, 1.4921875, 1.4375, 1.5, 0.5, 1.4921875, -1.0, 1.25]


def _eps_inputs():
    N, d = len(_EPS_A), 4
    q = np.zeros((1, N, d), np.float32)
    q[0, :, 0] = 1.0
    k = np.zeros((1, N, d), np.float32)
    k[0, :, 0] = _EPS_A
    v = bf16_bits_to_f32(bf16_bits(np.random.default_rng(5).standard_normal((1, N, d)).astype(np.float32)))
    return q, k, v


@pytest.mark.parametrize("scale,eps,count", [
    (1.0, 0.0, 2), (1.0, 0.005, 2), (1.0, 0.0078125, 4), (1.0, 0.01, 4), (1.0, 0.0625, 5),
    (1.0, 0.3, 6), (1.0, 3.0, 8),
    (0.5, 0.0038, 2), (0.5, 0.004, 4), (0.5, 0.03, 4), (0.5, 0.032, 5), (0.5, 0.12, 5), (0.5, 0.13, 6),
])
def test_near_tie_counts_by_construction(scale, eps, count):
    q, k, v = _eps_inputs()
    f = orc.fwd(q, k, v, 0, scale, 1, eps=eps)
    assert np.all(f["ties"] == count)


def test_near_tie_counts_causal_prefixes():
    # causal row i sees keys 0..i only: count the constructed distances by hand
    q, k, v = _eps_inputs()
    f = orc.fwd(q, k, v, 1, 1.0, 1, eps=0.01)
    # prefixes: [1.5] -> 1; +1.4921875 -> 2; +1.4375 (2^-4 away) -> 2; +1.5 -> 3
    # (two maxima, one near); +0.5 -> 3; +1.4921875 -> 4; +(-1) -> 4; +1.25 -> 4
    assert f["ties"].reshape(-1).tolist() == [1, 2, 2, 3, 3, 4, 4, 4]


def test_near_tie_shift_keeps_the_exact_output():
    # a shift decided by near ties is still a shift: O and LSE do not move
    q, k, v = _eps_inputs()
    base = orc.fwd(q, k, v, 0, 1.0, 0)
    for eps in (0.0, 0.01, 3.0):
        f = orc.fwd(q, k, v, 0, 1.0, 1, eps=eps)
        np.testing.assert_allclose(f["o"], base["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(f["lse"], base["lse"], rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        orc.fwd(q, k, v, 0, 1.0, 1, eps=-1e-3)


# ---- decomposition of the delta error (delta_lp - delta_hp) -------------------

def test_delta_split_sums_to_the_delta_error():
    # one + rest + out = sum_c dO (o - O_hp) for any stored output o, by
    # construction; checked with an arbitrary o and the oracle's exact O_hp
    from precision_flash_attention_attn_gb300.inputs import make_case
    c = make_case("tiny")
    BH = c.B * c.H
    qf, kf, vf, gf = (c.f64(n).reshape(BH, c.N, c.d).astype(np.float32) for n in ("q", "k", "v", "do"))
    ex = orc.fwd(qf, kf, vf, c.causal, c.scale, 0)
    rng = np.random.default_rng(9)
    o = (ex["o"] + rng.standard_normal(ex["o"].shape) * 1e-2).astype(np.float32)
    want = (gf.astype(np.float64) * (o.astype(np.float64) - ex["o"])).sum(-1)
    for mode in (0, 1, 2):
        sp = orc.delta_split(qf, kf, vf, o, gf, c.causal, c.scale, mode)
        np.testing.assert_allclose(sp["one"] + sp["rest"] + sp["out"], want, rtol=0, atol=1e-12)


def test_delta_split_uniform_row():
    # all scores equal and zero: every Pbar is exactly 1 in the baseline, so
    # nothing falls in `rest`; b_j / l = 1/n = p_j, so `one` is 0 too, and the
    # whole error is the output's own rounding
    N, d = 8, 4
    q = np.zeros((1, N, d), np.float32)
    k = np.zeros((1, N, d), np.float32)
    v = np.random.default_rng(3).standard_normal((1, N, d)).astype(np.float32)
    g = np.random.default_rng(4).standard_normal((1, N, d)).astype(np.float32)
    o = np.random.default_rng(5).standard_normal((1, N, d)).astype(np.float32)
    sp = orc.delta_split(q, k, v, o, g, 0, 0.5, 0)
    assert np.all(sp["one"] == 0.0) and np.all(sp["rest"] == 0.0)
    want = (g.astype(np.float64) * (o.astype(np.float64) - v.astype(np.float64).mean(1, keepdims=True))).sum(-1)
    np.testing.assert_allclose(sp["out"], want, rtol=0, atol=1e-12)


def test_delta_split_stabilised_tied_row_has_no_unit_part():
    # a row whose maximum rm > 0 is tied: the stabilised shift 2*rm puts
    # every Pbar below 1 (here exp(-1) at most), so `one` is exactly 0, while
    # the baseline feeds 1.0 on both tied keys and `one` is not 0
    N, d = 6, 4
    q = np.zeros((1, N, d), np.float32)
    q[0, :, 0] = 1.0
    k = np.zeros((1, N, d), np.float32)
    k[0, :, 0] = [2.0, 0.5, 2.0, -1.0, 1.0, 0.25]
    v = np.random.default_rng(6).standard_normal((1, N, d)).astype(np.float32)
    g = np.random.default_rng(7).standard_normal((1, N, d)).astype(np.float32)
    o = np.random.default_rng(8).standard_normal((1, N, d)).astype(np.float32)
    s1 = orc.delta_split(q, k, v, o, g, 0, 0.5, 1)
    s0 = orc.delta_split(q, k, v, o, g, 0, 0.5, 0)
    assert np.all(s1["one"] == 0.0)
    assert np.all(s0["one"] != 0.0)


# Running maximum M and count C across key tiles, worked by hand.  One query
# e0 against keys whose first component is the chosen score (every value
# BF16-exact), scale 1, two keys per tile, all keys visible.  Per tile: M and
# C update with the tile's max; the shift m = f(M, C) is re-taken; a changed
# m rescales the accumulator and restarts the count of keys whose final
# weight is 1; then Pbar = exp(s - m).  (p_one0, p_one1) per mode:
#   [1, .5 | 1, 2 | 2, 0]   baseline: tile 1 feeds key 0 as 1, tile 2 raises
#       M to 2 (key 3 fed as 1), tile 3 ties it (key 4 fed as 1): (3, 2);
#       stabilised: tiles 1, 2 as baseline (C = 1), tile 3 makes C = 2 so
#       m = 2*2 = 4, a rescale, and no unit entry: (2, 0).
#   [1, 1 | 2, .5 | 2, 0]   baseline: (4, 2).  stabilised: tile 1 has C = 2,
#       m = 2; tile 2 raises M to 2 with C = 1, m = 2 unchanged (no rescale),
#       key 2 fed as 1; tile 3: C = 2, m = 4, rescale: (1, 0).
#   [-1, -3 | -1, -2]        baseline: (2, 2).  stabilised: tile 2 makes
#       C = 2 with M < 0, so m = 0 and the first key's 1 is rescaled: (1, 0).
@pytest.mark.parametrize("scores,base,stab", [
    ([1.0, 0.5, 1.0, 2.0, 2.0, 0.0], (3, 2), (2, 0)),
    ([1.0, 1.0, 2.0, 0.5, 2.0, 0.0], (4, 2), (1, 0)),
    ([-1.0, -3.0, -1.0, -2.0], (2, 2), (1, 0)),
])
def test_emulation_multi_tile_counts_hand_worked(scores, base, stab):
    N, d = len(scores), 4
    q = np.zeros((1, N, d), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, N, d), np.float32)
    k[0, :, 0] = scores
    v = np.random.default_rng(11).standard_normal((1, N, d)).astype(np.float32)
    ex = orc.fwd(q, k, v, False, 1.0, 0)
    for mode, want in ((0, base), (1, stab)):
        em = orc.fwd_emul(q, k, v, False, 1.0, mode, beta=2.0, block_n=2)
        assert np.all(em["p_one0"] == want[0]), (mode, em["p_one0"])
        assert np.all(em["p_one1"] == want[1]), (mode, em["p_one1"])
        # the shift is exact in real arithmetic: LSE and O stay the exact ones
        np.testing.assert_allclose(em["lse"], ex["lse"], rtol=0, atol=1e-6)
        assert np.abs(em["o"] - ex["o"]).max() <= 2.0 ** -8 * np.abs(v).max() + 2.0 ** -9 * np.abs(ex["o"]).max()

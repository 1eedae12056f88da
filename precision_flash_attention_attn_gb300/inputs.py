"""Seeded synthetic inputs for the attention forward/backward workloads.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It holds none of the attention arithmetic (no softmax, no shift rule,
no output or gradient): it draws Gaussian tensors, rounds them to BF16, and
plants rows whose largest pre-softmax score is tied exactly between several
keys, which is the condition studied in "Why Low-Precision Transformer
Training Fails: An Analysis on Flash Attention" (section 3.4.4, "Why P[T,t]=1
is the critical condition").  To plant and to check ties it forms raw dot
products q.k, nothing more.

Tie semantics.  Ties are made by copying a key row bit for bit, so every
arithmetic that evaluates q.k the same way for equal operands ties them.  After
planting, every checked row must satisfy a gap condition: every key whose score
is within B_i of the row maximum has a key row identical to the maximising one,
where B_i = 2**-20 * d * |q_i|_2 * max_j |k_j|_2.  B_i is 16x the textbook
worst-case bound gamma_d * sum_c |q_c k_c| of FP32 recursive summation (the
products of two BF16 values are exact in FP32), so any FP32 evaluation of the
scores has exactly the tie sets of exact arithmetic on those rows.  Rows that
fail are redrawn (their query resampled, and re-planted if they were planted).

Workloads (B, H, N, d, causal; distributions) follow the GPT-2 shapes of the
paper's section 3.4.1 and the five cases of the benchmark definition:

  tiny   1, 2, 128,  64, causal    Q,K,V,dO ~ N(0,1)*0.5, 25% planted rows, 2-4 ties
  gpt2s  8, 12, 1024, 64, causal   N(0,1), 5% planted rows, 2-4 ties
  gpt2m  8, 16, 1024, 64, causal   Q,K rank-4 (U W, W*0.5) + N(0,0.05^2), 10%, 2-4 ties
  long   1, 16, 16384, 128, causal N(0,1), 1% planted rows, 2-4 ties
  ties   4, 16, 4096, 64, full     Q,K ~ N(0,1)*3, V,dO ~ N(0,1), 50% planted, 2-16 ties

The softmax scale is 1/sqrt(d) throughout.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "CaseSpec", "CASES", "Case", "make_case", "make_custom",
    "bf16_bits", "bf16_bits_to_f64", "bf16_bits_to_f32",
]


@dataclasses.dataclass(frozen=True)
class CaseSpec:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    qk_sigma: float = 1.0
    v_sigma: float = 1.0
    do_sigma: float = 1.0
    low_rank: int = 0            # >0: Q and K are rank-r factors plus noise
    low_rank_noise: float = 0.05
    plant_frac: float = 0.0
    ties_min: int = 2
    ties_max: int = 4
    min_plant_row: int = 0       # causal: smallest row index that may be planted
    neg_v_cols: bool = False     # invariant fixture: a quarter of V columns ~ N(-2, 1)
    check_all_rows: bool = True  # gap-check every row (else planted + a sample)
    sample_rows_per_head: int = 256

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


CASES = {
    "tiny": CaseSpec("tiny", 1, 2, 128, 64, True, 101, qk_sigma=0.5, v_sigma=0.5,
                     do_sigma=0.5, plant_frac=0.25, min_plant_row=3),
    "gpt2s": CaseSpec("gpt2s", 8, 12, 1024, 64, True, 102, plant_frac=0.05, min_plant_row=3),
    "gpt2m": CaseSpec("gpt2m", 8, 16, 1024, 64, True, 103, low_rank=4, plant_frac=0.10,
                      min_plant_row=3),
    "long": CaseSpec("long", 1, 16, 16384, 128, True, 104, plant_frac=0.01, min_plant_row=3,
                     check_all_rows=False),
    "ties": CaseSpec("ties", 4, 16, 4096, 64, False, 105, qk_sigma=3.0, plant_frac=0.5,
                     ties_max=16, check_all_rows=False, sample_rows_per_head=512),
}


# ---------------------------------------------------------------------------
# BF16 storage helpers (the generator's own quantiser; round to nearest even)
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to BF16 (nearest, ties to even) and return the raw
    16-bit patterns.  Inputs are finite Gaussian draws, so no NaN handling."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + (((u >> 16) & 1) + 0x7FFF)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------------------
# Case container
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Case:
    spec: CaseSpec
    q: np.ndarray        # uint16 BF16 bits, [B, H, N, d]
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    planted: np.ndarray  # bool [B, H, N]: rows given a planted tie
    checked: np.ndarray  # bool [B, H, N]: rows that passed the gap check
    ties: np.ndarray     # int32 [B, H, N]: exact tie count at the row max (checked rows), else -1

    @property
    def B(self): return self.spec.B
    @property
    def H(self): return self.spec.H
    @property
    def N(self): return self.spec.N
    @property
    def d(self): return self.spec.d
    @property
    def causal(self): return self.spec.causal
    @property
    def scale(self): return self.spec.scale

    def f64(self, name: str) -> np.ndarray:
        return bf16_bits_to_f64(getattr(self, name))

    def realised(self) -> dict:
        """Realised planting statistics (reported, not asserted)."""
        chk = self.checked
        t = self.ties[chk]
        return {
            "rows": int(chk.size),
            "checked_rows": int(chk.sum()),
            "planted_rows": int(self.planted.sum()),
            "rows_with_tied_max": int((t > 1).sum()),
            "tied_fraction_of_checked": float((t > 1).mean()) if t.size else 0.0,
            "max_ties": int(t.max()) if t.size else 0,
        }


# ---------------------------------------------------------------------------
# Generation
# ---------------------------------------------------------------------------

def _draw_qk(rng, spec: CaseSpec, n: int, d: int) -> np.ndarray:
    if spec.low_rank > 0:
        r = spec.low_rank
        U = rng.standard_normal((n, r))
        W = rng.standard_normal((r, d)) * 0.5
        return (U @ W + rng.standard_normal((n, d)) * spec.low_rank_noise).astype(np.float32)
    return (rng.standard_normal((n, d)) * spec.qk_sigma).astype(np.float32)


def _draw_q_rows(rng, spec: CaseSpec, qfactor, n: int, d: int) -> np.ndarray:
    """Fresh query rows.  For low-rank cases the head's query factor W is kept
    so a redrawn row has the same structure as its neighbours."""
    if spec.low_rank > 0:
        W = qfactor
        U = rng.standard_normal((n, spec.low_rank))
        return (U @ W + rng.standard_normal((n, d)) * spec.low_rank_noise).astype(np.float32)
    return (rng.standard_normal((n, d)) * spec.qk_sigma).astype(np.float32)


def _row_ids(kbits: np.ndarray) -> np.ndarray:
    """Integer id per key row; equal ids <=> bit-identical rows."""
    kb = np.ascontiguousarray(kbits)
    view = kb.view(np.dtype((np.void, kb.dtype.itemsize * kb.shape[1]))).ravel()
    _, inv = np.unique(view, return_inverse=True)
    return inv.astype(np.int64)


class _Head:
    """Scores of one head, kept dense for N <= 4096, otherwise per row."""

    def __init__(self, qf, kf, causal, dense):
        self.qf, self.kf, self.causal, self.dense = qf, kf, causal, dense
        self.N = qf.shape[0]
        self.S = (qf @ kf.T) if dense else None

    def nvis(self, i):
        return i + 1 if self.causal else self.N

    def row(self, i):
        n = self.nvis(i)
        if self.dense:
            return self.S[i, :n]
        return self.kf[:n] @ self.qf[i]

    def copy_key(self, dst, src):
        self.kf[dst] = self.kf[src]
        if self.dense:
            self.S[:, dst] = self.S[:, src]

    def set_query(self, i, qrow):
        self.qf[i] = qrow
        if self.dense:
            self.S[i] = self.kf @ qrow

    def scores_rows(self, rows):
        if self.dense:
            return self.S[rows]
        return self.qf[rows] @ self.kf.T


def _plant_row(rng, spec, hd: _Head, kbits, ids, protected, i):
    s = hd.row(i)
    n = s.shape[0]
    jmax = int(np.argmax(s))
    same = ids[:n] == ids[jmax]
    t0 = int(same.sum())
    t = int(rng.integers(spec.ties_min, spec.ties_max + 1))
    need = t - t0
    pos = np.empty(0, dtype=np.int64)
    if need > 0:
        cand = np.flatnonzero(~protected[:n] & ~same)
        need = min(need, cand.size)
        if need > 0:
            pos = rng.choice(cand, size=need, replace=False)
            for j in pos:
                kbits[j] = kbits[jmax]
                hd.copy_key(j, jmax)
                ids[j] = ids[jmax]
    protected[jmax] = True
    protected[:n][same] = True
    protected[pos] = True


def _gap_check(hd: _Head, ids, rows, d):
    """Return (failing rows, tie counts) for the given rows."""
    knorm_max = float(np.sqrt((hd.kf * hd.kf).sum(1)).max())
    fails, ties = [], np.zeros(len(rows), dtype=np.int32)
    chunk = 512
    for c0 in range(0, len(rows), chunk):
        rr = rows[c0:c0 + chunk]
        S = hd.scores_rows(rr)
        if hd.causal:
            S = np.where(np.arange(hd.N)[None, :] <= rr[:, None], S, -np.inf)
        am = np.argmax(S, axis=1)
        mx = S[np.arange(len(rr)), am]
        qn = np.sqrt((hd.qf[rr] * hd.qf[rr]).sum(1))
        bound = 2.0 ** -20 * d * qn * knorm_max + 1e-300
        near = (mx[:, None] - S) <= bound[:, None]
        bad = near & (ids[None, :] != ids[am][:, None])
        f = bad.any(axis=1)
        fails.extend(rr[f].tolist())
        ties[c0:c0 + len(rr)] = near.sum(axis=1)
    return np.array(fails, dtype=np.int64), ties


def _make_head(rng, spec: CaseSpec):
    N, d = spec.N, spec.d
    qfactor = None
    if spec.low_rank > 0:
        qfactor = rng.standard_normal((spec.low_rank, d)) * 0.5
        U = rng.standard_normal((N, spec.low_rank))
        q32 = (U @ qfactor + rng.standard_normal((N, d)) * spec.low_rank_noise).astype(np.float32)
        k32 = _draw_qk(rng, spec, N, d)
    else:
        q32 = _draw_qk(rng, spec, N, d)
        k32 = _draw_qk(rng, spec, N, d)
    qbits, kbits = bf16_bits(q32), bf16_bits(k32)
    hd = _Head(bf16_bits_to_f64(qbits), bf16_bits_to_f64(kbits), spec.causal, dense=N <= 4096)
    ids = _row_ids(kbits)

    planted = np.zeros(N, dtype=bool)
    n_plant = int(round(spec.plant_frac * N))
    lo = spec.min_plant_row if spec.causal else 0
    lo = max(lo, spec.ties_min - 1) if spec.causal else lo
    if n_plant > 0:
        rows = rng.choice(np.arange(lo, N), size=min(n_plant, N - lo), replace=False)
        planted[rows] = True
        protected = np.zeros(N, dtype=bool)
        for i in rows:
            _plant_row(rng, spec, hd, kbits, ids, protected, int(i))
    else:
        protected = np.zeros(N, dtype=bool)

    if spec.check_all_rows:
        check = np.arange(N)
    else:
        extra = rng.choice(N, size=min(spec.sample_rows_per_head, N), replace=False)
        check = np.union1d(np.flatnonzero(planted), extra)
    checked = np.zeros(N, dtype=bool)
    checked[check] = True

    todo = check
    ties = np.full(N, -1, dtype=np.int32)
    for _ in range(64):
        fails, t = _gap_check(hd, ids, todo, d)
        ties[todo] = t
        if fails.size == 0:
            break
        newq = bf16_bits(_draw_q_rows(rng, spec, qfactor, fails.size, d))
        for r, i in enumerate(fails):
            qbits[i] = newq[r]
            hd.set_query(int(i), bf16_bits_to_f64(newq[r]))
        for i in fails:
            if planted[i]:
                _plant_row(rng, spec, hd, kbits, ids, protected, int(i))
        # re-planting may overwrite another row's maximiser, so check all again
        todo = check
    else:
        raise RuntimeError("gap check did not converge")
    return qbits, kbits, planted, checked, ties


def make_custom(spec: CaseSpec) -> Case:
    rng = np.random.default_rng(spec.seed)
    B, H, N, d = spec.B, spec.H, spec.N, spec.d
    q = np.empty((B, H, N, d), np.uint16)
    k = np.empty_like(q)
    planted = np.zeros((B, H, N), bool)
    checked = np.zeros((B, H, N), bool)
    ties = np.full((B, H, N), -1, np.int32)
    for b in range(B):
        for h in range(H):
            qb, kb, pl, ch, t = _make_head(rng, spec)
            q[b, h], k[b, h], planted[b, h], checked[b, h], ties[b, h] = qb, kb, pl, ch, t
    v32 = rng.standard_normal((B, H, N, d)).astype(np.float32) * np.float32(spec.v_sigma)
    if spec.neg_v_cols:
        cols = rng.choice(d, size=d // 4, replace=False)
        v32[..., cols] = (rng.standard_normal((B, H, N, cols.size)) - 2.0).astype(np.float32)
    do32 = rng.standard_normal((B, H, N, d)).astype(np.float32) * np.float32(spec.do_sigma)
    return Case(spec, q, k, bf16_bits(v32), bf16_bits(do32), planted, checked, ties)


def make_case(name: str, **overrides) -> Case:
    """Build one of the named workloads; keyword overrides change any CaseSpec
    field (e.g. a smaller B, another seed, the negative-mean V fixture)."""
    spec = dataclasses.replace(CASES[name], **overrides) if overrides else CASES[name]
    return make_custom(spec)

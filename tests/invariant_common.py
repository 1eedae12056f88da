"""Shared pieces of the stabilised-softmax invariant checks on the
negative-mean-V fixture (a quarter of V's columns drawn from N(-2, 1), after
the mostly negative V column the paper traces: section 5, V[:, 20] in
[-6, +2]).  Same-sign V columns are the condition under which the paper's
bias mechanism acts ("Cause 2: Biased Rounding Error Leads to Positive
(delta_lp - delta_hp)[T]").

Rows judged: planted rows whose exact maximum is tied (count > 1), excluding
rows with |scale * rm| <= 2^-8 (there bf16(exp(-x)) rounds to 1 whatever the
shift) and rm = 0 (both conditions of the rule are strict)."""
import math

import numpy as np

from gpu_helpers import f32


def fixture(name, **kw):
    from conftest import case
    seeds = {"tiny": 1101, "ties": 1105}
    return case(name, neg_v_cols=True, seed=seeds[name], **kw)


def neg_cols(c):
    """The columns drawn from N(-2, 1) (their sample mean sits near -2)."""
    v = f32(c.v).reshape(-1, c.d)
    return np.flatnonzero(v.mean(0) < -1.0)


def judged_rows(c, tie_count, limit=None, seed=0):
    """Flat row ids of the judged rows (optionally a seeded sample of them)."""
    BH = c.B * c.H
    rows = np.flatnonzero(c.planted.reshape(-1) & (tie_count.reshape(-1) > 1))
    if limit is not None and rows.size > limit:
        rows = np.sort(np.random.default_rng(seed).choice(rows, size=limit, replace=False))
    qf = f32(c.q).reshape(BH, c.N, c.d).astype(np.float64)
    kf = f32(c.k).reshape(BH, c.N, c.d).astype(np.float64)
    keep = []
    for r in rows:
        h, i = divmod(int(r), c.N)
        n = i + 1 if c.causal else c.N
        rm = float((kf[h, :n] @ qf[h, i]).max())
        if rm != 0.0 and abs(c.scale * rm) > 2.0 ** -8:
            keep.append(r)
    return np.array(keep, dtype=np.int64)


def mean_se(x):
    x = np.asarray(x, dtype=np.float64)
    if x.size < 2:
        return {"mean": float(x.mean()) if x.size else None, "se": None, "n": int(x.size)}
    return {"mean": float(x.mean()), "se": float(x.std(ddof=1) / math.sqrt(x.size)), "n": int(x.size)}

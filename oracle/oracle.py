"""Python access to the FP64 CPU attention oracle (``attn_ref.c``).

TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this module.  It never imports the
CUDA package and the CUDA package never imports it.

Every function takes float32 arrays that hold BF16 values exactly, shaped
[BH, N, d] (contiguous), and returns float64 results.  See ``attn_ref.c`` for
the passages of "Why Low-Precision Transformer Training Fails: An Analysis on
Flash Attention" each routine follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

BETA = 2.0  # section 4 / Figure 7 of the paper uses beta = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, IEEE arithmetic)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_fwd.argtypes = [P, P, P, P, i64, i32, i32, i32, f64, i32, f64, f64, P, i64, P, P, P, P]
        L.oracle_bwd_dq.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, f64, P, i64, P]
        L.oracle_bwd_dkdv.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, f64, P, i64, P, P]
        L.oracle_bf16_round.argtypes = [P, P, i64]
        L.oracle_fwd_emul.argtypes = [P, P, P, i64, i32, i32, i32, f64, i32, f64, i32, P, i64,
                                      P, P, P, P, P, P, P]
        L.oracle_delta_split.argtypes = [P, P, P, P, P, i64, i32, i32, i32, f64, i32, f64, f64, P, i64,
                                         P, P, P]
        L.oracle_delta_split.restype = ctypes.c_int
        L.oracle_row_shift.argtypes = [f64, ctypes.c_long, i32, f64]
        L.oracle_row_shift.restype = f64
        for f in (L.oracle_fwd, L.oracle_bwd_dq, L.oracle_bwd_dkdv, L.oracle_fwd_emul,
                  L.oracle_num_threads):
            f.restype = ctypes.c_int
        L.oracle_bf16_round.restype = None
        _lib = L
    return _lib


def row_shift(rmz: float, rs: int, mode: int, beta: float = BETA) -> float:
    """The per-row shift m of the mode (scaled units)."""
    return float(lib().oracle_row_shift(float(rmz), int(rs), int(mode), float(beta)))


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    assert a.ndim == 3
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    return r, r.size


def bf16_round(x) -> np.ndarray:
    """Round FP32 values to BF16 (nearest, ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().oracle_bf16_round(_ptr(x), _ptr(y), x.size)
    return y


def fwd(q, k, v, causal, scale, mode=0, beta=BETA, rows=None, dout=None, eps=0.0):
    """Exact attention forward.  Returns dict(o, lse, ties[, delta]); with
    rows=None every row of every head in [BH, N] order, else the listed flat
    rows (bh*N + i) in that order.  ties is the row's rs of section 3.4.5:
    keys at the maximum (eps = 0) or within eps of it in scaled units."""
    if not eps >= 0.0:
        raise ValueError("eps must be >= 0")
    q, k, v = _f32(q), _f32(k), _f32(v)
    BH, N, d = q.shape
    r, nr = _rows(rows)
    n = BH * N if r is None else nr
    o = np.empty((n, d), np.float64)
    lse = np.empty(n, np.float64)
    ties = np.empty(n, np.int32)
    delta = np.empty(n, np.float64) if dout is not None else None
    g = _f32(dout) if dout is not None else None
    rc = lib().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), BH, N, d, int(causal), float(scale),
                          int(mode), float(beta), float(eps), _ptr(r), nr, _ptr(o), _ptr(lse), _ptr(ties),
                          _ptr(delta))
    if rc:
        raise MemoryError("oracle_fwd failed")
    out = {"o": o, "lse": lse, "ties": ties}
    if delta is not None:
        out["delta"] = delta
    if r is None:
        out = {kk: (vv.reshape(BH, N, d) if kk == "o" else vv.reshape(BH, N)) for kk, vv in out.items()}
    return out


def bwd(q, k, v, dout, causal, scale, q_rows=None, k_rows=None, lse=None, delta=None):
    """Exact gradients of sum(dO o O).  Needs the exact LSE and delta of every
    row of the heads involved (computed here if not given, as [BH*N]).
    Returns dict(dq, dk, dv) for the requested query rows / key rows (all if
    None, shaped [BH, N, d])."""
    q, k, v, g = _f32(q), _f32(k), _f32(v), _f32(dout)
    BH, N, d = q.shape
    if lse is None or delta is None:
        f = fwd(q, k, v, causal, scale, 0, rows=None, dout=g)
        lse = f["lse"].reshape(-1)
        delta = f["delta"].reshape(-1)
    lse = np.ascontiguousarray(lse, np.float64).ravel()
    delta = np.ascontiguousarray(delta, np.float64).ravel()
    qr, nq = _rows(q_rows)
    kr, nk = _rows(k_rows)
    dq = np.empty(((BH * N) if qr is None else nq, d), np.float64)
    dk = np.empty(((BH * N) if kr is None else nk, d), np.float64)
    dv = np.empty_like(dk)
    L = lib()
    L.oracle_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lse), _ptr(delta), BH, N, d,
                    int(causal), float(scale), _ptr(qr), nq, _ptr(dq))
    L.oracle_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lse), _ptr(delta), BH, N, d,
                      int(causal), float(scale), _ptr(kr), nk, _ptr(dk), _ptr(dv))
    if qr is None:
        dq = dq.reshape(BH, N, d)
    if kr is None:
        dk, dv = dk.reshape(BH, N, d), dv.reshape(BH, N, d)
    return {"dq": dq, "dk": dk, "dv": dv}


def fwd_emul(q, k, v, causal, scale, mode=0, beta=BETA, block_n=128, rows=None):
    """BF16-rounding emulation of the tiled forward (see attn_ref.c).  Returns
    dict(o, lse, p_one0, p_one1, p_amb, o_peradd, p_max)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    BH, N, d = q.shape
    r, nr = _rows(rows)
    n = BH * N if r is None else nr
    o = np.empty((n, d), np.float64)
    op = np.empty((n, d), np.float64)
    lse = np.empty(n, np.float64)
    p0 = np.empty(n, np.int32)
    p1 = np.empty(n, np.int32)
    pa = np.empty(n, np.int32)
    pm = np.empty(n, np.float32)
    rc = lib().oracle_fwd_emul(_ptr(q), _ptr(k), _ptr(v), BH, N, d, int(causal), float(scale),
                               int(mode), float(beta), int(block_n), _ptr(r), nr, _ptr(o),
                               _ptr(lse), _ptr(p0), _ptr(p1), _ptr(pa), _ptr(op), _ptr(pm))
    if rc:
        raise RuntimeError("oracle_fwd_emul failed")
    out = {"o": o, "lse": lse, "p_one0": p0, "p_one1": p1, "p_amb": pa, "o_peradd": op,
           "p_max": pm}
    if r is None:
        out = {kk: (vv.reshape(BH, N, d) if vv.ndim == 2 else vv.reshape(BH, N))
               for kk, vv in out.items()}
    return out


def delta_split(q, k, v, o, dout, causal, scale, mode=0, beta=BETA, eps=0.0, rows=None):
    """Decomposition of sum_c dO (o - O_hp) per row (see attn_ref.c):
    returns dict(one, rest, out) -- the keys whose BF16 probability is 1, the
    other keys, and the output rounding.  o is a stored output [BH, N, d]
    (float32 values), dout the loss gradient."""
    q, k, v, o, g = _f32(q), _f32(k), _f32(v), _f32(o), _f32(dout)
    BH, N, d = q.shape
    r, nr = _rows(rows)
    n = BH * N if r is None else nr
    one, rest, out = (np.empty(n, np.float64) for _ in range(3))
    rc = lib().oracle_delta_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(g), BH, N, d, int(causal),
                                  float(scale), int(mode), float(beta), float(eps), _ptr(r), nr,
                                  _ptr(one), _ptr(rest), _ptr(out))
    if rc:
        raise MemoryError("oracle_delta_split failed")
    res = {"one": one, "rest": rest, "out": out}
    if r is None:
        res = {kk: vv.reshape(BH, N) for kk, vv in res.items()}
    return res

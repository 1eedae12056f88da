"""Thin Python binding of libfa (include/fa.h): argument marshalling only.

The names mirror the C ABI: ``fa_fwd``, ``fa_bwd``, ``fa_tie_stats``,
``fa_device_status`` and ``fa_status_string``.  Tensor arguments are torch
CUDA tensors (their data pointers are passed through) or raw integer device
addresses; every step of the computation runs in the library's kernels.  A
non-zero status raises :class:`FAError`.  ``attention_fwd`` / ``attention_bwd``
/ ``tie_stats`` additionally allocate the outputs with torch.

If the shared library has not been built this module raises on import: there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import INCLUDE, LIB

MODES = {"baseline": 0, "stabilised": 1, "fp32_out": 2}
FA_OK = 0

if not os.path.exists(LIB):
    raise ImportError(f"libfa.so is not built ({LIB}); run __graft_entry__.build() first")

_lib = ctypes.CDLL(LIB)
_P = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float

_lib.fa_fwd.argtypes = [_P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _P]
_lib.fa_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _P]
_lib.fa_bwd_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _P]
_lib.fa_bwd_noalloc.restype = ctypes.c_int
_lib.fa_tie_stats.argtypes = [_P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _P, _P, _P, _P]


class StabParams(ctypes.Structure):
    """fa_stab_params_t: beta (> 1) and eps (only 0 is supported)."""
    _fields_ = [("beta", ctypes.c_float), ("eps", ctypes.c_float)]


BETA_DEFAULT = 2.0
_SP = ctypes.POINTER(StabParams)
_lib.fa_fwd_ex.argtypes = [_P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _SP, _P]
_lib.fa_bwd_ex.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _i, _P]
DELTA_STORED_O = 0            # delta from the caller's o (fa_bwd)
DELTA_RECOMPUTED_O_FP32 = 1   # delta from O recomputed as P V in FP32 inside the backward
DELTA_FROM_DP_P = 2           # delta = rowsum(dP o P), no output read
_lib.fa_tie_stats_ex.argtypes = [_P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _SP, _P, _P, _P, _P, _P, _P]
_lib.fa_delta_error_split.argtypes = [_P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _SP, _P, _P, _P, _P]
_lib.fa_fwd_layout.argtypes = [_P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _SP, _i, _P]
_lib.fa_bwd_layout.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _i, _i, _P]
LAYOUT_BHND = 0   # [B, H, N, d]
LAYOUT_BNHD = 1   # [B, N, H, d]
_lib.fa_fwd_heads.argtypes = [_P, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _P, _SP, _P]
_lib.fa_bwd_heads.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _f, _P, _P]
_lib.fa_device_status.argtypes = [_P, _i]
_lib.fa_profile_start.argtypes = []
_lib.fa_profile_stop.argtypes = [_i, _P, _P]
_lib.fa_last_error.argtypes = []
_lib.fa_last_error.restype = ctypes.c_char_p
_lib.fa_status_string.argtypes = [_i]
_lib.fa_status_string.restype = ctypes.c_char_p
for _fn in (_lib.fa_fwd, _lib.fa_bwd, _lib.fa_tie_stats, _lib.fa_device_status, _lib.fa_profile_start,
            _lib.fa_profile_stop, _lib.fa_fwd_ex, _lib.fa_tie_stats_ex, _lib.fa_bwd_ex, _lib.fa_delta_error_split,
            _lib.fa_fwd_heads, _lib.fa_bwd_heads, _lib.fa_fwd_layout, _lib.fa_bwd_layout):
    _fn.restype = ctypes.c_int


class FAError(RuntimeError):
    def __init__(self, fn, status):
        detail = fa_last_error() if status in (3, 4) else ""
        super().__init__(f"{fn} returned {status} ({fa_status_string(status)})" + (f": {detail}" if detail else ""))
        self.status = status


def fa_last_error() -> str:
    return _lib.fa_last_error().decode()


def library_path() -> str:
    return LIB


def declared_symbols() -> list[str]:
    """Function names declared in include/fa.h."""
    with open(os.path.join(INCLUDE, "fa.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(fa_\w+)\s*\(", text, re.M)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != FA_OK:
        raise FAError(fn, rc)
    return rc


def fa_status_string(status: int) -> str:
    return _lib.fa_status_string(int(status)).decode()


def fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, mode, stream=None, check=True):
    rc = _lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(causal),
                     float(scale), int(mode), _stream(stream))
    return _check("fa_fwd", rc) if check else rc


def _params(beta, eps):
    if beta is None and eps is None:
        return None
    return ctypes.pointer(StabParams(BETA_DEFAULT if beta is None else float(beta),
                                     0.0 if eps is None else float(eps)))


def fa_fwd_ex(q, k, v, o, lse, B, H, N, d, causal, scale, mode, beta=None, eps=None, stream=None,
              check=True):
    """fa_fwd with stabilised-softmax parameters (None: the library default)."""
    rc = _lib.fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(causal),
                        float(scale), int(mode), _params(beta, eps), _stream(stream))
    return _check("fa_fwd_ex", rc) if check else rc


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, stream=None, check=True):
    rc = _lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                     _ptr(dv), B, H, N, d, int(causal), float(scale), int(mode), _stream(stream))
    return _check("fa_bwd", rc) if check else rc


def fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, delta_source=DELTA_STORED_O,
              stream=None, check=True):
    """fa_bwd with a choice of the output delta is formed from (o may be None
    with DELTA_RECOMPUTED_O_FP32)."""
    rc = _lib.fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, H, N, d, int(causal), float(scale), int(mode), int(delta_source), _stream(stream))
    return _check("fa_bwd_ex", rc) if check else rc


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, stream=None,
                   check=True):
    """fa_bwd with its workspace in the library's static scratch array
    (FA_NOALLOC_SCRATCH_BYTES per device) instead of a device allocation, for
    callers that must not allocate; overlapping calls race on the scratch."""
    rc = _lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                             _ptr(dv), B, H, N, d, int(causal), float(scale), int(mode), _stream(stream))
    return _check("fa_bwd_noalloc", rc) if check else rc


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def fa_tie_stats(q, k, v, o, B, H, N, d, causal, scale, mode, tie_count, pv_err, p_one=None,
                 stream=None, check=True):
    rc = _lib.fa_tie_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, d, int(causal), float(scale),
                           int(mode), _ptr(tie_count), _ptr(pv_err), _ptr(p_one), _stream(stream))
    return _check("fa_tie_stats", rc) if check else rc


def fa_tie_stats_ex(q, k, v, o, B, H, N, d, causal, scale, mode, tie_count, pv_err, p_one=None,
                    dO=None, delta_err=None, beta=None, eps=None, stream=None, check=True):
    """fa_tie_stats with stabilised-softmax parameters (None: the library
    default) and, with dO and delta_err, the per-row delta error."""
    rc = _lib.fa_tie_stats_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, d, int(causal), float(scale),
                              int(mode), _params(beta, eps), _ptr(tie_count), _ptr(pv_err), _ptr(p_one),
                              _ptr(dO), _ptr(delta_err), _stream(stream))
    return _check("fa_tie_stats_ex", rc) if check else rc


def fa_delta_error_split(q, k, v, o, dO, B, H, N, d, causal, scale, mode, err_one, err_rest, err_out,
                         beta=None, eps=None, stream=None, check=True):
    rc = _lib.fa_delta_error_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), B, H, N, d, int(causal),
                                   float(scale), int(mode), _params(beta, eps), _ptr(err_one), _ptr(err_rest),
                                   _ptr(err_out), _stream(stream))
    return _check("fa_delta_error_split", rc) if check else rc


def fa_fwd_layout(q, k, v, o, lse, B, H, N, d, causal, scale, mode, layout, beta=None, eps=None, stream=None,
                  check=True):
    """fa_fwd_ex with a tensor layout (LAYOUT_BHND or LAYOUT_BNHD)."""
    rc = _lib.fa_fwd_layout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(causal), float(scale),
                            int(mode), _params(beta, eps), int(layout), _stream(stream))
    return _check("fa_fwd_layout", rc) if check else rc


def fa_bwd_layout(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, layout, stream=None,
                  check=True):
    """fa_bwd with a tensor layout (LAYOUT_BHND or LAYOUT_BNHD)."""
    rc = _lib.fa_bwd_layout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                            B, H, N, d, int(causal), float(scale), int(mode), int(layout), _stream(stream))
    return _check("fa_bwd_layout", rc) if check else rc


def _head_modes(head_modes):
    arr = (ctypes.c_int * len(head_modes))(*[int(m) for m in head_modes])
    return arr


def fa_fwd_heads(q, k, v, o_bf16, o_fp32, lse, B, H, N, d, causal, scale, head_modes, beta=None, eps=None,
                 stream=None, check=True):
    """Forward with a mode per head (host list of H modes)."""
    hm = _head_modes(head_modes)
    rc = _lib.fa_fwd_heads(_ptr(q), _ptr(k), _ptr(v), _ptr(o_bf16), _ptr(o_fp32), _ptr(lse), B, H, N, d,
                           int(causal), float(scale), ctypes.cast(hm, _P), _params(beta, eps), _stream(stream))
    return _check("fa_fwd_heads", rc) if check else rc


def fa_bwd_heads(q, k, v, o_bf16, o_fp32, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, head_modes,
                 stream=None, check=True):
    """Backward with a mode per head: delta from each head's own output."""
    hm = _head_modes(head_modes)
    rc = _lib.fa_bwd_heads(_ptr(q), _ptr(k), _ptr(v), _ptr(o_bf16), _ptr(o_fp32), _ptr(lse), _ptr(dO), _ptr(dq),
                           _ptr(dk), _ptr(dv), B, H, N, d, int(causal), float(scale), ctypes.cast(hm, _P),
                           _stream(stream))
    return _check("fa_bwd_heads", rc) if check else rc


def fa_device_status(stream=None, reset=True) -> int:
    return int(_lib.fa_device_status(_stream(stream), int(reset)))


KERNELS = ["fwd", "fwd_stats", "bwd_pre", "bwd_main", "dq_convert", "pv_err"]


def fa_profile_start() -> None:
    _check("fa_profile_start", _lib.fa_profile_start())


def fa_profile_stop() -> dict:
    """{kernel: (launches, total_ms)} for the session just ended."""
    n = len(KERNELS)
    launches = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    _check("fa_profile_stop", _lib.fa_profile_stop(n, launches, ms))
    return {k: (int(launches[i]), float(ms[i])) for i, k in enumerate(KERNELS)}


# --------------------------------------------------------------------------
# Allocating conveniences (torch tensors in, torch tensors out)
# --------------------------------------------------------------------------

def _shape(q):
    B, H, N, d = q.shape
    return B, H, N, d


def attention_fwd(q, k, v, causal=True, scale=None, mode=0, stream=None, beta=None):
    """Returns (o, lse).  o is BF16, or FP32 in mode 2.  beta: mode 1's shift
    factor (None: the library default)."""
    import torch
    B, H, N, d = _shape(q)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty((B, H, N, d), device=q.device,
                    dtype=torch.float32 if mode == 2 else torch.bfloat16)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    fa_fwd_ex(q, k, v, o, lse, B, H, N, d, causal, scale, mode, beta=beta, stream=stream)
    return o, lse


def attention_bwd(q, k, v, o, lse, dO, causal=True, scale=None, mode=0, stream=None,
                  delta_source=DELTA_STORED_O):
    """Returns (dq, dk, dv), BF16."""
    import torch
    B, H, N, d = _shape(q)
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, delta_source, stream)
    return dq, dk, dv


def tie_stats(q, k, v, o, causal=True, scale=None, mode=0, with_p_one=True, stream=None, beta=None):
    """Returns (tie_count, pv_err, p_one or None).  beta as for attention_fwd."""
    import torch
    B, H, N, d = _shape(q)
    scale = d ** -0.5 if scale is None else scale
    tc = torch.empty((B, H, N), device=q.device, dtype=torch.int32)
    pe = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    po = torch.empty((2, B, H, N), device=q.device, dtype=torch.int32) if with_p_one else None
    fa_tie_stats_ex(q, k, v, o, B, H, N, d, causal, scale, mode, tc, pe, po, beta=beta, stream=stream)
    return tc, pe, po


def delta_error(q, k, v, o, dO, causal=True, scale=None, mode=0, stream=None, beta=None):
    """Per-row delta_lp - delta_hp = sum_c dO (o - O_ref) of the stored output
    o (FP32 [B, H, N]), from fa_tie_stats_ex."""
    import torch
    B, H, N, d = _shape(q)
    scale = d ** -0.5 if scale is None else scale
    tc = torch.empty((B, H, N), device=q.device, dtype=torch.int32)
    pe = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    de = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    fa_tie_stats_ex(q, k, v, o, B, H, N, d, causal, scale, mode, tc, pe, None, dO=dO, delta_err=de, beta=beta,
                    stream=stream)
    return de


def delta_error_split(q, k, v, o, dO, causal=True, scale=None, mode=0, stream=None, beta=None, eps=None):
    """(err_one, err_rest, err_out), FP32 [B, H, N]: delta_lp - delta_hp of the
    stored output o split into keys with BF16 probability 1, the other keys,
    and the output rounding (fa_delta_error_split)."""
    import torch
    B, H, N, d = _shape(q)
    scale = d ** -0.5 if scale is None else scale
    outs = [torch.empty((B, H, N), device=q.device, dtype=torch.float32) for _ in range(3)]
    fa_delta_error_split(q, k, v, o, dO, B, H, N, d, causal, scale, mode, *outs, beta=beta, eps=eps,
                         stream=stream)
    return tuple(outs)

"""Helpers shared by the GPU parity tests: device copies of seeded inputs and
the tolerance rules."""
import numpy as np

from precision_flash_attention_attn_gb300.inputs import bf16_bits_to_f32

# Tolerances against the FP64 oracle (max abs on O; rel. Frobenius on grads).
O_TOL_BF16 = 1e-2
O_TOL_FP32 = 2e-3
LSE_TOL = 1e-4
GRAD_REL_TOL = 1e-2


def torch_mod():
    import torch
    return torch


def dev_bf16(bits: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def o_bound(o_exact: np.ndarray, mode: int) -> np.ndarray:
    """Per-element bound on |O_gpu - O_exact|.  FP32 output: 2e-3.  BF16
    output: 1e-2, except where half a BF16 ulp of the exact value plus 4e-3
    exceeds it (|O| >= 4: no BF16 value lies within 1e-2 of every real)."""
    if mode == 2:
        return np.full(o_exact.shape, O_TOL_FP32)
    a = np.abs(o_exact)
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    half_ulp = np.exp2(e - 8)          # BF16 has 8 significant bits
    return np.maximum(O_TOL_BF16, half_ulp + 4e-3)


def rel_fro(a, b, floor=0.0) -> float:
    """||a - b|| / max(||b||, floor).  Where an exact gradient is identically
    zero (dQ and dK when every row sees a single key, since dP - delta = 0
    there) the caller passes a floor at the scale of the other gradients, so
    the FP32 rounding residue is judged against that scale."""
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), floor, 1e-300))


def sample_rows(BH, N, n, seed=0, must=None):
    rng = np.random.default_rng(seed)
    rows = rng.choice(BH * N, size=min(n, BH * N), replace=False)
    # always include the first and last rows of every head tile edge region
    edge = np.array([0, N - 1, min(127, N - 1), min(128, N - 1)])
    rows = np.concatenate([rows, edge, (BH - 1) * N + edge])
    if must is not None:
        rows = np.concatenate([rows, must])
    return np.unique(rows)


def f32(bits):
    return bf16_bits_to_f32(bits)

"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/fa.h declares, and rejects invalid arguments with
the documented status before touching any device."""
import ctypes
import subprocess

import pytest

import __graft_entry__

__graft_entry__.build()
from precision_flash_attention_attn_gb300 import fa  # noqa: E402

FAKE = 1 << 20          # 16-byte aligned, never dereferenced: validation fails first
MISALIGNED = FAKE + 8


def test_library_exports_every_declared_symbol():
    declared = fa.declared_symbols()
    assert set(declared) == {"fa_fwd", "fa_bwd", "fa_tie_stats", "fa_device_status", "fa_status_string",
                             "fa_profile_start", "fa_profile_stop", "fa_last_error", "fa_bwd_noalloc",
                             "fa_fwd_ex", "fa_tie_stats_ex", "fa_bwd_ex", "fa_delta_error_split",
                             "fa_fwd_heads", "fa_bwd_heads", "fa_fwd_layout", "fa_bwd_layout"}
    lib = ctypes.CDLL(fa.library_path())
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared) <= exported


def test_status_strings():
    names = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_ALLOC", "FA_ERR_CUDA",
             "FA_ERR_TIMEOUT", "FA_ERR_NONFINITE"]
    for code, name in enumerate(names):
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


def _fwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, causal=1, scale=0.125,
             mode=0, stream=0, check=False)
    a.update(kw)
    return fa.fa_fwd(**a)


def _bwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=1,
             N=128, d=64, causal=1, scale=0.125, mode=0, stream=0, check=False)
    a.update(kw)
    return fa.fa_bwd(**a)


def _stats(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, H=1, N=128, d=64, causal=1, scale=0.125, mode=0,
             tie_count=FAKE, pv_err=FAKE, p_one=None, stream=0, check=False)
    a.update(kw)
    return fa.fa_tie_stats(**a)


INVALID = [
    dict(q=0), dict(k=0), dict(v=0), dict(q=MISALIGNED), dict(B=0), dict(H=0), dict(N=0), dict(N=-5),
    dict(causal=2), dict(causal=-1), dict(mode=3), dict(mode=-1), dict(scale=0.0), dict(scale=-1.0),
    dict(scale=float("inf")), dict(scale=float("nan")), dict(B=1 << 14, H=1 << 10, N=1024),
    dict(N=65535 * 128 + 1),
]


@pytest.mark.parametrize("kw", INVALID)
def test_invalid_arguments_rejected(kw):
    assert _fwd(**kw) == 1
    assert _bwd(**kw) == 1
    assert _stats(**kw) == 1


@pytest.mark.parametrize("kw", [dict(o=0), dict(lse=0), dict(o=MISALIGNED)])
def test_fwd_output_pointers(kw):
    assert _fwd(**kw) == 1


@pytest.mark.parametrize("name", ["dO", "dq", "dk", "dv", "lse", "o"])
def test_bwd_pointers(name):
    assert _bwd(**{name: 0}) == 1


def test_stats_pointers():
    assert _stats(tie_count=0) == 1
    assert _stats(pv_err=0) == 1
    assert _stats(p_one=MISALIGNED) == 1


@pytest.mark.parametrize("d", [32, 96, 256, 100])
def test_unsupported_head_dim(d):
    assert _fwd(d=d) == 2
    assert _bwd(d=d) == 2
    assert _stats(d=d) == 2


def test_binding_raises_on_error():
    with pytest.raises(fa.FAError) as ei:
        fa.fa_fwd(0, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 1, 0.125, 0, stream=0)
    assert ei.value.status == 1


def _fwd_ex(beta, eps, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, causal=1, scale=0.125,
             mode=1, beta=beta, eps=eps, stream=0, check=False)
    a.update(kw)
    return fa.fa_fwd_ex(**a)


def _stats_ex(beta, eps, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, H=1, N=128, d=64, causal=1, scale=0.125, mode=1,
             tie_count=FAKE, pv_err=FAKE, p_one=None, beta=beta, eps=eps, stream=0, check=False)
    a.update(kw)
    return fa.fa_tie_stats_ex(**a)


# "The modified safe softmax" requires beta > 1 and a tolerance eps >= 0
BAD_PARAMS = [
    (1.0, 0.0, 1), (0.5, 0.0, 1), (-2.0, 0.0, 1), (float("nan"), 0.0, 1), (float("inf"), 0.0, 1),
    (2.0, -1e-3, 1), (2.0, float("nan"), 1), (2.0, float("inf"), 1),
]


@pytest.mark.parametrize("beta,eps,code", BAD_PARAMS)
def test_stab_params_rejected(beta, eps, code):
    for mode in (0, 1, 2):  # checked in every mode, used only in mode 1
        assert _fwd_ex(beta, eps, mode=mode) == code
        assert _stats_ex(beta, eps, mode=mode) == code


@pytest.mark.parametrize("beta,eps", [(2.0, 1e-3), (8.0, 1.0), (4.0, 0.0)])
def test_valid_stab_params_pass_validation(beta, eps):
    # accepted parameters get past argument checking: without a GPU the call
    # then fails on the device, never with FA_ERR_INVALID_ARG / UNSUPPORTED
    for mode in (0, 1, 2):
        assert _fwd_ex(beta, eps, mode=mode) not in (0, 1, 2)
        assert _stats_ex(beta, eps, mode=mode) not in (0, 1, 2)


def test_argument_errors_precede_parameter_errors():
    assert _fwd_ex(1.0, 0.0, q=0) == 1
    assert _fwd_ex(2.0, 1e-3, d=96) == 2
    assert _stats_ex(2.0, 1e-3, tie_count=0) == 1


def test_delta_err_needs_dO():
    # delta_err is nullable; when set, dO must be a 16-byte aligned pointer too
    assert _stats_ex(2.0, 0.0, delta_err=FAKE, dO=None) == 1
    assert _stats_ex(2.0, 0.0, delta_err=FAKE, dO=MISALIGNED) == 1
    assert _stats_ex(2.0, 0.0, delta_err=MISALIGNED, dO=FAKE) == 1


def _bwd_ex(source, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=1,
             N=128, d=64, causal=1, scale=0.125, mode=0, delta_source=source, stream=0, check=False)
    a.update(kw)
    return fa.fa_bwd_ex(**a)


@pytest.mark.parametrize("source", [3, -1, 100])
def test_bwd_ex_unknown_delta_source(source):
    assert _bwd_ex(source) == 1


@pytest.mark.parametrize("source", [0, 1, 2])
@pytest.mark.parametrize("kw", [dict(q=0), dict(dO=0), dict(dq=MISALIGNED), dict(lse=0), dict(N=0), dict(mode=3)])
def test_bwd_ex_invalid_arguments(source, kw):
    assert _bwd_ex(source, **kw) == 1


def test_bwd_ex_stored_o_still_needs_o():
    assert _bwd_ex(0, o=0) == 1


def _fwd_heads(modes, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o_bf16=FAKE, o_fp32=FAKE, lse=FAKE, B=1, H=len(modes), N=128, d=64, causal=1,
             scale=0.125, head_modes=modes, stream=0, check=False)
    a.update(kw)
    return fa.fa_fwd_heads(**a)


def _bwd_heads(modes, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o_bf16=FAKE, o_fp32=FAKE, lse=FAKE, dO=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1,
             H=len(modes), N=128, d=64, causal=1, scale=0.125, head_modes=modes, stream=0, check=False)
    a.update(kw)
    return fa.fa_bwd_heads(**a)


@pytest.mark.parametrize("modes", [[0, 3], [-1, 1], [2, 2, 7]])
def test_head_modes_out_of_range(modes):
    assert _fwd_heads(modes) == 1
    assert _bwd_heads(modes) == 1


def test_head_modes_need_their_output_buffer():
    # BF16 heads need o_bf16, FP32 heads o_fp32; an unused one may be NULL
    assert _fwd_heads([0, 2], o_bf16=0) == 1
    assert _fwd_heads([0, 2], o_fp32=0) == 1
    assert _bwd_heads([1, 2], o_fp32=MISALIGNED) == 1
    assert _fwd_heads([2, 2], o_bf16=0) not in (1, 2)
    assert _fwd_heads([0, 1], o_fp32=0) not in (1, 2)


def test_head_modes_at_most_64_heads():
    assert _fwd_heads([0] * 65) == 2
    assert _bwd_heads([2] * 65) == 2


@pytest.mark.parametrize("layout", [2, -1])
def test_unknown_layout_rejected(layout):
    assert fa.fa_fwd_layout(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 1, 0.125, 0, layout, stream=0,
                            check=False) == 1
    assert fa.fa_bwd_layout(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 1, 0.125, 0,
                            layout, stream=0, check=False) == 1

"""The C-ABI library loads, exports what include/fa.h declares, and rejects bad
arguments on the host before touching a device (CPU only, no GPU needed)."""

import ctypes
import os
import re
import subprocess

import pytest

import online_softmax_14_b300 as fa
from online_softmax_14_b300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_ex", "fa_check_device_error", "fa_status_string", "fa_last_error_string"):
        assert n in names


@pytest.mark.parametrize("name", declared_functions())
def test_library_exports_declared_symbol(name):
    lib = ctypes.CDLL(B.library_path())
    assert hasattr(lib, name)
    out = subprocess.run(["nm", "-D", "--defined-only", B.library_path()], capture_output=True, text=True).stdout
    assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_status_strings_and_version():
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_UNKNOWN_STATUS"
    assert fa.fa_version() >= 100
    fa.fa_set_wait_timeout_ms(0)  # clamps, no crash
    fa.fa_set_wait_timeout_ms(1000)
    fa.fa_debug_inject(0)


P = 0x10000  # a fake, 16-byte-aligned address: these calls must fail before using it


def _fwd_ex(dtype=0, q=P, k=P, v=P, o=P, lse=None, kv=None, Bs=1, H=1, N=16, d=64, scale=0.125, causal=0):
    return B.fa_status_raw("fa_fwd_ex", dtype, q, k, v, o, lse, kv, Bs, H, N, d, ctypes.c_float(scale), causal, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), B.FA_ERR_INVALID),
    (dict(o=None), B.FA_ERR_INVALID),
    (dict(Bs=0), B.FA_ERR_INVALID),
    (dict(N=0), B.FA_ERR_INVALID),
    (dict(H=-1), B.FA_ERR_INVALID),
    (dict(scale=0.0), B.FA_ERR_INVALID),
    (dict(scale=-1.0), B.FA_ERR_INVALID),
    (dict(scale=float("nan")), B.FA_ERR_INVALID),
    (dict(scale=float("inf")), B.FA_ERR_INVALID),
    (dict(q=P + 8), B.FA_ERR_INVALID),          # bf16 needs 16-byte alignment (TMA)
    (dict(lse=P + 2), B.FA_ERR_INVALID),
    (dict(d=96), B.FA_ERR_UNSUPPORTED),         # bf16 serves d in {64, 128}
    (dict(d=32), B.FA_ERR_UNSUPPORTED),
    (dict(dtype=1, d=129), B.FA_ERR_UNSUPPORTED),
    (dict(dtype=1, v=P + 2), B.FA_ERR_INVALID),  # fp32 needs 4-byte alignment
    (dict(dtype=7), B.FA_ERR_INVALID),
    (dict(causal=3), B.FA_ERR_INVALID),          # causal is 0, 1 or 2
    (dict(causal=-1), B.FA_ERR_INVALID),
])
def test_host_validation(kw, status):
    assert _fwd_ex(**kw) == status
    assert fa.fa_last_error_string() != ""


def test_valid_call_without_gpu_fails_loudly():
    """On a machine without a usable GPU a well-formed call reports FA_ERR_CUDA
    (or FA_ERR_UNSUPPORTED for a non-sm_103 device) instead of doing anything on
    the CPU."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _fwd_ex()
    assert st in (B.FA_ERR_CUDA, B.FA_ERR_UNSUPPORTED)
    assert fa.fa_last_error_string()
    with pytest.raises(B.FaError):
        fa.fa_fwd(P, P, P, P, None, 1, 1, 16, 64, 0.125, False, stream=0)


def _bwd(q=P, k=P, v=P, o=P, do=P, lse=P, kv=None, dq=P, dk=P, dv=P, ws=P, ws_bytes=1 << 20, Bs=1, H=1, N=16, d=128,
         scale=0.125, causal=0):
    return B.fa_status_raw("fa_bwd_ex", q, k, v, o, do, lse, kv, dq, dk, dv, ws, ctypes.c_size_t(ws_bytes), Bs, H, N,
                           d, ctypes.c_float(scale), causal, None)


def test_bwd_workspace_size():
    # two float32 arrays of B*H*Np, Np = N rounded up to 128 (the query tile)
    assert fa.fa_bwd_workspace_size(2, 3, 100, 128) == 2 * 2 * 3 * 128 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 64, 128) == 2 * 128 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 129, 128) == 2 * 256 * 4
    assert fa.fa_bwd_workspace_size(0, 1, 64, 128) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(do=None), B.FA_ERR_INVALID),
    (dict(lse=None), B.FA_ERR_INVALID),
    (dict(dq=None), B.FA_ERR_INVALID),
    (dict(ws=None), B.FA_ERR_INVALID),
    (dict(dk=P + 4), B.FA_ERR_INVALID),
    (dict(ws=P + 8), B.FA_ERR_INVALID),
    (dict(ws_bytes=16), B.FA_ERR_INVALID),      # smaller than fa_bwd_workspace_size
    (dict(N=0), B.FA_ERR_INVALID),
    (dict(scale=float("nan")), B.FA_ERR_INVALID),
    (dict(d=64), B.FA_ERR_UNSUPPORTED),
    (dict(causal=5), B.FA_ERR_INVALID),
])
def test_bwd_host_validation(kw, status):
    assert _bwd(**kw) == status
    assert fa.fa_last_error_string() != ""


def _bwd_qk(q=P, k=P, v=P, o=P, do=P, lse=P, kv=None, dq=P, dk=P, dv=P, ws=P, ws_bytes=1 << 20, Bs=1, H=1, Nq=16,
            Nk=48, d=128, scale=0.125, causal=1):
    return B.fa_status_raw("fa_bwd_qk", q, k, v, o, do, lse, kv, dq, dk, dv, ws, ctypes.c_size_t(ws_bytes), Bs, H,
                           Nq, Nk, d, ctypes.c_float(scale), causal, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Nk=0), B.FA_ERR_INVALID),
    (dict(Nq=0), B.FA_ERR_INVALID),
    (dict(do=None), B.FA_ERR_INVALID),
    (dict(dv=P + 4), B.FA_ERR_INVALID),
    (dict(ws_bytes=16), B.FA_ERR_INVALID),      # smaller than fa_bwd_workspace_size(B, H, Nq, d)
    (dict(d=64), B.FA_ERR_UNSUPPORTED),
    (dict(causal=3), B.FA_ERR_INVALID),
])
def test_bwd_qk_host_validation(kw, status):
    assert _bwd_qk(**kw) == status
    assert fa.fa_last_error_string() != ""


def _merge(dtype=0, op=P, lp=P, n=2, o=P, lse=None, Bs=1, H=1, N=16, d=64):
    return B.fa_status_raw("fa_merge", dtype, op, lp, n, o, lse, Bs, H, N, d, None)


@pytest.mark.parametrize("kw,status", [
    (dict(op=None), B.FA_ERR_INVALID),
    (dict(lp=None), B.FA_ERR_INVALID),
    (dict(o=None), B.FA_ERR_INVALID),
    (dict(n=0), B.FA_ERR_INVALID),
    (dict(N=0), B.FA_ERR_INVALID),
    (dict(dtype=5), B.FA_ERR_INVALID),
    (dict(dtype=1, op=P + 2), B.FA_ERR_INVALID),   # fp32 parts need 4-byte alignment
    (dict(lp=P + 2), B.FA_ERR_INVALID),
    (dict(d=257), B.FA_ERR_UNSUPPORTED),
    (dict(n=4097), B.FA_ERR_UNSUPPORTED),
])
def test_merge_host_validation(kw, status):
    assert _merge(**kw) == status
    assert fa.fa_last_error_string() != ""

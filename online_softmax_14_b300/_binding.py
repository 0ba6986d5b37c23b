"""ctypes binding over libfa.so (include/fa.h).  Argument marshalling only.

Each C entry point has a Python function of the same name taking the same
arguments; a tensor argument may be a torch tensor (its ``data_ptr()`` is passed)
or a raw integer address, and ``stream`` defaults to PyTorch's current CUDA
stream.  A non-OK status raises ``FaError``.  ``attention_fwd`` is a convenience
wrapper that allocates the outputs with PyTorch and calls ``fa_fwd_ex``.

There is no fallback: if libfa.so has not been built, importing this module
raises ImportError naming the build command.
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with `python -m online_softmax_14_b300.build` "
        "(or __graft_entry__.build()); there is no CPU fallback")
_lib = ctypes.CDLL(_LIB_PATH)

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_BF16, FA_FP32 = 0, 1

_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_lib.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_fwd.restype = _i
_lib.fa_fwd_ex.argtypes = [_i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_fwd_ex.restype = _i
_lib.fa_fwd_qk.argtypes = [_i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_fwd_qk.restype = _i
_lib.fa_status_string.argtypes = [_i]
_lib.fa_status_string.restype = ctypes.c_char_p
_lib.fa_last_error_string.argtypes = []
_lib.fa_last_error_string.restype = ctypes.c_char_p
_lib.fa_check_device_error.argtypes = [_vp]
_lib.fa_check_device_error.restype = _i
_lib.fa_set_wait_timeout_ms.argtypes = [_i]
_lib.fa_set_wait_timeout_ms.restype = None
_lib.fa_debug_inject.argtypes = [_i]
_lib.fa_debug_inject.restype = None
_lib.fa_version.argtypes = []
_lib.fa_version.restype = _i
_sz = ctypes.c_size_t
_lib.fa_bwd_workspace_size.argtypes = [_i, _i, _i, _i]
_lib.fa_bwd_workspace_size.restype = _sz
_lib.fa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_bwd.restype = _i
_lib.fa_bwd_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_bwd_ex.restype = _i
_lib.fa_bwd_qk.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_bwd_qk.restype = _i
_lib.fa_merge.argtypes = [_i, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _vp]
_lib.fa_merge.restype = _i
_lib.fa_bwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_bwd_noalloc.restype = _i
FA_BWD_NOALLOC_MAX_ROWS = 524288
_lib.fa_std_workspace_size.argtypes = [_i, _i, _i]
_lib.fa_std_workspace_size.restype = _sz
_lib.fa_std_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _vp]
_lib.fa_std_fwd.restype = _i


class FaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{fa_status_string(status)}: {detail}")


def library_path() -> str:
    return _LIB_PATH


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _causal(causal) -> int:
    """0/False: no mask; 1/True: key j visible to query i iff j <= i; 2 or
    "strict": iff j < i (a query does not see its own key)."""
    if causal == "strict":
        return 2
    if isinstance(causal, bool) or causal is None:
        return int(bool(causal))
    return int(causal)


def _check(status: int):
    if status != FA_OK:
        raise FaError(status, _lib.fa_last_error_string().decode())


def fa_status_string(status: int) -> str:
    return _lib.fa_status_string(int(status)).decode()


def fa_last_error_string() -> str:
    return _lib.fa_last_error_string().decode()


def fa_version() -> int:
    return _lib.fa_version()


def fa_set_wait_timeout_ms(ms: int) -> None:
    _lib.fa_set_wait_timeout_ms(int(ms))


def fa_debug_inject(code: int) -> None:
    _lib.fa_debug_inject(int(code))


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream=None) -> None:
    _check(_lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale), _causal(causal),
                       _stream(stream)))


def fa_fwd_ex(dtype, q, k, v, o, lse, kv_len, B, H, N, d, scale, causal, stream=None) -> None:
    _check(_lib.fa_fwd_ex(int(dtype), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(kv_len), B, H, N, d,
                          float(scale), _causal(causal), _stream(stream)))


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(_lib.fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
           stream=None) -> None:
    _check(_lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                       _ptr(workspace), int(workspace_bytes), B, H, N, d, float(scale), _causal(causal),
                       _stream(stream)))


def fa_bwd_ex(q, k, v, o, do, lse, kv_len, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
              stream=None) -> None:
    _check(_lib.fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(kv_len), _ptr(dq),
                          _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), B, H, N, d, float(scale),
                          _causal(causal), _stream(stream)))


def fa_merge(dtype, o_parts, lse_parts, n_parts, o, lse, B, H, N, d, stream=None) -> None:
    _check(_lib.fa_merge(int(dtype), _ptr(o_parts), _ptr(lse_parts), int(n_parts), _ptr(o), _ptr(lse), B, H, N, d,
                         _stream(stream)))


def attention_merge(o_parts, lse_parts, stream=None):
    """O, lse of the merge of partial results: o_parts [P, B, H, N, d] (bf16 or
    fp32), lse_parts [P, B, H, N] fp32, CUDA tensors.  Allocates the outputs with
    PyTorch and runs ``fa_merge``."""
    if o_parts.dtype not in (torch.bfloat16, torch.float32) or lse_parts.dtype != torch.float32:
        raise TypeError("o_parts must be bf16 or fp32 and lse_parts fp32")
    if not (o_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_contiguous()
            and lse_parts.shape == o_parts.shape[:-1]):
        raise ValueError("o_parts [P, B, H, N, d] and lse_parts [P, B, H, N] must be contiguous CUDA tensors")
    P, B, H, N, d = o_parts.shape
    o = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
    lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    fa_merge(FA_BF16 if o_parts.dtype == torch.bfloat16 else FA_FP32, o_parts, lse_parts, P, o, lse, B, H, N, d,
             stream)
    return o, lse


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, causal, stream=None) -> None:
    """fa_bwd without a workspace argument: the library uses its own fixed
    device scratch (for callers that cannot allocate device memory)."""
    _check(_lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, H, N, d, float(scale), _causal(causal), _stream(stream)))


def fa_fwd_qk(dtype, q, k, v, o, lse, kv_len, B, H, Nq, Nk, d, scale, causal, stream=None) -> None:
    _check(_lib.fa_fwd_qk(int(dtype), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(kv_len), B, H, Nq, Nk, d,
                          float(scale), _causal(causal), _stream(stream)))


def fa_check_device_error(stream=None) -> None:
    _check(_lib.fa_check_device_error(_stream(stream)))


def fa_status_raw(fn_name: str, *args) -> int:
    """Call a C entry point by name with raw (already marshalled) arguments and
    return its status code without raising (for tests of the error paths)."""
    return getattr(_lib, fn_name)(*args)


def attention_fwd(q, k, v, scale=None, causal=False, kv_len=None, stream=None):
    """O, lse = attention of q [B, H, Nq, d] over k, v [B, H, Nk, d] (CUDA
    tensors, bf16 or fp32, contiguous; Nq may differ from Nk, see fa_fwd_qk).

    Allocates O (same dtype as q) and lse (fp32) with PyTorch, then runs
    ``fa_fwd_qk`` on ``stream`` (default: the current stream).
    """
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q, k, v must be bfloat16 or float32")
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == q.dtype and t.dim() == 4):
            raise ValueError("q, k, v must be contiguous 4-D CUDA tensors of one dtype")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q [B, H, Nq, d] and k, v [B, H, Nk, d] must agree in B, H and d")
    B, H, N, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    fa_fwd_qk(FA_BF16 if q.dtype == torch.bfloat16 else FA_FP32, q, k, v, o, lse, kv_len, B, H, N, Nk, d, scale,
              causal, stream)
    return o, lse


def fa_bwd_qk(q, k, v, o, do, lse, kv_len, dq, dk, dv, workspace, workspace_bytes, B, H, Nq, Nk, d, scale, causal,
              stream=None) -> None:
    _check(_lib.fa_bwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(kv_len), _ptr(dq),
                          _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), B, H, Nq, Nk, d, float(scale),
                          _causal(causal), _stream(stream)))


def attention_bwd(q, k, v, o, lse, do, scale=None, causal=False, kv_len=None, stream=None):
    """dQ, dK, dV (float32) of attention over bf16 CUDA tensors: q, o, do
    [B, H, Nq, d] and k, v [B, H, Nk, d] (Nq may differ from Nk; a causal mask is
    then aligned bottom-right, as in ``attention_fwd``).

    ``o`` and ``lse`` are the forward's outputs for the same inputs.  Allocates
    the gradients and the workspace with PyTorch, then runs ``fa_bwd_qk``.
    """
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    for t, shape in ((q, q.shape), (o, q.shape), (do, q.shape), (k, (B, H, Nk, d)), (v, (B, H, Nk, d))):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16 and tuple(t.shape) == tuple(shape)):
            raise ValueError("q, o, do must be contiguous bf16 CUDA tensors of shape [B, H, Nq, d] and k, v of "
                             "shape [B, H, Nk, d]")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty_like(dk)
    ws_bytes = fa_bwd_workspace_size(B, H, Nq, d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    fa_bwd_qk(q, k, v, o, do, lse.contiguous(), kv_len, dq, dk, dv, ws, ws_bytes, B, H, Nq, Nk, d, scale, causal,
              stream)
    return dq, dk, dv


def fa_std_workspace_size(B, H, N) -> int:
    return int(_lib.fa_std_workspace_size(B, H, N))


def fa_std_fwd(q, k, v, o, lse, kv_len, workspace, workspace_bytes, B, H, N, d, scale, causal, stream=None) -> None:
    _check(_lib.fa_std_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(kv_len), _ptr(workspace),
                           int(workspace_bytes), B, H, N, d, float(scale), _causal(causal), _stream(stream)))


def standard_attention_fwd(q, k, v, scale=None, causal=False, kv_len=None, stream=None):
    """O, lse by standard attention (S and P written to device memory in full):
    the comparator of the tiled kernels.  q, k, v bf16 [B, H, N, d] CUDA tensors.
    Allocates the outputs and the S / P workspace with PyTorch, then runs
    ``fa_std_fwd``."""
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    nbytes = fa_std_workspace_size(B, H, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    fa_std_fwd(q, k, v, o, lse, kv_len, ws, nbytes, B, H, N, d, scale, causal, stream)
    return o, lse

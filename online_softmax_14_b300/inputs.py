"""Seeded synthetic inputs for the attention kernels and for the CPU oracle.

This module holds no attention arithmetic: it only draws random tensors, so both
the CUDA path and the oracle can be fed the very same values.  Importing it does
not load the CUDA library.

Recipe (fixed, so every run sees identical inputs):
  * one CPU ``torch.Generator`` seeded with ``seed`` (default 0);
  * float32 standard-normal draws of shape [B, H, N, d] in the order Q, K, V, then
    dO when a backward pass is wanted;
  * Q and K multiplied by ``qk_mul`` (8 for the overflow-stress workload: a power
    of two, so the scaling is exact before and after rounding to bfloat16);
  * then cast to the workload dtype (bfloat16 or float32) -- the oracle receives
    these rounded values, converted exactly to float64;
  * key-padding lengths, when wanted, drawn last as integers uniform in [0, N],
    with kv_len[0] = 0 and kv_len[1] = N forced so that a fully masked batch and an
    unpadded batch always occur;
  * scale = 1/sqrt(d) rounded to float32.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One attention problem shape.  ``name`` describes it in words."""

    name: str
    dtype: str  # "bf16" or "fp32"
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qk_mul: float = 1.0
    padded: bool = False
    backward: bool = False
    note: str = field(default="", compare=False)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# The five workloads the performance and parity targets are quoted on.
WORKLOADS = {
    "fp32_B1_H1_N256_d64": Workload("fp32_B1_H1_N256_d64", "fp32", 1, 1, 256, 64, False,
                                    note="single-head float32 correctness case"),
    "bf16_causal_B4_H16_N2048_d64": Workload("bf16_causal_B4_H16_N2048_d64", "bf16", 4, 16, 2048, 64, True),
    "bf16_causal_B2_H32_N8192_d128": Workload("bf16_causal_B2_H32_N8192_d128", "bf16", 2, 32, 8192, 128, True,
                                              note="long-sequence throughput case"),
    "bf16_padded_stress_B8_H16_N1024_d128": Workload("bf16_padded_stress_B8_H16_N1024_d128", "bf16", 8, 16, 1024,
                                                     128, False, qk_mul=8.0, padded=True,
                                                     note="logits near +-500 and per-batch key padding"),
    "bf16_causal_fwdbwd_B4_H16_N4096_d128": Workload("bf16_causal_fwdbwd_B4_H16_N4096_d128", "bf16", 4, 16, 4096,
                                                     128, True, backward=True),
}


def default_scale(d: int) -> float:
    """1/sqrt(d) rounded to float32, returned as the exact Python float of that value."""
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32).item())


def make_problem(B, H, N, d, dtype="bf16", seed=0, qk_mul=1.0, padded=False, backward=False,
                 kv_len=None):
    """Draw one problem on the CPU.

    Returns a dict with q, k, v (and do when ``backward``) as CPU tensors of the
    requested dtype, ``kv_len`` (int32 tensor [B] or None) and ``scale``.
    ``kv_len`` may be given explicitly (a list) instead of drawn (``padded``).
    """
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32) if backward else None
    if qk_mul != 1.0:
        q.mul_(qk_mul)
        k.mul_(qk_mul)
    out = {
        "q": q.to(tdt).contiguous(),
        "k": k.to(tdt).contiguous(),
        "v": v.to(tdt).contiguous(),
        "do": None if do is None else do.to(tdt).contiguous(),
        "scale": default_scale(d),
        "kv_len": None,
    }
    if kv_len is not None:
        out["kv_len"] = torch.tensor(list(kv_len), dtype=torch.int32)
    elif padded:
        kl = torch.randint(0, N + 1, (B,), generator=g, dtype=torch.int64)
        if B >= 1:
            kl[0] = 0
        if B >= 2:
            kl[1] = N
        out["kv_len"] = kl.to(torch.int32)
    return out


def make_workload(w: Workload, seed=0):
    """Draw the inputs of a named workload (see ``WORKLOADS``)."""
    return make_problem(w.B, w.H, w.N, w.d, w.dtype, seed, w.qk_mul, w.padded, w.backward)

"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc when they need a gradient: code running
inside an allocator's own hooks, runtimes whose device pool is fixed and fully
handed out at start-up, and hosts that forbid allocation after initialisation.
fa_bwd_noalloc serves them with a fixed device array inside the library instead
of a caller workspace.  These tests check that it gives the same gradients as
fa_bwd with a workspace, and that both match the float64 oracle, on two calls in
a row (the second call finds the first call's data still in the shared array),
and that a problem too large for the fixed array is refused with a clear
error.

This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from online_softmax_14_b300 import _binding as B
from online_softmax_14_b300.inputs import make_problem

G_MAX, G_MEAN = 2e-2, 2e-3  # the backward parity bar used by the other GPU tests
DEV = "cuda:0"


def _grads_both_ways(pr, causal):
    import online_softmax_14_b300 as fa

    q, k, v, do = (pr[n].to(DEV) for n in ("q", "k", "v", "do"))
    Bs, H, N, d = q.shape
    o, lse = fa.attention_fwd(q, k, v, pr["scale"], causal=causal)
    ref = fa.attention_bwd(q, k, v, o, lse, do, pr["scale"], causal=causal)  # fa_bwd_ex with a workspace
    out = [torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV) for _ in range(3)]
    fa.fa_bwd_noalloc(q, k, v, o, do, lse, out[0], out[1], out[2], Bs, H, N, d, pr["scale"], causal)
    fa.fa_check_device_error()
    return [t.cpu().numpy() for t in out], [t.cpu().numpy() for t in ref]


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice():
    cases = [((2, 2, 200), True, 21), ((1, 3, 384), False, 22)]
    for (Bs, H, N), causal, seed in cases:
        pr = make_problem(Bs, H, N, 128, "bf16", seed=seed, backward=True)
        got, ref = _grads_both_ways(pr, causal)
        exact = oracle.attention_bwd(pr["q"], pr["k"], pr["v"], pr["do"], pr["scale"], causal=causal)
        for name, g, r, x in zip(("dQ", "dK", "dV"), got, ref, exact):
            assert np.all(np.isfinite(g)), f"{name} (N={N}): non-finite"
            for other, label in ((r, "fa_bwd"), (x, "oracle")):
                err = np.abs(g - other)
                assert err.max() <= G_MAX and err.mean() <= G_MEAN, \
                    f"{name} (N={N}) vs {label}: max err {err.max():.3g}, mean {err.mean():.3g}"


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    """B*H*Np above the fixed limit is refused before any device work (no GPU needed)."""
    P = 0x10000  # a fake aligned address: the call must fail before using it
    H = B.FA_BWD_NOALLOC_MAX_ROWS // 4096 + 1  # N = 4096 is already a multiple of 64
    st = B.fa_status_raw("fa_bwd_noalloc", P, P, P, P, P, P, P, P, P, 1, H, 4096, 128, ctypes.c_float(0.088), 1,
                         None)
    assert st == B.FA_ERR_UNSUPPORTED
    assert "fa_bwd_noalloc" in B.fa_last_error_string() and "fa_bwd" in B.fa_last_error_string()

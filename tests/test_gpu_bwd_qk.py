"""GPU parity of the backward for queries and keys of different lengths (needs a B300).

Nq queries and Nk keys per head, the queries read as the last Nq positions of the
key sequence, so a causal mask is aligned bottom-right: the reading the forward
(fa_fwd_qk) and the oracle (visible_mask) use for Nq != Nk.  The CUDA path runs
our forward for O and lse, then fa_bwd_qk; the oracle differentiates the exact
definition on the same bf16-rounded inputs.  The bar is the backward's bf16 bar
(max-abs 2e-2, mean-abs 2e-3 per gradient tensor).
"""

import numpy as np
import pytest
import torch

import oracle
from online_softmax_14_b300.inputs import make_problem

pytestmark = pytest.mark.gpu

G_MAX, G_MEAN = 2e-2, 2e-3
DEV = "cuda:0"
GUARD = 1 << 16
PATTERN = 0xA5


def fa():
    import online_softmax_14_b300 as m
    return m


def problem(B, H, Nq, Nk, seed, kv_len=None):
    pq = make_problem(B, H, Nq, 128, "bf16", seed=seed, backward=True)
    pk = make_problem(B, H, Nk, 128, "bf16", seed=seed + 1000)
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32)
    return pq["q"], pk["k"], pk["v"], pq["do"], pq["scale"], kv


def check(got, ref, label):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert g.shape == r.shape, f"{label} {name}: shape {g.shape} vs {r.shape}"
        assert np.all(np.isfinite(g)), f"{label} {name}: non-finite"
        err = np.abs(g - r)
        assert err.max() <= G_MAX, f"{label} {name}: max err {err.max():.3g} (|ref| max {np.abs(r).max():.3g})"
        assert err.mean() <= G_MEAN, f"{label} {name}: mean err {err.mean():.3g}"


@pytest.mark.parametrize("B,H,Nq,Nk,causal,kv_len", [
    (1, 2, 128, 384, 1, None),       # three key tiles, one query tile, bottom-right diagonal
    (2, 2, 256, 512, 1, None),
    (1, 2, 1, 300, 1, None),         # one decode query sees every key
    (2, 1, 200, 131, 1, None),       # more queries than keys: the first 69 rows see no key
    (1, 2, 77, 257, 2, None),        # strictly causal, ragged
    (2, 1, 130, 260, 0, [260, 100]),  # no causal mask, key padding
    (2, 1, 96, 300, 1, [0, 250]),    # a batch with no keys at all
])
def test_bwd_qk_parity(B, H, Nq, Nk, causal, kv_len):
    q, k, v, do, scale, kv = problem(B, H, Nq, Nk, seed=Nq + 7 * Nk + causal, kv_len=kv_len)
    m = fa()
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    kvd = None if kv is None else kv.to(DEV)
    o, lse = m.attention_fwd(qd, kd, vd, scale, causal=causal, kv_len=kvd)
    dq, dk, dv = m.attention_bwd(qd, kd, vd, o, lse, dod, scale, causal=causal, kv_len=kvd)
    m.fa_check_device_error()
    got = tuple(t.cpu().numpy().astype(np.float64) for t in (dq, dk, dv))
    ref = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv_len)
    check(got, ref, f"B{B} H{H} Nq{Nq} Nk{Nk} c{causal} kv{kv_len}")


def test_bwd_qk_equal_lengths_matches_fa_bwd():
    """fa_bwd_qk with Nq = Nk gives exactly what fa_bwd gives (same kernels)."""
    B, H, N = 2, 2, 200
    q, k, v, do, scale, _ = problem(B, H, N, N, seed=3)
    m = fa()
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = m.attention_fwd(qd, kd, vd, scale, causal=True)
    a = m.attention_bwd(qd, kd, vd, o, lse, dod, scale, causal=True)
    ws_bytes = m.fa_bwd_workspace_size(B, H, N, 128)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    b = [torch.empty(B, H, N, 128, dtype=torch.float32, device=DEV) for _ in range(3)]
    m.fa_bwd(qd, kd, vd, o, dod, lse, *b, ws, ws_bytes, B, H, N, 128, scale, True)
    m.fa_check_device_error()
    # dQ is summed with floating-point reductions in any order: compare to rounding
    for x, y in zip(a, b):
        assert torch.allclose(x, y, rtol=0, atol=1e-5)


class Guarded:
    """A float32 tensor inside a byte buffer with guards on both sides."""

    def __init__(self, shape):
        n = int(np.prod(shape)) * 4
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + n].view(torch.float32).view(shape)
        self.n = n

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.n:] == PATTERN).all())


@pytest.mark.parametrize("Nq,Nk,causal", [(1, 300, 1), (200, 131, 1), (77, 257, 2), (129, 513, 0)])
def test_bwd_qk_writes_stay_inside_outputs(Nq, Nk, causal):
    B, H = 2, 2
    q, k, v, do, scale, _ = problem(B, H, Nq, Nk, seed=Nq + Nk)
    m = fa()
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = m.attention_fwd(qd, kd, vd, scale, causal=causal)
    dq = Guarded((B, H, Nq, 128))
    dk, dv = Guarded((B, H, Nk, 128)), Guarded((B, H, Nk, 128))
    ws_bytes = m.fa_bwd_workspace_size(B, H, Nq, 128)
    ws = Guarded((ws_bytes // 4,))
    m.fa_bwd_qk(qd, kd, vd, o, dod, lse, None, dq.t, dk.t, dv.t, ws.t, ws_bytes, B, H, Nq, Nk, 128, scale, causal)
    m.fa_check_device_error()
    assert dq.intact() and dk.intact() and dv.intact() and ws.intact()

"""The backward oracle pinned by finite differences and by torch.autograd (CPU only)."""

import math

import numpy as np
import pytest
import torch

import oracle

CASES = [
    (1, 1, 5, 3, False, None),
    (1, 2, 6, 4, True, None),
    (2, 1, 7, 2, False, [3, 7]),
    (2, 1, 6, 4, True, [0, 5]),
    (1, 2, 6, 3, 2, None),           # strictly causal (Worked examples, Cell D2's setting)
]


def _inputs(seed, B, H, N, d):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, H, N, d)) for _ in range(4)]


@pytest.mark.parametrize("case", CASES)
def test_bwd_matches_central_differences(case):
    B, H, N, d, causal, kv = case
    q, k, v, do = _inputs(CASES.index(case), B, H, N, d)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal=causal, kv_len=kv)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(num - g)) < 2e-7, name


@pytest.mark.parametrize("case", CASES)
def test_bwd_matches_autograd(case):
    B, H, N, d, causal, kv = case
    q, k, v, do = _inputs(10 + CASES.index(case), B, H, N, d)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    vis = torch.ones(B, 1, N, N, dtype=torch.bool)
    if causal:  # inclusive (j <= i) or, for causal = 2, strict (j < i)
        vis &= torch.ones(N, N, dtype=torch.bool).tril(-1 if causal == 2 else 0)
    if kv is not None:
        for b in range(B):
            vis[b, :, :, kv[b]:] = False
    s = s.masked_fill(~vis, float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)  # fully masked rows -> 0
    o = p @ tv
    (o * torch.tensor(do)).sum().backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_bwd_delta_identity():
    """D_i = sum_j P_ij dP_ij equals rowsum(dO * O): both sides of the identity the
    GPU preprocess step relies on, computed from the oracle's forward."""
    q, k, v, do = _inputs(9, 1, 2, 9, 4)
    o, _ = oracle.attention_fwd(q, k, v, 0.5, causal=True)
    s = 0.5 * q @ np.swapaxes(k, -1, -2)
    s = np.where(np.tril(np.ones((9, 9), bool)), s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True)); p /= p.sum(-1, keepdims=True)
    dp = do @ np.swapaxes(v, -1, -2)
    assert np.allclose((p * dp).sum(-1), (do * o).sum(-1), atol=1e-13)

# Queries and keys of different lengths (the decode / chunked-prefill reading of the
# forward: queries are the last Nq positions of the key sequence, so a causal mask is
# aligned bottom-right).  (B, H, Nq, Nk, d, causal, kv_len)
CASES_QK = [
    (1, 1, 3, 7, 2, True, None),
    (1, 2, 1, 6, 3, True, None),       # one decode query sees every key
    (1, 1, 6, 4, 2, True, None),       # more queries than keys: the first two see none
    (2, 1, 4, 6, 2, 2, [6, 3]),        # strictly causal with key padding
    (1, 1, 2, 5, 3, False, None),
]


def _inputs_qk(seed, B, H, Nq, Nk, d):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, H, Nq, d)), rng.standard_normal((B, H, Nk, d)),
            rng.standard_normal((B, H, Nk, d)), rng.standard_normal((B, H, Nq, d)))


@pytest.mark.parametrize("case", CASES_QK)
def test_bwd_qk_matches_central_differences(case):
    B, H, Nq, Nk, d, causal, kv = case
    q, k, v, do = _inputs_qk(20 + CASES_QK.index(case), B, H, Nq, Nk, d)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal=causal, kv_len=kv)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(num - g)) < 2e-7, name


@pytest.mark.parametrize("case", CASES_QK)
def test_bwd_qk_matches_autograd(case):
    B, H, Nq, Nk, d, causal, kv = case
    q, k, v, do = _inputs_qk(40 + CASES_QK.index(case), B, H, Nq, Nk, d)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    vis = torch.ones(B, 1, Nq, Nk, dtype=torch.bool)
    if causal:  # query i sits at key position i + (Nk - Nq)
        vis &= torch.ones(Nq, Nk, dtype=torch.bool).tril(Nk - Nq - (1 if causal == 2 else 0))
    if kv is not None:
        for b in range(B):
            vis[b, :, :, kv[b]:] = False
    s = s.masked_fill(~vis, float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)  # fully masked rows -> 0
    o = p @ tv
    (o * torch.tensor(do)).sum().backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-12)

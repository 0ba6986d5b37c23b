"""The oracle pinned to what the pages and the mathematics fix (CPU only)."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import online
from pins import ALL_CHECKS, load_golden


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_passes_pin(check):
    fails = check(oracle.attention_fwd)
    assert not fails, "\n".join(fails)


@pytest.mark.parametrize("case", load_golden()["merges"], ids=lambda c: c["id"])
def test_merge_rule_against_page(case):
    """The block-state merge reproduces the Exercises / Worked examples merges."""
    rtol = case["rtol"]
    if "states" in case:
        states = [(s[0], s[1], np.asarray(s[2], float)) for s in case["states"]]
        st = states[0]
        for i, nxt in enumerate(states[1:]):
            st = online.merge_states(st, nxt)
            if i == 0 and "intermediate_l" in case:
                assert st[1] == pytest.approx(case["intermediate_l"], rel=rtol)
        # any other grouping and order gives the same state (associativity)
        rev = states[-1]
        for nxt in reversed(states[:-1]):
            rev = online.merge_states(nxt, rev)
        assert rev[0] == st[0] and rev[1] == pytest.approx(st[1], rel=1e-14)
    else:
        states = [online.block_state(s, v) for s, v in zip(case["block_scores"], case["block_values"])]
        st = online.merge_states(states[0], states[1])
    assert st[0] == case["m"]
    assert st[1] == pytest.approx(case["l"], rel=rtol)
    if "acc" in case:
        assert np.allclose(st[2], case["acc"], rtol=rtol)
    if "out" in case:
        out, _ = online.finish(st)
        assert np.allclose(out, case["out"], rtol=rtol)


def test_overflow_naive_vs_safe():
    """Exercises, overflow exercise: exp(800) overflows in float64, so the naive
    softmax is NaN, while the oracle's max-shifted result stays finite (17.3106)."""
    s = np.array([800.0, 801.0])
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.exp(s) / np.exp(s).sum()
    assert np.all(np.isnan(naive))
    q = np.ones((1, 1, 2, 1)); k = s.reshape(1, 1, 2, 1); v = np.array([10.0, 20.0]).reshape(1, 1, 2, 1)
    o, lse = oracle.attention_fwd(q, k, v, 1.0)
    assert np.all(np.isfinite(o)) and o[0, 0, 0, 0] == pytest.approx(17.3106, rel=5e-6)
    assert lse[0, 0, 0] == pytest.approx(801 + math.log(1 + math.exp(-1)), rel=1e-15)


def test_library_softmax_agrees():
    """A library routine for the same definition (torch.softmax, float64) agrees."""
    g = torch.Generator().manual_seed(3)
    B, H, N, d = 2, 3, 33, 8
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    scale = 1 / math.sqrt(d)
    for causal in (False, True):
        s = scale * q @ k.transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        want = torch.softmax(s, dim=-1) @ v
        lse_want = torch.logsumexp(s, dim=-1)
        o, lse = oracle.attention_fwd(q.numpy(), k.numpy(), v.numpy(), scale, causal=causal)
        assert np.allclose(o, want.numpy(), rtol=1e-12, atol=1e-13)
        assert np.allclose(lse, lse_want.numpy(), rtol=1e-13)


def test_rows_entry_matches_full():
    """attention_fwd_rows (sampled rows) equals the full evaluation row by row."""
    rng = np.random.default_rng(11)
    B, H, N, d = 2, 2, 40, 8
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    kv = [17, 40]
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, 0.3, causal=causal, kv_len=kv)
        rows = [(0, 1, 0), (0, 0, 16), (0, 0, 17), (1, 1, 39), (1, 0, 5)]
        ro, rl = oracle.attention_fwd_rows(q, k, v, 0.3, causal, kv, rows)
        for n, (b, h, i) in enumerate(rows):
            assert np.allclose(ro[n], o[b, h, i], rtol=1e-14, atol=1e-15)
            assert rl[n] == pytest.approx(lse[b, h, i], rel=1e-14)


def test_bf16_inputs_convert_exactly():
    """bfloat16 tensors reach the oracle exactly (every bf16 value is a float64)."""
    t = torch.randn(1, 1, 4, 4).to(torch.bfloat16)
    from oracle.attention import _f64
    a = _f64(t)
    assert a.dtype == np.float64
    assert np.array_equal(a, t.float().numpy().astype(np.float64))


def test_strictly_causal_cell_d2():
    """Worked examples, Cell D2: in a strictly causal setup query 0 has no earlier
    token, every score is -inf, l = 0, and the output is the zero vector (lse is
    -inf).  Every later query i attends exactly to keys 0 .. i-1."""
    rng = np.random.default_rng(21)
    N, d = 6, 3
    q, k, v = (rng.standard_normal((1, 1, N, d)) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.5, causal=oracle.STRICT)
    assert np.array_equal(o[0, 0, 0], np.zeros(d)) and np.isneginf(lse[0, 0, 0])
    for i in range(1, N):
        # the same row computed without a mask over the i earlier keys only
        oi, li = oracle.attention_fwd(q[:, :, i:i + 1], k[:, :, :i], v[:, :, :i], 0.5)
        assert np.allclose(o[0, 0, i], oi[0, 0, 0], rtol=1e-14) and lse[0, 0, i] == pytest.approx(li[0, 0, 0])
    # inclusive causal differs from strict exactly by the diagonal key
    o1, _ = oracle.attention_fwd(q, k, v, 0.5, causal=True)
    assert not np.allclose(o1[0, 0, 1:], o[0, 0, 1:])
    # the recurrence model and the backward agree with the definition in this mode
    oo, lo = online.online_attention(q, k, v, 0.5, causal=oracle.STRICT, block_size=2)
    assert np.allclose(oo, o, atol=1e-14) and np.array_equal(np.isneginf(lo), np.isneginf(lse))
    do = rng.standard_normal(q.shape)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.5, causal=oracle.STRICT)
    assert np.all(dq[0, 0, 0] == 0)                       # query 0 took part in nothing
    assert np.all(dk[0, 0, N - 1] == 0) and np.all(dv[0, 0, N - 1] == 0)  # the last key is seen by no query


@pytest.mark.parametrize("nq,nk", [(1, 9), (3, 9), (9, 4), (5, 5)])
@pytest.mark.parametrize("causal", [1, 2])
def test_fewer_or_more_queries_than_keys(nq, nk, causal):
    """With Nq != Nk the queries are the last Nq positions: query i sits at key
    position i + Nk - Nq.  Each row must equal unmasked attention over exactly
    the keys it may see (brute force by slicing); a row that sees no key gives
    O = 0, lse = -inf.  A single query with every key visible is plain
    attention over all keys (the decode case)."""
    rng = np.random.default_rng(nq * 10 + nk + causal)
    d = 3
    q = rng.standard_normal((1, 2, nq, d))
    k, v = (rng.standard_normal((1, 2, nk, d)) for _ in range(2))
    o, lse = oracle.attention_fwd(q, k, v, 0.6, causal=causal)
    assert o.shape == (1, 2, nq, d) and lse.shape == (1, 2, nq)
    for i in range(nq):
        last = i + nk - nq if causal == 1 else i + nk - nq - 1   # last visible key
        if last < 0:
            assert np.all(o[0, :, i] == 0) and np.all(np.isneginf(lse[0, :, i]))
            continue
        oi, li = oracle.attention_fwd(q[:, :, i:i + 1], k[:, :, :last + 1], v[:, :, :last + 1], 0.6)
        assert np.allclose(o[:, :, i], oi[:, :, 0], rtol=1e-14) and np.allclose(lse[:, :, i], li[:, :, 0])
    if nq == 1 and causal == 1:
        o_all, lse_all = oracle.attention_fwd(q, k, v, 0.6)
        assert np.allclose(o, o_all, rtol=1e-14) and np.allclose(lse, lse_all, rtol=1e-14)
    rows = [(0, h, i) for h in range(2) for i in range(nq)]
    o_r, l_r = oracle.attention_fwd_rows(q, k, v, 0.6, causal, None, rows)
    assert np.allclose(o_r, o[0].reshape(-1, d), rtol=1e-14)
    assert np.array_equal(np.isneginf(l_r), np.isneginf(lse[0].reshape(-1)))

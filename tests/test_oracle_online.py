"""The streaming recurrence model against the two-pass definition (CPU only).

Restates the live check of "The Flash Attention" page: flash and naive agree to
1e-10 in double precision on a fixed-seed d = 4 problem for every block size, the
flash path stays finite where a naive softmax without the max shift overflows,
and dropping the rescale factor c = exp(m_old - m_new) makes them disagree.
"""

import numpy as np
import pytest

import oracle
from oracle import online


def _problem(seed, N=24, d=4, scale_mul=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, 2, N, d)) * scale_mul
    k = rng.standard_normal((1, 2, N, d)) * scale_mul
    v = rng.standard_normal((1, 2, N, d))
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_every_block_size_matches_definition(causal):
    q, k, v = _problem(1)
    scale = 0.5
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, scale, causal=causal, kv_len=[19])
    for bs in range(1, q.shape[2] + 1):
        o, lse = online.online_attention(q, k, v, scale, causal=causal, kv_len=[19], block_size=bs)
        assert np.max(np.abs(o - o_ref)) < 1e-10, bs
        assert np.max(np.abs(lse - lse_ref)) < 1e-10, bs


def test_extreme_regime_naive_overflows_flash_finite():
    q, k, v = _problem(2, scale_mul=30.0)  # logits of several hundred
    scale = 0.5
    s = scale * q[0, 0] @ k[0, 0].T
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(s)
        naive = (e / e.sum(axis=1, keepdims=True)) @ v[0, 0]
    assert not np.all(np.isfinite(naive))
    o, _ = online.online_attention(q, k, v, scale, block_size=5)
    o_ref, _ = oracle.attention_fwd(q, k, v, scale)
    assert np.all(np.isfinite(o))
    assert np.max(np.abs(o - o_ref)) < 1e-10


def test_dropping_rescale_breaks_exactness():
    """The page's red-team move: forget c.  The result must no longer match."""
    q, k, v = _problem(3)
    o_ref, _ = oracle.attention_fwd(q, k, v, 0.5)
    o_bad, _ = online.online_attention(q, k, v, 0.5, block_size=4, drop_rescale=True)
    assert np.max(np.abs(o_bad - o_ref)) > 1e-3


def test_block_order_invariance():
    """Worked examples, Cell H: any block order gives the same result."""
    rng = np.random.default_rng(5)
    s = rng.standard_normal(37) * 3
    vals = rng.standard_normal((37, 3))
    base = online.online_row(s, vals, 6)
    nblk = (37 + 5) // 6
    for _ in range(10):
        order = rng.permutation(nblk)
        got = online.online_row(s, vals, 6, order=order)
        assert np.allclose(got[0], base[0], rtol=1e-13, atol=1e-14)
        assert got[1] == pytest.approx(base[1], rel=1e-14)


def test_masked_block_contributes_nothing():
    """Worked examples, Cell D: a block of -inf scores leaves (m, l, acc) as it was."""
    st = online.block_state([2.0, 1.0], [[10.0], [20.0]])
    masked = (-np.inf, 0.0, np.zeros(1))
    merged = online.merge_states(st, masked)
    assert merged[0] == st[0] and merged[1] == st[1] and np.array_equal(merged[2], st[2])
    both = online.merge_states(masked, masked)
    assert both[0] == -np.inf and both[1] == 0.0 and np.all(both[2] == 0.0)
    out, lse = online.finish(both)
    assert np.all(out == 0.0) and lse == -np.inf

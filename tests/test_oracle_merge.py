"""The merge of normalised partial results (oracle.merge_outputs), pinned.

A part (O_p, lse_p) over a key subset is the block state (m = lse_p, l = 1,
O~ = O_p), so the pages' merges pin it directly: each printed state
(m, l, O~) becomes (O~ / l, m + ln l), and the merged O and lse must reproduce
the printed merged output and m_new + ln l_new.  Brute force then checks it
against the definition: attention over all keys equals the merge of attention
over any split of the keys.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import online
from pins import load_golden


def _as_parts(states):
    o = np.stack([np.asarray(acc, float) / l for (m, l, acc) in states])
    lse = np.array([m + math.log(l) for (m, l, acc) in states])
    return o, lse


@pytest.mark.parametrize("case", load_golden()["merges"], ids=lambda c: c["id"])
def test_merge_outputs_against_page(case):
    if "states" in case:
        states = [(s[0], s[1], s[2]) for s in case["states"]]
    else:
        states = [online.block_state(s, v) for s, v in zip(case["block_scores"], case["block_values"])]
    o, lse = _as_parts(states)
    out, out_lse = oracle.merge_outputs(o, lse)
    rtol = case["rtol"]
    assert out_lse == pytest.approx(case["m"] + math.log(case["l"]), rel=rtol)
    if "out" in case:
        assert np.allclose(out, case["out"], rtol=rtol)
    # any order of the parts gives the same result
    out_r, lse_r = oracle.merge_outputs(o[::-1], lse[::-1])
    assert np.allclose(out_r, out, rtol=1e-14) and lse_r == pytest.approx(out_lse, rel=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cuts", [[4], [1, 5], [3, 6, 7], [2, 2, 5]])
def test_split_keys_then_merge_equals_full_attention(cuts, causal):
    """Attention over every key is the merge of attention over disjoint key
    ranges (each range evaluated by the definition with the other keys masked)."""
    rng = np.random.default_rng(len(cuts) + 10 * causal)
    N, d = 9, 3
    q, k, v = (rng.standard_normal((1, 2, N, d)) for _ in range(3))
    o_full, lse_full = oracle.attention_fwd(q, k, v, 0.7, causal=causal)
    bounds = [0] + cuts + [N]
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o_p = np.zeros_like(o_full)
        l_p = np.full(lse_full.shape, -np.inf)
        for i in range(N):
            s = 0.7 * (k[0, :, a:b] @ q[0, :, i, :, None])[..., 0]      # [H, b - a]
            vis = np.arange(a, b) <= i if causal else np.ones(b - a, bool)
            if not vis.any():
                continue
            s = np.where(vis[None], s, -np.inf)
            mx = s.max(axis=-1, keepdims=True)
            e = np.exp(s - mx)
            l_p[0, :, i] = mx[:, 0] + np.log(e.sum(-1))
            o_p[0, :, i] = (e[..., None] * v[0, :, a:b]).sum(1) / e.sum(-1, keepdims=True)
        parts_o.append(o_p)
        parts_l.append(l_p)
    o_m, lse_m = oracle.merge_outputs(np.stack(parts_o), np.stack(parts_l))
    assert np.allclose(o_m, o_full, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse_m, lse_full, rtol=1e-13)


def test_merge_special_cases():
    o = np.array([[1.0, -2.0], [3.0, 5.0]])
    # a part that saw no key carries no weight
    out, lse = oracle.merge_outputs(np.stack([o, 7 * o]), np.array([[0.3, -1.0], [-np.inf, -np.inf]]))
    assert np.array_equal(out, o) and np.array_equal(lse, [0.3, -1.0])
    # every part empty: O = 0, lse = -inf (Worked examples, Cell D2)
    out, lse = oracle.merge_outputs(np.stack([o, o]), np.full((2, 2), -np.inf))
    assert np.array_equal(out, np.zeros_like(o)) and np.all(np.isneginf(lse))
    # two identical parts: the same output, the normaliser doubles
    out, lse = oracle.merge_outputs(np.stack([o, o]), np.array([[0.5, 2.0], [0.5, 2.0]]))
    assert np.allclose(out, o, rtol=1e-15) and np.allclose(lse, np.array([0.5, 2.0]) + math.log(2), rtol=1e-15)
    # logits far apart (exp would overflow without the max shift)
    out, lse = oracle.merge_outputs(np.stack([o[:1], 2 * o[:1]]), np.array([[800.0], [801.0]]))
    w = 1 / (1 + math.e)
    assert np.allclose(out, w * o[:1] + (1 - w) * 2 * o[:1], rtol=1e-14)
    assert lse[0] == pytest.approx(801 + math.log(1 + math.exp(-1)), rel=1e-15)


@pytest.mark.parametrize("mutant", ["drop_weight", "max_not_logsumexp", "no_division"])
def test_pins_catch_planted_merge_mistakes(mutant, monkeypatch):
    """A plausible mistake planted in the merge must fail the page pins."""
    real = online.merge_outputs

    def broken(o_parts, lse_parts):
        o = np.asarray(o_parts, float)
        lse = np.asarray(lse_parts, float)
        if mutant == "drop_weight":                # plain average of the parts
            return o.mean(0), np.log(np.exp(lse).sum(0))
        out, out_lse = real(o, lse)
        if mutant == "max_not_logsumexp":          # lse taken as the largest part's
            return out, lse.max(0)
        m = lse.max(0)
        f = np.exp(lse - m)
        return (f[..., None] * o).sum(0), out_lse   # forgot to divide by l

    monkeypatch.setattr(oracle, "merge_outputs", broken)
    failed = 0
    for case in load_golden()["merges"]:
        try:
            test_merge_outputs_against_page(case)
        except AssertionError:
            failed += 1
    assert failed > 0

"""Pin checks for the attention oracle.

Each ``check_*`` function takes a forward implementation with the oracle's
signature ``fwd(q, k, v, scale, causal=False, kv_len=None) -> (O, lse)`` and returns
a list of failure messages (empty = pinned).  They compare against things other
than the oracle itself: numbers the source pages print, closed forms,
invariants, and high-precision brute force.  ``test_oracle_pins`` asserts every
check passes on the real oracle; ``test_oracle_mutations`` plants mistakes in the
oracle and asserts that some check catches each one.
"""

from __future__ import annotations

import json
import math
import os

import mpmath
import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _scores_problem(scores, values, n_queries=1):
    """Build Q, K, V with d_k = 1, q_i = 1, k_j = score_j, so that scale = 1 gives
    S[i, j] = score_j for every query row i."""
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64).reshape(len(s), -1)
    n = max(n_queries, len(s))
    q = np.ones((1, 1, n, 1))
    k = np.zeros((1, 1, n, 1))
    k[0, 0, : len(s), 0] = s
    vv = np.zeros((1, 1, n, v.shape[1]))
    vv[0, 0, : len(s)] = v
    return q, k, vv, len(s)


def _rel_ok(got, want, rtol, atol=0.0):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return bool(np.all(np.abs(got - want) <= atol + rtol * np.abs(want)))


def check_worked_examples(fwd):
    """Single-row worked examples printed by the Exercises and Worked examples pages."""
    g = load_golden()
    fails = []
    for c in g["cases"]:
        n = len(c["scores"])
        q, k, v, _ = _scores_problem(c["scores"], c["values"])
        # kv_len = n restricts the row to the case's own keys (no padding keys).
        o, lse = fwd(q, k, v, 1.0, causal=False, kv_len=[n])
        rtol = c.get("rtol", 5e-4)
        out = o[0, 0, 0]
        if not _rel_ok(out, c["out"], rtol, atol=1e-12):
            fails.append(f"{c['id']}: out {out} != page {c['out']} (rtol {rtol})")
        ell = math.exp(lse[0, 0, 0] - c["m"])
        if not _rel_ok(ell, c["l"], max(rtol, 5e-5)):
            fails.append(f"{c['id']}: l {ell} != page {c['l']}")
        if "exact" in c and not _rel_ok(out, c["exact"]["out"], 1e-12):
            fails.append(f"{c['id']}: out {out} != closed form {c['exact']['out']}")
    return fails


def check_masked_examples(fwd):
    """Cell D (causal) and Cell D2 (fully masked) of the Worked examples page."""
    g = load_golden()
    fails = []
    for c in g["masked_cases"]:
        n = len(c["scores"])
        q, k, v, _ = _scores_problem(c["scores"], c["values"])
        i = c["query_position"]
        o, lse = fwd(q, k, v, 1.0, causal=c.get("causal", False), kv_len=[c.get("kv_len", n)])
        out = o[0, 0, i]
        rtol = c.get("rtol", 5e-4)
        if c["l"] == 0.0:
            if not (np.all(out == 0.0) and np.isneginf(lse[0, 0, i])):
                fails.append(f"{c['id']}: fully masked row gave out {out}, lse {lse[0, 0, i]}")
            continue
        if not _rel_ok(out, c["out"], rtol):
            fails.append(f"{c['id']}: out {out} != page {c['out']}")
        ell = math.exp(lse[0, 0, i] - c["m"])
        if not _rel_ok(ell, c["l"], rtol):
            fails.append(f"{c['id']}: l {ell} != page {c['l']}")
    return fails


def _mp_attention(q, k, v, scale, causal, kv_len):
    """Brute force in 40-digit arithmetic, no max shift, no vectorisation.

    For tiny inputs only.  exp() never overflows in mpmath, so the plain
    definition softmax(s)_j = e^{s_j} / sum_k e^{s_k} is used directly.
    """
    mpmath.mp.dps = 40
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, N, dv))
    lse = np.zeros((B, H, N))
    sc = mpmath.mpf(float(scale))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                vis = [j for j in range(N)
                       if (not causal or j <= i) and (kv_len is None or j < kv_len[b])]
                if not vis:
                    o[b, h, i] = 0.0
                    lse[b, h, i] = -math.inf
                    continue
                w = {}
                for j in vis:
                    s = sc * mpmath.fsum(mpmath.mpf(float(q[b, h, i, c])) * mpmath.mpf(float(k[b, h, j, c]))
                                         for c in range(dk))
                    w[j] = mpmath.exp(s)
                tot = mpmath.fsum(w.values())
                for c in range(dv):
                    o[b, h, i, c] = float(mpmath.fsum(w[j] * mpmath.mpf(float(v[b, h, j, c])) for j in vis) / tot)
                lse[b, h, i] = float(mpmath.log(tot))
    return o, lse


def brute_force_cases():
    """Seeded tiny problems covering plain, causal, padded and fully masked rows."""
    rng = np.random.default_rng(20240611)
    cases = []
    for (B, H, N, dk, dv, causal, kv) in [
        (1, 1, 1, 1, 1, False, None),
        (1, 2, 5, 3, 2, False, None),
        (2, 1, 7, 4, 4, True, None),
        (2, 2, 8, 4, 3, False, [3, 8]),
        (2, 1, 6, 2, 4, True, [0, 4]),
        (1, 1, 8, 4, 4, True, [5]),
    ]:
        q = rng.standard_normal((B, H, N, dk)) * 1.5
        k = rng.standard_normal((B, H, N, dk)) * 1.5
        v = rng.standard_normal((B, H, N, dv))
        cases.append((q, k, v, 1.0 / math.sqrt(dk), causal, kv))
    return cases


def check_brute_force(fwd):
    """The oracle equals a 40-digit brute force on tiny inputs to 1e-12."""
    fails = []
    for n, (q, k, v, scale, causal, kv) in enumerate(brute_force_cases()):
        o, lse = fwd(q, k, v, scale, causal=causal, kv_len=kv)
        o_ref, lse_ref = _mp_attention(q, k, v, scale, causal, kv)
        if not np.allclose(o, o_ref, rtol=1e-12, atol=1e-12):
            fails.append(f"brute case {n}: O max diff {np.max(np.abs(o - o_ref))}")
        fin = np.isfinite(lse_ref)
        if not (np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
                and np.allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-12)):
            fails.append(f"brute case {n}: lse mismatch")
    return fails


def check_closed_forms(fwd):
    """Closed forms and invariants that hold exactly (up to rounding)."""
    rng = np.random.default_rng(7)
    fails = []
    B, H, N, d = 2, 2, 9, 4
    v = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    kv = [4, 9]
    # Uniform rows (Exercises, equal-scores exercise; Question bank, uniform item):
    # Q = 0 makes every score 0, so O_i = mean of the visible values, lse = ln(#visible).
    q0 = np.zeros((B, H, N, d))
    for causal in (False, True):
        o, lse = fwd(q0, k, v, 0.5, causal=causal, kv_len=kv)
        for b in range(B):
            for i in range(N):
                nvis = min(kv[b], i + 1) if causal else kv[b]
                want = v[b, :, :nvis].mean(axis=1)
                if not np.allclose(o[b, :, i], want, rtol=1e-13, atol=1e-13):
                    fails.append(f"uniform row b={b} i={i} causal={causal}: not the mean")
                if not np.allclose(lse[b, :, i], math.log(nvis), rtol=1e-13):
                    fails.append(f"uniform row b={b} i={i}: lse != ln({nvis})")
    # Shift invariance (Exercises, equal-scores exercise: a common shift cancels):
    # adding c to every score of a row leaves O unchanged and moves lse by c.
    q = rng.standard_normal((B, H, N, d))
    o1, lse1 = fwd(q, k, v, 0.5)
    # a constant key component that every query sees with weight 1 shifts all scores
    q_ext = np.concatenate([q, np.full((B, H, N, 1), 2.0)], axis=-1)
    k_ext = np.concatenate([k, np.full((B, H, N, 1), 3.0)], axis=-1)
    o2, lse2 = fwd(q_ext, k_ext, v, 0.5)
    if not np.allclose(o1, o2, rtol=1e-12, atol=1e-12):
        fails.append("shift invariance: O changed under a constant score shift")
    if not np.allclose(lse2 - lse1, 0.5 * 6.0, rtol=1e-12):
        fails.append("shift invariance: lse did not move by the shift")
    # Block order / key order (Worked examples, Cell H): permuting K and V rows
    # jointly leaves a non-causal, unpadded output unchanged.
    perm = rng.permutation(N)
    o3, lse3 = fwd(q, k[:, :, perm], v[:, :, perm], 0.5)
    if not (np.allclose(o1, o3, rtol=1e-12, atol=1e-12) and np.allclose(lse1, lse3, rtol=1e-12)):
        fails.append("key permutation changed the output")
    # A masked key contributes exactly zero (Worked examples, Cell D): padding to
    # kv_len equals running on the first kv_len keys only.
    o4, _ = fwd(q[:1], k[:1], v[:1], 0.5, kv_len=[5])
    for i in range(N):
        s = 0.5 * (k[0, 0, :5] @ q[0, 0, i])
        w = np.exp(s - s.max())
        want = (w @ v[0, 0, :5]) / w.sum()
        if not np.allclose(o4[0, 0, i], want, rtol=1e-12, atol=1e-12):
            fails.append(f"padding row {i}: masked keys leaked")
            break
    # Scale: the score multiplier is applied once (Foundations section 9):
    # scale s on Q equals scale 1 on s*Q.
    o6, _ = fwd(q * 0.5, k, v, 1.0)
    if not np.allclose(o1, o6, rtol=1e-12, atol=1e-12):
        fails.append("scale not applied as a plain multiplier of Q K^T")
    # One-hot limit (Worked examples, Cell F): a huge single logit selects its value.
    qh = np.zeros((1, 1, 3, 1)); qh[...] = 1.0
    kh = np.array([0.0, 1000.0, 0.0]).reshape(1, 1, 3, 1)
    vh = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]]).reshape(1, 1, 3, 2)
    oh, lseh = fwd(qh, kh, vh, 1.0)
    if not (np.allclose(oh[0, 0], [[3.0, 4.0]] * 3, rtol=0, atol=1e-300) and np.allclose(lseh, 1000.0)):
        fails.append("one-hot limit: output is not the dominating value")
    return fails


ALL_CHECKS = [check_worked_examples, check_masked_examples, check_closed_forms, check_brute_force]

"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each.

Each mutant replaces one step function of ``oracle.attention`` for the duration of
one test.  The pins of ``pins.py`` must then report at least one failure: a pin set
that a dropped term, a wrong sign or index, or a transposed operand slips past would
not be worth trusting.
"""

import numpy as np
import pytest

import oracle.attention as A
from pins import ALL_CHECKS

NEG_INF = -np.inf


MUTANTS = {
    "scale_dropped": ("score_matrix", lambda q, k, scale: q @ k.T),
    "scale_squared": ("score_matrix", lambda q, k, scale: scale * scale * (q @ k.T)),
    "operand_transposed": ("score_matrix", lambda q, k, scale: scale * (k @ q.T)),
    "causal_strict": ("visible_mask", lambda nq, nk, causal, kv: (
        (np.arange(nk)[None, :] < np.arange(nq)[:, None]) if causal else np.ones((nq, nk), bool))
        & ((np.arange(nk)[None, :] < kv) if kv is not None else True)),
    "causal_off_by_one": ("visible_mask", lambda nq, nk, causal, kv: (
        (np.arange(nk)[None, :] <= np.arange(nq)[:, None] + 1) if causal else np.ones((nq, nk), bool))
        & ((np.arange(nk)[None, :] < kv) if kv is not None else True)),
    "padding_ignored": ("visible_mask", lambda nq, nk, causal, kv: (
        (np.arange(nk)[None, :] <= np.arange(nq)[:, None]) if causal else np.ones((nq, nk), bool))),
    "mask_to_zero_not_neginf": ("apply_mask", lambda s, vis: np.where(vis, s, 0.0)),
    "min_instead_of_max": ("row_max", lambda s: np.where(np.isneginf(s), np.inf, s).min(axis=-1)),
    "shift_sign_flipped": ("shifted_exp", lambda s, m: np.exp(s + np.where(np.isneginf(m), 0.0, m)[..., None])),
    "no_shift_overflow": ("shifted_exp", lambda s, m: np.exp(s)),
    "guard_dropped": ("normalise", lambda e, v: ((e @ v) / e.sum(-1)[:, None], e.sum(-1))),
    "normaliser_dropped": ("normalise", lambda e, v: (e @ v, e.sum(-1))),
    "one_value_dropped": ("normalise", lambda e, v: (
        np.where((e.sum(-1) > 0)[:, None], (e[:, :-1] @ v[:-1]) / np.where(e.sum(-1) > 0, e.sum(-1), 1)[:, None], 0.0),
        e.sum(-1))),
    "lse_sign": ("row_lse", lambda m, l: np.where(l > 0, m - np.log(np.where(l > 0, l, 1.0)), NEG_INF)),
    "lse_without_max": ("row_lse", lambda m, l: np.where(l > 0, np.log(np.where(l > 0, l, 1.0)), NEG_INF)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    fn_name, mutant = MUTANTS[name]
    monkeypatch.setattr(A, fn_name, mutant)
    fails = []
    with np.errstate(all="ignore"):
        for check in ALL_CHECKS:
            try:
                fails += check(A.attention_fwd)
            except Exception as e:  # a crash is also a caught mistake
                fails.append(f"{check.__name__} raised {type(e).__name__}")
    assert fails, f"mutant {name} passed every pin"

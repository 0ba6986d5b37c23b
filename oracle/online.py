"""Model of the tiled one-pass softmax (float64) -- TEST INFRASTRUCTURE.

Only tests, the smoke check and the benchmark's CPU-baseline leg may use this
module; the CUDA product path never does.

Two forms of the same algorithm, each in the pages' notation:

* ``merge_states`` -- the generic merge of two partial block states
  (m1, l1, O~1) and (m2, l2, O~2) against the common max m_new = max(m1, m2):
      l_new  = e^(m1 - m_new) l1  + e^(m2 - m_new) l2
      O~_new = e^(m1 - m_new) O~1 + e^(m2 - m_new) O~2
  ("Exercises -- Flash attention and efficient attention", the two- and
  three-block merge exercises; "Flash attention and efficient attention: Worked
  examples", Cells A, B and H; "Question bank", the rescale items).

* ``online_row`` -- the streaming recurrence over key blocks, one query row,
  running registers m, l, acc initialised to (-inf, 0, 0):
      m_new = max(m, m'),  c = exp(m - m_new),
      l   <- l * c   + sum_j exp(s_j - m_new)
      acc <- acc * c + sum_j exp(s_j - m_new) V_j
      out  = acc / l   once, after the last block
  ("The Flash Attention" page, the online recurrence panel).  ``drop_rescale``
  removes the factor c, the page's red-team mutation, which must break exactness.

The division is guarded: l == 0 (every key masked) returns the zero vector
(Worked examples, Cell D2).  Where both maxima are -inf, Cell D2 lets the merge
go ahead with every term equal to zero; with IEEE arithmetic exp(-inf - (-inf))
is NaN, so the common reference is taken as 0 when m_new = -inf, which makes
every term exactly 0 as the page describes.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -math.inf


def _ref(m_new: float) -> float:
    return 0.0 if m_new == NEG_INF else m_new


def merge_states(a, b):
    """Merge two block states (m, l, O~) into one, rescaling both to max(m_a, m_b).

    Each state is a tuple (m: float, l: float, acc: 1-D array).  Returns the merged
    (m, l, acc).  Commutative and associative up to rounding (Worked examples,
    Cell H; Question bank, associativity item).
    """
    ma, la, acca = a
    mb, lb, accb = b
    m_new = max(ma, mb)
    r = _ref(m_new)
    fa = math.exp(ma - r)
    fb = math.exp(mb - r)
    return m_new, fa * la + fb * lb, fa * np.asarray(acca, float) + fb * np.asarray(accb, float)


def block_state(scores, values):
    """State of one block measured against its own max (Worked examples, Cell A,
    'Block 1' step): m = max s, l = sum e^(s - m), O~ = sum e^(s - m) v."""
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64).reshape(len(s), -1)
    m = float(s.max()) if len(s) else NEG_INF
    e = np.exp(s - _ref(m))
    return m, float(e.sum()), e @ v


def finish(state):
    """Divide once at the end, guarded for l == 0 (Cell D2).  Returns (out, lse)."""
    m, l, acc = state
    if l == 0.0:
        return np.zeros_like(np.asarray(acc, float)), NEG_INF
    return np.asarray(acc, float) / l, m + math.log(l)


def online_row(scores, values, block_size: int, order=None, drop_rescale: bool = False):
    """Stream one query row's scores in blocks of ``block_size`` keys.

    scores: [Nk] (masked entries already -inf); values: [Nk, dv].
    order: optional permutation of the block indices (blocks may be processed in
    any order -- Worked examples, Cell H).
    Returns (out [dv], lse, m, l).
    """
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64).reshape(len(s), -1)
    nblk = (len(s) + block_size - 1) // block_size
    blocks = list(range(nblk)) if order is None else list(order)
    m, l, acc = NEG_INF, 0.0, np.zeros(v.shape[1])
    for bi in blocks:
        sj = s[bi * block_size : (bi + 1) * block_size]
        vj = v[bi * block_size : (bi + 1) * block_size]
        m_blk = float(sj.max())
        m_new = max(m, m_blk)
        r = _ref(m_new)
        c = math.exp(m - r)
        p = np.exp(sj - r)
        if drop_rescale:
            c = 1.0
        l = l * c + float(p.sum())
        acc = acc * c + p @ vj
        m = m_new
    out, lse = finish((m, l, acc))
    return out, lse, m, l


def online_attention(q, k, v, scale: float, causal: bool = False, kv_len=None,
                     block_size: int = 128, drop_rescale: bool = False):
    """Full attention by the streaming recurrence, row by row (slow; small inputs).

    Same arguments and results as ``attention.attention_fwd``.  The score row is
    formed one query at a time and consumed block by block.
    """
    from .attention import _f64, key_visible

    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, _ = q.shape
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                s = scale * (k[b, h] @ q[b, h, i])
                j = np.arange(N)
                if causal:
                    s = np.where(key_visible(j, i, causal), s, NEG_INF)
                if kv_len is not None:
                    s = np.where(j < int(kv_len[b]), s, NEG_INF)
                o[b, h, i], lse[b, h, i], _, _ = online_row(s, v[b, h], block_size,
                                                             drop_rescale=drop_rescale)
    return o, lse


def merge_outputs(o_parts, lse_parts):
    """Merge normalised partial results computed over disjoint key sets.

    A part with output O_p (already divided by its own normaliser) and
    log-normaliser lse_p is the block state (m = lse_p, l = 1, O~ = O_p): dividing
    O~ by l gives O_p and m + ln l gives lse_p.  The generic merge rule of the
    Exercises page (two-block and three-block merges) then applies unchanged:
        m = max_p lse_p,   f_p = e^(lse_p - m),   l = sum_p f_p,
        O = sum_p f_p O_p / l,   lse = m + ln l.
    Parts with lse_p = -inf (no visible key) carry zero weight; if every part
    has lse = -inf the result is O = 0 and lse = -inf (Worked examples, Cell D2).

    o_parts: [P, ..., dv]; lse_parts: [P, ...].  Returns (O [..., dv], lse [...])
    in float64.
    """
    o = np.asarray(o_parts, dtype=np.float64)
    lse = np.asarray(lse_parts, dtype=np.float64)
    m = lse.max(axis=0)
    m_ref = np.where(np.isneginf(m), 0.0, m)
    f = np.exp(lse - m_ref[None])
    l = f.sum(axis=0)
    num = (f[..., None] * o).sum(axis=0)
    safe = np.where(l > 0, l, 1.0)
    out = np.where((l > 0)[..., None], num / safe[..., None], 0.0)
    with np.errstate(divide="ignore"):
        out_lse = np.where(l > 0, m_ref + np.log(safe), NEG_INF)
    return out, out_lse

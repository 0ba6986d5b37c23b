"""The attention definition, written out plainly in float64 -- TEST INFRASTRUCTURE.

Only tests, the smoke check and the benchmark's CPU-baseline leg may use this
module; the CUDA product path never does.

What is computed (per batch b and head h, every matrix row-major, d innermost):

    S   = scale * Q K^T                          (N x N, materialised)
    S_ij = -inf  where key j is masked for query i
    m_i = max_j S_ij                             (pass 1)
    l_i = sum_j exp(S_ij - m_i)                  (pass 2)
    P_ij = exp(S_ij - m_i) / l_i,   O_i = sum_j P_ij V_j,   lse_i = m_i + ln l_i
    l_i == 0 (every key masked)  ->  O_i = 0, lse_i = -inf

Sources (page title, then section):
  * "Foundations -- Flash attention and efficient attention", sections 4 (Q K^T is
    N x N: one score per query/key pair), 7 (softmax: exponentiate, divide by the
    sum), 8 (subtract the max; same result, no overflow) and 9 (divide the scores by
    sqrt(d_k); the caller passes scale = 1/sqrt(d_k)).
  * "Exercises -- Flash attention and efficient attention", the safe-softmax and
    weighted-output exercises (scores [3,5,5,2]): the two passes written above.
  * "Flash attention and efficient attention: Worked examples", Cell D (a causal
    query at position t sees keys j <= t, future keys set to -inf before the
    exponential) and Cell D2 (all keys masked: l = 0, return the zero vector).
  * "The Flash Attention" page, table "path / scores held / output": the naive
    path forms the full n x n score matrix, as this module does.

Readings where the pages are silent (each is listed in the design notes):
  * causal is inclusive (j <= i) with queries and keys indexed alike; the
    strictly causal mode (j < i) is Cell D2's setting; with Nq != Nk the queries
    are the last Nq positions (query i at position i + Nk - Nq);
  * key padding: keys j >= kv_len[b] are masked for every head and query of batch
    b (the pages do not mention padding; it is the same -inf mask as Cell D);
  * lse is the natural log of sum_j exp(S_ij) over visible keys, i.e. m + ln l,
    and is -inf for a fully masked row.

The step functions (``score_matrix``, ``visible_mask``, ``apply_mask``,
``row_max``, ``shifted_exp``, ``normalise``, ``row_lse``) are module-level so that tests can plant a mistake
in one of them and check that the pins catch it.
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Return ``x`` as a float64 ndarray (accepts numpy arrays and CPU torch tensors,
    including bfloat16 ones, whose values convert exactly)."""
    if hasattr(x, "detach"):  # a torch tensor: convert through float32/64 exactly
        t = x.detach().to("cpu")
        if str(t.dtype) in ("torch.bfloat16", "torch.float16"):
            t = t.float()
        x = t.double().numpy()
    return np.asarray(x, dtype=np.float64)


def score_matrix(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T for one head (Foundations sections 4 and 9).

    q: [Nq, dk], k: [Nk, dk] float64 -> [Nq, Nk] float64.
    """
    return scale * (q @ k.T)


STRICT = 2  # causal mode: a query may not attend to itself


def key_visible(j, i, causal) -> np.ndarray:
    """Causal rule for key index j and query index i (arrays broadcast).

    causal = 0/False: every key.  1/True (Worked examples, Cell D): keys j <= i,
    the token sees itself.  2 (Cell D2's "strictly causal setup"): keys j < i
    only, so query 0 sees no key at all.
    """
    j = np.asarray(j)
    if not causal:
        return np.ones(np.broadcast(j, np.asarray(i)).shape, dtype=bool)
    if causal == STRICT:
        return j < i
    return j <= i


def visible_mask(nq: int, nk: int, causal, kv_len: int | None) -> np.ndarray:
    """Boolean [Nq, Nk]: True where query i may attend to key j.

    Causal (Worked examples, Cell D): key j is visible to query i iff j <= i;
    strictly causal (Cell D2) iff j < i.  When there are fewer (or more) queries
    than keys, the queries are taken to be the last Nq positions of the key
    sequence -- query i sits at position i + (Nk - Nq) -- so the last query sees
    every key (a reading: the pages only treat Nq = Nk, where this is the rule
    above).  Key padding (a reading; the pages have no padding): key j is
    visible iff j < kv_len.
    """
    vis = np.ones((nq, nk), dtype=bool)
    if causal:
        vis &= key_visible(np.arange(nk)[None, :], np.arange(nq)[:, None] + (nk - nq), causal)
    if kv_len is not None:
        vis &= np.arange(nk)[None, :] < int(kv_len)
    return vis


def apply_mask(s: np.ndarray, vis: np.ndarray) -> np.ndarray:
    """Set masked scores to -inf before the exponential (Worked examples, Cell D)."""
    return np.where(vis, s, NEG_INF)


def row_max(s: np.ndarray) -> np.ndarray:
    """Pass 1 of the safe softmax: m_i = max_j S_ij (Foundations section 8)."""
    return s.max(axis=-1)


def shifted_exp(s: np.ndarray, m: np.ndarray) -> np.ndarray:
    """exp(S_ij - m_i), with exp(-inf) = 0 for masked entries (Foundations section 8).

    A fully masked row has m_i = -inf; its reference is taken as 0 so that every
    term is exp(-inf) = 0 rather than exp(-inf - (-inf)) = NaN (Worked examples,
    Cell D2: the running state never leaves its empty start).
    """
    m_ref = np.where(np.isneginf(m), 0.0, m)
    return np.exp(s - m_ref[..., None])


def normalise(e: np.ndarray, v: np.ndarray):
    """Pass 2 and the output: l_i = sum_j e_ij; O_i = (sum_j e_ij V_j) / l_i.

    Guard (Worked examples, Cell D2): l_i == 0 -> O_i = 0 (no division).
    Returns (O [Nq, dv], l [Nq]).
    """
    l = e.sum(axis=-1)
    num = e @ v
    safe = np.where(l > 0, l, 1.0)
    o = np.where((l > 0)[:, None], num / safe[:, None], 0.0)
    return o, l


def row_lse(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """lse_i = m_i + ln l_i = ln sum_j exp(S_ij); -inf for a fully masked row."""
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)


def _head_fwd(q, k, v, scale, causal, kv_len):
    s = score_matrix(q, k, scale)
    s = apply_mask(s, visible_mask(q.shape[0], k.shape[0], causal, kv_len))
    m = row_max(s)
    e = shifted_exp(s, m)
    o, l = normalise(e, v)
    return o, row_lse(m, l)


def attention_fwd(q, k, v, scale: float, causal: bool = False, kv_len=None):
    """Exact attention forward over every (b, h).

    q: [B, H, Nq, dk]; k: [B, H, Nk, dk]; v: [B, H, Nk, dv] (Nq may differ from
    Nk; any float type, converted exactly to float64); scale: the score
    multiplier (1/sqrt(dk) in the pages); causal: 0 (none), 1 (inclusive,
    j <= i + Nk - Nq) or 2 (strict, j < i + Nk - Nq); kv_len: None or B integers
    in [0, Nk].

    Returns (O [B, H, Nq, dv] float64, lse [B, H, Nq] float64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, _ = q.shape
    o = np.zeros(q.shape[:3] + (v.shape[-1],), dtype=np.float64)
    lse = np.zeros((B, H, N), dtype=np.float64)
    scale = float(scale)
    for b in range(B):
        kl = None if kv_len is None else int(kv_len[b])
        for h in range(H):
            o[b, h], lse[b, h] = _head_fwd(q[b, h], k[b, h], v[b, h], scale, causal, kl)
    return o, lse


def attention_fwd_rows(q, k, v, scale: float, causal: bool, kv_len, rows):
    """The same definition evaluated for selected query rows only.

    rows: iterable of (b, h, i).  Each row needs only q[b,h,i], all of K and V of
    head (b, h) and the row's own mask, so full-size problems can be checked on a
    sample of rows.  Returns (O [R, dv], lse [R]) float64.
    """
    out_o, out_lse = [], []
    scale = float(scale)
    nq = q.shape[2]
    for (b, h, i) in rows:
        qi = _f64(q[b, h, i : i + 1])
        kk = _f64(k[b, h])
        vv = _f64(v[b, h])
        nk = kk.shape[0]
        s = score_matrix(qi, kk, scale)
        vis = np.ones((1, nk), dtype=bool)
        if causal:
            vis &= key_visible(np.arange(nk)[None, :], i + (nk - nq), causal)
        if kv_len is not None:
            vis &= np.arange(nk)[None, :] < int(kv_len[b])
        s = apply_mask(s, vis)
        m = row_max(s)
        e = shifted_exp(s, m)
        o, l = normalise(e, vv)
        out_o.append(o[0])
        out_lse.append(float(row_lse(m, l)[0]))
    return np.stack(out_o), np.asarray(out_lse)


def attention_bwd(q, k, v, do, scale: float, causal: bool = False, kv_len=None):
    """Gradient of L = sum(O * dO) with respect to Q, K, V, for the forward above.

    The pages fix only that the backward pass recomputes S and P rather than
    storing them ("Question bank -- Flash attention and efficient attention",
    the recomputation items); the formulas are the textbook softmax-attention
    gradient, written out from the chain rule:

        P = softmax(S) (rows; masked entries 0),   dV = P^T dO,   dP = dO V^T,
        D_i = sum_j P_ij dP_ij,   dS = P * (dP - D),
        dQ = scale * dS K,         dK = scale * dS^T Q.

    A fully masked row has P = 0 and contributes nothing.  q and do may have a
    different length Nq from k and v (Nk); the mask is then visible_mask's
    (queries are the last Nq positions of the key sequence), as in the forward.
    Returns (dQ, dK, dV) float64 with the shapes of (q, k, v).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    scale = float(scale)
    for b in range(B):
        kl = None if kv_len is None else int(kv_len[b])
        for h in range(H):
            s = score_matrix(q[b, h], k[b, h], scale)
            s = apply_mask(s, visible_mask(Nq, Nk, causal, kl))
            m = row_max(s)
            e = shifted_exp(s, m)
            l = e.sum(axis=-1)
            p = np.where((l > 0)[:, None], e / np.where(l > 0, l, 1.0)[:, None], 0.0)
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            dd = (p * dp).sum(axis=-1)
            ds = p * (dp - dd[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv

"""GPU parity of the forward kernels against the float64 oracle (needs a B300).

Tolerances (from the accuracy targets of the attention forward):
  float32 inputs : max |O - O_ref| <= 1e-5
  bf16 inputs    : max |O - O_ref| <= 2e-2 and mean |O - O_ref| <= 2e-3
  lse            : max |lse - lse_ref| <= 1e-3 (and -inf exactly where the oracle has -inf)
The oracle receives the same bf16-rounded inputs, converted exactly to float64.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_14_b300.inputs import WORKLOADS, make_problem, make_workload

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, FP32_MAX, LSE_MAX = 2e-2, 2e-3, 1e-5, 1e-3
DEV = "cuda:0"


def fa():
    import online_softmax_14_b300 as m
    return m


def run(pr, causal, kv_len=None):
    q, k, v = (pr[n].to(DEV) for n in ("q", "k", "v"))
    kl = kv_len if kv_len is not None else pr.get("kv_len")
    o, lse = fa().attention_fwd(q, k, v, pr["scale"], causal=causal, kv_len=kl)
    fa().fa_check_device_error()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check(o, lse, o_ref, lse_ref, fp32=False, label=""):
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), f"{label}: non-finite output"
    if fp32:
        assert err.max() <= FP32_MAX, f"{label}: max|dO| {err.max():.3g}"
    else:
        assert err.max() <= BF16_MAX, f"{label}: max|dO| {err.max():.3g}"
        assert err.mean() <= BF16_MEAN, f"{label}: mean|dO| {err.mean():.3g}"
    ninf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), ninf), f"{label}: -inf pattern of lse differs"
    if (~ninf).any():
        lerr = np.abs(lse[~ninf] - lse_ref[~ninf]).max()
        assert lerr <= LSE_MAX, f"{label}: max|dlse| {lerr:.3g}"


def full_parity(B, H, N, d, causal, dtype="bf16", seed=0, kv_len=None, qk_mul=1.0, padded=False):
    pr = make_problem(B, H, N, d, dtype, seed=seed, qk_mul=qk_mul, padded=padded, kv_len=kv_len)
    o, lse = run(pr, causal)
    kl = None if pr["kv_len"] is None else pr["kv_len"].tolist()
    o_ref, lse_ref = oracle.attention_fwd(pr["q"], pr["k"], pr["v"], pr["scale"], causal=causal, kv_len=kl)
    check(o, lse, o_ref, lse_ref, fp32=(dtype == "fp32"), label=f"B{B} H{H} N{N} d{d} c{causal} kv{kl}")
    return o, lse


# --------------------------------------------------------------- bf16, small
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("padded", [False, True])
def test_bf16_multi_tile_ragged(d, causal, padded):
    # N = 300: three 128-row tiles, the last one ragged (44 rows)
    full_parity(3, 2, 300, d, causal, padded=padded, seed=d + causal + 2 * padded)


@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 257, 640])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_sequence_lengths(N, d):
    full_parity(1, 2, N, d, causal=(N % 2 == 1), seed=N)


@pytest.mark.parametrize("N", [200, 384])
def test_bf16_kv_len_extremes(N):
    kv = [0, 1, N - 1, N, 127, 128, 129]
    for causal in (False, True):
        o, lse = full_parity(len(kv), 2, N, 128, causal, kv_len=kv, seed=N)
        assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))  # no visible key: O = 0, lse = -inf


def test_bf16_uniform_rows_give_mean():
    """Q = 0 makes every score equal: each row's output is the mean of its visible
    values (Exercises, equal-scores exercise; Worked examples, Cell C)."""
    B, H, N, d = 2, 2, 260, 128
    pr = make_problem(B, H, N, d, "bf16", seed=3)
    pr["q"] = torch.zeros_like(pr["q"])
    for causal in (False, True):
        o, lse = run(pr, causal)
        v = pr["v"].double().numpy()
        if causal:
            want = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
            lwant = np.log(np.arange(1, N + 1))[None, None, :]
        else:
            want = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
            lwant = np.full((1, 1, N), math.log(N))
        assert np.abs(o - want).max() <= BF16_MAX and np.abs(o - want).mean() <= BF16_MEAN
        assert np.abs(lse - lwant).max() <= LSE_MAX


def test_bf16_one_hot_limit():
    """A single dominating logit selects its value row (Worked examples, Cell F)."""
    B, H, N, d = 1, 1, 256, 64
    pr = make_problem(B, H, N, d, "bf16", seed=4)
    q = torch.zeros(B, H, N, d)
    q[..., 0] = 1.0
    k = torch.zeros(B, H, N, d)
    k[0, 0, 77, 0] = 512.0  # score 512 * scale = 64 above every other key
    pr["q"], pr["k"] = q.to(torch.bfloat16), k.to(torch.bfloat16)
    o, lse = run(pr, causal=False)
    want = pr["v"][0, 0, 77].double().numpy()
    assert np.abs(o[0, 0] - want[None, :]).max() <= BF16_MAX


def test_bf16_key_permutation_invariance():
    """Streaming the key blocks in another order does not change the answer
    (Worked examples, Cell H): permuting K and V rows jointly leaves a
    non-causal output unchanged, within bf16 rounding."""
    pr = make_problem(1, 2, 384, 128, "bf16", seed=5)
    o1, l1 = run(pr, causal=False)
    perm = torch.randperm(384, generator=torch.Generator().manual_seed(0))
    pr2 = dict(pr, k=pr["k"][:, :, perm].contiguous(), v=pr["v"][:, :, perm].contiguous())
    o2, l2 = run(pr2, causal=False)
    assert np.abs(o1 - o2).max() <= BF16_MAX and np.abs(l1 - l2).max() <= LSE_MAX


def test_bf16_overflow_regime_is_finite():
    """Logits of several hundred (the stress workload's x8 inputs) stay finite
    where a softmax without the max shift overflows (Exercises, overflow exercise)."""
    full_parity(2, 2, 256, 128, causal=False, qk_mul=8.0, padded=True, seed=6)


# ---------------------------------------------------------------- fp32 path
def test_fp32_workload_full():
    w = WORKLOADS["fp32_B1_H1_N256_d64"]
    pr = make_workload(w)
    o, lse = run(pr, w.causal)
    o_ref, lse_ref = oracle.attention_fwd(pr["q"], pr["k"], pr["v"], pr["scale"], causal=w.causal)
    check(o, lse, o_ref, lse_ref, fp32=True, label=w.name)


@pytest.mark.parametrize("d", [1, 16, 33, 64, 100, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_shapes(d, causal):
    full_parity(2, 2, 77, d, causal, dtype="fp32", padded=True, seed=d)


# ------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["bf16_causal_B4_H16_N2048_d64", "bf16_padded_stress_B8_H16_N1024_d128"])
def test_full_size_workload_every_element(name):
    """The exact launch the benchmark times, compared with the oracle on every
    output element of every head: max-abs and mean-abs over the whole output,
    lse on every row, and the -inf pattern of lse exactly (the stress workload's
    kv_len[0] = 0 batch: "Flash attention and efficient attention: Worked
    examples", Cell D2)."""
    w = WORKLOADS[name]
    pr = make_workload(w)
    o, lse = run(pr, w.causal)
    kl = None if pr["kv_len"] is None else pr["kv_len"].tolist()
    o_ref, lse_ref = oracle.attention_fwd(pr["q"], pr["k"], pr["v"], pr["scale"], causal=w.causal, kv_len=kl)
    check(o, lse, o_ref, lse_ref, label=name)
    if kl is not None:
        for b, n in enumerate(kl):
            if n == 0:
                assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b]))
            else:
                assert np.all(np.isfinite(lse[b]))


def _rows_every_head(B, H, N, seed, per_head=6):
    """A few rows of every head: the first and last row of the head, rows at
    128-row tile edges, and random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(B):
        for h in range(H):
            fixed = {0, N - 1, 127, 128, N // 2 - 1, N // 2}
            rows += [(b, h, i) for i in sorted(fixed | {int(x) for x in rng.integers(0, N, per_head)})]
    return rows


def test_full_size_long_sequence_sampled_every_head():
    """The long-sequence workload (B=2 H=32 N=8192 d=128, causal): the oracle needs
    2.2e12 float64 FLOPs for the whole output, so it is evaluated row by row on
    about a dozen rows of every one of the 64 heads; every output is checked
    finite."""
    name = "bf16_causal_B2_H32_N8192_d128"
    w = WORKLOADS[name]
    pr = make_workload(w)
    o, lse = run(pr, w.causal)
    rows = _rows_every_head(w.B, w.H, w.N, seed=1)
    o_ref, lse_ref = oracle.attention_fwd_rows(pr["q"], pr["k"], pr["v"], pr["scale"], w.causal, None, rows)
    got = np.stack([o[b, h, i] for (b, h, i) in rows])
    gl = np.array([lse[b, h, i] for (b, h, i) in rows])
    check(got, gl, o_ref, lse_ref, label=name)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


# ---------------------------------------------------------- bounded waits
def test_starved_pipeline_times_out_and_recovers():
    """The test hook makes the producer stop after the first K/V tile; every
    bounded wait downstream must give up, the launch must report FA_ERR_TIMEOUT,
    and the context must stay usable for a correct run afterwards."""
    m = fa()
    pr = make_problem(1, 2, 512, 128, "bf16", seed=8)
    q, k, v = (pr[n].to(DEV) for n in ("q", "k", "v"))
    m.fa_set_wait_timeout_ms(50)
    m.fa_debug_inject(1)
    try:
        m.attention_fwd(q, k, v, pr["scale"], causal=False)
        with pytest.raises(m.FaError) as ei:
            m.fa_check_device_error()
        assert ei.value.status == m.FA_ERR_TIMEOUT
    finally:
        m.fa_debug_inject(0)
        m.fa_set_wait_timeout_ms(1000)
    m.fa_check_device_error()  # status word was cleared
    full_parity(1, 2, 512, 128, causal=False, seed=8)


# ------------------------------------------------- strictly causal (Cell D2)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 130, 300, 513])
def test_bf16_strictly_causal(N, d):
    """Key j is visible to query i only when j < i (Worked examples, Cell D2's
    strictly causal setup): query 0 sees no key, so O = 0 and lse = -inf."""
    o, lse = full_parity(2, 2, N, d, causal=2, seed=N + d)
    assert np.all(o[:, :, 0] == 0.0) and np.all(np.isneginf(lse[:, :, 0]))
    if N > 1:
        assert np.all(np.isfinite(lse[:, :, 1:]))


def test_bf16_strictly_causal_with_padding():
    full_parity(4, 2, 260, 128, causal=2, kv_len=[0, 1, 2, 260], seed=31)


@pytest.mark.parametrize("d", [16, 64, 128])
def test_fp32_strictly_causal(d):
    o, lse = full_parity(2, 2, 77, d, causal=2, dtype="fp32", seed=d + 1)
    assert np.all(o[:, :, 0] == 0.0) and np.all(np.isneginf(lse[:, :, 0]))


# -------------------------------- queries and keys of different lengths
def _qk_problem(B, H, Nq, Nk, d, dtype, seed, padded=False):
    """q from one draw of length Nq, k and v from another of length Nk."""
    pq = make_problem(B, H, Nq, d, dtype, seed=seed)
    pk = make_problem(B, H, Nk, d, dtype, seed=seed + 1000, padded=padded)
    return pq["q"], pk["k"], pk["v"], pq["scale"], pk["kv_len"]


def qk_parity(B, H, Nq, Nk, d, causal, dtype="bf16", seed=0, padded=False):
    q, k, v, scale, kl = _qk_problem(B, H, Nq, Nk, d, dtype, seed, padded)
    o, lse = fa().attention_fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale, causal=causal,
                                kv_len=None if kl is None else kl.to(DEV))
    fa().fa_check_device_error()
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    kll = None if kl is None else kl.tolist()
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, scale, causal=causal, kv_len=kll)
    check(o, lse, o_ref, lse_ref, fp32=(dtype == "fp32"), label=f"Nq{Nq} Nk{Nk} d{d} c{causal} kv{kll}")
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("Nq,Nk", [(1, 300), (64, 513), (200, 130), (129, 1000), (384, 256)])
def test_bf16_queries_and_keys_differ(Nq, Nk, causal, d):
    """Nq != Nk: the queries are the last Nq positions of the key sequence."""
    qk_parity(2, 2, Nq, Nk, d, causal, seed=Nq + Nk + causal)


def test_bf16_queries_and_keys_differ_padded():
    qk_parity(5, 2, 100, 400, 128, 1, seed=41, padded=True)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_fp32_queries_and_keys_differ(causal):
    qk_parity(2, 2, 37, 101, 64, causal, dtype="fp32", seed=42 + causal)
    qk_parity(2, 2, 101, 37, 64, causal, dtype="fp32", seed=45 + causal)


def test_decode_single_query_sees_every_key():
    """One query per head under the causal mask is the last position: it attends
    to every key, i.e. equals attention with no mask."""
    q, k, v, scale, _ = _qk_problem(3, 4, 1, 777, 128, "bf16", seed=50)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o_c, l_c = fa().attention_fwd(qd, kd, vd, scale, causal=True)
    o_n, l_n = fa().attention_fwd(qd, kd, vd, scale, causal=False)
    fa().fa_check_device_error()
    assert torch.equal(o_c, o_n) and torch.equal(l_c, l_n)

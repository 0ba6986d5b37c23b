"""GPU parity of the split-key merge (fa_merge) against the float64 oracle.

Tolerances: float32 parts -> max |O - O_ref| <= 1e-5 and |lse - lse_ref| <= 1e-5
relative; bf16 parts -> the bf16 bar (2e-2 max-abs, 2e-3 mean-abs), lse 1e-3.
The oracle merges the same (bf16-rounded) parts in float64.
"""

import numpy as np
import pytest
import torch

import oracle
from online_softmax_14_b300.inputs import make_problem

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def fa():
    import online_softmax_14_b300 as m
    return m


def _random_parts(P, B, H, N, d, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(P, B, H, N, d, generator=g).to(dtype)
    lse = torch.randn(P, B, H, N, generator=g) * 30.0               # logits far apart
    lse[0, 0, 0, :5] = -float("inf")                                # an empty part in some rows
    lse[:, 0, 0, 7] = -float("inf")                                 # a row with no visible key at all
    return o, lse


def _check(o, lse, o_ref, lse_ref, fp32):
    ninf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), ninf)
    err = np.abs(o - o_ref)
    if fp32:
        assert err.max() <= 1e-5
        assert np.allclose(lse[~ninf], lse_ref[~ninf], rtol=1e-6, atol=1e-5)
    else:
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        assert np.abs(lse[~ninf] - lse_ref[~ninf]).max() <= 1e-3


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("P,d", [(1, 64), (2, 128), (5, 128), (3, 33), (40, 256)])
def test_merge_random_parts(P, d, dtype):
    B, H, N = 2, 3, 77
    o_p, lse_p = _random_parts(P, B, H, N, d, seed=P * 1000 + d, dtype=dtype)
    o_dev = o_p.clone()
    o_dev[0, 0, 0, :5] = float("nan")     # an empty part's values must never be read
    o, lse = fa().attention_merge(o_dev.to(DEV), lse_p.to(DEV))
    fa().fa_check_device_error()
    o_ref, lse_ref = oracle.merge_outputs(o_p.double().numpy(), lse_p.double().numpy())
    _check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, dtype == torch.float32)
    assert np.all(o.float().cpu().numpy()[0, 0, 7] == 0)          # no visible key anywhere: O = 0


@pytest.mark.parametrize("cuts", [[256], [100, 300], [128, 256, 384]])
def test_split_key_attention_end_to_end(cuts):
    """Attention over every key, computed as the merge of attention over disjoint
    key ranges [a, b): each range is a forward call over K/V rotated so that the
    range comes first, with kv_len = b - a masking the rest."""
    B, H, N, d = 2, 2, 448, 128
    pr = make_problem(B, H, N, d, "bf16", seed=len(cuts))
    q, k, v = (pr[n].to(DEV) for n in ("q", "k", "v"))
    bounds = [0] + cuts + [N]
    o_parts, l_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        kr = torch.cat([k[:, :, a:], k[:, :, :a]], dim=2).contiguous()
        vr = torch.cat([v[:, :, a:], v[:, :, :a]], dim=2).contiguous()
        kl = torch.full((B,), b - a, dtype=torch.int32, device=DEV)
        o_p, l_p = fa().attention_fwd(q, kr, vr, pr["scale"], causal=False, kv_len=kl)
        o_parts.append(o_p)
        l_parts.append(l_p)
    o, lse = fa().attention_merge(torch.stack(o_parts).contiguous(), torch.stack(l_parts).contiguous())
    o_full, lse_full = fa().attention_fwd(q, k, v, pr["scale"], causal=False)
    fa().fa_check_device_error()
    o_ref, lse_ref = oracle.attention_fwd(pr["q"], pr["k"], pr["v"], pr["scale"], causal=False)
    _check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, fp32=False)
    # and the merged result agrees with the single-pass kernel
    assert np.abs(o.float().cpu().numpy() - o_full.float().cpu().numpy()).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - lse_full.cpu().numpy()).max() <= 1e-3


def test_split_key_decode():
    """Decoding with the keys split across parts: each part is a forward of the
    same queries over one key range (queries fewer than keys), then fa_merge."""
    B, H, Nq, Nk, d = 2, 4, 3, 1000, 128
    pq = make_problem(B, H, Nq, d, "bf16", seed=60)
    pk = make_problem(B, H, Nk, d, "bf16", seed=61)
    q, k, v = pq["q"].to(DEV), pk["k"].to(DEV), pk["v"].to(DEV)
    bounds = [0, 250, 600, Nk]
    o_parts, l_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o_p, l_p = fa().attention_fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(), pq["scale"])
        o_parts.append(o_p)
        l_parts.append(l_p)
    o, lse = fa().attention_merge(torch.stack(o_parts).contiguous(), torch.stack(l_parts).contiguous())
    fa().fa_check_device_error()
    o_ref, lse_ref = oracle.attention_fwd(pq["q"], pk["k"], pk["v"], pq["scale"])
    _check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, fp32=False)

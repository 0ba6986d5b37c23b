"""The seeded input generator: deterministic, and shaped as the workloads say (CPU)."""

import torch

from online_softmax_14_b300.inputs import WORKLOADS, default_scale, make_problem


def test_deterministic_and_ordered():
    a = make_problem(2, 3, 17, 8, "bf16", seed=5, backward=True)
    b = make_problem(2, 3, 17, 8, "bf16", seed=5, backward=True)
    for key in ("q", "k", "v", "do"):
        assert torch.equal(a[key], b[key])
    # Q, K, V are consecutive draws from one generator, in that order
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, 3, 17, 8, generator=g)
    assert torch.equal(a["q"], q.to(torch.bfloat16))
    c = make_problem(2, 3, 17, 8, "bf16", seed=6)
    assert not torch.equal(a["q"], c["q"])


def test_stress_scaling_is_exact_and_padding_forced():
    p = make_problem(8, 2, 64, 16, "bf16", seed=0, qk_mul=8.0, padded=True)
    g = torch.Generator().manual_seed(0)
    q = torch.randn(8, 2, 64, 16, generator=g)
    assert torch.equal(p["q"], (q * 8).to(torch.bfloat16))
    assert torch.equal(p["q"].float() / 8, q.to(torch.bfloat16).float())
    kl = p["kv_len"]
    assert kl.dtype == torch.int32 and kl.shape == (8,)
    assert kl[0] == 0 and kl[1] == 64 and bool(((kl >= 0) & (kl <= 64)).all())


def test_workloads_and_scale():
    w = WORKLOADS["bf16_causal_B2_H32_N8192_d128"]
    assert (w.B, w.H, w.N, w.d, w.causal) == (2, 32, 8192, 128, True)
    s = default_scale(128)
    assert s == float(torch.tensor(128 ** -0.5, dtype=torch.float32))
    assert WORKLOADS["fp32_B1_H1_N256_d64"].dtype == "fp32"

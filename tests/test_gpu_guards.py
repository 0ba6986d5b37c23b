"""Out-of-bounds write checks with guard regions (needs a B300).

Each output tensor is carved out of the middle of a larger device buffer whose
head and tail are filled with a byte pattern.  The kernels run on ragged shapes
(N not a multiple of any tile, padded and strictly causal masks, d = 64 and
128) and the test asserts that every guard byte is still intact, so a write past
either end of an output is caught without a memory checker.
"""

import pytest
import torch

from online_softmax_14_b300.inputs import make_problem

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 1 << 16  # bytes on each side
PATTERN = 0xA5


def fa():
    import online_softmax_14_b300 as m
    return m


class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer with guards on both sides."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
        self.nbytes = nbytes

    def intact(self):
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("fp32", 33), ("fp32", 128)])
@pytest.mark.parametrize("N,causal", [(1, 1), (131, 0), (300, 2), (513, 1)])
def test_forward_writes_stay_inside_outputs(dtype, d, N, causal):
    B, H = 3, 2
    pr = make_problem(B, H, N, d, dtype, seed=N + d, padded=True)
    q, k, v = (pr[n].to(DEV) for n in ("q", "k", "v"))
    kv = pr["kv_len"].to(DEV)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o = Guarded((B, H, N, d), tdt)
    lse = Guarded((B, H, N), torch.float32)
    m = fa()
    m.fa_fwd_ex(m.FA_BF16 if dtype == "bf16" else m.FA_FP32, q, k, v, o.t, lse.t, kv, B, H, N, d, pr["scale"],
                causal)
    m.fa_check_device_error()
    assert o.intact() and lse.intact()


@pytest.mark.parametrize("N,causal", [(1, 1), (65, 0), (200, 2), (300, 1)])
@pytest.mark.parametrize("noalloc", [False, True])
def test_backward_writes_stay_inside_outputs(N, causal, noalloc):
    B, H, d = 2, 2, 128
    pr = make_problem(B, H, N, d, "bf16", seed=N, backward=True)
    q, k, v, do = (pr[n].to(DEV) for n in ("q", "k", "v", "do"))
    m = fa()
    o, lse = m.attention_fwd(q, k, v, pr["scale"], causal=causal)
    grads = [Guarded((B, H, N, d), torch.float32) for _ in range(3)]
    if noalloc:
        m.fa_bwd_noalloc(q, k, v, o, do, lse, *(g.t for g in grads), B, H, N, d, pr["scale"], causal)
    else:
        ws_bytes = m.fa_bwd_workspace_size(B, H, N, d)
        ws = Guarded((ws_bytes // 4,), torch.float32)
        m.fa_bwd(q, k, v, o, do, lse, *(g.t for g in grads), ws.t, ws_bytes, B, H, N, d, pr["scale"], causal)
        assert ws.intact()
    m.fa_check_device_error()
    assert all(g.intact() for g in grads)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 128), (torch.bfloat16, 40)])
def test_merge_writes_stay_inside_outputs(dtype, d):
    P, B, H, N = 3, 2, 2, 77
    g = torch.Generator().manual_seed(d)
    o_p = torch.randn(P, B, H, N, d, generator=g).to(dtype).to(DEV)
    l_p = torch.randn(P, B, H, N, generator=g).to(DEV)
    o = Guarded((B, H, N, d), dtype)
    lse = Guarded((B, H, N), torch.float32)
    m = fa()
    m.fa_merge(m.FA_BF16 if dtype == torch.bfloat16 else m.FA_FP32, o_p, l_p, P, o.t, lse.t, B, H, N, d)
    m.fa_check_device_error()
    assert o.intact() and lse.intact()


@pytest.mark.parametrize("Nq,Nk", [(1, 300), (200, 131), (129, 513)])
def test_forward_different_lengths_stays_inside_outputs(Nq, Nk):
    B, H, d = 2, 2, 128
    pq = make_problem(B, H, Nq, d, "bf16", seed=Nq)
    pk = make_problem(B, H, Nk, d, "bf16", seed=Nk)
    q, k, v = pq["q"].to(DEV), pk["k"].to(DEV), pk["v"].to(DEV)
    o = Guarded((B, H, Nq, d), torch.bfloat16)
    lse = Guarded((B, H, Nq), torch.float32)
    m = fa()
    m.fa_fwd_qk(m.FA_BF16, q, k, v, o.t, lse.t, None, B, H, Nq, Nk, d, pq["scale"], 1)
    m.fa_check_device_error()
    assert o.intact() and lse.intact()

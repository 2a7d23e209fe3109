"""CPU pins of the oracle's backward (gradients of O with respect to Q, K, V).

"Tensor Core 迁移计划" (phase 2) names the backward's contractions dV = P^T dO,
dP = dO V^T and dQ, dK from dS; the oracle fills in dS by the softmax's
Jacobian.  The pins tie it to things other than itself:
  * central differences of the oracle's forward (pinned separately), on inputs
    whose perturbed values stay exactly representable in fp16, with Richardson
    extrapolation (error O(h^4));
  * torch's fp64 autograd through softmax(scale Q K^T + mask) V on the CPU;
  * closed forms: identical keys give dQ = 0; sum_j dK_j = 0 (shifting every
    key by one vector shifts a row's visible scores alike, which the softmax
    ignores); sum_j dV_j = sum_i dO_i (every P row sums to 1).
"""
import numpy as np
import pytest
import torch

from exact_attention_05_gb300.workloads import FP16, bits


def _grid16(gen, shape, lo=-2.0, hi=2.0):
    """fp16 values on a 1/16 grid in [lo, hi): x +- 2^-6 and x +- 2^-7 stay exact in fp16."""
    n = int((hi - lo) * 16)
    x = torch.randint(0, n, shape, generator=gen).to(torch.float64) / 16.0 + lo
    return x.to(torch.float16)


def _loss(oracle_mod, q, k, v, w, causal, scale):
    o, _ = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, causal, scale)
    return float((o * w.to(torch.float64).numpy()).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(oracle_mod, causal):
    gen = torch.Generator().manual_seed(201 + causal)
    B, N, M, Hq, Hkv, d = 1, 3, 4, 2, 1, 4
    q = _grid16(gen, (B, N, Hq, d))
    k = _grid16(gen, (B, M, Hkv, d))
    v = _grid16(gen, (B, M, Hkv, d))
    w = _grid16(gen, (B, N, Hq, d))   # upstream gradient dO
    scale = 0.5
    dq, dk, dv = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(w), FP16, causal,
                                               scale)
    grads = {"q": dq, "k": dk, "v": dv}
    for name in ("q", "k", "v"):
        base = {"q": q, "k": k, "v": v}
        x = base[name]
        flat = x.reshape(-1)
        for idx in range(flat.numel()):
            def diff(h):
                plus, minus = flat.clone(), flat.clone()
                plus[idx] = (flat[idx].to(torch.float64) + h).to(torch.float16)
                minus[idx] = (flat[idx].to(torch.float64) - h).to(torch.float16)
                assert float(plus[idx]) - float(flat[idx]) == h   # exact step
                args = dict(base)
                args[name] = plus.view_as(x)
                lp = _loss(oracle_mod, args["q"], args["k"], args["v"], w, causal, scale)
                args[name] = minus.view_as(x)
                lm = _loss(oracle_mod, args["q"], args["k"], args["v"], w, causal, scale)
                return (lp - lm) / (2 * h)
            d1, d2 = diff(2.0 ** -6), diff(2.0 ** -7)
            fd = (4.0 * d2 - d1) / 3.0
            an = grads[name].reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * (1.0 + abs(an)), (name, idx, fd, an)


def _torch_reference(q, k, v, dout, causal, scale):
    """fp64 autograd through softmax(scale Q K^T + mask) V with GQA head sharing."""
    B, N, Hq, d = q.shape
    M, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    qd = q.to(torch.float64).requires_grad_(True)
    kd = k.to(torch.float64).requires_grad_(True)
    vd = v.to(torch.float64).requires_grad_(True)
    qh = qd.permute(0, 2, 1, 3)                                  # [B,Hq,N,d]
    kh = kd.permute(0, 2, 1, 3).repeat_interleave(g, dim=1)      # [B,Hq,M,d]
    vh = vd.permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    s = scale * qh @ kh.transpose(-1, -2)
    if causal:
        mask = torch.ones(N, M, dtype=torch.bool).tril()
        s = s.masked_fill(~mask, float("-inf"))
    o = torch.softmax(s, dim=-1) @ vh
    o.permute(0, 2, 1, 3).backward(dout.to(torch.float64))
    return qd.grad.numpy(), kd.grad.numpy(), vd.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,N,M,Hq,Hkv,d", [(1, 37, 37, 4, 2, 64), (2, 20, 29, 2, 2, 32),
                                           (1, 33, 17, 3, 1, 16)])
def test_backward_matches_torch_autograd(oracle_mod, B, N, M, Hq, Hkv, d, causal):
    gen = torch.Generator().manual_seed(300 + N + M + causal)
    q = torch.randn((B, N, Hq, d), generator=gen).to(torch.float16)
    k = torch.randn((B, M, Hkv, d), generator=gen).to(torch.float16)
    v = torch.randn((B, M, Hkv, d), generator=gen).to(torch.float16)
    dout = torch.randn((B, N, Hq, d), generator=gen).to(torch.float16)
    scale = d ** -0.5
    dq, dk, dv = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(dout), FP16,
                                               causal, scale)
    rq, rk, rv = _torch_reference(q, k, v, dout, causal, scale)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11)


def test_backward_identical_keys_give_zero_dq(oracle_mod):
    gen = torch.Generator().manual_seed(401)
    B, N, M, H, d = 1, 9, 12, 2, 32
    q = torch.randn((B, N, H, d), generator=gen).to(torch.float16)
    row = torch.randn((1, 1, H, d), generator=gen).to(torch.float16)
    k = row.expand(B, M, H, d).contiguous()
    v = torch.randn((B, M, H, d), generator=gen).to(torch.float16)
    dout = torch.randn((B, N, H, d), generator=gen).to(torch.float16)
    for causal in (False, True):
        dq, _, dv = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(dout), FP16,
                                                  causal, 0.3)
        assert np.abs(dq).max() < 1e-13
        if not causal:
            # uniform P: every key receives the mean upstream gradient of the rows
            want = dout.to(torch.float64).sum(dim=1, keepdim=True).numpy() / M
            np.testing.assert_allclose(dv, np.broadcast_to(want, dv.shape), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(oracle_mod, causal):
    gen = torch.Generator().manual_seed(402 + causal)
    B, N, M, Hq, Hkv, d = 2, 24, 24, 4, 2, 64
    q = torch.randn((B, N, Hq, d), generator=gen).to(torch.float16)
    k = torch.randn((B, M, Hkv, d), generator=gen).to(torch.float16)
    v = torch.randn((B, M, Hkv, d), generator=gen).to(torch.float16)
    dout = torch.randn((B, N, Hq, d), generator=gen).to(torch.float16)
    dq, dk, dv = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(dout), FP16,
                                               causal, 0.125)
    # sum over keys of dK is zero for every (b, kv head)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12
    # sum over keys of dV equals the sum of the upstream gradients of the heads reading it
    g = Hq // Hkv
    do64 = dout.to(torch.float64).numpy()
    want = do64.reshape(B, N, Hkv, g, d).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_dq_rows_equal_full_backward(oracle_mod, causal):
    """The sampled-row dQ used at full size equals the pinned full backward's rows."""
    gen = torch.Generator().manual_seed(410 + causal)
    B, N, M, Hq, Hkv, d = 2, 40, 33, 4, 2, 64
    q = torch.randn((B, N, Hq, d), generator=gen).to(torch.bfloat16)
    k = torch.randn((B, M, Hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((B, M, Hkv, d), generator=gen).to(torch.bfloat16)
    dout = torch.randn((B, N, Hq, d), generator=gen).to(torch.bfloat16)
    dq, _, _ = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(dout), 1, causal, 0.2)
    rows = np.array([(0, 0, 0), (1, 3, 39), (0, 2, 17), (1, 1, 32), (1, 0, 5)], np.int64)
    got = oracle_mod.attention_backward_dq_rows(bits(q), bits(k), bits(v), bits(dout), 1, causal,
                                                0.2, rows)
    want = np.stack([dq[b, i, h] for b, h, i in rows])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)

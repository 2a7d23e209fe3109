"""GPU parity of the backward (fa_bwd through the C ABI) against the oracle.

The GPU forward (fa_fwd) produces O and LSE, as a training step would; fa_bwd
then gives dQ, dK, dV, which are compared element by element with the
oracle's fp64 gradients of the same inputs (the oracle recomputes everything
from Q, K, V, dO).  Tolerance (per tensor, max |gpu - oracle| <= tol * max
|oracle|): P and dS enter the tensor core rounded to the input type (relative
error up to 2^-11 for fp16, 2^-8 for bf16 per element), O and the outputs are
rounded once more, so the gradients carry a few units of the type's rounding
relative to their own scale: tol = 8 * 2^-11 ~ 4e-3 for fp16 and 8 * 2^-8 ~
3e-2 for bf16.  The scale is max |oracle|, floored at 1: where the gradients
vanish (one key: P = 1, dS = dP - D = 0) what is left is the fp32 rounding of
dP and D, whose size is that of dO . V, i.e. 1 for unit-variance inputs.
"""
import numpy as np
import pytest

from exact_attention_05_gb300.workloads import BF16, FP16, bits, make_dout, make_inputs
from parity import torch_cuda

pytestmark = pytest.mark.gpu

TOL = {FP16: 8 * 2.0 ** -11, BF16: 8 * 2.0 ** -8}


def run_backward(q, k, v, dout, causal, scale):
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, lse = fa.attention_forward(qd, kd, vd, causal, scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    return [t.double().cpu().numpy() for t in (dq, dk, dv)]


def check(oracle_mod, B, Hq, Hkv, N, M, d, dtype, causal, seed=11):
    scale = 1.0 / np.sqrt(d)
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, dtype, seed)
    dout = make_dout(B, N, Hq, d, dtype, seed + 1000)
    got = run_backward(q, k, v, dout, causal, scale)
    ref = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(dout), dtype, causal,
                                        scale)
    errs = []
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.isfinite(g).all(), f"{name}: non-finite"
        e = float(np.abs(g - r).max())
        scl = max(float(np.abs(r).max()), 1.0)
        errs.append((name, e, scl))
        assert e <= TOL[dtype] * scl, f"{name}: max|err| {e:.3e} > {TOL[dtype]:.1e} * {scl:.3e}"
    return errs


CASES = [
    # B, Hq, Hkv, N, M, d, dtype, causal
    (1, 2, 2, 256, 256, 64, FP16, False),
    (1, 2, 2, 256, 256, 128, BF16, True),
    (2, 4, 4, 384, 384, 128, FP16, True),
    (1, 8, 2, 512, 512, 128, BF16, True),
    (1, 4, 1, 256, 256, 64, FP16, False),
    (1, 2, 2, 300, 300, 128, FP16, True),
    (1, 2, 2, 200, 333, 128, BF16, False),
    (1, 2, 2, 130, 1, 64, FP16, False),
    (1, 2, 2, 256, 400, 128, FP16, True),
    (1, 2, 1, 400, 256, 64, BF16, True),
    # odd GQA group, ragged
    (1, 6, 2, 333, 333, 128, BF16, True),
    (1, 3, 1, 200, 260, 64, FP16, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}x{}_N{}_M{}_d{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "f16" if c[6] == FP16 else "bf16",
    "causal" if c[7] else "full"))
def test_backward_parity(oracle_mod, case):
    errs = check(oracle_mod, *case)
    print(case, errs)


def test_backward_headline_shape(oracle_mod):
    """The causal MHA prefill shape B=2, H=16, N=M=2048, d=128, bf16, in full."""
    errs = check(oracle_mod, 2, 16, 16, 2048, 2048, 128, BF16, True, seed=1002)
    print(errs)


def test_backward_deterministic_dk_dv():
    """dK and dV accumulate in TMEM in a fixed order: two runs agree bit for bit."""
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    q, k, v = (t.cuda() for t in make_inputs(1, 4, 2, 512, 512, 128, FP16, 5))
    dout = make_dout(1, 512, 4, 128, FP16, 6).cuda()
    o, lse = fa.attention_forward(q, k, v, True, 0.088)
    a = fa.attention_backward(q, k, v, o, lse, dout, True, 0.088)
    b = fa.attention_backward(q, k, v, o, lse, dout, True, 0.088)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_backward_gqa_workload_full(oracle_mod):
    """The causal GQA workload (Hq=32, Hkv=8, N=M=8192, fp16, 1% of K rows x8) as the
    bench runs its backward, every element of dQ, dK and dV against the oracle."""
    from exact_attention_05_gb300.workloads import WORKLOADS, workload_inputs
    w = WORKLOADS["prefill_causal_gqa32x8_n8192_f16_peaky"]
    q, k, v = workload_inputs(w)
    dout = make_dout(w.B, w.N, w.Hq, w.d, w.dtype, w.seed + 7)
    got = run_backward(q, k, v, dout, w.causal, w.scale)
    ref = oracle_mod.attention_backward(bits(q), bits(k), bits(v), bits(dout), w.dtype, w.causal,
                                        w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.isfinite(g).all(), f"{name}: non-finite"
        e = float(np.abs(g - r).max())
        scl = max(float(np.abs(r).max()), 1.0)
        print(f"PARITY backward {w.name} {name}: max|err| = {e:.3e}, scale {scl:.3e}")
        assert e <= TOL[w.dtype] * scl, f"{name}: max|err| {e:.3e} > {TOL[w.dtype]:.1e} * {scl:.3e}"


@pytest.mark.parametrize("name", ["prefill_causal_h16_n32768_bf16"])
def test_backward_workload_full_sampled(oracle_mod, name):
    """The long causal workload at full size, as the bench runs its backward (its
    full fp64 backward would take the oracle several minutes on 16 cores, as it is
    parallel over (b, kv head) only): dQ on sampled rows against the oracle (dQ_i
    depends on row i alone), and dK, dV through properties that hold at any size:
    sum_j dK_j = 0 for every (b, kv head)
    (the softmax ignores a common shift of the keys), and sum_j dV_j equals the sum of
    dO over the rows of the query heads that read the kv head (every P row sums to 1).
    The sums are checked within 8 ulp of the type times sum_j |dK_j| (resp. |dV_j|),
    the per-element bound added up."""
    import exact_attention_05_gb300 as fa
    from exact_attention_05_gb300.workloads import WORKLOADS, sample_rows, workload_inputs
    torch = torch_cuda()
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    dout = make_dout(w.B, w.N, w.Hq, w.d, w.dtype, w.seed + 7)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, lse = fa.attention_forward(qd, kd, vd, w.causal, w.scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, w.causal, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    tol = TOL[w.dtype]
    rows = sample_rows(w, 96, seed=17)
    ref = oracle_mod.attention_backward_dq_rows(bits(q), bits(k), bits(v), bits(dout), w.dtype,
                                                w.causal, w.scale, rows)
    got = dq.double().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    e = float(np.abs(got - ref).max())
    assert e <= tol * max(float(np.abs(ref).max()), 1.0), f"dQ rows: {e:.3e}"
    dk64 = dk.double().cpu().numpy()
    dv64 = dv.double().cpu().numpy()
    ksum = np.abs(dk64.sum(axis=1))
    kbound = tol * np.abs(dk64).sum(axis=1)
    assert bool((ksum <= kbound + 1e-30).all()), float((ksum / np.maximum(kbound, 1e-30)).max())
    g = w.Hq // w.Hkv
    want = dout.double().numpy().reshape(w.B, w.N, w.Hkv, g, w.d).sum(axis=(1, 3))
    vdiff = np.abs(dv64.sum(axis=1) - want)
    vbound = tol * np.abs(dv64).sum(axis=1)
    assert bool((vdiff <= vbound + 1e-30).all()), float((vdiff / np.maximum(vbound, 1e-30)).max())

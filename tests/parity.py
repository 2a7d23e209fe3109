"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle element by element.

Tolerances are the ones the method's target states: max |O_gpu - O_oracle|
<= 2e-3 for fp16 inputs and 1e-2 for bf16 inputs, and max |LSE_gpu -
LSE_oracle| <= 1e-3, over every compared element.
"""
import numpy as np
import pytest

from exact_attention_05_gb300.workloads import BF16, FP16, bits, make_inputs

O_TOL = {FP16: 2e-3, BF16: 1e-2}
LSE_TOL = 1e-3


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def run_prefill(q, k, v, causal, scale, stream=None):
    """fa_fwd on host tensors; returns (O float64 numpy, LSE numpy)."""
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.attention_forward(qd, kd, vd, causal, scale, stream=stream)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def run_decode(q, k, v, chunk, scale, single_launch=False):
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    o, lse = fa.decode(q.cuda(), k.cuda(), v.cuda(), chunk, scale, single_launch=single_launch)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    assert np.isfinite(lse_gpu).all(), f"{what}: non-finite LSE"
    eo = float(np.abs(o_gpu - o_ref).max())
    el = float(np.abs(lse_gpu - lse_ref).max())
    assert eo <= O_TOL[dtype], f"{what}: max|dO| = {eo:.3e} > {O_TOL[dtype]:.0e}"
    assert el <= LSE_TOL, f"{what}: max|dLSE| = {el:.3e} > {LSE_TOL:.0e}"
    return eo, el


def prefill_case(oracle_mod, B, Hq, Hkv, N, M, d, dtype, causal, scale=None, seed=5,
                 peaky_frac=0.0):
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, dtype, seed, peaky_frac)
    o, lse = run_prefill(q, k, v, causal, scale)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, causal, scale)
    return assert_close(o, lse, o_ref, lse_ref, dtype, f"prefill {B,Hq,Hkv,N,M,d,dtype,causal}")

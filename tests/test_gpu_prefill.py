"""GPU parity of the prefill path (fa_fwd through the C ABI) against the fp64 oracle.

Small cases are compared element by element: several tiles, ragged tails in
N and M, N != M with the top-left causal mask, GQA ratios 1-8, d = 64 and 128,
fp16 and bf16, the degenerate N = M = 1.  The four prefill workloads are run
at full size in the launch configuration the bench times, and every one of
them is compared with the oracle on every element of O and LSE (the long
causal workload's oracle takes about 75 s on 16 host cores).
"""
import pytest

from exact_attention_05_gb300.workloads import BF16, FP16, WORKLOADS, bits, workload_inputs
from parity import assert_close, prefill_case, run_prefill

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, N, M, d, dtype, causal
    (1, 2, 2, 256, 256, 64, FP16, False),
    (1, 2, 1, 300, 300, 128, BF16, True),
    (2, 4, 2, 200, 333, 64, FP16, False),
    (1, 4, 4, 130, 400, 128, FP16, True),
    (1, 2, 2, 400, 130, 128, BF16, True),
    (1, 8, 1, 129, 129, 128, FP16, True),
    (1, 8, 4, 257, 257, 64, BF16, True),
    (1, 1, 1, 1, 1, 64, BF16, False),
    (1, 1, 1, 1, 1, 128, FP16, True),
    (2, 2, 2, 5, 1000, 128, FP16, False),
    (1, 2, 2, 1000, 5, 64, BF16, False),
    (1, 3, 3, 384, 384, 128, FP16, False),
    (2, 4, 2, 384, 384, 128, BF16, True),
    (1, 2, 2, 127, 129, 64, FP16, True),
    # causal with an even GQA group (two query heads per CTA) and N != M
    (1, 4, 2, 130, 400, 128, FP16, True),
    (2, 8, 2, 400, 131, 64, BF16, True),
    # causal with an odd GQA group
    (1, 6, 2, 333, 333, 128, FP16, True),
    (2, 9, 3, 257, 300, 64, BF16, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}x{}_N{}_M{}_d{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "f16" if c[6] == FP16 else "bf16",
    "causal" if c[7] else "full"))
def test_prefill_parity_small(oracle_mod, case):
    prefill_case(oracle_mod, *case)


# K/V larger than the prefill's L2 group budget (64 MB): the CTAs are dispatched
# in several groups of heads (MHA with a ragged last row pair; causal GQA with
# two query heads per CTA)
GROUPED = [
    (1, 10, 10, 12900, 12900, 128, BF16, True),
    (1, 32, 16, 8200, 8200, 128, FP16, True),
    # an odd GQA group (one query head per Q tile pair, three per kv head)
    (1, 48, 16, 8200, 8200, 128, FP16, True),
    # non-causal: few query rows against a long key range
    (1, 4, 4, 300, 36000, 128, BF16, False),
]


@pytest.mark.parametrize("case", GROUPED, ids=lambda c: "B{}_H{}x{}_N{}_{}".format(
    c[0], c[1], c[2], c[3], "f16" if c[6] == FP16 else "bf16"))
def test_prefill_parity_l2_groups(oracle_mod, case):
    prefill_case(oracle_mod, *case)


# More work items (Q tile pairs) than SMs: resident CTAs take over the items of
# CTAs that have not started, one after the other, so each of these runs items
# back to back on one CTA -- including items whose second Q tile lies wholly
# below the last row (an odd number of row tiles, rows paired), non-causal,
# d = 64, and causal GQA with two query heads per item and N != M.
MANY_ITEMS = [
    (8, 24, 24, 300, 300, 128, BF16, True),
    (4, 24, 8, 640, 640, 64, FP16, False),
    (6, 32, 8, 520, 700, 128, FP16, True),
    (3, 40, 40, 1100, 1100, 64, BF16, True),
    # one KV tile per item (N <= 128, two query heads per item): no steady iterations
    (12, 32, 16, 100, 100, 128, FP16, True),
    # tile 0 walks one KV tile, tile 1 two (the diagonal), d = 64
    (2, 100, 100, 200, 200, 64, BF16, True),
    # every item's second Q tile lies below the last row (N <= 128, rows paired)
    (4, 48, 48, 100, 300, 128, FP16, False),
]


@pytest.mark.parametrize("case", MANY_ITEMS, ids=lambda c: "B{}_H{}x{}_N{}_M{}_d{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[7] else "full"))
def test_prefill_parity_many_items(oracle_mod, case):
    prefill_case(oracle_mod, *case)


@pytest.mark.parametrize("scale", [0.02, 1.0])
def test_prefill_scale_values(oracle_mod, scale):
    prefill_case(oracle_mod, 1, 2, 2, 300, 300, 128, FP16, True, scale=scale)


def test_prefill_peaky_keys(oracle_mod):
    """1% of key rows x8: the row max jumps mid-sequence and O must be rescaled."""
    prefill_case(oracle_mod, 1, 8, 2, 640, 640, 128, FP16, True, peaky_frac=0.01, seed=9)


@pytest.mark.parametrize("name", ["prefill_mha_n256_d64_f16", "prefill_causal_b2_h16_n2048_bf16",
                                  "prefill_causal_gqa32x8_n8192_f16_peaky",
                                  "prefill_causal_h16_n32768_bf16"])
def test_prefill_workload_full(oracle_mod, name):
    """Every element of O [B,N,Hq,d] and LSE [B,Hq,N] of a full-size workload."""
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    o, lse = run_prefill(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), w.dtype, w.causal, w.scale)
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    assert_close(o, lse, o_ref, lse_ref, w.dtype, name)

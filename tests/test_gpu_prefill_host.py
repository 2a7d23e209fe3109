"""GPU checks of fa_fwd_host: the forward on host tensors, with the transfers
overlapped with the kernels, chunk by chunk.

Each chunk runs fa_fwd on a contiguous slice of (b, kv heads) and the kernel
treats heads independently, so the results must equal fa_fwd on device tensors
bit for bit (fa_fwd itself is checked against the oracle in test_gpu_prefill).
"""
import pytest
import torch

import exact_attention_05_gb300 as fa
from exact_attention_05_gb300.workloads import BF16, FP16, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, N, M, d, dtype, causal
    (1, 16, 16, 512, 512, 128, BF16, True),     # one batch entry: four head groups
    (2, 8, 2, 300, 333, 128, FP16, True),       # GQA, ragged N != M, two groups per entry
    (5, 4, 4, 200, 200, 64, FP16, False),       # B >= 4: one chunk per batch entry
    (3, 6, 3, 129, 257, 128, BF16, False),      # kv-head groups of uneven size
    (1, 2, 1, 1, 1, 64, BF16, True),            # degenerate N = M = 1
]


def device_reference(q, k, v, causal, scale):
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}x{}_N{}_M{}_d{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "f16" if c[6] == FP16 else "bf16",
    "causal" if c[7] else "full"))
def test_host_forward_equals_device_forward(case):
    B, Hq, Hkv, N, M, d, dtype, causal = case
    scale = 1.0 / d ** 0.5
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, dtype, seed=77 + N)
    o_ref, lse_ref = device_reference(q, k, v, causal, scale)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    for _ in range(2):  # the second call reuses the streams, events and staging
        o, lse = fa.attention_forward_host(qp, kp, vp, causal, scale)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, lse_ref)


def test_host_forward_pageable_memory_and_no_lse():
    q, k, v = make_inputs(2, 4, 2, 256, 256, 128, FP16, seed=5)
    o_ref, _ = device_reference(q, k, v, True, 0.088)
    o = torch.empty_like(q)  # pageable
    fa.attention_forward_host(q, k, v, True, 0.088, out=o, with_lse=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)


def test_host_forward_on_a_side_stream():
    q, k, v = (t.pin_memory() for t in make_inputs(2, 8, 8, 384, 384, 128, BF16, seed=6))
    o_ref, lse_ref = device_reference(q, k, v, False, 0.1)
    s = torch.cuda.Stream()
    o, lse = fa.attention_forward_host(q, k, v, False, 0.1, stream=s)
    s.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)

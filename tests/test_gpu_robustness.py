"""GPU robustness checks that need no sanitizer: guard bands around every output
(no write lands outside the caller's buffers), bitwise determinism, a
non-default stream, a NULL lse, and the bounded-wait path (a wait that nobody
releases expires after its limit, the timeout is reported through
fa_get_last_device_status, and the context stays usable).
"""
import numpy as np
import pytest

import exact_attention_05_gb300 as fa
from exact_attention_05_gb300.workloads import BF16, FP16, bits, make_inputs
from parity import assert_close, run_prefill, torch_cuda

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side (a multiple of 8, so the interior stays 16-byte aligned)


def guarded(torch, numel, dtype, pattern):
    buf = torch.empty(numel + 2 * GUARD, dtype=dtype, device="cuda")
    iview = buf.view(torch.int16) if dtype != torch.float32 else buf.view(torch.int32)
    iview.fill_(pattern)
    return buf, buf[GUARD:GUARD + numel]


def guards_intact(torch, buf, dtype, pattern):
    iv = (buf.view(torch.int16) if dtype != torch.float32 else buf.view(torch.int32)).cpu()
    return bool((iv[:GUARD] == pattern).all()) and bool((iv[-GUARD:] == pattern).all())


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_writes_stay_inside_outputs(oracle_mod, causal):
    torch = torch_cuda()
    B, Hq, Hkv, N, M, d = 2, 4, 2, 300, 333, 128
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, BF16, seed=41)
    obuf, o = guarded(torch, B * N * Hq * d, torch.bfloat16, 0x7E7E)
    lbuf, lse = guarded(torch, B * Hq * N, torch.float32, 0x7F7F7F7F)
    fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), o, lse, B, Hq, Hkv, N, M, d, int(causal), 0.1, BF16)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    assert guards_intact(torch, obuf, torch.bfloat16, 0x7E7E)
    assert guards_intact(torch, lbuf, torch.float32, 0x7F7F7F7F)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), BF16, causal, 0.1)
    assert_close(o.view(B, N, Hq, d).double().cpu().numpy(),
                 lse.view(B, Hq, N).double().cpu().numpy(), o_ref, lse_ref, BF16, "guarded")


def test_decode_writes_stay_inside_outputs(oracle_mod):
    torch = torch_cuda()
    B, Hq, Hkv, M, d = 2, 8, 2, 1000, 128
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=42)
    obuf, o = guarded(torch, B * Hq * d, torch.float16, 0x7E7E)
    lbuf, lse = guarded(torch, B * Hq, torch.float32, 0x7F7F7F7F)
    fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), o, lse, B, Hq, Hkv, M, d, 128, 0.08, FP16)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    assert guards_intact(torch, obuf, torch.float16, 0x7E7E)
    assert guards_intact(torch, lbuf, torch.float32, 0x7F7F7F7F)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, False, 0.08)
    assert_close(o.view(B, 1, Hq, d).double().cpu().numpy(),
                 lse.view(B, Hq).double().cpu().numpy(), o_ref, lse_ref[:, :, 0], FP16, "guarded")


def test_prefill_is_deterministic():
    torch = torch_cuda()
    q, k, v = make_inputs(1, 4, 4, 700, 700, 128, FP16, seed=43)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.attention_forward(qd, kd, vd, True, 0.09)
    o2, l2 = fa.attention_forward(qd, kd, vd, True, 0.09)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_non_default_stream_and_null_lse():
    torch = torch_cuda()
    q, k, v = make_inputs(1, 2, 2, 500, 500, 64, BF16, seed=44)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ref, _ = fa.attention_forward(qd, kd, vd, True, 0.125)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.attention_forward(qd, kd, vd, True, 0.125, with_lse=False, stream=s)
    s.synchronize()
    assert lse is None
    assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    od, _ = fa.decode(qd[:, :1].contiguous(), kd, vd, 64, 0.125, stream=s, with_lse=False)
    s.synchronize()
    assert torch.isfinite(od.float()).all()


def test_unsupported_shape_is_rejected_on_device():
    torch = torch_cuda()
    q = torch.zeros((1, 4, 2, 96), dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.attention_forward(q, q, q, False, 0.1)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


def test_bounded_wait_expires_and_context_survives(oracle_mod):
    torch = torch_cuda()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    fa.fa_set_wait_timeout_ns(2_000_000)  # 2 ms
    try:
        assert fa.fa_selftest_wait_timeout() == fa.FA_OK
        assert fa.fa_get_last_device_status() == fa.FA_ERR_TIMEOUT
        assert fa.fa_get_last_device_status() == fa.FA_OK   # read clears it
    finally:
        fa.fa_set_wait_timeout_ns(0)
    # the context is still healthy: a normal call still matches the oracle
    q, k, v = make_inputs(1, 2, 1, 200, 200, 128, FP16, seed=45)
    o, lse = run_prefill(q, k, v, True, 0.1)
    o_ref, lse_ref = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, True, 0.1)
    assert_close(o, lse, o_ref, lse_ref, FP16, "after timeout")
    assert np.isfinite(o).all()


def test_prefill_many_items_inside_a_captured_cuda_graph():
    """A prefill grid with more work items than SMs (resident CTAs take over the
    items of CTAs that have not started) captured into a CUDA graph and replayed
    with new query values: every replay equals an eager call, bit for bit."""
    torch = torch_cuda()
    B, Hq, Hkv, N, M, d = 4, 16, 8, 1024, 1024, 128
    scale = 1.0 / d ** 0.5
    q0, k, v = (t.cuda() for t in make_inputs(B, Hq, Hkv, N, M, d, BF16, seed=81))
    q = q0.clone()
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    fa.attention_forward(q, k, v, True, scale, out=o, lse=lse)  # kernel set-up before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.attention_forward(q, k, v, True, scale, out=o, lse=lse)
    for seed in (82, 83):
        qn, _, _ = make_inputs(B, Hq, Hkv, N, M, d, BF16, seed=seed)
        q.copy_(qn.cuda())
        graph.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = fa.attention_forward(q, k, v, True, scale)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), seed
    assert fa.fa_get_last_device_status() == fa.FA_OK


def test_prefill_grids_on_two_streams_at_once():
    """Two prefill grids, each with more work items than SMs, enqueued on two
    streams without ordering between them: CTAs only take over items of their
    own grid, so each result equals its own call made alone, bit for bit."""
    torch = torch_cuda()
    shapes = [(4, 16, 16, 1024, 1024, 128, BF16, True), (3, 24, 8, 700, 900, 64, FP16, False)]
    inputs, alone = [], []
    for i, (B, Hq, Hkv, N, M, d, dt, causal) in enumerate(shapes):
        q, k, v = (t.cuda() for t in make_inputs(B, Hq, Hkv, N, M, d, dt, seed=90 + i))
        inputs.append((q, k, v, causal, 1.0 / d ** 0.5))
        o, lse = fa.attention_forward(q, k, v, causal, 1.0 / d ** 0.5)
        torch.cuda.synchronize()
        alone.append((o.clone(), lse.clone()))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = []
    for rep in range(3):
        for s, (q, k, v, causal, scale) in zip(streams, inputs):
            with torch.cuda.stream(s):
                outs.append(fa.attention_forward(q, k, v, causal, scale, stream=s))
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    for i, (o, lse) in enumerate(outs):
        o_ref, lse_ref = alone[i % 2]
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), i

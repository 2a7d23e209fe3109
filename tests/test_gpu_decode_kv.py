"""GPU parity of the FP8 (e4m3) K/V decode and the paged-KV decode.

fa_decode_fp8 is compared with the oracle's exact attention over the
dequantised cache (k_scale[h] * e4m3(k8), likewise V), fa_decode_paged with
the oracle's block-table gather; both at the O/LSE tolerances of the 16-bit
path (the GPU result and the oracle describe the same real-valued attention,
so only fp32 rounding separates them).  Cases: both decode workloads at full
size, ragged key counts (partial 128-key sub-tiles and partial chunks), d = 64
and 128, fp16 and bf16 queries, GQA groups of 1 to 16 heads, page sizes 8 to
1024, sequences of 0 and 1 keys, shuffled pages and a pool larger than needed.
"""
import numpy as np
import pytest

from exact_attention_05_gb300.workloads import BF16, FP16, WORKLOADS, bits, \
    make_fp8_decode_inputs, make_inputs, make_paged, workload_decode_inputs
from parity import assert_close, torch_cuda

pytestmark = pytest.mark.gpu


def run_fp8(q, k8, v8, ks, vs, chunk, scale):
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    o, lse = fa.decode_fp8(q.cuda(), k8.cuda(), v8.cuda(), ks.cuda(), vs.cuda(), chunk, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def run_paged(q, kc, vc, bt, seq_lens, max_seq_len, chunk, scale):
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    o, lse = fa.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), seq_lens.cuda(),
                             max_seq_len, chunk, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


# ---- FP8 -----------------------------------------------------------------------

FP8_CASES = [
    # B, Hq, Hkv, M, d, dtype (of q and o), chunk
    (1, 8, 8, 512, 128, FP16, 128),
    (2, 8, 2, 1000, 128, BF16, 128),
    (1, 4, 4, 301, 64, FP16, 128),
    (1, 16, 2, 1000, 64, BF16, 256),
    (2, 4, 4, 777, 128, FP16, 100),
    (1, 2, 1, 129, 128, FP16, 1),
    (1, 6, 3, 4097, 64, FP16, 500),
    (1, 4, 4, 1, 128, BF16, 128),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "B{}_H{}x{}_M{}_d{}_{}_c{}".format(
    c[0], c[1], c[2], c[3], c[4], "f16" if c[5] == FP16 else "bf16", c[6]))
def test_fp8_decode_parity(oracle_mod, case):
    B, Hq, Hkv, M, d, dtype, chunk = case
    scale = 1.0 / d ** 0.5
    q, k8, v8, ks, vs = make_fp8_decode_inputs(B, Hq, Hkv, M, d, dtype, seed=61 + M)
    o, lse = run_fp8(q, k8, v8, ks, vs, chunk, scale)
    o_ref, lse_ref = oracle_mod.decode_fp8(bits(q), k8.numpy(), v8.numpy(), ks.numpy(),
                                           vs.numpy(), dtype, scale)
    assert_close(o, lse, o_ref, lse_ref, dtype, f"fp8 decode {case}")


def test_fp8_decode_workload_full(oracle_mod):
    w = WORKLOADS["decode_fp8_b2_h8_m65536_f16"]
    x = workload_decode_inputs(w)
    o, lse = run_fp8(x["q"], x["k"], x["v"], x["k_scale"], x["v_scale"], w.chunk, w.scale)
    o_ref, lse_ref = oracle_mod.decode_fp8(bits(x["q"]), x["k"].numpy(), x["v"].numpy(),
                                           x["k_scale"].numpy(), x["v_scale"].numpy(), w.dtype,
                                           w.scale)
    assert_close(o, lse, o_ref, lse_ref, w.dtype, w.name)


def test_fp8_decode_scales_per_head(oracle_mod):
    """Very different scales per kv head (1e-3 .. 1e2 on K, 1e-2 .. 10 on V):
    a scale taken from the wrong head or swapped between K and V shows."""
    torch = torch_cuda()
    B, Hq, Hkv, M, d = 1, 8, 4, 600, 128
    q, k8, v8, _, _ = make_fp8_decode_inputs(B, Hq, Hkv, M, d, FP16, seed=71)
    ks = torch.tensor([1e-3, 3e-2, 0.5, 1e2 / 448.0], dtype=torch.float32)
    vs = torch.tensor([10.0, 1e-2, 0.3, 2.0], dtype=torch.float32)
    o, lse = run_fp8(q, k8, v8, ks, vs, 128, 1.0 / d ** 0.5)
    o_ref, lse_ref = oracle_mod.decode_fp8(bits(q), k8.numpy(), v8.numpy(), ks.numpy(),
                                           vs.numpy(), FP16, 1.0 / d ** 0.5)
    # O scales with v_scale (up to 10): compare relative to each row's magnitude
    rel = np.abs(o - o_ref).max(axis=-1) / np.maximum(np.abs(o_ref).max(axis=-1), 1e-30)
    assert float(rel.max()) <= 2e-3, float(rel.max())
    assert float(np.abs(lse - lse_ref).max()) <= 1e-3


# ---- paged ---------------------------------------------------------------------

PAGED_CASES = [
    # B, Hq, Hkv, max_seq_len, d, dtype, page, chunk, seq_lens (None = all max)
    (2, 8, 8, 1000, 128, FP16, 16, 128, None),
    (3, 8, 2, 1500, 128, BF16, 8, 128, [1500, 17, 640]),
    (2, 4, 4, 777, 64, FP16, 64, 64, [777, 300]),
    (2, 16, 2, 2000, 64, BF16, 128, 256, [1999, 129]),
    (1, 4, 4, 3000, 128, FP16, 256, 128, None),
    (2, 2, 2, 5000, 128, FP16, 1024, 384, [5000, 1100]),
    (4, 4, 1, 300, 128, FP16, 32, 32, [300, 0, 1, 33]),
    (1, 6, 3, 129, 64, FP16, 16, 16, None),
]


@pytest.mark.parametrize("case", PAGED_CASES, ids=lambda c: "B{}_H{}x{}_M{}_d{}_{}_p{}_c{}".format(
    c[0], c[1], c[2], c[3], c[4], "f16" if c[5] == FP16 else "bf16", c[6], c[7]))
def test_paged_decode_parity(oracle_mod, case):
    torch = torch_cuda()
    B, Hq, Hkv, M, d, dtype, page, chunk, lens = case
    scale = 1.0 / d ** 0.5
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, dtype, seed=91 + M)
    kc, vc, bt = make_paged(k, v, page, seed=5 + page, extra_pages=3)
    # one more table column than needed, never read (the entry is out of range)
    bt = torch.cat([bt, torch.full((B, 1), -1, dtype=torch.int32)], dim=1).contiguous()
    seq = torch.tensor(lens if lens is not None else [M] * B, dtype=torch.int32)
    o, lse = run_paged(q, kc, vc, bt, seq, M, chunk, scale)
    o_ref, lse_ref = oracle_mod.decode_paged(bits(q), bits(kc), bits(vc), bt.numpy(),
                                             seq.numpy(), dtype, M, scale)
    empty = seq.numpy() <= 0
    if empty.any():
        assert np.all(o[empty] == 0.0) and np.all(np.isneginf(lse[empty]))
        o, lse, o_ref, lse_ref = o[~empty], lse[~empty], o_ref[~empty], lse_ref[~empty]
    assert_close(o, lse, o_ref, lse_ref, dtype, f"paged decode {case}")


def test_paged_decode_workload_full(oracle_mod):
    w = WORKLOADS["decode_paged_b2_h8_m65536_p16_f16"]
    x = workload_decode_inputs(w)
    o, lse = run_paged(x["q"], x["k_cache"], x["v_cache"], x["block_table"], x["seq_lens"], w.M,
                       w.chunk, w.scale)
    o_ref, lse_ref = oracle_mod.attention(bits(x["q"]), bits(x["k"]), bits(x["v"]), w.dtype,
                                          False, w.scale)
    assert_close(o, lse, o_ref, lse_ref[:, :, 0], w.dtype, w.name)


def test_paged_equals_contiguous_decode():
    """The same keys through a shuffled page pool and contiguously give the same
    result up to the order of fp32 rounding.  Both read the same rows into the
    same tile positions; the paged path merges each stripe's chunks on the fly
    and the contiguous two-kernel path merges per-chunk partials, which Step 2
    of the flash-decoding page's section 2.2 makes the same sum in another order."""
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    B, Hq, Hkv, M, d = 2, 8, 8, 4096, 128
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=123)
    kc, vc, bt = make_paged(k, v, 64, seed=3)
    seq = torch.full((B,), M, dtype=torch.int32)
    o1, l1 = fa.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), seq.cuda(), M, 128,
                             d ** -0.5)
    o2, l2 = fa.decode(q.cuda(), k.cuda(), v.cuda(), 128, d ** -0.5)
    torch.cuda.synchronize()
    # a few fp32 roundings of the merge apart: far below the parity tolerances
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-4
    assert (l1 - l2).abs().max().item() <= 2e-5


def test_paged_decode_rejects_bad_geometry():
    import exact_attention_05_gb300 as fa
    torch = torch_cuda()
    q = torch.zeros((1, 1, 2, 128), dtype=torch.float16, device="cuda")
    kc = torch.zeros((4, 24, 2, 128), dtype=torch.float16, device="cuda")   # page 24
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    sl = torch.full((1,), 64, dtype=torch.int32, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.decode_paged(q, kc, kc, bt, sl, 64, 48, 0.1)
    assert e.value.status == fa.FA_ERR_INVALID_ARG

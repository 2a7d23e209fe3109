"""Pins of the fp64 CPU oracle against facts that do not come from the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, an off-by-one mask, a wrong GQA index, a transposed operand, a
wrong LSE base) fails at least one of them:

* decoders vs numpy/torch's own float16/bfloat16 conversion (library routines);
* the invariants the method fixes: rows of P sum to 1; constant V returns V;
  M = 1 returns V[0]; causal row 0 returns V[0];
* closed forms: uniform attention for Q = 0 (mean of V, LSE = ln #keys), an
  exactly solvable one-hot case, shift invariance of O with LSE moving by the
  shift, GQA equal to MHA with repeated K/V heads;
* the chunked decode of "CUDA 实现 Flash Decoding" section 2.2 against the
  unchunked softmax, for several chunk sizes with a ragged last chunk;
* an independent formulation (numpy exp(S)/sum exp(S) without the max
  subtraction, safe at these sizes) and torch's float64 CPU
  scaled_dot_product_attention (a library special case).
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_05_gb300.workloads import BF16, FP16, bits, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def dec(oracle_mod, t, dtype):
    return oracle_mod.decode(bits(t), dtype)


def as16(x, dtype):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(
        torch.float16 if dtype == FP16 else torch.bfloat16)


# ---------------------------------------------------------------------------
# the bit decoders against library conversions, all 65536 patterns
# ---------------------------------------------------------------------------

def test_fp16_decoder_matches_numpy(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = oracle_mod.decode(pats, FP16)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_bf16_decoder_matches_torch(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = oracle_mod.decode(pats, BF16)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_softmax_rows_sum_to_one(oracle_mod, causal, dtype):
    q, k, v = make_inputs(2, 4, 2, 9, 9 if causal else 13, 8, dtype, seed=11)
    o, lse, p = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, causal, 0.3,
                                     with_probs=True)
    assert np.allclose(p.sum(axis=-1), 1.0, atol=1e-14, rtol=0)
    assert (p >= 0).all()
    if causal:
        N = p.shape[2]
        upper = np.triu(np.ones((N, p.shape[3]), bool), k=1)
        assert (p[..., upper] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_returns_v(oracle_mod, causal):
    q, k, _ = make_inputs(1, 2, 1, 7, 7, 16, FP16, seed=12)
    row = np.linspace(-2, 2, 16).astype(np.float32)
    v = as16(np.broadcast_to(row, (1, 7, 1, 16)).copy(), FP16)
    o, _ = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, causal, 0.25)
    vrow = oracle_mod.decode(bits(v[0, 0, 0]), FP16)
    assert np.abs(o - vrow).max() < 1e-14


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_single_key_returns_v0_and_scaled_logit(oracle_mod, dtype):
    q, k, v = make_inputs(2, 3, 3, 5, 1, 8, dtype, seed=13)
    scale = 0.37
    o, lse = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, False, scale)
    qd, kd, vd = dec(oracle_mod, q, dtype), dec(oracle_mod, k, dtype), dec(oracle_mod, v, dtype)
    for b in range(2):
        for h in range(3):
            for i in range(5):
                assert np.abs(o[b, i, h] - vd[b, 0, h]).max() < 1e-15
                assert abs(lse[b, h, i] - scale * float(qd[b, i, h] @ kd[b, 0, h])) < 1e-12


def test_causal_row_zero_returns_v0(oracle_mod):
    q, k, v = make_inputs(1, 2, 2, 6, 6, 8, BF16, seed=14)
    scale = 0.5
    o, lse = oracle_mod.attention(bits(q), bits(k), bits(v), BF16, True, scale)
    qd, kd, vd = dec(oracle_mod, q, BF16), dec(oracle_mod, k, BF16), dec(oracle_mod, v, BF16)
    for h in range(2):
        assert np.abs(o[0, 0, h] - vd[0, 0, h]).max() < 1e-15
        assert abs(lse[0, h, 0] - scale * float(qd[0, 0, h] @ kd[0, 0, h])) < 1e-12


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_one_hot_closed_form(oracle_mod):
    """q = t e_0, k_{j*} = e_0 and every other k_j has a zero first component.

    Then s_{j*} = scale*t and s_j = 0 otherwise, so exactly
    O = (e^{scale t} v_{j*} + sum_{j != j*} v_j) / (e^{scale t} + M - 1),
    LSE = ln(e^{scale t} + M - 1); O tends to v_{j*} as t grows.
    """
    M, d, jstar, scale = 11, 8, 6, 0.125
    _, k, v = make_inputs(1, 1, 1, 1, M, d, FP16, seed=15)
    k = k.clone()
    k[..., 0] = 0
    k[0, jstar, 0] = torch.tensor([1.0], dtype=torch.float16)
    k[0, jstar, 0, 1:] = 0
    vd = dec(oracle_mod, v, FP16)[0, :, 0]
    prev_err = None
    for t in (8.0, 32.0, 64.0, 128.0):
        q = torch.zeros((1, 1, 1, d), dtype=torch.float16)
        q[..., 0] = t
        o, lse = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, False, scale)
        e = math.exp(scale * t)
        want = (e * vd[jstar] + vd.sum(0) - vd[jstar]) / (e + M - 1)
        assert np.abs(o[0, 0, 0] - want).max() < 1e-13
        assert abs(lse[0, 0, 0] - math.log(e + M - 1)) < 1e-13
        err = np.abs(o[0, 0, 0] - vd[jstar]).max()
        assert err <= (M - 1) * math.exp(-scale * t) * np.abs(vd).max() * 2 + 1e-15
        if prev_err is not None:
            assert err < prev_err
        prev_err = err


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_is_uniform(oracle_mod, causal):
    N = M = 9
    _, k, v = make_inputs(1, 2, 2, N, M, 8, BF16, seed=16)
    q = torch.zeros((1, N, 2, 8), dtype=torch.bfloat16)
    o, lse = oracle_mod.attention(bits(q), bits(k), bits(v), BF16, causal, 0.7)
    vd = dec(oracle_mod, v, BF16)
    for h in range(2):
        for i in range(N):
            n = i + 1 if causal else M
            assert np.abs(o[0, i, h] - vd[0, :n, h].mean(0)).max() < 1e-14
            assert abs(lse[0, h, i] - math.log(n)) < 1e-14


def test_shift_invariance(oracle_mod):
    """Adding c to every logit of a row leaves O unchanged and moves LSE by c."""
    N, M, d, scale = 5, 7, 6, 0.5
    q, k, v = make_inputs(1, 1, 1, N, M, d, FP16, seed=17)
    q0, k0 = q.clone(), k.clone()
    q0[..., 0] = 0
    k0[..., 0] = 0
    q1, k1 = q0.clone(), k0.clone()
    q1[..., 0] = 3.0
    k1[..., 0] = 1.0              # every logit gains scale * 3
    oa, la = oracle_mod.attention(bits(q0), bits(k0), bits(v), FP16, False, scale)
    ob, lb = oracle_mod.attention(bits(q1), bits(k1), bits(v), FP16, False, scale)
    assert np.abs(oa - ob).max() < 1e-14
    assert np.abs((lb - la) - scale * 3.0).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_heads(oracle_mod, causal):
    B, Hq, Hkv, N, M, d = 2, 8, 2, 6, 6, 8
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, FP16, seed=18)
    g = Hq // Hkv
    krep = k.repeat_interleave(g, dim=2)
    vrep = v.repeat_interleave(g, dim=2)
    o1, l1 = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, causal, 0.3)
    o2, l2 = oracle_mod.attention(bits(q), bits(krep), bits(vrep), FP16, causal, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # a wrong mapping (h % Hkv) would give a different answer on these inputs
    kmod = k.repeat(1, 1, g, 1)
    vmod = v.repeat(1, 1, g, 1)
    o3, _ = oracle_mod.attention(bits(q), bits(kmod), bits(vmod), FP16, causal, 0.3)
    assert np.abs(o1 - o3).max() > 1e-3


# ---------------------------------------------------------------------------
# split-KV decode: chunk partials and the LSE-weighted merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("chunk", [1, 3, 7, 128, 300, 301])
def test_chunked_merge_equals_unchunked(oracle_mod, chunk):
    B, Hq, Hkv, M, d = 2, 4, 2, 301, 16
    q, k, v = make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=19)
    scale = 1 / 4
    op, lp, o, lse = oracle_mod.decode_chunked(bits(q), bits(k), bits(v), FP16, chunk, scale)
    o_ref, l_ref = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, False, scale)
    assert np.abs(o - o_ref).max() < 1e-13
    assert np.abs(lse - l_ref[:, :, 0]).max() < 1e-12
    nc = -(-M // chunk)
    assert op.shape == (B, Hq, nc, d)
    # each partial is plain attention over its own chunk of keys
    for c in sorted({0, nc // 2, nc - 1}):
        j0, j1 = c * chunk, min(M, (c + 1) * chunk)
        oc, lc = oracle_mod.attention(bits(q), bits(k[:, j0:j1].contiguous()),
                                      bits(v[:, j0:j1].contiguous()), FP16, False, scale)
        assert np.abs(op[:, :, c] - oc[:, 0]).max() < 1e-13
        assert np.abs(lp[:, :, c] - lc[:, :, 0]).max() < 1e-12


# ---------------------------------------------------------------------------
# independent formulations on tiny inputs
# ---------------------------------------------------------------------------

def brute_force(qd, kd, vd, causal, scale):
    B, N, Hq, d = qd.shape
    _, M, Hkv, _ = kd.shape
    g = Hq // Hkv
    o = np.zeros_like(qd)
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            S = scale * qd[b, :, h] @ kd[b, :, h // g].T          # [N, M]
            E = np.exp(S)                                       # no max subtraction
            if causal:
                E = E * (np.arange(M)[None, :] <= np.arange(N)[:, None])
            o[b, :, h] = (E / E.sum(1, keepdims=True)) @ vd[b, :, h // g]
            lse[b, h] = np.log(E.sum(1))
    return o, lse


@pytest.mark.parametrize("shape", [(2, 2, 2, 17, 17, 4), (1, 4, 2, 5, 13, 64),
                                   (2, 2, 1, 16, 9, 64), (1, 1, 1, 1, 17, 4)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_brute_force_without_max_subtraction(oracle_mod, shape, causal, dtype):
    B, Hq, Hkv, N, M, d = shape
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, dtype, seed=20 + N + M)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attention(bits(q), bits(k), bits(v), dtype, causal, scale)
    qd, kd, vd = dec(oracle_mod, q, dtype), dec(oracle_mod, k, dtype), dec(oracle_mod, v, dtype)
    ob, lb = brute_force(qd, kd, vd, causal, scale)
    assert np.abs(o - ob).max() < 1e-12
    assert np.abs(lse - lb).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(oracle_mod, causal):
    B, Hq, Hkv, N, M, d = 2, 4, 2, 17, 17, 64
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, BF16, seed=21)
    o, _ = oracle_mod.attention(bits(q), bits(k), bits(v), BF16, causal, 1 / 8)
    g = Hq // Hkv
    qt = q.double().permute(0, 2, 1, 3)
    kt = k.double().repeat_interleave(g, dim=2).permute(0, 2, 1, 3)
    vt = v.double().repeat_interleave(g, dim=2).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                           scale=1 / 8)
    assert np.abs(o - ref.permute(0, 2, 1, 3).numpy()).max() < 1e-12


def test_rows_entry_matches_full(oracle_mod):
    B, Hq, Hkv, N, M, d = 2, 4, 2, 21, 21, 16
    q, k, v = make_inputs(B, Hq, Hkv, N, M, d, FP16, seed=22)
    o, lse = oracle_mod.attention(bits(q), bits(k), bits(v), FP16, True, 0.25)
    rows = np.array([(0, 0, 0), (1, 3, 20), (0, 2, 7), (1, 1, 13)])
    orr, lrr = oracle_mod.attention_rows(bits(q), bits(k), bits(v), FP16, True, 0.25, rows)
    for r, (b, h, i) in enumerate(rows):
        assert np.array_equal(orr[r], o[b, i, h])
        assert lrr[r] == lse[b, h, i]


# ---------------------------------------------------------------------------
# the measurement conventions, against the pages' printed numbers
# ---------------------------------------------------------------------------

def _rows(path):
    import os
    here = os.path.join(os.path.dirname(__file__), "golden", path)
    out = []
    with open(here) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                out.append(line.split())
    return out


def test_flop_convention_reproduces_printed_tflops():
    from exact_attention_05_gb300.workloads import Workload
    for seq, impl, ms, tflops in _rows("fmha_sm120_benchmark.txt"):
        w = Workload("t", "prefill", 1, 32, 32, int(seq), int(seq), 128, BF16, True, 1.0, 0)
        got = w.flops / (float(ms) * 1e-3) / 1e12
        assert abs(got - float(tflops)) < 0.006, (seq, impl, got, tflops)


def test_decode_byte_count_reproduces_printed_model():
    from exact_attention_05_gb300.workloads import Workload
    for d, mb, gbs, ms in _rows("flash_decoding_bandwidth.txt"):
        w = Workload("t", "decode", 2, 8, 8, 1, 65536, int(d), FP16, False, 1.0, 0, chunk=128)
        kv_bytes = w.decode_bytes - 2 * w.B * w.Hq * w.d * 2
        assert abs(kv_bytes / 1e6 - float(mb)) < 1.0
        assert abs(kv_bytes / (float(gbs) * 1e9) * 1e3 - float(ms)) < 0.01

"""CPU pins of the oracle's FP8 (e4m3) and paged K/V decode.

The FP8 KV cache and the paged ("kv cache block") cache are the next steps
named in the closing "TODO" section of "[CUDA 优化实战] fmha sm120 : 超越
torch.sdpa(flash-attention-2)"; lever 1 of section 8 of "CUDA 实现 Flash
Decoding：解码阶段并行度重建与性能剖析" is the FP8 cache.  Each oracle function is
tied to something other than itself: torch's own float8_e4m3fn conversion,
hand-computed values of the OCP E4M3 format, the 16-bit attention oracle (pinned
in test_oracle_pins.py) on inputs where both describe the same real numbers,
closed forms, and the contiguous layout recovered through a shuffled page pool.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_05_gb300 import workloads as W


def _bits16(t):
    return W.bits(t)


# ---- E4M3 decoding -----------------------------------------------------------


def test_e4m3_all_patterns_match_torch(oracle_mod):
    b = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.e4m3(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(mine, ref, equal_nan=True)


@pytest.mark.parametrize("byte,value", [
    (0x00, 0.0),                 # +0
    (0x38, 1.0),                 # exponent 7 = bias, mantissa 0
    (0x3C, 1.5),                 # mantissa 4/8
    (0x40, 2.0),
    (0x7E, 448.0),               # largest finite: 1.75 * 2^8
    (0x08, 2.0 ** -6),           # smallest normal
    (0x01, 2.0 ** -9),           # smallest subnormal: 1/8 * 2^-6
    (0x07, 7 * 2.0 ** -9),       # largest subnormal
    (0xB8, -1.0),
    (0xFE, -448.0),
])
def test_e4m3_hand_values(oracle_mod, byte, value):
    assert oracle_mod.e4m3(np.array([byte], np.uint8))[0] == value


def test_e4m3_nan_and_negative_zero(oracle_mod):
    v = oracle_mod.e4m3(np.array([0x7F, 0xFF, 0x80], np.uint8))
    assert math.isnan(v[0]) and math.isnan(v[1])
    assert v[2] == 0.0 and math.copysign(1.0, v[2]) < 0


# ---- FP8 decode ----------------------------------------------------------------


def _random_e4m3(gen, shape):
    """Random finite e4m3 bytes (NaN patterns 0x7f/0xff excluded)."""
    x = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32)
    x = torch.where((x & 0x7F) == 0x7F, x - 1, x)
    return x.to(torch.uint8)


def _dequant16(b8, scales):
    """k_scale[h] * e4m3(b8) as an fp16 tensor; exact when the scales are powers of two."""
    val = b8.view(torch.float8_e4m3fn).to(torch.float64) * scales.to(torch.float64).view(1, 1, -1, 1)
    t = val.to(torch.float16)
    assert torch.equal(t.to(torch.float64), val)  # exactly representable
    return t


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_fp8_decode_equals_16bit_oracle_on_exact_values(oracle_mod, Hq, Hkv):
    # Scales are powers of two and different per head and between K and V, so a
    # scale taken from the wrong head, or K's scale used for V, shows.
    gen = torch.Generator().manual_seed(31)
    B, M, d = 2, 50, 64
    q = torch.randn((B, 1, Hq, d), generator=gen).to(torch.float16)
    k8 = _random_e4m3(gen, (B, M, Hkv, d))
    v8 = _random_e4m3(gen, (B, M, Hkv, d))
    ks = torch.tensor([2.0 ** -(5 + h) for h in range(Hkv)], dtype=torch.float32)
    vs = torch.tensor([2.0 ** -(3 + 2 * h) for h in range(Hkv)], dtype=torch.float32)
    scale = 0.125
    o8, l8 = oracle_mod.decode_fp8(_bits16(q), k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy(),
                                   W.FP16, scale)
    k16, v16 = _dequant16(k8, ks), _dequant16(v8, vs)
    o16, l16 = oracle_mod.attention(_bits16(q), _bits16(k16), _bits16(v16), W.FP16, False, scale)
    np.testing.assert_allclose(o8, o16, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, l16[:, :, 0], rtol=0, atol=1e-12)


def test_fp8_decode_uniform_keys_closed_form(oracle_mod):
    # Every key row equal: softmax is uniform, O = mean_j V_j and
    # LSE = scale * q.k + ln M, with V dequantised by torch's own cast.
    gen = torch.Generator().manual_seed(32)
    B, M, Hq, Hkv, d = 1, 37, 2, 1, 64
    q = torch.randn((B, 1, Hq, d), generator=gen).to(torch.float16)
    row = _random_e4m3(gen, (d,))
    k8 = row.view(1, 1, 1, d).expand(B, M, Hkv, d).contiguous()
    v8 = _random_e4m3(gen, (B, M, Hkv, d))
    ks = torch.tensor([0.03], dtype=torch.float32)
    vs = torch.tensor([0.7], dtype=torch.float32)
    scale = 0.2
    o, lse = oracle_mod.decode_fp8(_bits16(q), k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy(),
                                   W.FP16, scale)
    kf = row.view(torch.float8_e4m3fn).to(torch.float64) * float(ks[0])
    vf = v8.view(torch.float8_e4m3fn).to(torch.float64) * float(vs[0])
    qf = q.to(torch.float64)
    for h in range(Hq):
        np.testing.assert_allclose(o[0, 0, h], vf[0, :, 0].mean(0).numpy(), rtol=0, atol=1e-12)
        want = scale * float(qf[0, 0, h] @ kf) + math.log(M)
        assert abs(lse[0, h] - want) < 1e-12


def test_fp8_quantiser_roundtrip_bounds():
    # The input recipe's quantiser: the largest magnitude of each head maps to
    # 448, and dequantised values are within half an e4m3 step (2^-4 relative
    # for normals) of the float32 input.
    gen = torch.Generator().manual_seed(33)
    x = torch.randn((2, 300, 3, 64), generator=gen)
    b8, s = W.quantize_e4m3(x)
    deq = b8.view(torch.float8_e4m3fn).to(torch.float32) * s.view(1, 1, -1, 1)
    for h in range(3):
        amax = x[:, :, h].abs().max()
        assert torch.isclose(s[h] * 448.0, amax, rtol=1e-6)
        err = (deq[:, :, h] - x[:, :, h]).abs()
        bound = torch.maximum(x[:, :, h].abs() * 2.0 ** -4, s[h] * 2.0 ** -10)
        assert bool((err <= bound * 1.0001).all())


# ---- paged decode --------------------------------------------------------------


@pytest.mark.parametrize("page", [1, 8, 16, 64])
def test_paged_decode_equals_contiguous(oracle_mod, page):
    gen = torch.Generator().manual_seed(40 + page)
    B, M, Hq, Hkv, d = 2, 100, 4, 2, 64
    q = torch.randn((B, 1, Hq, d), generator=gen).to(torch.bfloat16)
    k = torch.randn((B, M, Hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((B, M, Hkv, d), generator=gen).to(torch.bfloat16)
    kc, vc, bt = W.make_paged(k, v, page, seed=7, extra_pages=5)
    seq = np.full((B,), M, np.int32)
    o, lse = oracle_mod.decode_paged(_bits16(q), _bits16(kc), _bits16(vc), bt.numpy(), seq,
                                     W.BF16, M, 0.125)
    oc, lc = oracle_mod.attention(_bits16(q), _bits16(k), _bits16(v), W.BF16, False, 0.125)
    np.testing.assert_allclose(o, oc, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lc[:, :, 0], rtol=0, atol=1e-12)


def test_paged_decode_ragged_lengths_and_empty(oracle_mod):
    gen = torch.Generator().manual_seed(50)
    B, M, Hq, Hkv, d, page = 4, 80, 2, 2, 64, 16
    q = torch.randn((B, 1, Hq, d), generator=gen).to(torch.float16)
    k = torch.randn((B, M, Hkv, d), generator=gen).to(torch.float16)
    v = torch.randn((B, M, Hkv, d), generator=gen).to(torch.float16)
    kc, vc, bt = W.make_paged(k, v, page, seed=8)
    lens = [80, 17, 0, 1]
    o, lse = oracle_mod.decode_paged(_bits16(q), _bits16(kc), _bits16(vc), bt.numpy(),
                                     np.array(lens, np.int32), W.FP16, M, 0.1)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b]))
            continue
        ob, lb = oracle_mod.attention(_bits16(q[b:b + 1]), _bits16(k[b:b + 1, :L].contiguous()),
                                      _bits16(v[b:b + 1, :L].contiguous()), W.FP16, False, 0.1)
        np.testing.assert_allclose(o[b:b + 1], ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], lb[0, :, 0], rtol=0, atol=1e-12)
    # one key: O is that key's V row exactly, LSE its scaled logit
    vb = v[3, 0].to(torch.float64).numpy()
    np.testing.assert_array_equal(o[3, 0], np.stack([vb[h] for h in range(Hq)]))


def test_paged_decode_seq_len_clamped_to_max(oracle_mod):
    gen = torch.Generator().manual_seed(51)
    B, M, H, d, page = 1, 32, 1, 64, 8
    q = torch.randn((B, 1, H, d), generator=gen).to(torch.float16)
    k = torch.randn((B, M, H, d), generator=gen).to(torch.float16)
    v = torch.randn((B, M, H, d), generator=gen).to(torch.float16)
    kc, vc, bt = W.make_paged(k, v, page, seed=9)
    a = oracle_mod.decode_paged(_bits16(q), _bits16(kc), _bits16(vc), bt.numpy(),
                                np.array([1000], np.int32), W.FP16, M, 0.1)
    b = oracle_mod.decode_paged(_bits16(q), _bits16(kc), _bits16(vc), bt.numpy(),
                                np.array([M], np.int32), W.FP16, M, 0.1)
    np.testing.assert_array_equal(a[0], b[0])


def test_paged_decode_rejects_bad_table(oracle_mod):
    B, M, H, d, page = 1, 16, 1, 64, 8
    z = np.zeros((4, page, H, d), np.uint16)
    q = np.zeros((B, 1, H, d), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.decode_paged(q, z, z, np.array([[0, 4]], np.int32), np.array([M], np.int32),
                                W.FP16, M, 0.1)
    # the same bad entry is never read when the sequence ends before it
    oracle_mod.decode_paged(q, z, z, np.array([[0, 4]], np.int32), np.array([8], np.int32),
                            W.FP16, M, 0.1)

"""Seeded synthetic workloads shared by the tests, the bench and the smoke check.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it without sharing any of the method.

Recipe (the pages measure on random tensors, no dataset): one CPU
``torch.Generator`` per workload, seeded with the workload's seed; Q, K and V
are drawn in that order as iid N(0, 1) float32 and rounded to the workload's
16-bit type (round-to-nearest-even, ``Tensor.to``).  The "peaky" GQA prefill
workload additionally picks exactly floor(1% of B*M*Hkv) key rows -- a row is
one (b, m, h_kv) d-vector -- with a ``randperm`` drawn from the same generator
after V, and multiplies them by 8 in float32 before rounding.

FP8 K/V workloads (``kv="e4m3"``): K and V are drawn as above in float32 and
quantised per kv head the way a serving stack writes an FP8 cache: scale_h =
amax over that head's K (or V) values / 448 (the largest finite e4m3 value),
bytes = e4m3(x / scale_h) by torch's round-to-nearest-even cast, clamped to
+-448 first.  The attention kernels never see the float32 values, only the
bytes and the scales.

Paged workloads (``page > 0``): the contiguous K/V of a workload are cut into
pages of ``page`` keys and scattered to a random permutation of a pool of
pages (``randperm`` from the workload's generator, drawn after K and V); the
pool's unused pages, and the tail of a sequence's last page, hold N(0, 1)
noise so that a wrong gather cannot go unnoticed.  block_table [B,
pages_per_seq] int32 lists each sequence's pages in key order.

Layouts: q/o [B, N, Hq, d]; k/v [B, M, Hkv, d]; decode q/o [B, 1, Hq, d];
paged k/v cache [num_pages, page, Hkv, d].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

FP16 = 0
BF16 = 1
TORCH_DTYPE = {FP16: torch.float16, BF16: torch.bfloat16}
DTYPE_NAME = {FP16: "f16", BF16: "bf16"}


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" or "decode"
    B: int
    Hq: int
    Hkv: int
    N: int               # query rows per (b, h); 1 for decode
    M: int               # keys per (b, h_kv)
    d: int
    dtype: int
    causal: bool
    scale: float
    seed: int
    chunk: int = 0       # decode only
    peaky_frac: float = 0.0
    kv: str = "16bit"    # decode K/V format: "16bit" (dtype) or "e4m3"
    page: int = 0        # decode: keys per page of a paged cache (0 = contiguous K/V)
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H*N*M*d, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.M * self.d
        return f / 2.0 if self.causal else f

    @property
    def decode_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode call: K and V once per kv head, plus q and o."""
        esz = 1 if self.kv == "e4m3" else 2
        kv = 2 * self.B * self.Hkv * self.M * self.d * esz
        qo = 2 * self.B * self.Hq * self.d * 2
        extra = 0
        if self.kv == "e4m3":
            extra += 2 * self.Hkv * 4                       # k_scale, v_scale
        if self.page > 0:
            extra += self.B * (-(-self.M // self.page)) * 4 + self.B * 4  # block table, seq_lens
        return kv + qo + extra


INV_SQRT_64 = 1.0 / math.sqrt(64.0)
INV_SQRT_128 = 1.0 / math.sqrt(128.0)

# The five workloads the pages' measurements are shaped like (seeds fixed).
WORKLOADS = {
    "prefill_mha_n256_d64_f16": Workload(
        "prefill_mha_n256_d64_f16", "prefill", 1, 2, 2, 256, 256, 64, FP16, False,
        INV_SQRT_64, 1001, note="non-causal MHA, O and LSE"),
    "prefill_causal_b2_h16_n2048_bf16": Workload(
        "prefill_causal_b2_h16_n2048_bf16", "prefill", 2, 16, 16, 2048, 2048, 128, BF16, True,
        INV_SQRT_128, 1002, note="causal MHA"),
    "prefill_causal_gqa32x8_n8192_f16_peaky": Workload(
        "prefill_causal_gqa32x8_n8192_f16_peaky", "prefill", 1, 32, 8, 8192, 8192, 128, FP16,
        True, INV_SQRT_128, 1003, peaky_frac=0.01,
        note="causal GQA, 1% of K rows x8"),
    "prefill_causal_h16_n32768_bf16": Workload(
        "prefill_causal_h16_n32768_bf16", "prefill", 1, 16, 16, 32768, 32768, 128, BF16, True,
        INV_SQRT_128, 1004, note="long causal MHA"),
    "decode_b2_h8_m65536_f16": Workload(
        "decode_b2_h8_m65536_f16", "decode", 2, 8, 8, 1, 65536, 128, FP16, False,
        INV_SQRT_128, 1005, chunk=128, note="split-KV decode, chunk 128"),
    "decode_b1_h8_m512_f16": Workload(
        "decode_b1_h8_m512_f16", "decode", 1, 8, 8, 1, 512, 128, FP16, False,
        INV_SQRT_128, 1005, chunk=128, note="split-KV decode, small case"),
    "decode_fp8_b2_h8_m65536_f16": Workload(
        "decode_fp8_b2_h8_m65536_f16", "decode", 2, 8, 8, 1, 65536, 128, FP16, False,
        INV_SQRT_128, 1006, chunk=128, kv="e4m3",
        note="split-KV decode over e4m3 K/V with per-kv-head scales, chunk 128"),
    "decode_paged_b2_h8_m65536_p16_f16": Workload(
        "decode_paged_b2_h8_m65536_p16_f16", "decode", 2, 8, 8, 1, 65536, 128, FP16, False,
        INV_SQRT_128, 1007, chunk=128, page=16,
        note="split-KV decode over a paged cache, 16-key pages in shuffled order, chunk 128"),
}

E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor):
    """Per-kv-head e4m3 bytes and fp32 scales of a float32 [B, M, Hkv, d] tensor:
    returns (uint8 [B, M, Hkv, d], float32 [Hkv])."""
    Hkv = x.shape[2]
    amax = x.abs().permute(2, 0, 1, 3).reshape(Hkv, -1).amax(dim=1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    y = (x / scale.view(1, 1, Hkv, 1)).clamp(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), scale.contiguous()


def make_fp8_decode_inputs(B, Hq, Hkv, M, d, dtype, seed):
    """q [B,1,Hq,d] of the 16-bit dtype; k8, v8 uint8 [B,M,Hkv,d]; k_scale, v_scale [Hkv]."""
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, 1, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, M, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, M, Hkv, d), generator=g, dtype=torch.float32)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    return q.to(TORCH_DTYPE[dtype]), k8, v8, ks, vs


def make_paged(k: torch.Tensor, v: torch.Tensor, page: int, seed: int, extra_pages: int = 0):
    """Scatters contiguous k/v [B, M, Hkv, d] into a shuffled pool of pages.
    Returns (k_cache, v_cache [num_pages, page, Hkv, d], block_table int32
    [B, ceil(M / page)])."""
    B, M, Hkv, d = k.shape
    per_seq = -(-M // page)
    num_pages = B * per_seq + extra_pages
    g = torch.Generator().manual_seed(int(seed))
    perm = torch.randperm(num_pages, generator=g)[:B * per_seq].view(B, per_seq)
    caches = []
    for x in (k, v):
        pool = torch.randn((num_pages, page, Hkv, d), generator=g, dtype=torch.float32).to(x.dtype)
        pad = torch.randn((B, per_seq * page, Hkv, d), generator=g, dtype=torch.float32).to(x.dtype)
        pad[:, :M] = x
        pool[perm.reshape(-1)] = pad.view(B * per_seq, page, Hkv, d)
        caches.append(pool.contiguous())
    return caches[0], caches[1], perm.to(torch.int32).contiguous()


def workload_decode_inputs(w: Workload):
    """All host tensors of a decode workload, by name: q, k, v (contiguous, the
    16-bit or e4m3 bytes), k_scale/v_scale (e4m3), k_cache, v_cache,
    block_table, seq_lens (paged)."""
    if w.kv == "e4m3":
        q, k8, v8, ks, vs = make_fp8_decode_inputs(w.B, w.Hq, w.Hkv, w.M, w.d, w.dtype, w.seed)
        out = {"q": q, "k": k8, "v": v8, "k_scale": ks, "v_scale": vs}
    else:
        q, k, v = make_inputs(w.B, w.Hq, w.Hkv, 1, w.M, w.d, w.dtype, w.seed)
        out = {"q": q, "k": k, "v": v}
    if w.page > 0:
        kc, vc, bt = make_paged(out["k"], out["v"], w.page, w.seed + 1)
        out.update(k_cache=kc, v_cache=vc, block_table=bt,
                   seq_lens=torch.full((w.B,), w.M, dtype=torch.int32))
    return out


def make_inputs(B, Hq, Hkv, N, M, d, dtype, seed, peaky_frac=0.0):
    """Host (CPU) tensors q [B,N,Hq,d], k/v [B,M,Hkv,d] of the 16-bit dtype."""
    g = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPE[dtype]
    q = torch.randn((B, N, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, M, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, M, Hkv, d), generator=g, dtype=torch.float32)
    if peaky_frac > 0.0:
        nrows = B * M * Hkv
        count = int(math.floor(peaky_frac * nrows))
        pick = torch.randperm(nrows, generator=g)[:count]
        kr = k.view(nrows, d)
        kr[pick] *= 8.0
    return q.to(tdt), k.to(tdt), v.to(tdt)


def make_dout(B, N, Hq, d, dtype, seed):
    """Upstream gradient dO [B, N, Hq, d] for the backward: iid N(0, 1) float32
    from its own generator, rounded to the 16-bit dtype."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn((B, N, Hq, d), generator=g, dtype=torch.float32).to(TORCH_DTYPE[dtype])


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.Hq, w.Hkv, w.N, w.M, w.d, w.dtype, w.seed, w.peaky_frac)


def bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a CPU fp16/bf16 tensor, as numpy.uint16."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, count: int, seed: int = 7) -> np.ndarray:
    """Deterministic (b, h, i) query rows: first and last rows of every head, plus random ones."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        for h in range(w.Hq):
            rows.append((b, h, 0))
            rows.append((b, h, w.N - 1))
    extra = max(0, count - len(rows))
    if extra:
        rows.extend(zip(rng.integers(0, w.B, extra), rng.integers(0, w.Hq, extra),
                        rng.integers(0, w.N, extra)))
    return np.asarray(rows[:max(count, 2 * w.B * w.Hq)], dtype=np.int64)

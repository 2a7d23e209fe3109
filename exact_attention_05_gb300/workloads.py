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

Layouts: q/o [B, N, Hq, d]; k/v [B, M, Hkv, d]; decode q/o [B, 1, Hq, d].
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
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H*N*M*d, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.M * self.d
        return f / 2.0 if self.causal else f

    @property
    def decode_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode call: K and V once per kv head, plus q and o."""
        esz = 2
        kv = 2 * self.B * self.Hkv * self.M * self.d * esz
        qo = 2 * self.B * self.Hq * self.d * esz
        return kv + qo


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
}


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

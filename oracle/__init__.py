"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  The CUDA library never calls it and shares no code
with it.  The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over
query-row blocks); this module compiles it with gcc and marshals numpy arrays.

Every function takes the raw 16-bit patterns of the inputs (``numpy.uint16``
arrays, fp16 when ``dtype == 0``, bfloat16 when ``dtype == 1``) and decodes
them itself, so the oracle sees exactly the values the GPU path sees.

Definitions followed (see ``oracle.c`` for the passage each one restates):
softmax attention with materialised S and P ("[CUDA 优化实战] fmha sm120",
section 1), top-left causal mask and GQA head mapping (same page, section 2),
natural-log LSE of the scaled logits and the chunk-partial + LSE-weighted
merge of split-KV decoding ("CUDA 实现 Flash Decoding", section 2.2); the
OCP E4M3 decoding of an FP8 K/V cache and the block-table gather of a paged
cache (the fmha sm120 page's closing "TODO" section; lever 1 of the Flash
Decoding page's section 8).  The e4m3 functions take the raw bytes
(``numpy.uint8``) and fp32 per-kv-head scales.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FP16 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP if available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        I, D = ctypes.c_int, ctypes.c_double
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = D
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D
        lib.oracle_attention.argtypes = [u16p, u16p, u16p, I, I, I, I, I, I, I, I, D,
                                         f64p, f64p, f64p]
        lib.oracle_attention.restype = I
        lib.oracle_attention_rows.argtypes = [u16p, u16p, u16p, I, I, I, I, I, I, I, I, D,
                                              i64p, I, f64p, f64p]
        lib.oracle_attention_rows.restype = I
        lib.oracle_decode_chunked.argtypes = [u16p, u16p, u16p, I, I, I, I, I, I, I, D,
                                              f64p, f64p, f64p, f64p]
        lib.oracle_decode_chunked.restype = I
        lib.oracle_attention_backward.argtypes = [u16p, u16p, u16p, u16p, I, I, I, I, I, I, I,
                                                  I, D, f64p, f64p, f64p]
        lib.oracle_attention_backward.restype = I
        lib.oracle_attention_backward_dq_rows.argtypes = [u16p, u16p, u16p, u16p, I, I, I, I, I,
                                                          I, I, I, D, i64p, I, f64p]
        lib.oracle_attention_backward_dq_rows.restype = I
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        i32p = ctypes.POINTER(ctypes.c_int32)
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = D
        lib.oracle_decode_fp8.argtypes = [u16p, u8p, u8p, f32p, f32p, I, I, I, I, I, I, D,
                                          f64p, f64p]
        lib.oracle_decode_fp8.restype = I
        lib.oracle_decode_paged.argtypes = [u16p, u16p, u16p, i32p, i32p, I, I, I, I, I, I, I,
                                            I, I, D, f64p, f64p]
        lib.oracle_decode_paged.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        lib.oracle_set_num_threads.argtypes = [I]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _u16(a: np.ndarray):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are raw 16-bit patterns (numpy.uint16)")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _f64(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact fp64 value of each 16-bit pattern (the oracle's own decoder)."""
    lib = _load()
    fn = lib.oracle_fp16_to_double if dtype == FP16 else lib.oracle_bf16_to_double
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([fn(int(x)) for x in flat], dtype=np.float64).reshape(np.shape(bits))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def attention(q, k, v, dtype, causal, scale, with_probs=False):
    """Exact attention of q [B,N,Hq,d] against k/v [B,M,Hkv,d] (uint16 bit arrays).

    Returns (O [B,N,Hq,d] fp64, LSE [B,Hq,N] fp64) and, with ``with_probs``,
    the materialised P [B,Hq,N,M] as a third element.
    """
    lib = _load()
    B, N, Hq, d = q.shape
    Bk, M, Hkv, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch")
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    o = np.zeros((B, N, Hq, d), np.float64)
    lse = np.zeros((B, Hq, N), np.float64)
    probs = np.zeros((B, Hq, N, M), np.float64) if with_probs else None
    rc = lib.oracle_attention(qp, kp, vp, int(dtype), B, Hq, Hkv, N, M, d, int(bool(causal)),
                              float(scale), _f64(o), _f64(lse), _f64(probs))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return (o, lse, probs) if with_probs else (o, lse)


def attention_rows(q, k, v, dtype, causal, scale, rows):
    """The same definition for selected query rows only.

    ``rows`` is an int array [R, 3] of (b, h, i).  Returns (O [R, d], LSE [R]).
    """
    lib = _load()
    B, N, Hq, d = q.shape
    _, M, Hkv, _ = k.shape
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    o = np.zeros((rows.shape[0], d), np.float64)
    lse = np.zeros((rows.shape[0],), np.float64)
    rc = lib.oracle_attention_rows(qp, kp, vp, int(dtype), B, Hq, Hkv, N, M, d, int(bool(causal)),
                                   float(scale),
                                   rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   rows.shape[0], _f64(o), _f64(lse))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return o, lse


def decode_chunked(q, k, v, dtype, chunk, scale):
    """Split-KV decode: q [B,1,Hq,d], k/v [B,M,Hkv,d].

    Returns (O_part [B,Hq,nc,d], lse_part [B,Hq,nc], O [B,1,Hq,d], LSE [B,Hq]).
    """
    lib = _load()
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes a single query row per head")
    _, M, Hkv, _ = k.shape
    nc = -(-M // chunk)
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    op = np.zeros((B, Hq, nc, d), np.float64)
    lp = np.zeros((B, Hq, nc), np.float64)
    o = np.zeros((B, 1, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.oracle_decode_chunked(qp, kp, vp, int(dtype), B, Hq, Hkv, M, d, int(chunk),
                                   float(scale), _f64(op), _f64(lp), _f64(o), _f64(lse))
    if rc != 0:
        raise ValueError("oracle_decode_chunked rejected its arguments")
    return op, lp, o, lse


def attention_backward(q, k, v, dout, dtype, causal, scale):
    """Gradients of exact attention: q, dout [B,N,Hq,d], k/v [B,M,Hkv,d] (uint16
    bit arrays).  Returns (dQ [B,N,Hq,d], dK [B,M,Hkv,d], dV [B,M,Hkv,d]) fp64."""
    lib = _load()
    B, N, Hq, d = q.shape
    _, M, Hkv, _ = k.shape
    if dout.shape != q.shape or k.shape != v.shape:
        raise ValueError("shape mismatch")
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    dout, dp = _u16(dout)
    dq = np.zeros((B, N, Hq, d), np.float64)
    dk = np.zeros((B, M, Hkv, d), np.float64)
    dv = np.zeros((B, M, Hkv, d), np.float64)
    rc = lib.oracle_attention_backward(qp, kp, vp, dp, int(dtype), B, Hq, Hkv, N, M, d,
                                       int(bool(causal)), float(scale), _f64(dq), _f64(dk),
                                       _f64(dv))
    if rc != 0:
        raise ValueError("oracle_attention_backward rejected its arguments")
    return dq, dk, dv


def attention_backward_dq_rows(q, k, v, dout, dtype, causal, scale, rows):
    """dQ of selected query rows: ``rows`` is an int array [R, 3] of (b, h, i).
    Returns dQ [R, d] fp64 (the same definition as attention_backward)."""
    lib = _load()
    B, N, Hq, d = q.shape
    _, M, Hkv, _ = k.shape
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    dout, dp = _u16(dout)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    out = np.zeros((rows.shape[0], d), np.float64)
    rc = lib.oracle_attention_backward_dq_rows(
        qp, kp, vp, dp, int(dtype), B, Hq, Hkv, N, M, d, int(bool(causal)), float(scale),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.shape[0], _f64(out))
    if rc != 0:
        raise ValueError("oracle_attention_backward_dq_rows rejected its arguments")
    return out


def e4m3(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 value of each e4m3 byte (the oracle's own decoder)."""
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_double(int(x)) for x in flat],
                    dtype=np.float64).reshape(np.shape(bits))


def _typed(a, dt, ct, what):
    a = np.ascontiguousarray(a)
    if a.dtype != dt:
        raise TypeError(f"{what} must be {np.dtype(dt).name}")
    return a, a.ctypes.data_as(ctypes.POINTER(ct))


def decode_fp8(q, k8, v8, k_scale, v_scale, dtype, scale):
    """Decode of q [B,1,Hq,d] (uint16 bits) over e4m3 bytes k8/v8 [B,M,Hkv,d]
    (uint8) with float32 scales [Hkv].  Returns (O [B,1,Hq,d], LSE [B,Hq])."""
    lib = _load()
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes a single query row per head")
    _, M, Hkv, _ = k8.shape
    q, qp = _u16(q)
    k8, kp = _typed(k8, np.uint8, ctypes.c_uint8, "k8")
    v8, vp = _typed(v8, np.uint8, ctypes.c_uint8, "v8")
    ks, ksp = _typed(k_scale, np.float32, ctypes.c_float, "k_scale")
    vs, vsp = _typed(v_scale, np.float32, ctypes.c_float, "v_scale")
    if ks.shape != (Hkv,) or vs.shape != (Hkv,):
        raise ValueError("scales are [Hkv]")
    o = np.zeros((B, 1, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.oracle_decode_fp8(qp, kp, vp, ksp, vsp, int(dtype), B, Hq, Hkv, M, d, float(scale),
                               _f64(o), _f64(lse))
    if rc != 0:
        raise ValueError("oracle_decode_fp8 rejected its arguments")
    return o, lse


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, dtype, max_seq_len, scale):
    """Decode of q [B,1,Hq,d] over a paged cache k/v [num_pages, page, Hkv, d]
    (uint16 bits) through block_table [B, max_pages] and seq_lens [B] (int32).
    Returns (O [B,1,Hq,d], LSE [B,Hq]); an empty sequence gives O = 0, LSE = -inf."""
    lib = _load()
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes a single query row per head")
    num_pages, page, Hkv, _ = k_cache.shape
    q, qp = _u16(q)
    kc, kp = _u16(k_cache)
    vc, vp = _u16(v_cache)
    bt, btp = _typed(block_table, np.int32, ctypes.c_int32, "block_table")
    sl, slp = _typed(seq_lens, np.int32, ctypes.c_int32, "seq_lens")
    if bt.ndim != 2 or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("block_table is [B, max_pages], seq_lens [B]")
    o = np.zeros((B, 1, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.oracle_decode_paged(qp, kp, vp, btp, slp, int(dtype), B, Hq, Hkv, int(max_seq_len),
                                 num_pages, page, bt.shape[1], d, float(scale), _f64(o),
                                 _f64(lse))
    if rc != 0:
        raise ValueError("oracle_decode_paged rejected its arguments")
    return o, lse

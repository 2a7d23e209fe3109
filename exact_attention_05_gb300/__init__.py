"""Thin Python binding of libfa.so, the GB300 exact-attention C ABI (include/fa.h).

Only argument marshalling happens here: every step of the attention runs in the
library's CUDA kernels.  PyTorch is used for device memory and streams.  There
is no fallback: if the library is not built, every call raises.

The functions mirror the C entry points one to one (``fa_fwd``, ``fa_decode``,
``fa_status_string``, ``fa_get_last_device_status``, ...); pointer arguments
accept a torch tensor (its ``data_ptr()``), an int address, or None, and the
stream argument accepts a ``torch.cuda.Stream``, an int handle, or None for
torch's current stream.  ``attention_forward`` and ``decode`` are shape-checked
conveniences that allocate the outputs and call the same entry points.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from .workloads import BF16, FP16

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libfa.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_NO_MEMORY = 4
FA_ERR_TIMEOUT = 5
FA_ERR_SCRATCH_LIMIT = 6

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} ({status})")


def header_functions() -> list[str]:
    """Names of the functions include/fa.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(fa_\w+)\s*\(", text, flags=re.M)))


def load_library():
    """Loads libfa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with exact_attention_05_gb300.build.build() "
                "(the attention path has no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, fp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        I, F = ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, fp, I, I, I, I, I, I, I, F, I, vp]
        lib.fa_fwd.restype = I
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, fp, I, I, I, I, I, I, I, F, I, vp]
        lib.fa_fwd_host.restype = I
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, I, I, I, I, I, I, I, F, I, vp]
        lib.fa_bwd.restype = I
        lib.fa_decode.argtypes = [vp, vp, vp, vp, fp, I, I, I, I, I, I, F, I, vp]
        lib.fa_decode.restype = I
        lib.fa_decode_fused.argtypes = [vp, vp, vp, vp, fp, I, I, I, I, I, I, F, I, vp]
        lib.fa_decode_fused.restype = I
        lib.fa_decode_noalloc.argtypes = [vp, vp, vp, vp, fp, I, I, I, I, I, I, F, I, vp]
        lib.fa_decode_noalloc.restype = I
        lib.fa_decode_fp8.argtypes = [vp, vp, vp, fp, fp, vp, fp, I, I, I, I, I, I, F, I, vp]
        lib.fa_decode_fp8.restype = I
        lib.fa_decode_paged.argtypes = [vp, vp, vp, ip, ip, vp, fp, I, I, I, I, I, I, I, I, I, F,
                                        I, vp]
        lib.fa_decode_paged.restype = I
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_get_last_device_status.argtypes = [vp]
        lib.fa_get_last_device_status.restype = I
        lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        lib.fa_set_wait_timeout_ns.restype = None
        lib.fa_selftest_wait_timeout.argtypes = [vp]
        lib.fa_selftest_wait_timeout.restype = I
        lib.fa_release_workspaces.argtypes = []
        lib.fa_release_workspaces.restype = None
        lib.fa_abi_version.argtypes = []
        lib.fa_abi_version.restype = I
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> int:
    if status != FA_OK:
        raise FAError(status, where)
    return status


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, M, d, causal, scale, dtype, stream=None,
           check=True) -> int:
    st = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                               int(Hkv), int(N), int(M), int(d), int(causal), float(scale),
                               int(dtype), _stream(stream))
    return _check(st, "fa_fwd") if check else st


def fa_fwd_host(q, k, v, o, lse, B, Hq, Hkv, N, M, d, causal, scale, dtype, stream=None,
                check=True) -> int:
    """fa_fwd on host (CPU, preferably pinned) tensors, transfers overlapped with
    the kernels; synchronize `stream` before reading o and lse."""
    st = load_library().fa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                    int(Hq), int(Hkv), int(N), int(M), int(d), int(causal),
                                    float(scale), int(dtype), _stream(stream))
    return _check(st, "fa_fwd_host") if check else st


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, M, d, causal, scale, dtype,
           stream=None, check=True) -> int:
    """Backward of fa_fwd: dq [B,N,Hq,d], dk/dv [B,M,Hkv,d] from dout and the
    forward's o and lse."""
    st = load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                               _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(N),
                               int(M), int(d), int(causal), float(scale), int(dtype),
                               _stream(stream))
    return _check(st, "fa_bwd") if check else st


def fa_decode(q, k, v, o, lse, B, Hq, Hkv, M, d, chunk, scale, dtype, stream=None,
              check=True) -> int:
    st = load_library().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                                  int(Hkv), int(M), int(d), int(chunk), float(scale), int(dtype),
                                  _stream(stream))
    return _check(st, "fa_decode") if check else st


def fa_decode_fused(q, k, v, o, lse, B, Hq, Hkv, M, d, chunk, scale, dtype, stream=None,
                    check=True) -> int:
    """fa_decode in one launch: the chunk kernel merges its own partials."""
    st = load_library().fa_decode_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                        int(Hq), int(Hkv), int(M), int(d), int(chunk),
                                        float(scale), int(dtype), _stream(stream))
    return _check(st, "fa_decode_fused") if check else st


def fa_decode_noalloc(q, k, v, o, lse, B, Hq, Hkv, M, d, chunk, scale, dtype, stream=None,
                      check=True) -> int:
    """fa_decode with its partials in the library's static device scratch: for
    callers that cannot allocate device memory (no cudaMalloc is made)."""
    st = load_library().fa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                          int(Hq), int(Hkv), int(M), int(d), int(chunk),
                                          float(scale), int(dtype), _stream(stream))
    return _check(st, "fa_decode_noalloc") if check else st


def fa_decode_fp8(q, k8, v8, k_scale, v_scale, o, lse, B, Hq, Hkv, M, d, chunk, scale, dtype,
                  stream=None, check=True) -> int:
    """Split-KV decode over e4m3 K/V bytes with fp32 per-kv-head scales."""
    st = load_library().fa_decode_fp8(_ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale),
                                      _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(M),
                                      int(d), int(chunk), float(scale), int(dtype),
                                      _stream(stream))
    return _check(st, "fa_decode_fp8") if check else st


def fa_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, max_seq_len,
                    num_pages, page_size, max_pages_per_seq, d, chunk, scale, dtype, stream=None,
                    check=True) -> int:
    """Split-KV decode over a paged K/V cache [num_pages, page_size, Hkv, d]
    addressed through block_table [B, max_pages_per_seq] and seq_lens [B]."""
    st = load_library().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                        _ptr(seq_lens), _ptr(o), _ptr(lse), int(B), int(Hq),
                                        int(Hkv), int(max_seq_len), int(num_pages),
                                        int(page_size), int(max_pages_per_seq), int(d),
                                        int(chunk), float(scale), int(dtype), _stream(stream))
    return _check(st, "fa_decode_paged") if check else st


def fa_get_last_device_status(stream=None) -> int:
    return load_library().fa_get_last_device_status(_stream(stream))


def fa_set_wait_timeout_ns(ns: int) -> None:
    load_library().fa_set_wait_timeout_ns(int(ns))


def fa_selftest_wait_timeout(stream=None) -> int:
    return load_library().fa_selftest_wait_timeout(_stream(stream))


def fa_release_workspaces() -> None:
    load_library().fa_release_workspaces()


def fa_abi_version() -> int:
    return load_library().fa_abi_version()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FP16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: fp16 or bf16")


def attention_forward(q, k, v, causal: bool, scale: float, out=None, lse=None, with_lse=True,
                      stream=None):
    """O (and LSE) of q [B,N,Hq,d] against k/v [B,M,Hkv,d], all contiguous CUDA tensors."""
    import torch
    B, N, Hq, d = q.shape
    _, M, Hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    for t in (q, k, v, out):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    fa_fwd(q, k, v, out, lse, B, Hq, Hkv, N, M, d, int(bool(causal)), scale, _dtype_code(q),
           stream)
    return out, lse


def attention_forward_host(q, k, v, causal: bool, scale: float, out=None, lse=None,
                           with_lse=True, stream=None):
    """attention_forward on CPU tensors (pin them for the transfers to overlap the
    kernels): returns pinned CPU O [B,N,Hq,d] and LSE [B,Hq,N], complete once
    `stream` (default: the current CUDA stream) is synchronized."""
    import torch
    B, N, Hq, d = q.shape
    _, M, Hkv, _ = k.shape
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=True)
    for t in (q, k, v, out):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CPU tensors")
    fa_fwd_host(q, k, v, out, lse, B, Hq, Hkv, N, M, d, int(bool(causal)), scale, _dtype_code(q),
                stream)
    return out, lse


def decode(q, k, v, chunk: int, scale: float, out=None, lse=None, with_lse=True, stream=None,
           single_launch=False):
    """Split-KV decode of q [B,1,Hq,d] against k/v [B,M,Hkv,d] (fa_decode, or
    fa_decode_fused with ``single_launch``)."""
    import torch
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes q of shape [B, 1, Hq, d]")
    _, M, Hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    fn = fa_decode_fused if single_launch else fa_decode
    fn(q, k, v, out, lse, B, Hq, Hkv, M, d, chunk, scale, _dtype_code(q), stream)
    return out, lse


def decode_fp8(q, k8, v8, k_scale, v_scale, chunk: int, scale: float, out=None, lse=None,
               with_lse=True, stream=None):
    """Split-KV decode of q [B,1,Hq,d] against e4m3 k8/v8 [B,M,Hkv,d] (torch.uint8
    or torch.float8_e4m3fn) with fp32 scales [Hkv]: K = k_scale[h] * k8, V = v_scale[h] * v8."""
    import torch
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes q of shape [B, 1, Hq, d]")
    _, M, Hkv, _ = k8.shape
    for t in (k8, v8):
        if t.element_size() != 1:
            raise TypeError("k8 and v8 hold one byte per element")
    for t in (q, k8, v8, k_scale, v_scale):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("scales are float32")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    fa_decode_fp8(q, k8, v8, k_scale, v_scale, out, lse, B, Hq, Hkv, M, d, chunk, scale,
                  _dtype_code(q), stream)
    return out, lse


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, chunk: int,
                 scale: float, out=None, lse=None, with_lse=True, stream=None):
    """Split-KV decode of q [B,1,Hq,d] against a paged cache k_cache/v_cache
    [num_pages, page_size, Hkv, d] through block_table [B, max_pages_per_seq]
    and seq_lens [B] (both int32 on the device)."""
    import torch
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("decode takes q of shape [B, 1, Hq, d]")
    num_pages, page_size, Hkv, _ = k_cache.shape
    for t in (block_table, seq_lens):
        if t.dtype != torch.int32:
            raise TypeError("block_table and seq_lens are int32")
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    fa_decode_paged(q, k_cache, v_cache, block_table, seq_lens, out, lse, B, Hq, Hkv, max_seq_len,
                    num_pages, page_size, block_table.shape[1], d, chunk, scale, _dtype_code(q),
                    stream)
    return out, lse


def attention_backward(q, k, v, o, lse, dout, causal: bool, scale: float, dq=None, dk=None,
                       dv=None, stream=None):
    """dQ, dK, dV of attention_forward(q, k, v, causal, scale) -> (o, lse) for the
    upstream gradient dout [B,N,Hq,d]; all contiguous CUDA tensors."""
    import torch
    B, N, Hq, d = q.shape
    _, M, Hkv, _ = k.shape
    for t in (q, k, v, o, lse, dout):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, M, d, int(bool(causal)), scale,
           _dtype_code(q), stream)
    return dq, dk, dv

"""Host-side checks of the C ABI that need no GPU.

The library must build, load, export every function include/fa.h declares, and
turn every invalid argument into its documented status code before it makes
any CUDA call (all calls here are rejected by the argument checks, so none of
them reaches the driver).
"""
import ctypes
import subprocess

import pytest

import exact_attention_05_gb300 as fa
from exact_attention_05_gb300 import build as fa_build

GOOD = 0x100000          # a 16-byte aligned fake address; never dereferenced
MIS = 0x100008           # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def test_exports_every_declared_function(lib):
    names = fa.header_functions()
    assert {"fa_fwd", "fa_decode", "fa_status_string", "fa_get_last_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported
    # nothing but the C ABI leaks out of the library (the CUDA runtime is static and hidden)
    assert {n for n in exported if not n.startswith("fa_")} <= {"_init", "_fini"}


def test_status_strings(lib):
    for code in range(6):
        assert fa.fa_status_string(code)
    assert fa.fa_status_string(99) == "unknown fa_status"
    assert fa.fa_abi_version() == 1


def fwd(**kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=None, B=1, Hq=2, Hkv=2, N=128, M=128, d=128,
                causal=0, scale=0.1, dtype=0)
    args.update(kw)
    return fa.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                     args["Hq"], args["Hkv"], args["N"], args["M"], args["d"], args["causal"],
                     args["scale"], args["dtype"], stream=0, check=False)


def fwd_host(**kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=None, B=1, Hq=2, Hkv=2, N=128, M=128, d=128,
                causal=0, scale=0.1, dtype=0)
    args.update(kw)
    return fa.fa_fwd_host(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                          args["Hq"], args["Hkv"], args["N"], args["M"], args["d"], args["causal"],
                          args["scale"], args["dtype"], stream=0, check=False)


def dec(**kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=None, B=1, Hq=2, Hkv=2, M=128, d=128,
                chunk=128, scale=0.1, dtype=0)
    args.update(kw)
    return fa.fa_decode(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                        args["Hq"], args["Hkv"], args["M"], args["d"], args["chunk"],
                        args["scale"], args["dtype"], stream=0, check=False)


def bwd(**kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=GOOD, do=GOOD, dq=GOOD, dk=GOOD, dv=GOOD, B=1,
                Hq=2, Hkv=2, N=128, M=128, d=128, causal=0, scale=0.1, dtype=0)
    args.update(kw)
    return fa.fa_bwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["do"],
                     args["dq"], args["dk"], args["dv"], args["B"], args["Hq"], args["Hkv"],
                     args["N"], args["M"], args["d"], args["causal"], args["scale"], args["dtype"],
                     stream=0, check=False)


def dec8(**kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, ks=GOOD, vs=GOOD, o=GOOD, lse=None, B=1, Hq=2, Hkv=2,
                M=128, d=128, chunk=128, scale=0.1, dtype=0)
    args.update(kw)
    return fa.fa_decode_fp8(args["q"], args["k"], args["v"], args["ks"], args["vs"], args["o"],
                            args["lse"], args["B"], args["Hq"], args["Hkv"], args["M"], args["d"],
                            args["chunk"], args["scale"], args["dtype"], stream=0, check=False)


def decp(**kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, bt=GOOD, sl=GOOD, o=GOOD, lse=None, B=1, Hq=2, Hkv=2,
                M=128, num_pages=8, page=16, max_pages=8, d=128, chunk=128, scale=0.1, dtype=0)
    args.update(kw)
    return fa.fa_decode_paged(args["q"], args["k"], args["v"], args["bt"], args["sl"], args["o"],
                              args["lse"], args["B"], args["Hq"], args["Hkv"], args["M"],
                              args["num_pages"], args["page"], args["max_pages"], args["d"],
                              args["chunk"], args["scale"], args["dtype"], stream=0, check=False)


@pytest.mark.parametrize("call", [fwd, fwd_host, dec, dec8, decp, bwd])
@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=None), fa.FA_ERR_INVALID_ARG),
    (dict(v=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(M=0), fa.FA_ERR_INVALID_ARG),
    (dict(M=-5), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), fa.FA_ERR_INVALID_ARG),
    (dict(d=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=-1), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q=MIS), fa.FA_ERR_INVALID_ARG),
    (dict(k=MIS), fa.FA_ERR_INVALID_ARG),
    (dict(v=MIS), fa.FA_ERR_INVALID_ARG),
    (dict(o=MIS), fa.FA_ERR_INVALID_ARG),
    (dict(lse=GOOD + 2), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 20, Hq=1 << 10, Hkv=1 << 10), fa.FA_ERR_INVALID_ARG),   # > 2^39 elements
])
def test_invalid_arguments(lib, call, kw, code):
    assert call(**kw) == code


@pytest.mark.parametrize("kw", [dict(N=0), dict(N=-1), dict(causal=2), dict(causal=-1)])
def test_invalid_forward_only_arguments(lib, kw):
    assert fwd(**kw) == fa.FA_ERR_INVALID_ARG
    assert fwd_host(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(chunk=0), dict(chunk=-128),
                                dict(B=1 << 16, Hq=1 << 16, Hkv=1 << 16, M=1 << 10, d=64,
                                     chunk=1)])
def test_invalid_decode_only_arguments(lib, kw):
    assert dec(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(ks=None), dict(vs=None), dict(ks=GOOD + 2),
                                dict(vs=GOOD + 1), dict(chunk=0),
                                dict(B=1 << 16, Hkv=1 << 16, Hq=1 << 16, M=1 << 20, d=64)])
def test_invalid_fp8_decode_arguments(lib, kw):
    assert dec8(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [
    dict(bt=None), dict(sl=None), dict(bt=GOOD + 2), dict(sl=GOOD + 1),
    dict(page=0), dict(page=4), dict(page=24), dict(page=1 << 17), dict(page=-16),
    dict(num_pages=0), dict(max_pages=0),
    dict(max_pages=7),                    # 7 * 16 < max_seq_len 128
    dict(chunk=0), dict(chunk=8),         # chunk not a multiple of min(page, 128)
    dict(page=256, chunk=64), dict(page=256, chunk=192),
    dict(num_pages=1 << 30, page=1 << 16, max_pages=1),
])
def test_invalid_paged_decode_arguments(lib, kw):
    assert decp(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(lse=None), dict(do=None), dict(dq=None), dict(dk=None),
                                dict(dv=None), dict(do=MIS), dict(dq=MIS), dict(dk=MIS),
                                dict(dv=MIS), dict(lse=GOOD + 2), dict(causal=2), dict(N=0)])
def test_invalid_backward_arguments(lib, kw):
    assert bwd(**kw) == fa.FA_ERR_INVALID_ARG


def test_python_binding_raises_with_status(lib):
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(None, GOOD, GOOD, GOOD, None, 1, 1, 1, 1, 1, 64, 0, 0.1, 0, stream=0)
    assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_header_compiles_as_c(tmp_path):
    """include/fa.h is a plain C header (no CUDA or torch types needed to include it)."""
    src = tmp_path / "t.c"
    src.write_text('#include "fa.h"\nint main(void){ fa_status s = FA_OK; return (int)s; }\n')
    import os
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", inc, str(src)],
                   check=True)

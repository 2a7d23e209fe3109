"""fa_decode_noalloc, the decode entry point that allocates no device memory.

It exists for callers that cannot call cudaMalloc: code running while a CUDA
graph is being captured, processes whose device memory must all come from their
own pool, hosts that forbid allocation after start-up.  It runs the same split-KV
decode as fa_decode but keeps the chunk partials in a fixed array of static
device memory instead of an allocated workspace.  Here it is called through the
C ABI and compared, on two calls in a row (different shapes, so a stale partial
left in the shared array by the first call would show up in the second), with
the fp64 oracle and with fa_decode, within the tolerances the other parity
tests use; once captured inside a CUDA graph and replayed; and under a short
wait limit, with an expired wait reported (and cleared) through
fa_get_last_device_status, the status word these launches share with every
other entry point.

The file name makes pytest collect it last.
"""
import pytest

import exact_attention_05_gb300 as fa
from exact_attention_05_gb300 import build as fa_build
from exact_attention_05_gb300.workloads import BF16, FP16, make_inputs
from exact_attention_05_gb300.workloads import bits
from parity import LSE_TOL, O_TOL, assert_close, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def run_both(torch, oracle_mod, B, Hq, Hkv, M, d, dtype, chunk, seed):
    """fa_decode_noalloc against the oracle and against fa_decode."""
    scale = 1.0 / d ** 0.5
    qh, kh, vh = make_inputs(B, Hq, Hkv, 1, M, d, dtype, seed)
    q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_decode_noalloc(q, k, v, o, lse, B, Hq, Hkv, M, d, chunk, scale, dtype)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o64, lse64 = o.double().cpu().numpy(), lse.double().cpu().numpy()
    o_or, lse_or = oracle_mod.attention(bits(qh), bits(kh), bits(vh), dtype, False, scale)
    assert_close(o64, lse64, o_or, lse_or[:, :, 0], dtype, f"noalloc vs oracle {B, Hq, Hkv, M}")
    o_ref, lse_ref = fa.decode(q, k, v, chunk, scale)
    torch.cuda.synchronize()
    eo = (o.double() - o_ref.double()).abs().max().item()
    el = (lse.double() - lse_ref.double()).abs().max().item()
    assert eo <= O_TOL[dtype], f"max|dO| vs fa_decode {eo:.3e}"
    assert el <= LSE_TOL, f"max|dLSE| vs fa_decode {el:.3e}"


def test_noalloc_decode_matches_oracle_and_fa_decode_on_two_calls(lib, oracle_mod):
    torch = torch_cuda()
    run_both(torch, oracle_mod, 2, 8, 8, 65536, 128, FP16, 128, seed=1005)  # long decode workload
    run_both(torch, oracle_mod, 1, 8, 2, 1000, 64, BF16, 100, seed=61)      # second call, other shape
    assert fa.fa_get_last_device_status() == fa.FA_OK


def test_noalloc_wait_limit_and_timeout_report(lib, oracle_mod):
    """Under a 2 ms wait limit (fa_set_wait_timeout_ns, read at every call) the
    decode still completes and matches the oracle; a wait that expires under
    that limit (the self-test kernel's barrier that nobody arrives on, which
    returns by itself) is reported once by fa_get_last_device_status and then
    cleared, and the next allocation-free call is clean again."""
    torch = torch_cuda()
    fa.fa_set_wait_timeout_ns(2_000_000)
    try:
        run_both(torch, oracle_mod, 1, 8, 8, 512, 128, FP16, 128, seed=1005)
        assert fa.fa_selftest_wait_timeout() == fa.FA_OK
        assert fa.fa_get_last_device_status() == fa.FA_ERR_TIMEOUT
        assert fa.fa_get_last_device_status() == fa.FA_OK        # read once, then cleared
        run_both(torch, oracle_mod, 2, 4, 2, 3000, 64, FP16, 128, seed=62)
    finally:
        fa.fa_set_wait_timeout_ns(0)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    torch = torch_cuda()
    q = torch.zeros((4, 1, 32, 128), dtype=torch.float16, device="cuda")
    k = torch.zeros((4, 8192, 32, 128), dtype=torch.float16, device="cuda")
    # 4*32*ceil(8192/16)*(128+1) floats = 33.8 MB of partials > the 8 MiB array
    st = fa.fa_decode_noalloc(q, k, k, q, None, 4, 32, 32, 8192, 128, 16, 0.1, FP16, check=False)
    assert st == fa.FA_ERR_SCRATCH_LIMIT
    assert "scratch" in fa.fa_status_string(st)


def test_noalloc_decode_inside_a_captured_cuda_graph(lib):
    """Captured once into a CUDA graph (capture fails on any allocation), then
    replayed with new query values written into the same buffer: every replay
    must equal an eager fa_decode on those values."""
    torch = torch_cuda()
    B, Hq, Hkv, M, d, chunk = 2, 8, 2, 3000, 128, 128
    scale = 1.0 / d ** 0.5
    q0, k, v = (t.cuda() for t in make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=71))
    q = q0.clone()
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first call (looks up the array) before any capture
        fa.fa_decode_noalloc(q, k, v, o, lse, B, Hq, Hkv, M, d, chunk, scale, FP16, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_decode_noalloc(q, k, v, o, lse, B, Hq, Hkv, M, d, chunk, scale, FP16)
    for seed in (72, 73):
        qn, _, _ = make_inputs(B, Hq, Hkv, 1, M, d, FP16, seed=seed)
        q.copy_(qn.cuda())
        graph.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = fa.decode(q, k, v, chunk, scale)
        torch.cuda.synchronize()
        eo = (o.double() - o_ref.double()).abs().max().item()
        el = (lse.double() - lse_ref.double()).abs().max().item()
        assert eo <= O_TOL[FP16] and el <= LSE_TOL, (seed, eo, el)
    assert fa.fa_get_last_device_status() == fa.FA_OK

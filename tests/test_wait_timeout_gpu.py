"""Bounded pipeline waits ("Warp-specialised W4A4 kernel on the newest GPU
architecture", sections 3 and 7: the deadlock classes of a warp-specialised
pipeline, and a wait that cannot hang).

A GEMM called with a wait limit (bs_gemm_args.wait_timeout_us) far shorter
than its first hand-off -- the epilogue waits for a whole K = 8192 reduction
-- must give up: the kernel ends early on its own, after the copies and
tensor-core work it issued have drained, the device status word reads
BS_ERR_TIMEOUT with the id of the wait that ran out, and the next call with
the default limit computes the right result in the same context.  No fault,
trap or hang is involved: every wait of the kernels is bounded.
"""
import ctypes
import os
import subprocess

import pytest
import torch

import oracle
import workloads
from tests.helpers import gemm_errors

pytestmark = pytest.mark.gpu

# wait sites of the kernels (the id above the status code in the status word)
SITES = {1: {10, 20, 30, 31, 32, 40}, 2: {110, 120, 130, 131, 132, 140}}


@pytest.mark.parametrize("kernel", [1, 2], ids=["one_cta", "pair"])
def test_wait_runs_out_then_the_context_stays_usable(cuda_lib, kernel):
    bs = cuda_lib
    K = 8192
    d = workloads.dense_lowrank(M=256, N=256, K=K, lowrank=False, bias=False)
    xq, xs, _ = bs.q4_quantize(d["x"].cuda())
    wq, ws, _ = bs.q4_quantize(d["w"].cuda())
    torch.cuda.synchronize()
    bs.clear_device_status()

    with bs.kernel_options(fp4_kernel=kernel, wait_timeout_us=1):
        bs.gemm_fp4(xq, xs, wq, ws, K, out_dtype=torch.float32)
    torch.cuda.synchronize()           # returns: the kernel ended by itself
    st, detail = bs.device_status()
    assert st == bs.BS_ERR_TIMEOUT, (st, hex(detail))
    assert (detail >> 8) in SITES[kernel], hex(detail)

    bs.clear_device_status()
    with bs.kernel_options(fp4_kernel=kernel):
        y = bs.gemm_fp4(xq, xs, wq, ws, K, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == bs.BS_OK
    oa, osa = oracle.q4_quantize(d["x"])
    ob, osb = oracle.q4_quantize(d["w"])
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, K)
    ok, ratio, rel = gemm_errors(y.cpu().numpy(), yr, s, False)
    assert ok, (ratio, rel)


# wait sites of the FP8 and FP4-decode kernels.  (The grouped FP8 kernel
# orders all its warps behind griddepcontrol.wait -- its tile table needs the
# expert offsets first -- and afterwards hands off every 128-wide K block, so
# none of its waits can be made to run past a limit without withholding a
# producer; its timeout exits share the helpers exercised here.)
SITES_FP8 = {50, 60, 61, 62, 63, 70, 71, 72}
SITES_DECODE = {210, 220, 221, 230}

HOLD_NS = 5_000_000      # upstream kernel's hold: 5 ms, far past the limit
LIMIT_US = 10


@pytest.fixture(scope="module")
def pdl_hold(tmp_path_factory):
    """hold() enqueues, on the current stream, tests/native/pdl_hold.cu's
    kernel: it lets the next kernel start early (programmatic dependent
    launch) and keeps the stream's previous grid alive for HOLD_NS.  The
    library's kernels order their first reads of another kernel's data behind
    griddepcontrol.wait, so the tensor-core and epilogue waits of a kernel
    launched right behind the hold last the whole hold."""
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "native", "pdl_hold.cu")
    so = str(tmp_path_factory.mktemp("pdl_hold") / "pdl_hold.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    lib.pdl_hold.restype = ctypes.c_int
    lib.pdl_hold.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]

    def hold():
        assert lib.pdl_hold(HOLD_NS, torch.cuda.current_stream().cuda_stream) == 0
    return hold


def _timeout_then_same_result(bs, hold, run, sites):
    """run(opts, before) -> output tensor, calling before() right before the
    library call (nothing else may be enqueued in between, or the early
    start is lost).  A normal call; then one launched behind the hold with a
    short wait limit, which must end by itself with BS_ERR_TIMEOUT at one of
    `sites`; then a normal call that must reproduce the first result bit for
    bit (stream-K counters back at zero, nothing left behind in the
    context)."""
    bs.clear_device_status()
    ref = run({}, lambda: None).clone()
    torch.cuda.synchronize()
    assert bs.device_status()[0] == bs.BS_OK
    run({"wait_timeout_us": LIMIT_US}, hold)
    torch.cuda.synchronize()           # returns: the kernel ended by itself
    st, detail = bs.device_status()
    assert st == bs.BS_ERR_TIMEOUT, (st, hex(detail))
    assert (detail >> 8) in sites, hex(detail)
    bs.clear_device_status()
    again = run({}, lambda: None)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == bs.BS_OK
    assert torch.equal(again, ref)


@pytest.mark.parametrize("case", ["fp8_stream_k", "fp8_tiles", "w8a8", "fp8_prefill"])
def test_wait_runs_out_fp8(cuda_lib, pdl_hold, case):
    bs = cuda_lib
    g = torch.Generator().manual_seed(3)
    M = 256 if case == "fp8_prefill" else 16
    K, N = 8192, 1024
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    rowwise = case == "w8a8"
    mode = bs.Q8_ROW if rowwise else bs.Q8_TOKEN
    xq, xs = bs.q8_quantize(x, mode=mode)
    wq, ws = bs.q8_quantize(w, mode=bs.Q8_ROW if rowwise else bs.Q8_BLOCK)

    def run(opts, before):
        with bs.kernel_options(fp8_stream_k=2 if case == "fp8_tiles" else 1, **opts):
            before()
            return bs.gemm_fp8(xq, xs, wq, ws, rowwise=rowwise)

    _timeout_then_same_result(bs, pdl_hold, run, SITES_FP8)


def test_wait_runs_out_fp4_decode(cuda_lib, pdl_hold):
    bs = cuda_lib
    g = torch.Generator().manual_seed(4)
    K, N = 8192, 1024
    x = torch.randn(16, K, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    xq, xs, _ = bs.q4_quantize(x)
    wq, ws, _ = bs.q4_quantize(w)

    def run(opts, before):
        with bs.kernel_options(fp4_decode=1, **opts):
            before()
            return bs.gemm_fp4(xq, xs, wq, ws, K)

    _timeout_then_same_result(bs, pdl_hold, run, SITES_DECODE)



def test_wait_runs_out_fp8_multi(cuda_lib, pdl_hold):
    """The multi-weight kernel (three decode products in one grid)."""
    bs = cuda_lib
    g = torch.Generator().manual_seed(6)
    K, N = 4096, 1024
    x = torch.randn(16, K, generator=g).to(torch.bfloat16).cuda()
    xq, xs = bs.q8_quantize(x, mode=bs.Q8_TOKEN)
    wqs = [bs.q8_quantize((torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda(), mode=bs.Q8_BLOCK)
           for _ in range(3)]

    def run(opts, before):
        with bs.kernel_options(**opts):
            before()
            return torch.stack(bs.gemm_fp8_multi(xq, xs, wqs))

    _timeout_then_same_result(bs, pdl_hold, run, SITES_FP8)


def test_wait_runs_out_fp4_multi(cuda_lib, pdl_hold):
    """The FP4 decode kernel's multi-weight variant (three products)."""
    bs = cuda_lib
    g = torch.Generator().manual_seed(7)
    K, N = 4096, 1024
    x = torch.randn(16, K, generator=g).to(torch.bfloat16).cuda()
    xq, xs, _ = bs.q4_quantize(x)
    wqs = [bs.q4_quantize((torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda())[:2] for _ in range(3)]

    def run(opts, before):
        with bs.kernel_options(**opts):
            before()
            return torch.stack(bs.gemm_fp4_multi(xq, xs, wqs, K))

    _timeout_then_same_result(bs, pdl_hold, run, SITES_DECODE)

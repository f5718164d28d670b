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


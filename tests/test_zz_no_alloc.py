"""bs_moe_dispatch_noalloc: the expert grouping for callers that cannot
allocate device memory (a runtime that owns a fixed arena, a plugin enqueue
path that must not allocate, a latency-critical loop).  It keeps its scratch
in a static device array of the library, so it takes no workspace argument.

Called through the C ABI and compared, output by output, with bs_moe_dispatch
(which takes a caller workspace) on two calls in a row with different
routings, so contents left in the shared array by the first call cannot leak
into the second.  This file is collected last so that a failure here, under
-x, comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests.helpers import routing

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(T, k, E, dev):
    import fp8_quantized_gemm_q4_gb300 as bs
    rows = bs.moe_rows_bound(T, k, E)
    return dict(counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
                offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                pair_of_row=torch.full((rows,), -7, dtype=torch.int32, device=dev),
                token_of=torch.full((rows,), -7, dtype=torch.int32, device=dev),
                weight_of=torch.full((rows,), -7.0, dtype=torch.float32, device=dev))


def test_noalloc_dispatch_matches_workspace_dispatch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quantized_gemm_q4_gb300 as bs
    lib = bs.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two different routings, the second with more pairs and a different E
    for (T, E, k, seed) in [(4096, 64, 8, 11), (16384, 256, 8, 12)]:
        r = routing(T, E, k, index=seed)
        ids = torch.from_numpy(r["topk_ids"]).to(dev)
        w = torch.from_numpy(r["topk_w"]).to(dev)
        ref = bs.moe_dispatch(ids, w, E)
        got = _outputs(T, k, E, dev)
        st = lib.bs_moe_dispatch_noalloc(_ptr(ids), _ptr(w), T, k, E, _ptr(got["counts"]), _ptr(got["offsets"]),
                                         _ptr(got["pair_of_row"]), _ptr(got["token_of"]), _ptr(got["weight_of"]),
                                         stream)
        assert st == bs.BS_OK, lib.bs_last_error()
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "pair_of_row", "token_of", "weight_of"):
            assert torch.equal(got[key], ref[key]), key      # integer work / copied weights: exact
        assert bs.device_status()[0] == 0


def test_noalloc_dispatch_rejects_requests_above_the_static_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quantized_gemm_q4_gb300 as bs
    lib = bs.load()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check fails first
    T, k, E = 1 << 17, 8, 1024        # 1024 chunks x 1024 experts x 4 B = 4 MiB > 1 MiB
    assert lib.bs_moe_dispatch_workspace_bytes(T, k, E) > (1 << 20)
    st = lib.bs_moe_dispatch_noalloc(fake, fake, T, k, E, fake, fake, fake, fake, fake, None)
    assert st == bs.BS_ERR_INVALID
    assert b"static array" in lib.bs_last_error()

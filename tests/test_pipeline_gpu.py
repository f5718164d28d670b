"""CopyComputePipeline: host batches through the library's quantizer + FP4
GEMM with copies in, step and copies out overlapped on three streams.  Each
batch's host result must equal, bit for bit, the same step run directly on
that batch (no buffer reused too early, no result read too soon)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("depth", [1, 2, 3])
def test_pipeline_results_match_direct_calls(cuda_lib, depth):
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.pipeline import CopyComputePipeline
    g = torch.Generator().manual_seed(depth)
    M, N, K, nb = 256, 512, 1024, 7
    w = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16).cuda()
    wq, ws, _ = bs.q4_quantize(w)
    xq = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty(bs.sf_bytes(M, K), dtype=torch.uint8, device="cuda")

    def direct(x):
        bs.q4_quantize(x, out=(xq, xs, None))
        return bs.gemm_fp4(xq, xs, wq, ws, K)

    hosts = [torch.randn(M, K, generator=g).to(torch.bfloat16).pin_memory() for _ in range(nb)]
    outs = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    din = [[torch.empty(M, K, dtype=torch.bfloat16, device="cuda")] for _ in range(depth)]
    dout = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(depth)]

    def step(s):
        bs.q4_quantize(din[s][0], out=(xq, xs, None))
        bs.gemm_fp4(xq, xs, wq, ws, K, out=dout[s])

    pipe = CopyComputePipeline(step, din, dout)
    for h, o in zip(hosts, outs):
        pipe.submit([h], o)
    pipe.finish()
    torch.cuda.synchronize()
    for h, o in zip(hosts, outs):
        ref = direct(h.cuda()).cpu()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    assert bs.device_status()[0] == 0

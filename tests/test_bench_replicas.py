"""bench.py's N > 1 path (independent replicas, no data-path collective):
the job time is the max over ranks and the value counts every rank's work.
Run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank 1 is the slow replica
    step_ms, gemm_ms = bench.max_over_ranks([1.0 + rank, 0.5 + 0.25 * rank], "cpu")
    value = bench.job_throughput(1e12, world, step_ms)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, step_ms, gemm_ms, value))


def test_two_gloo_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, step_ms, gemm_ms, value in res:
        assert step_ms == 2.0 and gemm_ms == 0.75
        assert value == pytest.approx(2 * 1e12 / 2e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.job_throughput(10.0, 1, 1.0) == 10000.0


def test_traffic_record_tracks_code_not_comments(tmp_path, monkeypatch):
    """The recorded DRAM traffic of a kernel is reported only while the
    kernel's code (and the shared headers') matches the capture: editing a
    comment keeps it, editing code drops it to None."""
    import json
    import shutil

    import bench
    root = tmp_path
    csrc = root / "pkg" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "fp8_quantized_gemm_q4_gb300", "csrc")
    for name in ("gemm_fp4_pair.cu",) + bench.KERNEL_HEADERS:
        shutil.copy(os.path.join(src, name), csrc / name)
    monkeypatch.setattr(bench, "ROOT", str(root))
    kernel = "pkg/csrc/gemm_fp4_pair.cu"
    (root / "profiles").mkdir()
    rec = {"entries": [{"kernel_src": kernel, "source_sha1": bench.kernel_source_sha1(kernel),
                        "workload": "w", "dram_bytes_per_launch": 123}]}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_for(kernel, "w") == 123
    assert bench.traffic_for(kernel, "other workload") is None
    path = csrc / "gemm_fp4_pair.cu"
    text = path.read_text()
    path.write_text("// an added comment line\n" + text.replace("namespace bsk {", "namespace bsk {  /* note */", 1))
    assert bench.traffic_for(kernel, "w") == 123
    path.write_text(text.replace("constexpr int kThreads = 384;", "constexpr int kThreads = 383;"))
    assert bench.traffic_for(kernel, "w") is None
    (csrc / "ptx.cuh").write_text((csrc / "ptx.cuh").read_text() + "\nstatic int extra_code;\n")
    path.write_text(text)
    assert bench.traffic_for(kernel, "w") is None

"""Host logic of bench.py and the algorithmic counts, on CPU: the byte model
against the figures the pages print, the roofline arithmetic, and the
multi-rank aggregation (max of the timed region, sum of the work) over a
2-rank gloo group."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from tcgen05_tmem_bf16_gb300 import roofline as rf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bytes_model.json")


def test_bytes_model_matches_page_figures():
    g = json.load(open(GOLDEN))
    sw = g["swiglu_unfused_pointwise_read_bytes_per_token"]
    assert rf.swiglu_unfused_pointwise_read_bytes_per_token(sw["d_intermediate"]) == sw["bytes"]
    ratio = g["int4_over_bf16_weight_bytes"]["ratio"]
    assert rf.int4_weight_bytes(8192, 28672) / rf.bf16_weight_bytes(8192, 28672) == ratio


def test_counts_of_the_workloads():
    c = rf.gemm_counts(4096, 4096, 4096, has_bias=True, has_res=True)
    assert c.flops == 2 * 4096 ** 3
    assert c.fused_bytes == 4 * 4096 * 4096 * 2 + 4096 * 2
    assert c.unfused_bytes - c.fused_bytes == 2 * 4096 * 4096 * 2
    s = rf.swiglu_counts(2048, 14336, 4096)
    assert s.flops == 4 * 2048 * 14336 * 4096
    assert s.fused_bytes == 2048 * 4096 * 2 + 2 * 14336 * 4096 * 2 + 2048 * 14336 * 2
    w = rf.w4a16_counts(16, 28672, 8192, 128)
    assert w.fused_bytes == 16 * 8192 * 2 + 8192 * 28672 // 2 + 64 * 28672 * 2 + 16 * 28672 * 2
    assert w.unfused_bytes - w.fused_bytes == 2 * 8192 * 28672 * 2
    # bound: prefill is tensor-bound, decode W4A16 is HBM-bound at the measured peaks
    assert rf.bound(c, 1888.0, 6764.0) == "tensor"
    assert rf.bound(w, 1888.0, 6764.0) == "hbm"
    assert rf.roofline_seconds(c, 1888.0, 6764.0) == pytest.approx(c.flops / 1888e12)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = 1.0 + rank          # rank 1 is the slower one
    units = 10.0 * (rank + 1)
    t, u = bench.aggregate(secs, units, world)
    bench.barrier(world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
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
    for rank, t, u in res:
        assert t == 2.0      # max over ranks
        assert u == 30.0     # sum over ranks


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_source_hash_covers_code_not_comments(tmp_path, monkeypatch):
    # the hash that keys recorded DRAM traffic changes with the code of a
    # kernel's sources, not with their comments or layout
    a = "int f(int x) {  // the input\n  /* doubled */ return 2 * x;\n}\n"
    b = "// a header comment\nint f(int x) {\n  return 2 * x;  /* still doubled,\n  over two lines */\n}\n"
    c = "int f(int x) { return 3 * x; }\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    csrc = tmp_path / "tcgen05_tmem_bf16_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "api.cu").write_text("int plan();\n")
    (csrc / "common.cuh").write_text("// helpers\n")
    (csrc / "wq_gemm.cu").write_text(a)
    (csrc / "gemm_tc.cu").write_text("int g();\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha("wq_gemm_kernel")
    (csrc / "wq_gemm.cu").write_text(b)
    assert bench.kernel_source_sha("wq_gemm_kernel") == h0
    (csrc / "gemm_tc.cu").write_text("int g2();\n")  # another kernel's file
    assert bench.kernel_source_sha("wq_gemm_kernel") == h0
    (csrc / "wq_gemm.cu").write_text(c)
    assert bench.kernel_source_sha("wq_gemm_kernel") != h0
    (csrc / "wq_gemm.cu").write_text(a)
    (csrc / "common.cuh").write_text("// helpers\nint h();\n")  # a shared header
    assert bench.kernel_source_sha("wq_gemm_kernel") != h0

"""The five workloads at full size, through the same entry points the
benchmark times.  Small outputs are checked in full; large ones on a seeded
4096-element sample (corners, both sides of every 128 boundary, the ragged
last row/column, uniform positions) that the oracle computes one element at
a time.  The unfused compositions are run on the same inputs and checked the
same way, so every fused/unfused pair in the benchmark is parity-checked."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up

pytestmark = pytest.mark.gpu


def sampled(ref_fn, out_bits, M, N, what, count=4096):
    rows, cols = workloads.sample_indices(M, N, count)
    ref = ref_fn(rows, cols)
    assert_parity(out_bits[rows, cols], ref, what)


def ws_for(gbf, op, M, N, K):
    n = gbf.gbf_workspace_size(op, M, N, K, False)
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda"), n


def test_prefill_projection_bias_residual(cuda_lib):
    w = workloads.make("prefill")
    M, N, K = w["M"], w["N"], w["K"]
    A, W, bias, res = up(w["A"]), up(w["B"]), up(w["bias"]), up(w["residual"])
    ref_fn = lambda r, c: oracle.gemm_epilogue(w["A"], w["B"], "nk", None, w["bias"],
                                               w["residual"], M=M, N=N, K=K, rows=r, cols=c)
    out = poison_bf16(M, N)
    cuda_lib.gemm_epilogue(A, W, "nk", None, bias, res, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    sampled(ref_fn, down(out), M, N, "prefill fused")
    ws, nb = ws_for(cuda_lib, "gemm_epilogue", M, N, K)
    out2 = poison_bf16(M, N)
    cuda_lib.gemm_epilogue_unfused(A, W, "nk", None, bias, res, out2, M, N, K, workspace=ws,
                                   workspace_bytes=nb)
    assert cuda_lib.gbf_check_device_error() == 0
    D = down(ws[:M * N * 2].view(torch.bfloat16).reshape(M, N))
    rows, cols = workloads.sample_indices(M, N, 4096)
    assert_parity(D[rows, cols], oracle.gemm_epilogue(w["A"], w["B"], "nk", M=M, N=N, K=K,
                                                      rows=rows, cols=cols), "prefill D")
    want = oracle.pointwise_epilogue(D, None, w["bias"], w["residual"], M=M, N=N)
    assert_parity(down(out2), want, "prefill unfused pointwise")


def test_swiglu_workload(cuda_lib):
    w = workloads.make("swiglu")
    M, N, K = w["M"], w["N"], w["K"]
    x, wg, wu = up(w["x"]), up(w["w_gate"]), up(w["w_up"])
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm(x, wg, wu, "nk", h, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    sampled(lambda r, c: oracle.swiglu(w["x"], w["w_gate"], w["w_up"], "nk", M=M, N=N, K=K,
                                       rows=r, cols=c), down(h), M, N, "swiglu fused")
    ws, nb = ws_for(cuda_lib, "swiglu", M, N, K)
    h2 = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm_unfused(x, wg, wu, "nk", h2, M, N, K, workspace=ws,
                                      workspace_bytes=nb)
    assert cuda_lib.gbf_check_device_error() == 0
    sampled(lambda r, c: oracle.swiglu(w["x"], w["w_gate"], w["w_up"], "nk", M=M, N=N, K=K,
                                       unfused=True, rows=r, cols=c), down(h2), M, N,
            "swiglu unfused")


def test_w4a16_decode_workload(cuda_lib):
    w = workloads.make("w4a16")
    M, N, K, G = w["M"], w["N"], w["K"], w["group"]
    A, Wq, s = up(w["A"]), up(w["Wq"]), up(w["scales"])
    ref_fn = lambda r, c: oracle.w4a16(w["A"], w["Wq"], w["scales"], G, M=M, N=N, K=K,
                                       rows=r, cols=c)
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(A, Wq, s, G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    got = down(out)
    # every one of the 16 x 28672 outputs (3.8e9 multiply-adds in the oracle,
    # run on all host cores)
    with oracle.all_cores():
        ref = oracle.w4a16(w["A"], w["Wq"], w["scales"], G, M=M, N=N, K=K)
    assert_parity(got, ref, "w4a16 fused, full output")
    ws, nb = ws_for(cuda_lib, "w4a16", M, N, K)
    out2 = poison_bf16(M, N)
    cuda_lib.w4a16_gemm_unfused(A, Wq, s, G, None, None, None, out2, M, N, K, workspace=ws,
                                workspace_bytes=nb)
    assert cuda_lib.gbf_check_device_error() == 0
    sampled(ref_fn, down(out2), M, N, "w4a16 unfused")


@pytest.mark.parametrize("M", workloads.SWEEP_M)
def test_epilogue_sweep(cuda_lib, M):
    w = workloads.make("sweep", M=M)
    N, K = w["N"], w["K"]
    kw = dict(alpha=w["alpha"], beta=w["beta"], act=w["act"])
    A, B, C, bias = up(w["A"]), up(w["B"]), up(w["C"]), up(w["bias"])
    out = poison_bf16(M, N)
    cuda_lib.gemm_epilogue(A, B, "kn", C, bias, None, out, M, N, K, **kw)
    assert cuda_lib.gbf_check_device_error() == 0
    got = down(out)
    if M <= 16:
        ref = oracle.gemm_epilogue(w["A"], w["B"], "kn", w["C"], w["bias"], None, M=M, N=N, K=K,
                                   **kw)
        assert_parity(got, ref, f"sweep M={M} full")
    else:
        sampled(lambda r, c: oracle.gemm_epilogue(w["A"], w["B"], "kn", w["C"], w["bias"], None,
                                                  M=M, N=N, K=K, rows=r, cols=c, **kw),
                got, M, N, f"sweep M={M}")
    ws, nb = ws_for(cuda_lib, "gemm_epilogue", M, N, K)
    out2 = poison_bf16(M, N)
    cuda_lib.gemm_epilogue_unfused(A, B, "kn", C, bias, None, out2, M, N, K, workspace=ws,
                                   workspace_bytes=nb, **kw)
    assert cuda_lib.gbf_check_device_error() == 0
    D = down(ws[:M * N * 2].view(torch.bfloat16).reshape(M, N))
    rows, cols = workloads.sample_indices(M, N, 2048)
    assert_parity(D[rows, cols], oracle.gemm_epilogue(w["A"], w["B"], "kn", M=M, N=N, K=K,
                                                      rows=rows, cols=cols), f"sweep M={M} D")
    # the unfused result: the oracle's pointwise pass on the GPU's own D
    with oracle.all_cores():
        want = oracle.pointwise_epilogue(D, w["C"], w["bias"], None, M=M, N=N, **kw)
    assert_parity(down(out2), want, f"sweep M={M} unfused pointwise")

"""gemm_epilogue_unfused_noalloc, the entry point for callers that cannot
allocate device memory (code inside a host framework that owns every device
allocation, or under a policy that forbids new allocations), so they cannot
pass a workspace.  It must give the same result as gemm_epilogue_unfused
with a caller workspace, call after call, although every call reuses the
one scratch array built into the library; and that result is checked against
the fp64 oracle stage by stage, as the other unfused compositions are: the
product D against the oracle's product, the ending against the oracle's
pointwise pass applied to that D.

This file is named so that pytest collects it last; it must pass on its own
in a fresh process as well as after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up

pytestmark = pytest.mark.gpu

MAX_ELEMS = 1 << 22


def rand_bf16(seed, shape, std=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def noalloc(cuda_lib, A, B, layout, C, bias, res, out, M, N, K, alpha, beta, act):
    lib = cuda_lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    return lib.gemm_epilogue_unfused_noalloc(
        A.data_ptr(), B.data_ptr(), cuda_lib.LAYOUT[layout], C.data_ptr(), bias.data_ptr(),
        res.data_ptr(), out.data_ptr(), M, N, K, ctypes.c_float(alpha), ctypes.c_float(beta),
        cuda_lib.ACT[act], stream)


def test_matches_the_workspace_entry_point_and_the_oracle_on_two_calls_in_a_row(cuda_lib):
    cases = [(300, 520, 256, "nk", "gelu_tanh", 0.75, 0.25, 1),
             (64, 1040, 512, "kn", "silu", 1.5, -0.5, 2)]
    for M, N, K, layout, act, alpha, beta, seed in cases:
        hA = rand_bf16(seed, (M, K))
        hB = rand_bf16(seed + 1, (K, N) if layout == "kn" else (N, K), std=K ** -0.5)
        hC, hbias, hres = (rand_bf16(seed + 2, (M, N)), rand_bf16(seed + 3, (N,), std=0.3),
                           rand_bf16(seed + 4, (M, N)))
        A, B, C, bias, res = up(hA), up(hB), up(hC), up(hbias), up(hres)
        nbytes = cuda_lib.gbf_workspace_size("gemm_epilogue", M, N, K, False)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        want = poison_bf16(M, N)
        cuda_lib.gemm_epilogue_unfused(A, B, layout, C, bias, res, want, M, N, K, alpha, beta, act,
                                       workspace=ws, workspace_bytes=nbytes)
        got = poison_bf16(M, N)
        assert noalloc(cuda_lib, A, B, layout, C, bias, res, got, M, N, K, alpha, beta, act) == 0
        assert cuda_lib.gbf_check_device_error() == 0
        assert_parity(down(got), down(want), f"noalloc vs workspace M={M} N={N} K={K}")
        # against the oracle: D = A*B as the composition's first kernel computes
        # it (the same product kernel, identity ending), then the ending
        D = poison_bf16(M, N)
        cuda_lib.gemm_epilogue(A, B, layout, None, None, None, D, M, N, K)
        assert cuda_lib.gbf_check_device_error() == 0
        D = down(D)
        assert_parity(D, oracle.gemm_epilogue(hA, hB, layout, M=M, N=N, K=K),
                      f"noalloc product M={M} N={N} K={K}")
        assert_parity(down(got), oracle.pointwise_epilogue(D, hC, hbias, hres, M=M, N=N,
                                                           alpha=alpha, beta=beta, act=act),
                      f"noalloc ending M={M} N={N} K={K}")


def test_rejects_sizes_beyond_the_built_in_array(cuda_lib):
    lib = cuda_lib.load()
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream

    def call(M, N, K=64, act=0, layout=1):
        return lib.gemm_epilogue_unfused_noalloc(p, p, layout, None, None, None, p, M, N, K,
                                                 ctypes.c_float(1.0), ctypes.c_float(0.0), act,
                                                 stream)

    M, N = 2048, MAX_ELEMS // 2048 + 8
    assert call(M, N) == 4  # GBF_ERR_WORKSPACE, nothing launched
    # argument errors are reported as the workspace entry point reports them,
    # before the size limit
    assert call(M, N, act=9) == 1
    assert call(M, N, layout=5) == 1
    assert call(M, N + 4) == 3
    assert call(-1, 8) == 1
    torch.cuda.synchronize()
    assert torch.all(buf == 0)

"""gemm_epilogue_unfused_noalloc, the entry point for callers that cannot
allocate device memory (code inside a host framework that owns every device
allocation, or under a policy that forbids new allocations), so they cannot
pass a workspace.  It must give the same result as gemm_epilogue_unfused
with a caller workspace, call after call, although every call reuses the
one scratch array built into the library.

This file is named so that pytest collects it last; it must pass on its own
in a fresh process as well as after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_parity, down, poison_bf16, up

pytestmark = pytest.mark.gpu

MAX_ELEMS = 1 << 22


def rand_bf16(seed, shape, std=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def test_matches_the_workspace_entry_point_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(300, 520, 256, "nk", "gelu_tanh", 0.75, 0.25, 1),
             (64, 1040, 512, "kn", "silu", 1.5, -0.5, 2)]
    for M, N, K, layout, act, alpha, beta, seed in cases:
        A = up(rand_bf16(seed, (M, K)))
        B = up(rand_bf16(seed + 1, (K, N) if layout == "kn" else (N, K), std=K ** -0.5))
        C = up(rand_bf16(seed + 2, (M, N)))
        bias = up(rand_bf16(seed + 3, (N,), std=0.3))
        res = up(rand_bf16(seed + 4, (M, N)))
        nbytes = cuda_lib.gbf_workspace_size("gemm_epilogue", M, N, K, False)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        want = poison_bf16(M, N)
        cuda_lib.gemm_epilogue_unfused(A, B, layout, C, bias, res, want, M, N, K, alpha, beta, act,
                                       workspace=ws, workspace_bytes=nbytes)
        got = poison_bf16(M, N)
        st = lib.gemm_epilogue_unfused_noalloc(
            A.data_ptr(), B.data_ptr(), cuda_lib.LAYOUT[layout], C.data_ptr(), bias.data_ptr(),
            res.data_ptr(), got.data_ptr(), M, N, K, ctypes.c_float(alpha), ctypes.c_float(beta),
            cuda_lib.ACT[act], stream)
        assert st == 0
        assert cuda_lib.gbf_check_device_error() == 0
        assert_parity(down(got), down(want), f"noalloc vs workspace M={M} N={N} K={K}")


def test_rejects_sizes_beyond_the_built_in_array(cuda_lib):
    lib = cuda_lib.load()
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    M, N = 2048, MAX_ELEMS // 2048 + 8
    st = lib.gemm_epilogue_unfused_noalloc(p, p, 1, None, None, None, p, M, N, 64,
                                           ctypes.c_float(1.0), ctypes.c_float(0.0), 0,
                                           torch.cuda.current_stream().cuda_stream)
    assert st == 4  # GBF_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(buf == 0)

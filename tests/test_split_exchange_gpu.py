"""The split-K reductions of the decode kernels at every split count.

The swapped kernel and the weight-only kernel split K across a cluster of
2..8 CTAs.  The partial sums are exchanged one of two ways:

- push: the output rows are shared out among the ranks, and each rank
  bulk-copies the other ranks' rows to them.
- pull: for larger tiles (the swapped kernel at M > 64, the weight-only
  kernel at M > 16), each rank loads the other partials of its chunks
  through distributed shared memory.

The split count normally follows from the shape, so these tests force every
count from 2 to 8 (including counts that leave some ranks without rows) and
compare with the oracle element by element."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up

pytestmark = pytest.mark.gpu


def rand_bf16(seed, shape, std=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


@pytest.fixture
def forced(cuda_lib):
    def force(s):
        assert cuda_lib.gbf_debug_force_splits(s) == 0
    yield force
    cuda_lib.gbf_debug_force_splits(0)


@pytest.mark.parametrize("splits", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("M", [1, 13, 16, 32, 64, 100, 128])
def test_swapped_gemm_every_split_count(cuda_lib, forced, M, splits):
    N, K = 264, 1024  # 3 weight tiles, the last one ragged; 16 K blocks
    A = rand_bf16(100 + M, (M, K))
    W = rand_bf16(200 + M, (N, K), std=K ** -0.5)
    C = rand_bf16(300 + M, (M, N))
    bias = rand_bf16(400 + M, (N,))
    res = rand_bf16(500 + M, (M, N))
    forced(splits)
    assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk") == ("swap_splitk", splits)
    out = poison_bf16(M, N)
    cuda_lib.gemm_epilogue(up(A), up(W), "nk", up(C), up(bias), up(res), out, M, N, K,
                           alpha=0.75, beta=0.5, act="gelu_tanh")
    assert cuda_lib.gbf_check_device_error() == 0
    want = oracle.gemm_epilogue(A, W, "nk", C, bias, res, M=M, N=N, K=K, alpha=0.75, beta=0.5,
                                act="gelu_tanh")
    assert_parity(down(out), want, f"swapped M={M} splits={splits}")


@pytest.mark.parametrize("splits", [2, 3, 5, 8])
@pytest.mark.parametrize("M", [1, 16, 20, 32])
def test_swapped_gate_up_every_split_count(cuda_lib, forced, M, splits):
    N, K = 136, 512
    x = rand_bf16(600 + M, (M, K))
    wg = rand_bf16(700 + M, (N, K), std=K ** -0.5)
    wu = rand_bf16(800 + M, (N, K), std=K ** -0.5)
    C = rand_bf16(900 + M, (M, N))
    forced(splits)
    assert cuda_lib.gbf_kernel_path("swiglu", M, N, K, "nk") == ("swap_splitk", splits)
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm(up(x), up(wg), up(wu), "nk", h, M, N, K, alpha=0.5, beta=0.25,
                              C=up(C))
    assert cuda_lib.gbf_check_device_error() == 0
    want = oracle.swiglu(x, wg, wu, "nk", C, M=M, N=N, K=K, alpha=0.5, beta=0.25)
    assert_parity(down(h), want, f"gate/up M={M} splits={splits}")


@pytest.mark.parametrize("splits", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("M", [1, 16, 17, 32])
def test_weight_only_every_split_count(cuda_lib, forced, M, splits):
    N, K, G = 1024, 1024, 128
    rng = np.random.Generator(np.random.PCG64(1000 + M))
    A = workloads.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    S = workloads.to_bf16_bits(rng.uniform(0.002, 0.006, size=(K // G, N)).astype(np.float32))
    bias = rand_bf16(1100 + M, (N,))
    res = rand_bf16(1200 + M, (M, N))
    forced(splits)
    assert cuda_lib.gbf_kernel_path("w4a16", M, N, K)[1] == splits
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(S), G, None, up(bias), up(res), out, M, N, K,
                        act="silu")
    assert cuda_lib.gbf_check_device_error() == 0
    want = oracle.w4a16(A, Wq, S, G, None, bias, res, M=M, N=N, K=K, act="silu")
    assert_parity(down(out), want, f"w4a16 M={M} splits={splits}")

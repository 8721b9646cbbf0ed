"""Sizes at the large end: an output of more than 2^31 elements (64-bit
element offsets in every store of the ending), a weight-only product whose
packed weight is 2 GiB, and a long K on the split-K path.  Checked on a
seeded sample (corners, 128-boundaries, the last row and column) gathered on
the device, against the oracle element by element."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, up

pytestmark = pytest.mark.gpu


def rand_bf16(seed, shape, std=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def gather(out, rows, cols):
    r = torch.from_numpy(np.asarray(rows, dtype=np.int64)).cuda()
    c = torch.from_numpy(np.asarray(cols, dtype=np.int64)).cuda()
    return down(out[r, c])


def test_output_beyond_two_to_the_31_elements(cuda_lib):
    # 40000 x 57344 bf16 = 2.29e9 elements (4.6 GB): the CTA-pair kernel,
    # bias and residual broadcast, every row offset beyond 32 bits
    M, N, K = 40000, 57344, 64
    A = rand_bf16(1, (M, K))
    W = rand_bf16(2, (N, K), std=K ** -0.5)
    bias = rand_bf16(3, (N,))
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    out.fill_(float("nan"))
    res = torch.ones(M, N, dtype=torch.bfloat16, device="cuda")  # residual = 1
    cuda_lib.gemm_epilogue(up(A), up(W), "nk", None, up(bias), res, out, M, N, K, act="relu")
    assert cuda_lib.gbf_check_device_error() == 0
    rows, cols = workloads.sample_indices(M, N, 4096, seed=11)
    # residual = 1 everywhere: the oracle's fp64 value before rounding, + 1
    ref = oracle.gemm_epilogue(A, W, "nk", None, bias, None, M=M, N=N, K=K, act="relu",
                               rows=rows, cols=cols, want_f64=True)[1] + 1.0
    want = np.array([oracle.bf16_from_f64(v) for v in ref], dtype=np.uint16)
    assert_parity(gather(out, rows, cols), want, "output beyond 2^31 elements")
    del out, res
    torch.cuda.empty_cache()


def test_weight_only_product_with_a_two_gib_weight(cuda_lib):
    M, N, K, G = 16, 65536, 65536, 128
    rng = np.random.Generator(np.random.PCG64(21))
    A = workloads.to_bf16_bits((rng.standard_normal((M, K)) * 0.25).astype(np.float32))
    Wq = torch.randint(0, 256, (K, N // 2), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(5))
    S = workloads.to_bf16_bits(rng.uniform(0.002, 0.004, size=(K // G, N)).astype(np.float32))
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.w4a16_gemm(up(A), Wq, up(S), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    rows, cols = workloads.sample_indices(M, N, 512, seed=12)
    # a narrow packed weight holding the bytes of the sampled columns only:
    # byte column j = byte c // 2 of sampled column c, i.e. columns
    # c - c % 2 (high nibble) and c - c % 2 + 1 (low nibble)
    cols_u = np.unique(cols)
    narrow = Wq[:, torch.from_numpy(cols_u // 2).cuda()].cpu().numpy()
    Nn = 2 * cols_u.size
    s_n = np.zeros((K // G, Nn), dtype=np.uint16)
    col_map = {}
    for j, c in enumerate(cols_u):
        s_n[:, 2 * j] = S[:, c - (c % 2)]
        s_n[:, 2 * j + 1] = S[:, c - (c % 2) + 1]
        col_map[c] = 2 * j + (c % 2)
    ncols = np.array([col_map[c] for c in cols])
    want = oracle.w4a16(A, narrow, s_n, G, M=M, N=Nn, K=K, rows=rows, cols=ncols)
    assert_parity(gather(out, rows, cols), want, "2 GiB int4 weight")
    del Wq, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [1, 100])
def test_long_k_split_across_the_cluster(cuda_lib, M):
    N, K = 256, 131072
    A = rand_bf16(31 + M, (M, K), std=0.5)
    W = rand_bf16(32 + M, (N, K), std=K ** -0.5)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.gemm_epilogue(up(A), up(W), "nk", None, None, None, out, M, N, K, act="silu")
    assert cuda_lib.gbf_check_device_error() == 0
    path, splits = cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk")
    assert path == "swap_splitk" and splits == 8
    assert_parity(down(out), oracle.gemm_epilogue(A, W, "nk", M=M, N=N, K=K, act="silu"),
                  f"K = {K}")

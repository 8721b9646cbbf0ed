"""GPU parity of gemm_epilogue against the fp64 oracle, element by element.

Sizes span several tiles and ragged tails on both kernel families (the
small-M swapped split-K kernel for M <= 128, the persistent 128x256 kernel
above), both B layouts, every activation, every optional operand, the
in-place residual, and the degenerate sizes (M, N or K = 0)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, empty_bf16, poison_bf16, up

pytestmark = pytest.mark.gpu


def rand_bf16(seed, shape, std=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def case(M, N, K, layout, seed, c=True, bias=True, res=True):
    A = rand_bf16(seed, (M, K))
    B = rand_bf16(seed + 1, (K, N) if layout == "kn" else (N, K), std=K ** -0.5)
    C = rand_bf16(seed + 2, (M, N)) if c else None
    bi = rand_bf16(seed + 3, (N,), std=0.3) if bias else None
    r = rand_bf16(seed + 4, (M, N)) if res else None
    return A, B, C, bi, r


def run_and_check(gbf, M, N, K, layout, act, alpha, beta, seed, c=True, bias=True, res=True,
                  expect_path=None, force_path=None):
    A, B, C, bi, r = case(M, N, K, layout, seed, c, bias, res)
    if force_path:
        assert gbf.gbf_debug_force_path(force_path) == 0
    try:
        if expect_path:
            assert gbf.gbf_kernel_path("gemm_epilogue", M, N, K, layout)[0] == expect_path
        out = poison_bf16(M, N)
        gbf.gemm_epilogue(up(A), up(B), layout, up(C), up(bi), up(r), out, M, N, K, alpha, beta,
                          act)
    finally:
        if force_path:
            gbf.gbf_debug_force_path(None)
    assert gbf.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(A, B, layout, C, bi, r, M=M, N=N, K=K, alpha=alpha, beta=beta,
                               act=act)
    assert_parity(down(out), ref, f"gemm_epilogue M={M} N={N} K={K} {layout} {act}")


def test_tiny_workload_full_output(cuda_lib):
    w = workloads.make("tiny")
    M, N, K = w["M"], w["N"], w["K"]
    out = poison_bf16(M, N)
    cuda_lib.gemm_epilogue(up(w["A"]), up(w["B"]), "kn", up(w["C"]), up(w["bias"]), None, out,
                           M, N, K, w["alpha"], w["beta"], w["act"])
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(w["A"], w["B"], "kn", w["C"], w["bias"], None, M=M, N=N, K=K,
                               alpha=w["alpha"], beta=w["beta"], act=w["act"])
    assert_parity(down(out), ref, "tiny")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M", [1, 7, 16, 33, 64, 100, 128])
def test_small_m_swapped_kernel(cuda_lib, layout, M):
    run_and_check(cuda_lib, M, 264, 520, layout, "gelu_tanh", 0.75, 0.25, seed=100 + M,
                  expect_path="swap_splitk")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(129, 136, 72), (300, 520, 1000), (256, 512, 64),
                                   (511, 264, 128), (1030, 1048, 136)])
def test_persistent_kernel(cuda_lib, layout, M, N, K):
    run_and_check(cuda_lib, M, N, K, layout, "silu", 0.5, 1.5, seed=M + N + K,
                  expect_path="persistent", force_path="persistent")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(129, 136, 72), (300, 520, 1000), (511, 264, 200),
                                   (1030, 1048, 136), (1300, 2056, 256), (256, 4096, 4096)])
def test_persistent_splitk_kernel(cuda_lib, layout, M, N, K):
    # two CTAs per tile, each over half of K (ragged halves included), the
    # partial sums of the other CTA's 128 columns exchanged by bulk copies;
    # more clusters than fit at once in the last case but one
    run_and_check(cuda_lib, M, N, K, layout, "gelu_tanh", 0.75, -0.5, seed=M + 5 * N + K,
                  expect_path="persistent_splitk", force_path="persistent_splitk")


@pytest.mark.parametrize("act", ["identity", "relu", "silu", "gelu_tanh"])
@pytest.mark.parametrize("opts", [(False, False, False), (True, True, True)])
def test_persistent_splitk_every_ending(cuda_lib, act, opts):
    c, bias, res = opts
    run_and_check(cuda_lib, 200, 392, 384, "nk", act, 1.25, 0.5, seed=33, c=c, bias=bias,
                  res=res, expect_path="persistent_splitk", force_path="persistent_splitk")


def test_persistent_splitk_in_place_residual(cuda_lib):
    M, N, K = 300, 264, 512
    A, B, C, bi, r = case(M, N, K, "nk", 810)
    out = up(r)  # residual == out
    assert cuda_lib.gbf_debug_force_path("persistent_splitk") == 0
    try:
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk")[0] == "persistent_splitk"
        cuda_lib.gemm_epilogue(up(A), up(B), "nk", up(C), up(bi), out, out, M, N, K, 0.5, 1.0,
                               "silu")
    finally:
        cuda_lib.gbf_debug_force_path(None)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(A, B, "nk", C, bi, r, M=M, N=N, K=K, alpha=0.5, beta=1.0,
                               act="silu")
    assert_parity(down(out), ref, "split-K in-place residual")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(512, 4096, 512), (300, 520, 200), (257, 264, 136),
                                   (700, 1000, 1000), (256, 256, 128), (1030, 2056, 392)])
def test_cta_pair_kernel_split_k(cuda_lib, layout, M, N, K):
    # two CTA pairs per 256 x 256 tile (a cluster of four), each pair over
    # half of the K blocks (3 blocks split 1 + 2, ragged last blocks), each
    # CTA finishing half of its rows' columns after a bulk-copy exchange with
    # the CTA of the other pair; more clusters than fit at once in the last case
    run_and_check(cuda_lib, M, N, K, layout, "gelu_tanh", 0.75, 0.5, seed=M + 13 * N + K,
                  expect_path="pair_splitk", force_path="pair_splitk")


@pytest.mark.parametrize("act", ["identity", "relu", "silu", "gelu_tanh"])
@pytest.mark.parametrize("opts", [(False, False, False), (True, True, True)])
def test_cta_pair_split_k_every_ending(cuda_lib, act, opts):
    c, bias, res = opts
    run_and_check(cuda_lib, 384, 520, 384, "nk", act, 1.25, 0.5, seed=35, c=c, bias=bias,
                  res=res, expect_path="pair_splitk", force_path="pair_splitk")


def test_cta_pair_split_k_in_place_residual(cuda_lib):
    M, N, K = 300, 264, 512
    A, B, C, bi, r = case(M, N, K, "kn", 811)
    out = up(r)  # residual == out
    assert cuda_lib.gbf_debug_force_path("pair_splitk") == 0
    try:
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "kn")[0] == "pair_splitk"
        cuda_lib.gemm_epilogue(up(A), up(B), "kn", up(C), up(bi), out, out, M, N, K, 0.5, 1.0,
                               "silu")
    finally:
        cuda_lib.gbf_debug_force_path(None)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(A, B, "kn", C, bi, r, M=M, N=N, K=K, alpha=0.5, beta=1.0,
                               act="silu")
    assert_parity(down(out), ref, "pair split-K in-place residual")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(512, 2048, 256), (1000, 2000, 320)])
def test_cta_pair_kernel_224_wide_tiles(cuda_lib, layout, M, N, K):
    # shapes whose last round of 256-wide tiles is thin, so the planner takes
    # 224-wide tiles (for B as [K][N] the MMA reads 112 of the 128 columns each
    # CTA loads); N not a multiple of 224
    run_and_check(cuda_lib, M, N, K, layout, "gelu_tanh", 0.75, 0.25, seed=M + 11 * N + K,
                  expect_path="pair", force_path="pair")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(512, 256, 64), (515, 264, 256), (1030, 1048, 136),
                                   (777, 520, 328), (2048, 1024, 512), (129, 264, 128),
                                   (300, 520, 200), (400, 1048, 136)])
def test_cta_pair_kernel(cuda_lib, layout, M, N, K):
    run_and_check(cuda_lib, M, N, K, layout, "gelu_tanh", 0.75, -0.25, seed=M + 3 * N + K,
                  expect_path="pair", force_path="pair")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(257, 264, 136), (1030, 1048, 136), (640, 4096, 512),
                                   (2048, 2560, 192), (4100, 520, 64)])
def test_cta_pair_kernel_one_stream(cuda_lib, layout, M, N, K):
    # units of one 256-row M-tile, one MMA stream alternating between the two
    # accumulators; more units than pairs in the last two cases (the
    # accumulators are reused across rounds)
    run_and_check(cuda_lib, M, N, K, layout, "silu", 0.75, 0.5, seed=M + 7 * N + K,
                  expect_path="pair_1stream", force_path="pair_1stream")


@pytest.mark.parametrize("layout", ["nk"])
@pytest.mark.parametrize("M,N,K", [(1024, 4096, 256), (700, 2000, 200)])
def test_cta_pair_kernel_one_stream_224_wide_tiles(cuda_lib, layout, M, N, K):
    # one-stream units whose 256-wide tiles leave SM pairs idle, so the
    # planner takes 224-wide tiles for K-contiguous weights (16 -> 19
    # N-tiles; N = 2000 ragged)
    run_and_check(cuda_lib, M, N, K, layout, "gelu_tanh", 0.5, 0.75, seed=M + 5 * N + K,
                  expect_path="pair_1stream", force_path="pair_1stream")


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,N,K", [(512, 512, 64), (600, 1000, 72), (1024, 2048, 136),
                                   (777, 4096, 1000)])
def test_cta_pair_one_stream_two_k_streams(cuda_lib, layout, M, N, K):
    # one tile per pair: two MMA streams over the alternate K blocks of the
    # tile (one block: the second stream idle; an odd count: 2 + 1), the two
    # accumulators added in the ending
    run_and_check(cuda_lib, M, N, K, layout, "relu", 0.5, -0.75, seed=M + 17 * N + K,
                  expect_path="pair_1stream", force_path="pair_1stream")


@pytest.mark.parametrize("M,N,K", [(512, 4096, 256), (768, 2048, 192), (1024, 8192, 128),
                                   (3000, 1024, 64)])
def test_automatic_kernel_choice(cuda_lib, M, N, K):
    # whichever of the two kernels the planner picks for mid-size M
    run_and_check(cuda_lib, M, N, K, "nk", "relu", 1.25, 0.5, seed=M + N)


@pytest.mark.parametrize("act", ["identity", "relu", "silu", "gelu_tanh"])
@pytest.mark.parametrize("M", [48, 260, 600])
def test_every_activation(cuda_lib, act, M):
    run_and_check(cuda_lib, M, 392, 200, "nk", act, 1.25, -0.5, seed=7 + M)


@pytest.mark.parametrize("opts", [(False, False, False), (True, False, False),
                                  (False, True, False), (False, False, True)])
@pytest.mark.parametrize("M", [20, 200, 700])
def test_optional_operands(cuda_lib, opts, M):
    c, b, r = opts
    run_and_check(cuda_lib, M, 256, 128, "kn", "relu", 1.0, 2.0, seed=11 + M, c=c, bias=b, res=r)


@pytest.mark.parametrize("M", [1, 16, 128, 640])
def test_plain_product_matches_torch_matmul(cuda_lib, M):
    # alpha=1, beta=0, no bias/residual, identity: the plain product; cross-
    # checked against torch.matmul in fp32 as well as the oracle.
    N, K = 384, 512
    A, B, _, _, _ = case(M, N, K, "nk", 300 + M, False, False, False)
    out = poison_bf16(M, N)
    cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(A, B, "nk", M=M, N=N, K=K)
    assert_parity(down(out), ref, "plain product")
    t = (up(A).float() @ up(B).float().T).to(torch.bfloat16)
    assert_parity(down(out), down(t), "plain product vs torch")


@pytest.mark.parametrize("M", [5, 300, 520])
def test_in_place_residual(cuda_lib, M):
    N, K = 264, 128
    A, B, C, bi, r = case(M, N, K, "nk", 400 + M)
    out = up(r)  # residual == out
    cuda_lib.gemm_epilogue(up(A), up(B), "nk", up(C), up(bi), out, out, M, N, K, 0.5, 1.0, "silu")
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(A, B, "nk", C, bi, r, M=M, N=N, K=K, alpha=0.5, beta=1.0,
                               act="silu")
    assert_parity(down(out), ref, "in-place residual")


def test_identity_b_returns_a(cuda_lib):
    # B = I (K x N with N = K): out = A exactly.
    for M in (40, 300):
        n = 256
        A = rand_bf16(500 + M, (M, n))
        eye = workloads.to_bf16_bits(np.eye(n, dtype=np.float32))
        out = poison_bf16(M, n)
        cuda_lib.gemm_epilogue(up(A), up(eye), "kn", None, None, None, out, M, n, n)
        assert cuda_lib.gbf_check_device_error() == 0
        assert np.array_equal(down(out), A)


def test_degenerate_sizes(cuda_lib):
    # K = 0: empty sum, out = act(beta*C + bias) + residual.
    M, N = 24, 64
    _, _, C, bi, r = case(M, N, 8, "nk", 600)
    out = poison_bf16(M, N)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    cuda_lib.gemm_epilogue(dummy, dummy, "nk", up(C), up(bi), up(r), out, M, N, 0, 2.0, 0.5, "relu")
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(np.zeros((M, 0), np.uint16), np.zeros((N, 0), np.uint16), "nk",
                               C, bi, r, M=M, N=N, K=0, alpha=2.0, beta=0.5, act="relu")
    assert_parity(down(out), ref, "K=0")
    # M = 0 or N = 0: nothing to do, nothing written.
    sentinel = torch.full((4,), 7.0, dtype=torch.bfloat16, device="cuda")
    assert cuda_lib.gemm_epilogue(dummy, dummy, "nk", None, None, None, sentinel, 0, 8, 8) == 0
    assert cuda_lib.gemm_epilogue(dummy, dummy, "nk", None, None, None, sentinel, 8, 0, 8) == 0
    torch.cuda.synchronize()
    assert torch.all(sentinel == 7.0)


def test_writes_stay_inside_the_output(cuda_lib):
    # A ragged output inside a larger buffer: the guard rows/columns around it
    # must keep their values (out is written as a packed [M][N] block).
    M, N, K = 130, 264, 64
    A, B, C, bi, r = case(M, N, K, "kn", 700)
    buf = torch.full((M * N + 4096,), 3.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:M * N]
    cuda_lib.gemm_epilogue(up(A), up(B), "kn", up(C), up(bi), up(r), out, M, N, K, 1.0, 1.0, "silu")
    assert cuda_lib.gbf_check_device_error() == 0
    assert torch.all(buf[M * N:] == 3.0)
    ref = oracle.gemm_epilogue(A, B, "kn", C, bi, r, M=M, N=N, K=K, alpha=1.0, beta=1.0, act="silu")
    assert_parity(down(out).reshape(M, N), ref, "guard")


def test_inputs_under_both_readings_of_n0x(cuda_lib):
    # The variance reading (default) and the std reading of N(0, x).
    for sigma_is_std in (False, True):
        w = workloads.make("sweep", M=16, sigma_is_std=sigma_is_std,
                           shape=dict(N=512, K=1024))
        M, N, K = 16, 512, 1024
        out = poison_bf16(M, N)
        cuda_lib.gemm_epilogue(up(w["A"]), up(w["B"]), "kn", up(w["C"]), up(w["bias"]), None,
                               out, M, N, K, w["alpha"], w["beta"], w["act"])
        assert cuda_lib.gbf_check_device_error() == 0
        ref = oracle.gemm_epilogue(w["A"], w["B"], "kn", w["C"], w["bias"], None, M=M, N=N, K=K,
                                   alpha=w["alpha"], beta=w["beta"], act=w["act"])
        assert_parity(down(out), ref, f"sigma_is_std={sigma_is_std}")

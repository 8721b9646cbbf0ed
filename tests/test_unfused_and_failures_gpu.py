"""The unfused reference compositions, checked stage by stage against the
oracle (the bf16 intermediate is a rounding decision, so each stage is fed
the same bf16 inputs on both sides), fused vs unfused agreement, and the
bounded-wait failure path (a withheld signal makes the epilogue's wait run
out; the kernel records a timeout and exits, the context stays usable)."""
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


def workspace(gbf, op, M, N, K):
    n = gbf.gbf_workspace_size(op, M, N, K, False)
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda"), n


@pytest.mark.parametrize("M,layout", [(16, "kn"), (300, "nk"), (97, "kn")])
def test_gemm_epilogue_unfused_stagewise(cuda_lib, M, layout):
    N, K = 264, 384
    A = rand_bf16(1, (M, K))
    B = rand_bf16(2, (K, N) if layout == "kn" else (N, K), std=K ** -0.5)
    C, bias, res = rand_bf16(3, (M, N)), rand_bf16(4, (N,)), rand_bf16(5, (M, N))
    ws, nbytes = workspace(cuda_lib, "gemm_epilogue", M, N, K)
    out = poison_bf16(M, N)
    cuda_lib.gemm_epilogue_unfused(up(A), up(B), layout, up(C), up(bias), up(res), out, M, N, K,
                                   0.75, 0.5, "gelu_tanh", ws, nbytes)
    assert cuda_lib.gbf_check_device_error() == 0
    D = ws[:M * N * 2].view(torch.bfloat16).reshape(M, N)
    # stage 1: D = bf16(A*B~) against the oracle's plain product
    assert_parity(down(D), oracle.gemm_epilogue(A, B, layout, M=M, N=N, K=K), "unfused D")
    # stage 2: the pointwise pass on the GPU's own D
    ref = oracle.pointwise_epilogue(down(D), C, bias, res, M=M, N=N, alpha=0.75, beta=0.5,
                                    act="gelu_tanh")
    assert_parity(down(out), ref, "unfused pointwise")
    # fused result against the oracle (single rounding)
    fused = poison_bf16(M, N)
    cuda_lib.gemm_epilogue(up(A), up(B), layout, up(C), up(bias), up(res), fused, M, N, K, 0.75,
                           0.5, "gelu_tanh")
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(fused), oracle.gemm_epilogue(A, B, layout, C, bias, res, M=M, N=N, K=K,
                                                    alpha=0.75, beta=0.5, act="gelu_tanh"),
                  "fused")


@pytest.mark.parametrize("M", [8, 200])
def test_swiglu_unfused_stagewise(cuda_lib, M):
    N, K = 256, 320
    x = rand_bf16(11, (M, K))
    wg = rand_bf16(12, (N, K), std=K ** -0.5)
    wu = rand_bf16(13, (N, K), std=K ** -0.5)
    ws, nbytes = workspace(cuda_lib, "swiglu", M, N, K)
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm_unfused(up(x), up(wg), up(wu), "nk", h, M, N, K, workspace=ws,
                                      workspace_bytes=nbytes)
    assert cuda_lib.gbf_check_device_error() == 0
    off = (M * N * 2 + 255) // 256 * 256
    g = ws[:M * N * 2].view(torch.bfloat16).reshape(M, N)
    u = ws[off:off + M * N * 2].view(torch.bfloat16).reshape(M, N)
    assert_parity(down(g), oracle.gemm_epilogue(x, wg, "nk", M=M, N=N, K=K), "g")
    assert_parity(down(u), oracle.gemm_epilogue(x, wu, "nk", M=M, N=N, K=K), "u")
    assert_parity(down(h), oracle.swiglu_pointwise(down(g), down(u), M=M, N=N), "glu pass")


def test_w4a16_unfused_materialises_the_same_weight(cuda_lib):
    M, N, K, G = 16, 512, 512, 128
    rng = np.random.Generator(np.random.PCG64(21))
    A = rand_bf16(22, (M, K))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    s = workloads.to_bf16_bits(rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float32))
    ws, nbytes = workspace(cuda_lib, "w4a16", M, N, K)
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm_unfused(up(A), up(Wq), up(s), G, None, None, None, out, M, N, K,
                                workspace=ws, workspace_bytes=nbytes)
    assert cuda_lib.gbf_check_device_error() == 0
    w = ws[:K * N * 2].view(torch.bfloat16).reshape(K, N)
    # the materialised weight is bit-exact: one rounding of an exact product
    assert np.array_equal(down(w), oracle.dequant_int4(Wq, s, G, K=K, N=N))
    ref = oracle.w4a16(A, Wq, s, G, M=M, N=N, K=K)
    assert_parity(down(out), ref, "w4a16 unfused")
    fused = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, None, None, None, fused, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(fused), ref, "w4a16 fused")


def test_unfused_rejects_a_small_workspace(cuda_lib):
    M, N, K = 16, 64, 64
    A, B = up(rand_bf16(1, (M, K))), up(rand_bf16(2, (N, K)))
    out = poison_bf16(M, N)
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    st = cuda_lib.gemm_epilogue_unfused(A, B, "nk", None, None, None, out, M, N, K,
                                        workspace=ws, workspace_bytes=1024,
                                        raise_on_error=False)
    assert st == 4


@pytest.mark.parametrize("M", [8, 128, 256, 512])
def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib, M):
    N, K = 256, 128
    A = rand_bf16(31, (M, K))
    B = rand_bf16(32, (N, K), std=K ** -0.5)
    out = poison_bf16(M, N)
    if M <= 128:
        # the swapped kernel with a split-K exchange: an aborted rank must
        # still wait for its peers' copies before it leaves
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk")[1] > 1
    cuda_lib.gbf_set_wait_timeout_ns(20_000_000)  # 20 ms
    cuda_lib.gbf_debug_inject_timeout(True)
    try:
        cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
        assert cuda_lib.gbf_check_device_error() == 6  # GBF_ERR_TIMEOUT
    finally:
        cuda_lib.gbf_debug_inject_timeout(False)
        cuda_lib.gbf_set_wait_timeout_ns(2_000_000_000)
    assert cuda_lib.gbf_check_device_error() == 0  # the word was cleared
    cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), oracle.gemm_epilogue(A, B, "nk", M=M, N=N, K=K), "after timeout")


def test_stream_argument_is_honoured(cuda_lib):
    M, N, K = 200, 256, 256
    A, B = rand_bf16(41, (M, K)), rand_bf16(42, (N, K), std=K ** -0.5)
    s = torch.cuda.Stream()
    dA, dB = up(A), up(B)
    out = poison_bf16(M, N)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        cuda_lib.gemm_epilogue(dA, dB, "nk", None, None, None, out, M, N, K, stream=s)
    assert cuda_lib.gbf_check_device_error(s) == 0
    assert_parity(down(out), oracle.gemm_epilogue(A, B, "nk", M=M, N=N, K=K), "side stream")


@pytest.mark.parametrize("M", [16, 32])
def test_weight_only_kernel_timeout_is_reported_and_recoverable(cuda_lib, M):
    # a withheld accumulator-ready signal must end in GBF_ERR_TIMEOUT, with
    # the split-K exchange pushing partials (M = 16) or pulling them (M = 32),
    # and the next call on the same context must be correct
    N, K, G = 1024, 1024, 128
    assert cuda_lib.gbf_kernel_path("w4a16", M, N, K)[1] > 1
    w = workloads.make("w4a16", shape=dict(M=M, N=N, K=K, group=G))
    out = poison_bf16(M, N)
    cuda_lib.gbf_set_wait_timeout_ns(50_000_000)
    cuda_lib.gbf_debug_inject_timeout(True)
    try:
        cuda_lib.w4a16_gemm(up(w["A"]), up(w["Wq"]), up(w["scales"]), G, None, None, None, out,
                            M, N, K)
        assert cuda_lib.gbf_check_device_error() == 6
    finally:
        cuda_lib.gbf_debug_inject_timeout(False)
        cuda_lib.gbf_set_wait_timeout_ns(2_000_000_000)
    assert cuda_lib.gbf_check_device_error() == 0
    cuda_lib.w4a16_gemm(up(w["A"]), up(w["Wq"]), up(w["scales"]), G, None, None, None, out,
                        M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), oracle.w4a16(w["A"], w["Wq"], w["scales"], G, M=M, N=N, K=K),
                  "after timeout")


def test_split_k_persistent_kernel_timeout_is_reported_and_recoverable(cuda_lib):
    # the split-K form of the persistent kernel: a withheld accumulator-ready
    # signal in both CTAs of every cluster must end in GBF_ERR_TIMEOUT after
    # the partial-sum exchange has drained, and the next call must be correct
    M, N, K = 256, 512, 256
    A = rand_bf16(61, (M, K))
    B = rand_bf16(62, (N, K), std=K ** -0.5)
    out = poison_bf16(M, N)
    assert cuda_lib.gbf_debug_force_path("persistent_splitk") == 0
    try:
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk")[0] == "persistent_splitk"
        cuda_lib.gbf_set_wait_timeout_ns(20_000_000)
        cuda_lib.gbf_debug_inject_timeout(True)
        try:
            cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
            assert cuda_lib.gbf_check_device_error() == 6
        finally:
            cuda_lib.gbf_debug_inject_timeout(False)
            cuda_lib.gbf_set_wait_timeout_ns(2_000_000_000)
        assert cuda_lib.gbf_check_device_error() == 0
        cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
    finally:
        cuda_lib.gbf_debug_force_path(None)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), oracle.gemm_epilogue(A, B, "nk", M=M, N=N, K=K), "after timeout")


def test_one_stream_pair_kernel_timeout_is_reported_and_recoverable(cuda_lib):
    # the CTA-pair kernel with one MMA stream: a withheld accumulator-ready
    # signal for the first tile must end in GBF_ERR_TIMEOUT, and the next call
    # on the same context must be correct
    M, N, K = 1024, 1024, 256
    A = rand_bf16(71, (M, K))
    B = rand_bf16(72, (N, K), std=K ** -0.5)
    out = poison_bf16(M, N)
    assert cuda_lib.gbf_debug_force_path("pair_1stream") == 0
    try:
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk")[0] == "pair_1stream"
        cuda_lib.gbf_set_wait_timeout_ns(20_000_000)
        cuda_lib.gbf_debug_inject_timeout(True)
        try:
            cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
            assert cuda_lib.gbf_check_device_error() == 6
        finally:
            cuda_lib.gbf_debug_inject_timeout(False)
            cuda_lib.gbf_set_wait_timeout_ns(2_000_000_000)
        assert cuda_lib.gbf_check_device_error() == 0
        cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
    finally:
        cuda_lib.gbf_debug_force_path(None)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), oracle.gemm_epilogue(A, B, "nk", M=M, N=N, K=K), "after timeout")


def test_pair_split_k_timeout_is_reported_and_recoverable(cuda_lib):
    # the split-K form of the CTA-pair kernel (clusters of two pairs): a
    # withheld accumulator-ready signal must end in GBF_ERR_TIMEOUT (the
    # partial-sum exchange still completes), and the next call on the same
    # context must be correct
    M, N, K = 512, 1024, 256
    A = rand_bf16(73, (M, K))
    B = rand_bf16(74, (N, K), std=K ** -0.5)
    out = poison_bf16(M, N)
    assert cuda_lib.gbf_debug_force_path("pair_splitk") == 0
    try:
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, "nk")[0] == "pair_splitk"
        cuda_lib.gbf_set_wait_timeout_ns(20_000_000)
        cuda_lib.gbf_debug_inject_timeout(True)
        try:
            cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
            assert cuda_lib.gbf_check_device_error() == 6
        finally:
            cuda_lib.gbf_debug_inject_timeout(False)
            cuda_lib.gbf_set_wait_timeout_ns(2_000_000_000)
        assert cuda_lib.gbf_check_device_error() == 0
        cuda_lib.gemm_epilogue(up(A), up(B), "nk", None, None, None, out, M, N, K)
    finally:
        cuda_lib.gbf_debug_force_path(None)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), oracle.gemm_epilogue(A, B, "nk", M=M, N=N, K=K), "after timeout")

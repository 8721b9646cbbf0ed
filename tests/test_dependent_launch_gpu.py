"""Back-to-back dependent calls on one stream, with no host synchronisation in
between: the decode kernels (swapped split-K GEMM, weight-only GEMM) may start
while the previous kernel finishes and prefetch their weights, so each call
must still see the complete output of the call before it.  Every stage is
checked against the oracle on the GPU's own input of that stage."""
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


def test_chain_of_swapped_gemms_reads_each_previous_output(cuda_lib):
    # x_{i+1} = x_i * W_i^T + x_i (the residual is the previous output too)
    M, D, steps = 16, 2048, 6
    ws = [rand_bf16(100 + i, (D, D), std=D ** -0.5) for i in range(steps)]
    x0 = rand_bf16(99, (M, D))
    xs = [up(x0)] + [poison_bf16(M, D) for _ in range(steps)]
    dws = [up(w) for w in ws]
    for i in range(steps):
        cuda_lib.gemm_epilogue(xs[i], dws[i], "nk", None, None, xs[i], xs[i + 1], M, D, D)
    assert cuda_lib.gbf_check_device_error() == 0
    assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, D, D, "nk")[0] == "swap_splitk"
    for i in range(steps):
        xin = down(xs[i])
        want = oracle.gemm_epilogue(xin, ws[i], "nk", residual=xin, M=M, N=D, K=D)
        assert_parity(down(xs[i + 1]), want, f"chain step {i}")


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_chain_of_pair_gemms_reads_each_previous_output(cuda_lib, layout):
    # the CTA-pair kernel (forced: at this size the planner prefers the
    # one-SM kernel)
    M, D, steps = 1024, 1024, 4
    ws = [rand_bf16(200 + i, (D, D), std=D ** -0.5) for i in range(steps)]
    x0 = rand_bf16(199, (M, D))
    xs = [up(x0)] + [poison_bf16(M, D) for _ in range(steps)]
    dws = [up(w) for w in ws]
    assert cuda_lib.gbf_debug_force_path("pair") == 0
    try:
        assert cuda_lib.gbf_kernel_path("gemm_epilogue", M, D, D, layout)[0] == "pair"
        for i in range(steps):
            cuda_lib.gemm_epilogue(xs[i], dws[i], layout, None, None, xs[i], xs[i + 1], M, D, D)
    finally:
        cuda_lib.gbf_debug_force_path(None)
    assert cuda_lib.gbf_check_device_error() == 0
    for i in range(steps):
        xin = down(xs[i])
        want = oracle.gemm_epilogue(xin, ws[i], layout, residual=xin, M=M, N=D, K=D)
        assert_parity(down(xs[i + 1]), want, f"pair chain {layout} step {i}")


def test_chain_of_weight_only_gemms_reads_each_previous_output(cuda_lib):
    M, D, G, steps = 16, 2048, 128, 5
    rng = np.random.Generator(np.random.PCG64(7))
    qs = [rng.integers(0, 256, size=(D, D // 2), dtype=np.uint8) for _ in range(steps)]
    ss = [workloads.to_bf16_bits(rng.uniform(0.002, 0.006, size=(D // G, D)).astype(np.float32))
          for _ in range(steps)]
    x0 = rand_bf16(5, (M, D))
    xs = [up(x0)] + [poison_bf16(M, D) for _ in range(steps)]
    dq, ds = [up(q) for q in qs], [up(s) for s in ss]
    for i in range(steps):
        cuda_lib.w4a16_gemm(xs[i], dq[i], ds[i], G, None, None, None, xs[i + 1], M, D, D,
                            act="silu")
    assert cuda_lib.gbf_check_device_error() == 0
    for i in range(steps):
        want = oracle.w4a16(down(xs[i]), qs[i], ss[i], G, M=M, N=D, K=D, act="silu")
        assert_parity(down(xs[i + 1]), want, f"w4a16 chain step {i}")


def test_weight_only_gemm_after_a_plain_kernel_sees_its_writes(cuda_lib):
    # a torch kernel (no programmatic launch) writes the activations right
    # before the call
    M, N, K, G = 16, 1024, 1024, 128
    w = workloads.make("w4a16", shape=dict(M=M, N=N, K=K, group=G))
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    out = poison_bf16(M, N)
    src = up(w["A"])
    for _ in range(3):
        A.zero_()
        A.copy_(src)
        cuda_lib.w4a16_gemm(A, up(w["Wq"]), up(w["scales"]), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), oracle.w4a16(w["A"], w["Wq"], w["scales"], G, M=M, N=N, K=K),
                  "after a copy kernel")


@pytest.mark.parametrize("M1", [128, 640])
def test_weight_operand_written_by_the_previous_call(cuda_lib, M1):
    # the first call's output becomes the second call's B operand (W [N][K]),
    # so the second kernel must not fetch any operand before the first ends
    K1, N2, M2 = 256, 1024, 16
    X = rand_bf16(301, (M1, K1))
    Y = rand_bf16(302, (N2, K1), std=K1 ** -0.5)
    A = rand_bf16(303, (M2, N2))
    W = poison_bf16(M1, N2)  # written by call 1: [M1][N2] = W [N][K] of call 2
    out = poison_bf16(M2, M1)
    cuda_lib.gemm_epilogue(up(X), up(Y), "nk", None, None, None, W, M1, N2, K1)
    cuda_lib.gemm_epilogue(up(A), W, "nk", None, None, None, out, M2, M1, N2)
    assert cuda_lib.gbf_check_device_error() == 0
    w = down(W)
    assert_parity(w, oracle.gemm_epilogue(X, Y, "nk", M=M1, N=N2, K=K1), "first call")
    assert_parity(down(out), oracle.gemm_epilogue(A, w, "nk", M=M2, N=M1, K=N2),
                  "second call on the first call's output")

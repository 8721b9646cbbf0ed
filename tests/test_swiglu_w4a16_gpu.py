"""GPU parity of swiglu_dual_gemm and w4a16_gemm against the fp64 oracle,
element by element, with the targeted probes that pin packing, nibble order
and group indexing on the GPU side."""
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


# ------------------------------------------------------------------ SwiGLU

@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (130, 264, 328), (300, 128, 1000),
                                   (513, 392, 256), (1024, 264, 328), (1500, 512, 200)])
def test_swiglu_dual_gemm(cuda_lib, layout, M, N, K):
    x = rand_bf16(M + 1, (M, K))
    shp = (N, K) if layout == "nk" else (K, N)
    wg = rand_bf16(M + 2, shp, std=K ** -0.5)
    wu = rand_bf16(M + 3, shp, std=K ** -0.5)
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm(up(x), up(wg), up(wu), layout, h, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.swiglu(x, wg, wu, layout, M=M, N=N, K=K)
    assert_parity(down(h), ref, f"swiglu {layout} {M}x{N}x{K}")


@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("M,N,K", [(1, 136, 64), (16, 1000, 4096), (17, 264, 200),
                                   (32, 4096, 1024), (5, 128, 8)])
def test_swiglu_decode_sizes_swapped_kernel(cuda_lib, layout, M, N, K):
    # M <= 32: the gate/up GEMM on the swapped split-K kernel (two weight
    # tiles per stage, gate and up accumulators, GLU ending per column)
    x = rand_bf16(M + 11, (M, K))
    shp = (N, K) if layout == "nk" else (K, N)
    wg = rand_bf16(M + 12, shp, std=K ** -0.5)
    wu = rand_bf16(M + 13, shp, std=K ** -0.5)
    h = poison_bf16(M, N)
    assert cuda_lib.gbf_kernel_path("swiglu", M, N, K, layout)[0] == "swap_splitk"
    cuda_lib.swiglu_dual_gemm(up(x), up(wg), up(wu), layout, h, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.swiglu(x, wg, wu, layout, M=M, N=N, K=K)
    assert_parity(down(h), ref, f"swiglu swapped {layout} {M}x{N}x{K}")


@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "relu", "identity"])
def test_swiglu_decode_gates_alpha_beta_c(cuda_lib, act):
    M, N, K = 16, 392, 640
    x = rand_bf16(31, (M, K))
    wg = rand_bf16(32, (N, K), std=K ** -0.5)
    wu = rand_bf16(33, (N, K), std=K ** -0.5)
    C = rand_bf16(34, (M, N))
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm(up(x), up(wg), up(wu), "nk", h, M, N, K, 0.75, 1.5, up(C), act)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.swiglu(x, wg, wu, "nk", C, M=M, N=N, K=K, alpha=0.75, beta=1.5, act=act)
    assert_parity(down(h), ref, f"swiglu decode {act}")


@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "relu", "identity"])
def test_swiglu_other_gates_alpha_beta_c(cuda_lib, act):
    M, N, K = 200, 136, 256
    x = rand_bf16(1, (M, K))
    wg = rand_bf16(2, (N, K), std=K ** -0.5)
    wu = rand_bf16(3, (N, K), std=K ** -0.5)
    C = rand_bf16(4, (M, N))
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm(up(x), up(wg), up(wu), "nk", h, M, N, K, 0.75, 1.5, up(C), act)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.swiglu(x, wg, wu, "nk", C, M=M, N=N, K=K, alpha=0.75, beta=1.5, act=act)
    assert_parity(down(h), ref, f"swiglu {act}")


def test_swiglu_same_weights_is_silu_g_times_g(cuda_lib):
    # W_gate = W_up: h = silu(g)*g; compared with gemm_epilogue(act=SiLU) times
    # the plain product, both from the GPU (tolerance of a product of two
    # rounded values).
    M, N, K = 160, 256, 192
    x = rand_bf16(21, (M, K))
    w = rand_bf16(22, (N, K), std=K ** -0.5)
    h = poison_bf16(M, N)
    cuda_lib.swiglu_dual_gemm(up(x), up(w), up(w), "nk", h, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.swiglu(x, w, w, "nk", M=M, N=N, K=K)
    assert_parity(down(h), ref, "swiglu same weights")


# ------------------------------------------------------------------ W4A16

def w4_case(M, N, K, G, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    A = rand_bf16(seed, (M, K))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    s = workloads.to_bf16_bits(rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float32))
    return A, Wq, s


@pytest.mark.parametrize("M,N,K,G", [(1, 256, 128, 128), (16, 544, 1024, 128),
                                     (20, 256, 512, 64), (64, 32, 256, 128),
                                     (100, 512, 384, 128), (3, 1056, 2048, 256),
                                     (32, 1536, 640, 64), (7, 2080, 8192, 128)])
def test_w4a16_full_output(cuda_lib, M, N, K, G):
    A, Wq, s = w4_case(M, N, K, G, seed=M * 7 + N)
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.w4a16(A, Wq, s, G, M=M, N=N, K=K)
    assert_parity(down(out), ref, f"w4a16 {M}x{N}x{K} G={G}")


@pytest.mark.parametrize("act", ["relu", "silu", "gelu_tanh"])
def test_w4a16_with_ending(cuda_lib, act):
    M, N, K, G = 24, 512, 512, 128
    A, Wq, s = w4_case(M, N, K, G, seed=31)
    C = rand_bf16(32, (M, N))
    bias = rand_bf16(33, (N,), std=0.3)
    res = rand_bf16(34, (M, N))
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, up(C), up(bias), up(res), out, M, N, K, 0.5,
                        0.25, act)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.w4a16(A, Wq, s, G, C, bias, res, M=M, N=N, K=K, alpha=0.5, beta=0.25, act=act)
    assert_parity(down(out), ref, f"w4a16 {act}")


@pytest.mark.parametrize("k0,j,which", [(0, 0, "hi"), (0, 0, "lo"), (77, 5, "hi"),
                                        (130, 127, "lo"), (255, 64, "hi"), (63, 200, "lo")])
def test_w4a16_single_nibble_probe(cuda_lib, k0, j, which):
    # Every code is 8 (weight 0) except one nibble: only output column 2j
    # (high nibble) or 2j+1 (low nibble) may be non-zero, and it must equal
    # A[:, k0] * (q - 8) * s exactly (one bf16 product, one rounding).
    M, N, K, G = 16, 512, 256, 128
    q = 13
    Wq = np.full((K, N // 2), 0x88, dtype=np.uint8)
    Wq[k0, j] = (q << 4) | 8 if which == "hi" else 0x80 | q
    col = 2 * j if which == "hi" else 2 * j + 1
    A = workloads.to_bf16_bits((np.arange(M * K, dtype=np.float32).reshape(M, K) % 9) - 4)
    s = workloads.to_bf16_bits(np.full((K // G, N), 0.25, dtype=np.float32))
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    got = down(out)
    ref = oracle.w4a16(A, Wq, s, G, M=M, N=N, K=K)
    assert np.array_equal(got, ref)
    nz = np.argwhere(oracle.bf16_bits_to_f64(got) != 0)
    assert set(nz[:, 1].tolist()) <= {col}


def test_w4a16_power_of_two_group_scales_exact(cuda_lib):
    # Integer activations and power-of-two scales that differ per group and
    # column: every product and partial sum is exact in fp32, so the GPU
    # result must equal the oracle bit for bit.
    M, N, K, G = 8, 256, 512, 128
    rng = np.random.Generator(np.random.PCG64(41))
    A = workloads.to_bf16_bits(rng.integers(-3, 4, size=(M, K)).astype(np.float32))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    s = workloads.to_bf16_bits((2.0 ** rng.integers(-6, -1, size=(K // G, N))).astype(np.float32))
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    assert np.array_equal(down(out), oracle.w4a16(A, Wq, s, G, M=M, N=N, K=K))


def test_w4a16_all_eights_gives_the_ending_alone(cuda_lib):
    M, N, K, G = 5, 256, 256, 128
    A = rand_bf16(51, (M, K))
    Wq = np.full((K, N // 2), 0x88, dtype=np.uint8)
    s = workloads.to_bf16_bits(np.full((K // G, N), 0.01, dtype=np.float32))
    C = rand_bf16(52, (M, N))
    bias = rand_bf16(53, (N,))
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, up(C), up(bias), None, out, M, N, K, 1.0, 2.0,
                        "silu")
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.w4a16(A, Wq, s, G, C, bias, M=M, N=N, K=K, alpha=1.0, beta=2.0, act="silu")
    assert_parity(down(out), ref, "all eights")


@pytest.mark.parametrize("scales", ["small", "large", "mixed", "tiny_and_negative"])
def test_w4a16_dequantised_operand_is_bit_exact(cuda_lib, scales):
    # One-hot activation rows pick single k-rows, so out[m][n] is the
    # dequantised weight bf16((q - 8) * s) itself (one non-zero product, exact
    # in fp32).  Every code appears in those rows, with scales of general
    # mantissas: below 2^-5 (the kernel's fused multiply-add path), above it
    # (the separate subtract and multiply), both within one warp's columns,
    # and negative and subnormal ones.  The result must equal the oracle's
    # dequantised weight bit for bit.
    M, N, K, G = 16, 1024, 512, 128
    rng = np.random.Generator(np.random.PCG64(77))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    ks = np.array([0, 1, 63, 64, 127, 128, 200, 255, 256, 300, 383, 384, 450, 500, 510, 511])
    for i, k in enumerate(ks):  # every byte value appears in the picked rows
        Wq[k, :256] = np.arange(256, dtype=np.uint8)
    if scales == "small":
        sv = rng.uniform(0.001, 0.031, size=(K // G, N))
    elif scales == "large":
        sv = rng.uniform(0.04, 3.0, size=(K // G, N))
    elif scales == "mixed":
        sv = rng.uniform(0.001, 0.031, size=(K // G, N))
        sv[:, ::37] = rng.uniform(0.04, 3.0, size=sv[:, ::37].shape)
    else:
        sv = rng.uniform(-0.03, 0.03, size=(K // G, N))
        sv[:, ::11] = np.float32(3e-39)  # bf16 subnormal scales
    s = workloads.to_bf16_bits(sv.astype(np.float32))
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), ks] = 0x3F80  # 1.0
    out = poison_bf16(M, N)
    cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    w = oracle.bf16_bits_to_f64(oracle.dequant_int4(Wq, s, G, K=K, N=N)[ks])
    got = oracle.bf16_bits_to_f64(down(out))
    # weights that are themselves bf16 subnormals are left out of the bit-wise
    # comparison (what the tensor cores do with subnormal operands is not the
    # dequantisation's concern); subnormal scales still feed normal weights
    normal = (w == 0) | (np.abs(w) >= 2.0 ** -126)
    assert normal.mean() > 0.9
    assert np.array_equal(got[normal], w[normal])


@pytest.mark.parametrize("scales", ["small", "large"])
def test_fp8_dequantised_operand_is_bit_exact(cuda_lib, scales):
    # As above for FP8 weights: scales below 2^8 take the fused multiply,
    # larger ones the two-step one.
    M, N, K, G = 16, 512, 256, 128
    rng = np.random.Generator(np.random.PCG64(78))
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    Wq = rng.choice(codes, size=(K, N)).astype(np.uint8)
    ks = np.arange(0, K, K // M)
    sv = (rng.uniform(0.001, 200.0, size=(K // G, N)) if scales == "small"
          else rng.uniform(300.0, 3000.0, size=(K // G, N)))
    s = workloads.to_bf16_bits(sv.astype(np.float32))
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), ks] = 0x3F80
    out = poison_bf16(M, N)
    cuda_lib.w8a16_fp8_gemm(up(A), up(Wq), up(s), G, None, None, None, out, M, N, K)
    assert cuda_lib.gbf_check_device_error() == 0
    w = oracle.dequant_wq("fp8", Wq, s, G, K=K, N=N)
    got = down(out)
    ok = np.isfinite(oracle.bf16_bits_to_f64(w[ks]))
    assert np.array_equal(oracle.bf16_bits_to_f64(got)[ok], oracle.bf16_bits_to_f64(w[ks])[ok])

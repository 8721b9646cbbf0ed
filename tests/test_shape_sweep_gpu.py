"""Seeded random shapes through every dense kernel form, against the fp64 oracle.

Each case draws M, N, K (N and K multiples of 8, as the boundary requires),
the weight layout, the activation, alpha / beta and which of C, bias and
residual are present from its own seed, and runs the product twice: with the
planner's choice, and with one of the forms the tuning hook can force (the
one-SM kernel and its split-K form, the CTA-pair kernel with two M-tile
streams, one stream, or split K over two pairs).  The parametrised tests of
the other files pin chosen edge shapes; this file covers combinations of
ragged M, N and K tails, odd K-block counts and operand sets that nobody
picked by hand.  The weight-only kernel (all three weight formats), the
swapped small-M kernel (every split-K cluster size) and the gate/up dual
GEMM get the same treatment."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up
from test_gemm_gpu import case, rand_bf16

pytestmark = pytest.mark.gpu

FORMS = ["persistent", "persistent_splitk", "pair", "pair_1stream", "pair_splitk"]
ACTS = ["identity", "relu", "silu", "gelu_tanh"]


def draw(seed):
    rng = np.random.Generator(np.random.PCG64(9000 + seed))
    M = int(rng.integers(129, 900))           # above the swapped kernel's range
    N = 8 * int(rng.integers(1, 160))         # 8 .. 1272
    K = 8 * int(rng.integers(1, 100))         # 8 .. 792 (1 .. 13 K blocks)
    layout = ["kn", "nk"][int(rng.integers(0, 2))]
    act = ACTS[int(rng.integers(0, 4))]
    alpha = float(rng.choice([0.5, 1.0, 1.25]))
    beta = float(rng.choice([-0.5, 0.0, 0.75]))
    c, bias, res = (bool(x) for x in rng.integers(0, 2, size=3))
    form = FORMS[seed % len(FORMS)]
    return M, N, K, layout, act, alpha, beta, c, bias, res, form


@pytest.mark.parametrize("seed", range(20))
def test_random_shape_every_form(cuda_lib, seed):
    M, N, K, layout, act, alpha, beta, c, bias, res, form = draw(seed)
    A, B, C, bi, r = case(M, N, K, layout, 500 + seed, c, bias, res)
    ref = oracle.gemm_epilogue(A, B, layout, C, bi, r, M=M, N=N, K=K, alpha=alpha, beta=beta,
                               act=act)
    for forced in (None, form):
        assert cuda_lib.gbf_debug_force_path(forced) == 0
        try:
            path = cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, layout)[0]
            out = poison_bf16(M, N)
            cuda_lib.gemm_epilogue(up(A), up(B), layout, up(C), up(bi), up(r), out, M, N, K,
                                   alpha, beta, act)
        finally:
            cuda_lib.gbf_debug_force_path(None)
        assert cuda_lib.gbf_check_device_error() == 0
        assert_parity(down(out), ref, f"seed {seed}: {M}x{N}x{K} {layout} {act} via {path}")


def draw_wq(seed):
    rng = np.random.Generator(np.random.PCG64(9500 + seed))
    fmt = ["int4", "fp8", "nvfp4"][seed % 3]
    M = int(rng.integers(1, 70))
    N = 32 * int(rng.integers(1, 70))        # 32 .. 2208
    if fmt == "nvfp4":
        G = 16
        K = 16 * int(rng.integers(1, 80))    # 16 .. 1264
    else:
        G = int(rng.choice([64, 128, 256]))
        K = G * int(rng.integers(1, 10))
    act = ACTS[int(rng.integers(0, 4))]
    alpha = float(rng.choice([0.5, 1.0, 1.25]))
    beta = float(rng.choice([-0.5, 0.0, 0.75]))
    c, bias, res = (bool(x) for x in rng.integers(0, 2, size=3))
    return fmt, M, N, K, G, act, alpha, beta, c, bias, res, rng


@pytest.mark.parametrize("seed", range(15))
def test_random_shape_weight_only(cuda_lib, seed):
    # the weight-only kernel at random M (one or more 16 / 32-row M-tiles),
    # N and K, random scales and operand sets, in all three weight formats
    fmt, M, N, K, G, act, alpha, beta, c, bias, res, rng = draw_wq(seed)
    A = rand_bf16(700 + seed, (M, K))
    C = rand_bf16(720 + seed, (M, N)) if c else None
    bi = rand_bf16(740 + seed, (N,), std=0.3) if bias else None
    r = rand_bf16(760 + seed, (M, N)) if res else None
    if fmt == "fp8":
        Wq = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
        Wq[(Wq & 0x7F) == 0x7F] = 0x38  # no NaN codes (not valid weights)
        s = workloads.to_bf16_bits(rng.uniform(0.25, 2.0, (K // G, N)).astype(np.float32))
    elif fmt == "int4":
        Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
        s = workloads.to_bf16_bits(rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float32))
    else:
        Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
        s = rng.integers(0x28, 0x40, size=(K // 16, N), dtype=np.uint8)  # E4M3 0.25 .. 1.875
    ref = oracle.wq_gemm(fmt, A, Wq, s, G, C, bi, r, M=M, N=N, K=K, alpha=alpha, beta=beta,
                         act=act)
    out = poison_bf16(M, N)
    args = (up(C), up(bi), up(r), out, M, N, K, alpha, beta, act)
    if fmt == "int4":
        cuda_lib.w4a16_gemm(up(A), up(Wq), up(s), G, *args)
    elif fmt == "fp8":
        cuda_lib.w8a16_fp8_gemm(up(A), up(Wq), up(s), G, *args)
    else:
        cuda_lib.w4a16_nvfp4_gemm(up(A), up(Wq), up(s), *args)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(out), ref, f"seed {seed}: {fmt} {M}x{N}x{K} G={G} {act}")


@pytest.mark.parametrize("seed", range(15))
def test_random_shape_small_m_every_split_count(cuda_lib, seed):
    # the swapped kernel (M <= 128) at random shapes with the split-K
    # cluster size forced to a random 1..8 (0: the automatic choice)
    rng = np.random.Generator(np.random.PCG64(9800 + seed))
    M = int(rng.integers(1, 129))
    N = 8 * int(rng.integers(1, 140))
    K = 8 * int(rng.integers(1, 250))
    layout = ["kn", "nk"][int(rng.integers(0, 2))]
    act = ACTS[int(rng.integers(0, 4))]
    alpha, beta = float(rng.choice([0.5, 1.0])), float(rng.choice([0.0, 0.5]))
    c, bias, res = (bool(x) for x in rng.integers(0, 2, size=3))
    splits = int(rng.integers(0, 9))
    A, B, C, bi, r = case(M, N, K, layout, 800 + seed, c, bias, res)
    assert cuda_lib.gbf_debug_force_splits(splits) == 0
    try:
        path, S = cuda_lib.gbf_kernel_path("gemm_epilogue", M, N, K, layout)
        assert path == "swap_splitk"
        out = poison_bf16(M, N)
        cuda_lib.gemm_epilogue(up(A), up(B), layout, up(C), up(bi), up(r), out, M, N, K, alpha,
                               beta, act)
    finally:
        cuda_lib.gbf_debug_force_splits(0)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.gemm_epilogue(A, B, layout, C, bi, r, M=M, N=N, K=K, alpha=alpha, beta=beta,
                               act=act)
    assert_parity(down(out), ref, f"seed {seed}: {M}x{N}x{K} {layout} {act} S={S}")


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_gate_up(cuda_lib, seed):
    # the gate/up dual GEMM at random shapes on whichever kernel the planner
    # picks (swapped for M <= 32, else the persistent or CTA-pair kernel)
    rng = np.random.Generator(np.random.PCG64(9900 + seed))
    M = int(rng.integers(1, 600))
    N = 8 * int(rng.integers(1, 120))
    K = 8 * int(rng.integers(1, 120))
    layout = ["kn", "nk"][int(rng.integers(0, 2))]
    act = ["silu", "gelu_tanh", "relu"][int(rng.integers(0, 3))]
    alpha, beta = float(rng.choice([0.75, 1.0])), float(rng.choice([0.0, -0.5]))
    x = rand_bf16(900 + seed, (M, K))
    shp = (N, K) if layout == "nk" else (K, N)
    wg = rand_bf16(920 + seed, shp, std=K ** -0.5)
    wu = rand_bf16(940 + seed, shp, std=K ** -0.5)
    C = rand_bf16(960 + seed, (M, N)) if beta != 0.0 else None
    h = poison_bf16(M, N)
    path = cuda_lib.gbf_kernel_path("swiglu", M, N, K, layout)[0]
    cuda_lib.swiglu_dual_gemm(up(x), up(wg), up(wu), layout, h, M, N, K, alpha, beta, up(C), act)
    assert cuda_lib.gbf_check_device_error() == 0
    ref = oracle.swiglu(x, wg, wu, layout, C, M=M, N=N, K=K, alpha=alpha, beta=beta, act=act)
    assert_parity(down(h), ref, f"seed {seed}: swiglu {M}x{N}x{K} {layout} {act} via {path}")

"""GPU parity of the weight-only GEMMs with FP8 (E4M3, bf16 group scales) and
NVFP4 (E2M1 codes, E4M3 scales per 16 along K, per-tensor factor as alpha)
weights ("Fusion Thinking", Pattern 3: weight-only quantisation with BF16
activations, dequantised on-chip), and of their unfused compositions
(dequantise into a bf16 weight in HBM, then the bf16 GEMM)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up, widen

pytestmark = pytest.mark.gpu


def fp8_inputs(M, N, K, G, seed):
    w = workloads.make("w8a16_fp8", shape=dict(M=M, N=N, K=K, group=G))
    if seed:
        rng = np.random.Generator(np.random.PCG64(seed))
        w["A"] = workloads.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    return w


def nvfp4_inputs(M, N, K, seed):
    w = workloads.make("w4a16_nvfp4", shape=dict(M=M, N=N, K=K))
    if seed:
        rng = np.random.Generator(np.random.PCG64(seed))
        w["A"] = workloads.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    return w


def run(cuda_lib, kind, w, M, N, K, C=None, bias=None, residual=None, alpha=None, beta=0.0,
        act="identity", fused=True):
    out = poison_bf16(M, N)
    alpha = w["alpha"] if alpha is None else alpha
    args = dict(C=up(C), bias=up(bias), residual=up(residual), out=out, M=M, N=N, K=K,
                alpha=alpha, beta=beta, act=act)
    ws = None
    if not fused:
        nbytes = cuda_lib.gbf_workspace_size(kind, M, N, K, False)
        ws = torch.full((max(nbytes, 256),), 0xFF, dtype=torch.uint8, device="cuda")
        args.update(workspace=ws, workspace_bytes=nbytes)
    if kind == "w8a16_fp8":
        fn = cuda_lib.w8a16_fp8_gemm if fused else cuda_lib.w8a16_fp8_gemm_unfused
        fn(up(w["A"]), up(w["Wq"]), up(w["scales"]), w["group"], **args)
    else:
        fn = cuda_lib.w4a16_nvfp4_gemm if fused else cuda_lib.w4a16_nvfp4_gemm_unfused
        fn(up(w["A"]), up(w["Wq"]), up(w["scales"]), **args)
    assert cuda_lib.gbf_check_device_error() == 0
    return down(out), ws


def want(kind, w, M, N, K, **kw):
    fmt = "fp8" if kind == "w8a16_fp8" else "nvfp4"
    kw.setdefault("alpha", w["alpha"])
    return oracle.wq_gemm(fmt, w["A"], w["Wq"], w["scales"], w["group"], M=M, N=N, K=K, **kw)


@pytest.mark.parametrize("M,N,K,G", [(1, 512, 64, 64), (16, 1024, 1024, 128), (5, 32, 256, 64),
                                     (17, 544, 512, 512), (32, 4096, 2048, 128),
                                     (33, 1056, 384, 128)])
def test_fp8_fused(cuda_lib, M, N, K, G):
    w = fp8_inputs(M, N, K, G, seed=M + N)
    got, _ = run(cuda_lib, "w8a16_fp8", w, M, N, K)
    assert_parity(got, want("w8a16_fp8", w, M, N, K), f"fp8 {M}x{N}x{K} G{G}")


@pytest.mark.parametrize("M,N,K", [(1, 512, 16), (16, 1024, 1024), (5, 32, 48), (17, 544, 80),
                                   (32, 4096, 2048), (33, 1056, 400)])
def test_nvfp4_fused(cuda_lib, M, N, K):
    w = nvfp4_inputs(M, N, K, seed=M + N)
    got, _ = run(cuda_lib, "w4a16_nvfp4", w, M, N, K)
    assert_parity(got, want("w4a16_nvfp4", w, M, N, K), f"nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("scale", [2.0 ** -40, 2.0 ** 40])
def test_nvfp4_alpha_far_from_one(cuda_lib, scale):
    """The NVFP4 kernel carries its operand scaled by 2^-19 and multiplies
    alpha by 2^19; the result must not depend on where alpha sits."""
    M, N, K = 16, 1024, 1024
    w = nvfp4_inputs(M, N, K, seed=7)
    got1, _ = run(cuda_lib, "w4a16_nvfp4", w, M, N, K)
    assert_parity(got1, want("w4a16_nvfp4", w, M, N, K), "nvfp4")
    got, _ = run(cuda_lib, "w4a16_nvfp4", w, M, N, K, alpha=w["alpha"] * scale)
    # alpha * acc is one fp32 product, so a power-of-two factor on alpha
    # scales every output exactly (nothing here leaves the normal range)
    np.testing.assert_array_equal(widen(got), widen(got1) * scale)


@pytest.mark.parametrize("kind", ["w8a16_fp8", "w4a16_nvfp4"])
@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "relu"])
def test_full_ending(cuda_lib, kind, act):
    M, N, K = 16, 1024, 512
    w = fp8_inputs(M, N, K, 128, 3) if kind == "w8a16_fp8" else nvfp4_inputs(M, N, K, 3)
    rng = np.random.Generator(np.random.PCG64(7))
    C, bias, res = (workloads.to_bf16_bits(rng.standard_normal(s).astype(np.float32))
                    for s in ((M, N), (N,), (M, N)))
    kw = dict(C=C, bias=bias, residual=res, alpha=0.75, beta=0.5, act=act)
    got, _ = run(cuda_lib, kind, w, M, N, K, **kw)
    assert_parity(got, want(kind, w, M, N, K, **kw), f"{kind} {act}")


def test_fp8_every_code_including_subnormals_is_exact(cuda_lib):
    # A = one-hot rows picking k-rows; scale 1: out[m][n] = e4m3(q[k_m][n]),
    # bit-exact, for all 254 finite codes (the subnormals 0x01..0x07 and
    # 0x81..0x87 included).
    M, N, K, G = 16, 512, 64, 64
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    Wq = np.zeros((K, N), dtype=np.uint8)
    Wq[:16].flat[:codes.size] = codes
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), np.arange(M)] = 0x3F80  # 1.0
    s = np.full((K // G, N), 0x3F80, dtype=np.uint16)
    w = dict(A=A, Wq=Wq, scales=s, group=G, alpha=1.0)
    got, _ = run(cuda_lib, "w8a16_fp8", w, M, N, K)
    ref = want("w8a16_fp8", w, M, N, K)
    assert np.array_equal(oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(ref))
    vals = oracle.bf16_bits_to_f64(got).ravel()[:codes.size]
    assert np.array_equal(vals, [oracle.fp8_e4m3_to_f64(c) for c in codes])


def test_nvfp4_codes_nibble_order_and_block_scales_are_exact(cuda_lib):
    # one-hot A rows pick k-rows 0, 17, 33, 63; every byte value appears in
    # those rows; each 16-deep block has its own E4M3 scale (0.25, 1, 3, 448).
    M, N, K = 4, 512, 64
    Wq = np.zeros((K, N // 2), dtype=np.uint8)
    ks = [0, 17, 33, 63]
    for k in ks:
        Wq[k] = np.arange(256, dtype=np.uint8)
    S = np.zeros((K // 16, N), dtype=np.uint8)
    for b, c in enumerate((0x28, 0x38, 0x44, 0x7E)):
        S[b] = c
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), ks] = 0x3F80
    w = dict(A=A, Wq=Wq, scales=S, group=16, alpha=1.0)
    got, _ = run(cuda_lib, "w4a16_nvfp4", w, M, N, K)
    ref = want("w4a16_nvfp4", w, M, N, K)
    assert np.array_equal(oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(ref))
    e2m1 = [oracle.fp4_e2m1_to_f64(c) for c in range(16)]
    row = oracle.bf16_bits_to_f64(got)[1]  # k = 17: block 1, scale 1
    assert row[0] == e2m1[0] and row[2 * 0x5A] == e2m1[5] and row[2 * 0x5A + 1] == e2m1[0xA]


@pytest.mark.parametrize("kind", ["w8a16_fp8", "w4a16_nvfp4"])
def test_unfused_stagewise(cuda_lib, kind):
    M, N, K = 16, 1024, 512
    w = fp8_inputs(M, N, K, 128, 5) if kind == "w8a16_fp8" else nvfp4_inputs(M, N, K, 5)
    got, ws = run(cuda_lib, kind, w, M, N, K, fused=False)
    fmt = "fp8" if kind == "w8a16_fp8" else "nvfp4"
    W = down(ws[:K * N * 2].view(torch.bfloat16).view(K, N))
    # the dequantised weight is exact up to its one defined rounding: bit-exact
    want_w = oracle.dequant_wq(fmt, w["Wq"], w["scales"], w["group"], K=K, N=N)
    assert np.array_equal(oracle.bf16_bits_to_f64(W), oracle.bf16_bits_to_f64(want_w))
    assert_parity(got, oracle.gemm_epilogue(w["A"], W, "kn", M=M, N=N, K=K, alpha=w["alpha"]),
                  f"{kind} unfused")


@pytest.mark.parametrize("kind", ["w8a16_fp8", "w4a16_nvfp4"])
def test_decode_workload_full_output(cuda_lib, kind):
    # every one of the 16 x 28672 outputs (3.8e9 multiply-adds in the oracle,
    # run on all host cores)
    w = workloads.make(kind)
    M, N, K = w["M"], w["N"], w["K"]
    got, _ = run(cuda_lib, kind, w, M, N, K)
    with oracle.all_cores():
        ref = want(kind, w, M, N, K)
    assert_parity(got, ref, f"{kind} workload, full output")


def test_validation(cuda_lib):
    t = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    f8 = lambda **kw: cuda_lib.w8a16_fp8_gemm(**{**dict(
        A=t, Wq=q, scales=t, group_size=64, C=None, bias=None, residual=None, out=t, M=4,
        N=64, K=128), **kw}, raise_on_error=False)
    nv = lambda **kw: cuda_lib.w4a16_nvfp4_gemm(**{**dict(
        A=t, Wq=q, scales=q, C=None, bias=None, residual=None, out=t, M=4, N=64, K=128), **kw},
        raise_on_error=False)
    assert f8() == 0 and nv() == 0
    assert f8(group_size=32) == 3
    assert f8(K=96) == 3
    assert f8(N=48) == 3
    assert f8(group_size=0) == 1
    assert nv(K=24) == 3
    assert nv(N=48) == 3
    assert nv(scales=None) == 1
    assert nv(Wq=q[1:]) == 2
    ws_need = cuda_lib.gbf_workspace_size("w4a16_nvfp4", 4, 64, 128, False)
    assert ws_need == 64 * 128 * 2
    assert cuda_lib.w4a16_nvfp4_gemm_unfused(t, q, q, None, None, None, t, 4, 64, 128,
                                             workspace=None, raise_on_error=False) == 4
    torch.cuda.synchronize()

"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test ties one part of the oracle to something independent of it: a
hand-worked example under tests/golden/, a library routine (numpy matmul,
torch's bf16 cast and activations) in a special case, exact integer
arithmetic, or an invariant.  A plausible mistake in the oracle (a dropped
term, a wrong sign, a transposed operand, the other nibble order, a wrong
group index, a wrong GELU constant, round-half-up) fails at least one of
them.  CPU only.

Every pin runs twice: against the single-threaded build of the oracle and
against its OpenMP build (the same C file, the loop over output elements
shared among threads), and the two builds are also compared bit for bit on
the five workloads' shapes in miniature.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(autouse=True, params=["serial", "openmp"])
def oracle_build(request):
    prev = oracle.set_parallel(request.param == "openmp")
    yield request.param
    oracle.set_parallel(prev)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bits(x):
    """Exact bf16 bit patterns of values that are already bf16-exact."""
    arr = np.asarray(x, dtype=np.float32)
    b = to_bf16_bits(arr)
    assert np.array_equal(oracle.bf16_bits_to_f64(b), arr.astype(np.float64)), "value not bf16-exact"
    return b


# ---------------------------------------------------------------- bf16 rounding

@pytest.mark.parametrize("value,expected", [
    (1.0, 0x3F80),
    (-2.0, 0xC000),
    (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above the tie
    (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),    # just below the tie
    (2.0 ** -126, 0x0080),                     # smallest normal
    (2.0 ** -133, 0x0001),                     # smallest subnormal
    (2.0 ** -134, 0x0000),                     # tie between 0 and 2^-133 -> even
    (3 * 2.0 ** -134, 0x0002),                 # tie between 1 and 2 ulps -> even
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # tie at the top rounds to even = inf
    (float("inf"), 0x7F80),
    (-float("inf"), 0xFF80),
    (-0.0, 0x8000),
    (0.0, 0x0000),
])
def test_bf16_round_nearest_even_hand_values(value, expected):
    assert oracle.bf16_from_f64(value) == expected


def test_bf16_nan():
    h = oracle.bf16_from_f64(float("nan"))
    assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0


def test_bf16_round_matches_torch_cast_on_float32_values():
    # For values that are exact float32, one RNE step to bf16 is what torch's
    # float32 -> bf16 cast does; compare 20k random values spanning the range.
    rng = np.random.Generator(np.random.PCG64(1234))
    mant = rng.standard_normal(20000).astype(np.float32)
    expo = rng.integers(-140, 120, size=20000)
    vals = (mant * np.float32(2.0) ** expo.astype(np.float32)).astype(np.float32)
    vals = vals[np.isfinite(vals)]
    want = to_bf16_bits(vals)
    got = np.array([oracle.bf16_from_f64(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_widening_round_trip_all_patterns():
    lib = oracle._load()
    for h in range(0, 1 << 16, 7):
        if (h & 0x7F80) == 0x7F80 and (h & 0x7F):
            continue  # NaN payloads
        assert lib.oracle_bf16_from_f64(lib.oracle_bf16_to_f64(h)) == h


# ---------------------------------------------------------------- activations

def test_activation_special_values():
    assert oracle.act("silu", 0.0) == 0.0
    assert oracle.act("gelu_tanh", 0.0) == 0.0
    assert oracle.act("relu", -3.5) == 0.0
    assert oracle.act("relu", 2.25) == 2.25
    assert oracle.act("identity", -1.5) == -1.5
    assert oracle.act("silu", -800.0) == 0.0        # v * sigmoid(v) -> 0
    assert oracle.act("silu", 800.0) == 800.0


def test_silu_and_gelu_tanh_match_torch_float64():
    xs = torch.linspace(-12, 12, 4801, dtype=torch.float64)
    silu = torch.nn.functional.silu(xs)
    gelu = torch.nn.functional.gelu(xs, approximate="tanh")
    for x, s, g in zip(xs.tolist(), silu.tolist(), gelu.tolist()):
        assert oracle.act("silu", x) == pytest.approx(s, rel=1e-13, abs=1e-300)
        assert oracle.act("gelu_tanh", x) == pytest.approx(g, rel=1e-12, abs=1e-15)


def test_gelu_tanh_is_an_approximation_of_erf_gelu():
    # The tanh form stays within ~5e-4 of x*Phi(x) (textbook bound) and is
    # not the erf form itself.
    worst = 0.0
    for x in np.linspace(-6, 6, 1201):
        exact = 0.5 * x * (1 + math.erf(x / math.sqrt(2)))
        worst = max(worst, abs(oracle.act("gelu_tanh", float(x)) - exact))
    assert 1e-5 < worst < 5e-4


# ---------------------------------------------------------------- GEMM + epilogue

def test_epilogue_hand_worked_example():
    g = _golden("epilogue_hand.json")
    A, B, C = bits(g["A"]), bits(g["B_kn"]), bits(g["C"])
    bias, res = bits(g["bias"]), bits(g["residual"])
    W = np.ascontiguousarray(B.T)
    for act in ("relu", "identity"):
        want = np.array([int(h, 16) for h in g[act]["out_bits"]], dtype=np.uint16).reshape(2, 2)
        for layout, Bm in (("kn", B), ("nk", W)):
            got = oracle.gemm_epilogue(A, Bm, layout, C, bias, res, M=2, N=2, K=3,
                                       alpha=g["alpha"], beta=g["beta"], act=act)
            assert np.array_equal(got, want), (act, layout, got, want)
    plain = oracle.gemm_epilogue(A, B, "kn", M=2, N=2, K=3, want_f64=True)[1]
    assert np.array_equal(plain, np.array(g["AB"], dtype=np.float64))


def test_plain_product_matches_numpy_matmul():
    # alpha=1, beta=0, no bias/residual, identity: the plain product.
    rng = np.random.Generator(np.random.PCG64(7))
    M, N, K = 5, 7, 33
    A = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    B = to_bf16_bits(rng.standard_normal((K, N)).astype(np.float32))
    Af, Bf = oracle.bf16_bits_to_f64(A), oracle.bf16_bits_to_f64(B)
    _, got = oracle.gemm_epilogue(A, B, "kn", M=M, N=N, K=K, want_f64=True)
    np.testing.assert_allclose(got, Af @ Bf, rtol=1e-12, atol=1e-12)
    _, got_nk = oracle.gemm_epilogue(A, np.ascontiguousarray(B.T), "nk", M=M, N=N, K=K,
                                     want_f64=True)
    np.testing.assert_allclose(got_nk, Af @ Bf, rtol=1e-12, atol=1e-12)


def test_integer_inputs_are_exact_and_rounded_once():
    rng = np.random.Generator(np.random.PCG64(8))
    M, N, K = 9, 12, 200
    A = rng.integers(-16, 17, size=(M, K)).astype(np.float32)
    B = rng.integers(-16, 17, size=(K, N)).astype(np.float32)
    exact = A.astype(np.int64) @ B.astype(np.int64)
    _, f64 = oracle.gemm_epilogue(bits(A), bits(B), "kn", M=M, N=N, K=K, want_f64=True)
    assert np.array_equal(f64, exact.astype(np.float64))
    out = oracle.gemm_epilogue(bits(A), bits(B), "kn", M=M, N=N, K=K)
    assert np.array_equal(out, to_bf16_bits(exact.astype(np.float32)))


def test_identity_b_reduces_to_pointwise_of_a():
    # B = I: out = act(alpha*A + beta*C + bias) + residual, with torch's
    # float64 activation as the independent reference.
    rng = np.random.Generator(np.random.PCG64(9))
    n = 16
    A = to_bf16_bits(rng.standard_normal((n, n)).astype(np.float32))
    C = to_bf16_bits(rng.standard_normal((n, n)).astype(np.float32))
    bias = to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    res = to_bf16_bits(rng.standard_normal((n, n)).astype(np.float32))
    eye = bits(np.eye(n))
    f = oracle.bf16_bits_to_f64
    for act, fn in (("silu", torch.nn.functional.silu),
                    ("gelu_tanh", lambda t: torch.nn.functional.gelu(t, approximate="tanh")),
                    ("relu", torch.relu), ("identity", lambda t: t)):
        pre = torch.from_numpy(0.75 * f(A) + 0.25 * f(C) + f(bias)[None, :])
        want = fn(pre).numpy() + f(res)
        _, got = oracle.gemm_epilogue(A, eye, "kn", C, bias, res, M=n, N=n, K=n,
                                      alpha=0.75, beta=0.25, act=act, want_f64=True)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_zero_a_gives_closed_form_and_null_operands_are_zero():
    n = 8
    A = np.zeros((n, 5), dtype=np.uint16)
    B = bits(np.arange(40, dtype=np.float32).reshape(5, n))
    C = bits(np.full((n, n), 2.0))
    bias_v = np.arange(n) * 0.5 - 2.0
    bias = bits(bias_v)
    res = bits(np.full((n, n), -1.0))
    out = oracle.gemm_epilogue(A, B, "kn", C, bias, res, M=n, N=n, K=5, alpha=3.0,
                               beta=0.5, act="relu")
    want = np.maximum(1.0 + bias_v, 0)[None, :] - 1.0
    assert np.array_equal(out, to_bf16_bits(np.broadcast_to(want, (n, n)).astype(np.float32)))
    # Null C ignores beta entirely; K = 0 is an empty sum.
    out0 = oracle.gemm_epilogue(A[:, :0].copy(), B[:0].copy(), "kn", None, bias, None,
                                M=n, N=n, K=0, beta=123.0, act="identity")
    assert np.array_equal(out0, np.broadcast_to(bias, (n, n)))


def test_sampled_elements_equal_full_output():
    rng = np.random.Generator(np.random.PCG64(10))
    M, N, K = 6, 10, 17
    A = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    B = to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    C = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    full = oracle.gemm_epilogue(A, B, "nk", C, M=M, N=N, K=K, alpha=0.5, beta=2.0, act="silu")
    r = np.array([0, 5, 3, 2]); c = np.array([9, 0, 4, 4])
    part = oracle.gemm_epilogue(A, B, "nk", C, M=M, N=N, K=K, alpha=0.5, beta=2.0,
                                act="silu", rows=r, cols=c)
    assert np.array_equal(part, full[r, c])


def test_unfused_mode_rounds_the_product_first():
    # unfused = bf16(D) then the pointwise pass; with torch's bf16 cast of the
    # numpy product as D the two stages agree with the one-call unfused mode.
    rng = np.random.Generator(np.random.PCG64(11))
    M, N, K = 8, 16, 64
    A = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    B = to_bf16_bits(rng.standard_normal((K, N)).astype(np.float32))
    C = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    f = oracle.bf16_bits_to_f64
    D = torch.from_numpy(f(A) @ f(B)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    two_stage = oracle.pointwise_epilogue(D, C, M=M, N=N, alpha=0.5, beta=2.0, act="gelu_tanh")
    one_call = oracle.gemm_epilogue(A, B, "kn", C, M=M, N=N, K=K, alpha=0.5, beta=2.0,
                                    act="gelu_tanh", unfused=True)
    assert np.array_equal(two_stage, one_call)


# ---------------------------------------------------------------- SwiGLU

def test_swiglu_hand_worked_example():
    g = _golden("swiglu_hand.json")
    x, wg, wu, C = bits(g["x"]), bits(g["wg_kn"]), bits(g["wu_kn"]), bits(g["C"])
    for case in g["cases"]:
        for layout, a, b in (("kn", wg, wu), ("nk", np.ascontiguousarray(wg.T),
                                               np.ascontiguousarray(wu.T))):
            _, h = oracle.swiglu(x, a, b, layout, C if case["use_c"] else None, M=2, N=2, K=3,
                                 alpha=case["alpha"], beta=case["beta"], act="relu",
                                 want_f64=True)
            assert np.array_equal(h, np.array(case["h"], dtype=np.float64)), (case, layout)


def test_swiglu_silu_matches_library_composition():
    # alpha=1, beta=0: h = silu(g) * u with g, u from numpy matmul and torch's
    # float64 SiLU.
    rng = np.random.Generator(np.random.PCG64(12))
    M, N, K = 6, 9, 40
    x = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    wg = to_bf16_bits((rng.standard_normal((N, K)) / 4).astype(np.float32))
    wu = to_bf16_bits((rng.standard_normal((N, K)) / 4).astype(np.float32))
    f = oracle.bf16_bits_to_f64
    gm, um = f(x) @ f(wg).T, f(x) @ f(wu).T
    want = torch.nn.functional.silu(torch.from_numpy(gm)).numpy() * um
    _, h = oracle.swiglu(x, wg, wu, "nk", M=M, N=N, K=K, act="silu", want_f64=True)
    np.testing.assert_allclose(h, want, rtol=1e-12, atol=1e-14)
    # Same weights for gate and up: h = silu(g) * g.
    _, hh = oracle.swiglu(x, wg, wg, "nk", M=M, N=N, K=K, act="silu", want_f64=True)
    np.testing.assert_allclose(hh, torch.nn.functional.silu(torch.from_numpy(gm)).numpy() * gm,
                               rtol=1e-12, atol=1e-14)
    # Unfused mode: g and u rounded to bf16 first.
    gb = torch.from_numpy(gm).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ub = torch.from_numpy(um).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.swiglu_pointwise(gb, ub, M=M, N=N),
                          oracle.swiglu(x, wg, wu, "nk", M=M, N=N, K=K, unfused=True))


# ---------------------------------------------------------------- W4A16

def test_w4a16_hand_worked_example():
    g = _golden("w4a16_hand.json")
    A, s, bias = bits(g["A"]), bits(g["scales"]), bits(g["bias"])
    Wq = np.array(g["Wq"], dtype=np.uint8)
    w = oracle.dequant_int4(Wq, s, g["group_size"], K=2, N=2)
    assert np.array_equal(oracle.bf16_bits_to_f64(w), np.array(g["w"]))
    _, out = oracle.w4a16(A, Wq, s, 2, M=1, N=2, K=2, want_f64=True)
    assert np.array_equal(out, np.array(g["out_no_bias"]))
    _, out = oracle.w4a16(A, Wq, s, 2, None, bias, M=1, N=2, K=2, want_f64=True)
    assert np.array_equal(out, np.array(g["out_bias"]))


def test_w4a16_code_eight_is_zero_weight():
    rng = np.random.Generator(np.random.PCG64(13))
    M, N, K, G = 3, 8, 256, 128
    A = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    Wq = np.full((K, N // 2), 0x88, dtype=np.uint8)
    s = to_bf16_bits(rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float32))
    C = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    bias = to_bf16_bits(rng.standard_normal(N).astype(np.float32))
    res = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    assert not np.any(oracle.bf16_bits_to_f64(oracle.dequant_int4(Wq, s, G, K=K, N=N)))
    got = oracle.w4a16(A, Wq, s, G, C, bias, res, M=M, N=N, K=K, alpha=2.0, beta=0.5,
                       act="relu")
    zero_a = np.zeros_like(A)
    want = oracle.gemm_epilogue(zero_a, np.zeros((K, N), np.uint16), "kn", C, bias, res,
                                M=M, N=N, K=K, alpha=2.0, beta=0.5, act="relu")
    assert np.array_equal(got, want)


@pytest.mark.parametrize("which", ["hi", "lo"])
def test_w4a16_single_nibble_probe_fixes_nibble_order(which):
    # Only one code differs from 8: byte j of row k0.  The high nibble feeds
    # column 2j, the low nibble column 2j+1 (interleave(w_hi, w_lo)).
    M, N, K, G = 2, 16, 256, 128
    k0, j, q = 130, 5, 13
    Wq = np.full((K, N // 2), 0x88, dtype=np.uint8)
    Wq[k0, j] = (q << 4) | 8 if which == "hi" else (8 << 4) | q
    col = 2 * j if which == "hi" else 2 * j + 1
    A = bits(np.arange(M * K, dtype=np.float32).reshape(M, K) % 7 - 3)
    s = bits(np.full((K // G, N), 0.25))
    _, out = oracle.w4a16(A, Wq, s, G, M=M, N=N, K=K, want_f64=True)
    want = np.zeros((M, N))
    want[:, col] = oracle.bf16_bits_to_f64(A[:, k0]) * (q - 8) * 0.25
    assert np.array_equal(out, want)


def test_w4a16_group_scales_index_k_over_group_size():
    # Power-of-two scales, different per group and column, integer
    # activations: every product is exact, so the fp64 result is exact and
    # equals an independent numpy evaluation with the scales repeated G times
    # along K.
    rng = np.random.Generator(np.random.PCG64(14))
    M, N, K, G = 4, 32, 512, 128
    A = bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    expo = rng.integers(-8, -2, size=(K // G, N))
    s = bits((2.0 ** expo).astype(np.float32))
    codes = np.empty((K, N), dtype=np.int64)
    codes[:, 0::2] = Wq >> 4
    codes[:, 1::2] = Wq & 0xF
    w = (codes - 8) * np.repeat(2.0 ** expo, G, axis=0)
    want = oracle.bf16_bits_to_f64(A) @ w
    _, got = oracle.w4a16(A, Wq, s, G, M=M, N=N, K=K, want_f64=True)
    assert np.array_equal(got, want)


def test_w4a16_equals_dequantise_then_gemm():
    rng = np.random.Generator(np.random.PCG64(15))
    M, N, K, G = 5, 24, 384, 128
    A = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    s = to_bf16_bits(rng.uniform(0.005, 0.02, (K // G, N)).astype(np.float32))
    C = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    w = oracle.dequant_int4(Wq, s, G, K=K, N=N)
    a = oracle.w4a16(A, Wq, s, G, C, M=M, N=N, K=K, alpha=0.5, beta=1.5, act="gelu_tanh")
    b = oracle.gemm_epilogue(A, w, "kn", C, M=M, N=N, K=K, alpha=0.5, beta=1.5,
                             act="gelu_tanh")
    assert np.array_equal(a, b)
    # Each dequantised weight is one RNE rounding of the exact (q-8)*s.
    f = oracle.bf16_bits_to_f64
    codes = np.empty((K, N), dtype=np.int64)
    codes[:, 0::2] = Wq >> 4
    codes[:, 1::2] = Wq & 0xF
    exact = (codes - 8) * np.repeat(f(s), G, axis=0)
    assert np.array_equal(w, to_bf16_bits(exact.astype(np.float32)))


def test_oracle_rejects_bad_arguments():
    A = np.zeros((2, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.w4a16(A, np.zeros((4, 1), np.uint8), np.zeros((1, 2), np.uint16), 3,
                     M=2, N=2, K=4)
    with pytest.raises(ValueError):
        oracle.gemm_epilogue(A, np.zeros((4, 2), np.uint16), "kn", M=2, N=2, K=4,
                             rows=np.array([2]), cols=np.array([0]))


# ---------------------------------------------------------------- add + RMSNorm

def test_add_rmsnorm_hand_worked_example():
    g = _golden("add_rmsnorm_hand.json")
    a, x, w = bits(g["a"]), bits(g["x"]), bits(g["w"])
    norm, resid = oracle.add_rmsnorm(a, x, w, M=3, N=4, eps=0.0)
    assert np.array_equal(resid, bits(g["resid"]))
    want = workloads_bf16(np.array(g["norm"], dtype=np.float64))
    # compared as values: 0 * w with w < 0 is -0, equal to the fixture's 0
    assert np.array_equal(oracle.bf16_bits_to_f64(norm), oracle.bf16_bits_to_f64(want))


def workloads_bf16(v64):
    # one RNE rounding of exact float64 values (1.2 and 3.2 are not bf16-exact)
    return np.array([oracle.bf16_from_f64(float(t)) for t in v64.ravel()],
                    dtype=np.uint16).reshape(v64.shape)


def test_add_rmsnorm_matches_torch_rms_norm():
    rng = np.random.Generator(np.random.PCG64(31))
    M, N, eps = 7, 96, 1e-5
    a = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    x = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    w = to_bf16_bits(rng.uniform(0.5, 1.5, N).astype(np.float32))
    f = oracle.bf16_bits_to_f64
    r = torch.from_numpy(f(a) + f(x))
    want = torch.nn.functional.rms_norm(r, (N,), torch.from_numpy(f(w)), eps)
    want_bits = want.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    norm, resid = oracle.add_rmsnorm(a, x, w, M=M, N=N, eps=eps)
    assert np.array_equal(resid, r.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    # float64 torch vs fp64 oracle: equal after one bf16 rounding except at exact ties
    assert np.mean(norm == want_bits) > 0.999
    np.testing.assert_allclose(f(norm), want.numpy(), rtol=2 ** -8, atol=0)


def test_add_rmsnorm_scale_invariance_and_unfused_mode():
    rng = np.random.Generator(np.random.PCG64(32))
    M, N = 4, 64
    a = to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    zero = np.zeros_like(a)
    w = to_bf16_bits(np.ones(N, dtype=np.float32))
    # eps = 0: normalising 4*a gives the same as normalising a (power-of-two scale is exact)
    a4 = to_bf16_bits(oracle.bf16_bits_to_f64(a).astype(np.float32) * 4)
    n1, _ = oracle.add_rmsnorm(a, zero, w, M=M, N=N, eps=0.0)
    n4, _ = oracle.add_rmsnorm(a4, zero, w, M=M, N=N, eps=0.0)
    assert np.array_equal(n1, n4)
    # unfused normalises the stored bf16 residual: equal to fused when r is bf16-exact
    nf, rf = oracle.add_rmsnorm(a, zero, w, M=M, N=N)
    nu, ru = oracle.add_rmsnorm(a, zero, w, M=M, N=N, unfused=True)
    assert np.array_equal(rf, ru) and np.array_equal(nf, nu)


# ---------------------------------------------------------------- MLP block chain

def _bf16_from_f64_torch(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float64)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_mlp_chain_matches_library_composition():
    # h = bf16(silu(x Wg^T) * (x Wu^T)) from numpy matmuls and torch's SiLU;
    # out = h Wd^T + residual in float64 before the final rounding.
    rng = np.random.Generator(np.random.PCG64(21))
    M, D, F = 5, 24, 40
    x = to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
    wg = to_bf16_bits((rng.standard_normal((F, D)) / 5).astype(np.float32))
    wu = to_bf16_bits((rng.standard_normal((F, D)) / 5).astype(np.float32))
    wd = to_bf16_bits((rng.standard_normal((D, F)) / 6).astype(np.float32))
    r = to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
    f = oracle.bf16_bits_to_f64
    gm, um = f(x) @ f(wg).T, f(x) @ f(wu).T
    h_want = _bf16_from_f64_torch(torch.nn.functional.silu(torch.from_numpy(gm)).numpy() * um)
    (_, out64), h = oracle.mlp_swiglu_down(x, wg, wu, wd, r, M=M, D=D, F=F, want_f64=True)
    assert np.array_equal(h, h_want)
    np.testing.assert_allclose(out64, f(h_want) @ f(wd).T + f(r), rtol=1e-12, atol=1e-14)
    # without a residual the block is the bare down projection of h
    (_, bare), _ = oracle.mlp_swiglu_down(x, wg, wu, wd, None, M=M, D=D, F=F, want_f64=True)
    np.testing.assert_allclose(bare, f(h_want) @ f(wd).T, rtol=1e-12, atol=1e-14)
    # a row subset equals the same rows of the full result
    full, _ = oracle.mlp_swiglu_down(x, wg, wu, wd, r, M=M, D=D, F=F)
    sub, hs = oracle.mlp_swiglu_down(x, wg, wu, wd, r, M=M, D=D, F=F, rows=[4, 1])
    assert np.array_equal(sub, full[[4, 1]]) and np.array_equal(hs, h[[4, 1]])


def test_mlp_chain_identity_down_projection_adds_residual_to_h():
    # D == F and W_down = I: out = bf16(h + residual), with h, residual
    # small dyadic values so the sum is exact and the rounding is the only step.
    rng = np.random.Generator(np.random.PCG64(22))
    M, D = 3, 16
    x = bits(rng.integers(-4, 5, size=(M, D)) / 4.0)
    wg = bits(rng.integers(-2, 3, size=(D, D)) / 8.0)
    wu = bits(rng.integers(-2, 3, size=(D, D)) / 8.0)
    wd = bits(np.eye(D))
    r = bits(rng.integers(-8, 9, size=(M, D)) / 2.0)
    out, h = oracle.mlp_swiglu_down(x, wg, wu, wd, r, M=M, D=D, F=D)
    f = oracle.bf16_bits_to_f64
    want = np.array([[oracle.bf16_from_f64(v) for v in row] for row in f(h) + f(r)],
                    dtype=np.uint16)
    assert np.array_equal(out, want)
    assert not np.array_equal(out, h)  # the residual is really added
    out0, h0 = oracle.mlp_swiglu_down(x, wg, wu, wd, None, M=M, D=D, F=D)
    assert np.array_equal(out0, h0)


def test_mlp_chain_unfused_mode_rounds_every_intermediate():
    rng = np.random.Generator(np.random.PCG64(23))
    M, D, F = 4, 16, 32
    x = to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
    wg = to_bf16_bits((rng.standard_normal((F, D)) / 4).astype(np.float32))
    wu = to_bf16_bits((rng.standard_normal((F, D)) / 4).astype(np.float32))
    wd = to_bf16_bits((rng.standard_normal((D, F)) / 6).astype(np.float32))
    r = to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
    out, h = oracle.mlp_swiglu_down(x, wg, wu, wd, r, M=M, D=D, F=F, unfused=True)
    f = oracle.bf16_bits_to_f64
    gb = _bf16_from_f64_torch(f(x) @ f(wg).T)
    ub = _bf16_from_f64_torch(f(x) @ f(wu).T)
    assert np.array_equal(h, oracle.swiglu_pointwise(gb, ub, M=M, N=F))
    db = _bf16_from_f64_torch(f(h) @ f(wd).T)
    assert np.array_equal(out, oracle.pointwise_epilogue(db, residual=r, M=M, N=D))


# ---------------------------------------------------------------- FP8 / NVFP4 weights

# FP4 E2M1 element values by code 0..7 (OCP Microscaling Formats v1.0, FP4
# E2M1: sign bit, 2 exponent bits with bias 1, 1 mantissa bit; code 1 is the
# subnormal 0.5); codes 8..15 are their negatives.
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_fp8_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.fp8_e4m3_to_f64(c) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got).sum() == 2  # S.1111.111 only
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_fp4_e2m1_decode_table_and_symmetry():
    got = [oracle.fp4_e2m1_to_f64(c) for c in range(16)]
    assert got[:8] == E2M1
    assert got[8:] == [-v for v in E2M1]
    assert math.copysign(1.0, got[8]) == -1.0  # code 8 is -0
    # every E2M1 value is an exact E4M3 value (the scale format holds them all)
    e4 = {oracle.fp8_e4m3_to_f64(c) for c in range(256)}
    assert all(v in e4 for v in got)


def _wq_setup(seed, M, N, K):
    rng = np.random.Generator(np.random.PCG64(seed))
    A = to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    return rng, A


def test_wq_gemm_int4_kind_equals_w4a16():
    rng, A = _wq_setup(31, 5, 32, 256)
    Wq = rng.integers(0, 256, size=(256, 16), dtype=np.uint8)
    s = to_bf16_bits(rng.uniform(0.01, 0.05, size=(2, 32)).astype(np.float32))
    a = oracle.wq_gemm("int4", A, Wq, s, 128, M=5, N=32, K=256, act="silu", alpha=0.5)
    b = oracle.w4a16(A, Wq, s, 128, M=5, N=32, K=256, act="silu", alpha=0.5)
    assert np.array_equal(a, b)


def test_fp8_weights_match_torch_decode_then_numpy_matmul():
    M, N, K, G = 6, 24, 192, 64
    rng, A = _wq_setup(32, M, N, K)
    Wq = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
    Wq[(Wq & 0x7F) == 0x7F] = 0x3C  # no NaN codes in a weight
    s = to_bf16_bits(rng.uniform(0.01, 0.1, size=(K // G, N)).astype(np.float32))
    q = torch.from_numpy(Wq).view(torch.float8_e4m3fn).double()
    sc = torch.from_numpy(oracle.bf16_bits_to_f64(s)).repeat_interleave(G, dim=0)
    w = (q * sc).to(torch.bfloat16).double().numpy()  # 12 significant bits: one rounding
    want = oracle.bf16_bits_to_f64(A) @ w
    _, got = oracle.wq_gemm("fp8", A, Wq, s, G, M=M, N=N, K=K, want_f64=True)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.dequant_wq("fp8", Wq, s, G, K=K, N=N),
                          workloads_bf16(w))


@pytest.mark.parametrize("k0,n0,code", [(0, 0, 0x3), (17, 5, 0xE), (47, 30, 0x1), (63, 31, 0x9)])
def test_nvfp4_single_code_probe_fixes_nibble_order_and_block_scale(k0, n0, code):
    M, N, K = 3, 32, 64
    _, A = _wq_setup(33, M, N, K)
    Wq = np.zeros((K, N // 2), dtype=np.uint8)
    Wq[k0, n0 // 2] = (code << 4) if n0 % 2 == 0 else code
    # block scales 2^-1, 2^0, 2^1, 2^2 for k-blocks 0..3 (E4M3 codes 0x30, 0x38, 0x40, 0x48)
    S = np.zeros((K // 16, N), dtype=np.uint8)
    for b, c in enumerate((0x30, 0x38, 0x40, 0x48)):
        S[b, :] = c
    out = oracle.wq_gemm("nvfp4", A, Wq, S, M=M, N=N, K=K, want_f64=True)[1]
    v = (E2M1[code & 7] * (-1 if code & 8 else 1)) * 2.0 ** (k0 // 16 - 1)
    want = np.zeros((M, N))
    want[:, n0] = oracle.bf16_bits_to_f64(A)[:, k0] * v
    assert np.array_equal(out, want)


def test_nvfp4_alpha_is_the_per_tensor_scale():
    M, N, K = 4, 16, 32
    rng, A = _wq_setup(34, M, N, K)
    Wq = rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)
    S = rng.integers(0x28, 0x50, size=(K // 16, N), dtype=np.uint8)
    _, one = oracle.wq_gemm("nvfp4", A, Wq, S, M=M, N=N, K=K, want_f64=True)
    _, quarter = oracle.wq_gemm("nvfp4", A, Wq, S, M=M, N=N, K=K, alpha=0.25, want_f64=True)
    assert np.array_equal(quarter, one * 0.25)
    # the weight is exact: E2M1 x E4M3 needs at most 6 significant bits
    w = oracle.dequant_wq("nvfp4", Wq, S, K=K, N=N)
    codes = np.stack([(Wq >> 4) & 0xF, Wq & 0xF], axis=-1).reshape(K, N)
    vals = np.array([oracle.fp4_e2m1_to_f64(c) for c in range(16)])[codes]
    sv = np.array([oracle.fp8_e4m3_to_f64(c) for c in range(256)])[S].repeat(16, axis=0)
    assert np.array_equal(oracle.bf16_bits_to_f64(w), vals * sv)


# ---------------------------------------------------------------- the two builds

def _both(fn):
    prev = oracle.set_parallel(False)
    try:
        a = fn()
        oracle.set_parallel(True)
        b = fn()
    finally:
        oracle.set_parallel(prev)
    return a, b


def test_openmp_build_runs_on_several_threads(oracle_build):
    if oracle_build != "openmp":
        pytest.skip("checked once")
    prev = oracle.set_parallel(False)
    try:
        assert oracle.threads() == 1
        with oracle.all_cores():
            n = oracle.threads()
    finally:
        oracle.set_parallel(prev)
    assert 1 <= n <= (os.cpu_count() or 1)
    if (os.cpu_count() or 1) > 1 and "OMP_NUM_THREADS" not in os.environ:
        assert n > 1


@pytest.mark.parametrize("what", ["gemm", "gemm_unfused", "swiglu", "w4a16", "fp8", "nvfp4",
                                  "rmsnorm"])
def test_serial_and_openmp_builds_agree_bit_for_bit(oracle_build, what):
    if oracle_build != "serial":
        pytest.skip("checked once")
    import workloads
    if what.startswith("gemm"):
        w = workloads.make("sweep", M=37, shape=dict(N=136, K=200))
        fn = lambda: oracle.gemm_epilogue(w["A"], w["B"], "kn", w["C"], w["bias"], None,
                                          M=37, N=136, K=200, alpha=w["alpha"], beta=w["beta"],
                                          act=w["act"], unfused=what.endswith("unfused"),
                                          want_f64=True)
    elif what == "swiglu":
        w = workloads.make("swiglu", shape=dict(M=19, N=72, K=96))
        fn = lambda: oracle.swiglu(w["x"], w["w_gate"], w["w_up"], "nk", M=19, N=72, K=96,
                                   want_f64=True)
    elif what == "w4a16":
        w = workloads.make("w4a16", shape=dict(M=5, N=96, K=256))
        fn = lambda: oracle.w4a16(w["A"], w["Wq"], w["scales"], 128, M=5, N=96, K=256,
                                  want_f64=True)
    elif what in ("fp8", "nvfp4"):
        name = "w8a16_fp8" if what == "fp8" else "w4a16_nvfp4"
        w = workloads.make(name, shape=dict(M=3, N=64, K=128))
        fn = lambda: oracle.wq_gemm(what, w["A"], w["Wq"], w["scales"], w["group"], M=3, N=64,
                                    K=128, alpha=w["alpha"], want_f64=True)
    else:
        w = workloads.make("add_rmsnorm", shape=dict(M=9, N=64))
        fn = lambda: oracle.add_rmsnorm(w["a"], w["x"], w["weight"], M=9, N=64, eps=w["eps"])
    a, b = _both(fn)
    for x, y in zip(a, b):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))

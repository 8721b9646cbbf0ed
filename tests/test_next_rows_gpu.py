"""GPU parity of the rows added after the core path: the fused residual add +
RMSNorm ("Fusion Thinking", Pattern 1) with its unfused composition, and the
standalone level-1 gated ending ("Fusion Thinking", Pattern 2, level 1)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up

pytestmark = pytest.mark.gpu


def rand_bf16(seed, shape, std=1.0, mean=0.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return workloads.to_bf16_bits(
        (rng.standard_normal(shape) * std + mean).astype(np.float32))


# ------------------------------------------------------------------ add + RMSNorm

@pytest.mark.parametrize("M,N", [(1, 8), (7, 96), (64, 4096), (33, 4104), (5, 16384),
                                 (300, 2048), (129, 8192)])
def test_add_rmsnorm_fused(cuda_lib, M, N):
    a, x = rand_bf16(M, (M, N)), rand_bf16(M + 1, (M, N))
    w = rand_bf16(M + 2, (N,), std=0.2, mean=1.0)
    norm, resid = poison_bf16(M, N), poison_bf16(M, N)
    cuda_lib.add_rmsnorm(up(a), up(x), up(w), norm, resid, M, N, 1e-5)
    assert cuda_lib.gbf_check_device_error() == 0
    want_norm, want_resid = oracle.add_rmsnorm(a, x, w, M=M, N=N, eps=1e-5)
    assert_parity(down(resid), want_resid, f"resid {M}x{N}")
    assert_parity(down(norm), want_norm, f"norm {M}x{N}")


def test_add_rmsnorm_without_residual_output(cuda_lib):
    M, N = 16, 1024
    a, x = rand_bf16(1, (M, N)), rand_bf16(2, (M, N))
    w = rand_bf16(3, (N,), std=0.2, mean=1.0)
    norm = poison_bf16(M, N)
    cuda_lib.add_rmsnorm(up(a), up(x), up(w), norm, None, M, N, 1e-6)
    assert cuda_lib.gbf_check_device_error() == 0
    assert_parity(down(norm), oracle.add_rmsnorm(a, x, w, M=M, N=N, eps=1e-6)[0], "norm only")


@pytest.mark.parametrize("M,N", [(8, 4096), (200, 2048)])
def test_add_rmsnorm_unfused_stagewise(cuda_lib, M, N):
    a, x = rand_bf16(11, (M, N)), rand_bf16(12, (M, N))
    w = rand_bf16(13, (N,), std=0.2, mean=1.0)
    norm, resid = poison_bf16(M, N), poison_bf16(M, N)
    cuda_lib.add_rmsnorm_unfused(up(a), up(x), up(w), norm, resid, M, N, 1e-5)
    assert cuda_lib.gbf_check_device_error() == 0
    _, want_resid = oracle.add_rmsnorm(a, x, w, M=M, N=N, eps=1e-5)
    r = down(resid)
    assert_parity(r, want_resid, "unfused resid")
    # the second kernel normalises the stored bf16 residual
    want_norm, _ = oracle.add_rmsnorm(r, np.zeros_like(r), w, M=M, N=N, eps=1e-5)
    assert_parity(down(norm), want_norm, "unfused norm")


def test_add_rmsnorm_validation(cuda_lib):
    t = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    f = lambda **kw: cuda_lib.add_rmsnorm(**{**dict(a=t, x=t, weight=t, out_norm=t,
                                                    out_resid=t, M=2, N=16, eps=1e-5), **kw},
                                          raise_on_error=False)
    assert f(N=12) == 3
    assert f(N=16392) == 3
    assert f(eps=-1.0) == 1
    assert f(a=None) == 1
    assert cuda_lib.add_rmsnorm_unfused(t, t, t, t, None, 2, 16, 1e-5, raise_on_error=False) == 1


def test_add_rmsnorm_workload_full_output(cuda_lib):
    w = workloads.make("add_rmsnorm")
    M, N = w["M"], w["N"]
    norm, resid = poison_bf16(M, N), poison_bf16(M, N)
    cuda_lib.add_rmsnorm(up(w["a"]), up(w["x"]), up(w["weight"]), norm, resid, M, N, w["eps"])
    assert cuda_lib.gbf_check_device_error() == 0
    want_norm, want_resid = oracle.add_rmsnorm(w["a"], w["x"], w["weight"], M=M, N=N,
                                               eps=w["eps"])
    assert_parity(down(resid), want_resid, "workload resid")
    assert_parity(down(norm), want_norm, "workload norm")


# ------------------------------------------------------------------ level-1 gated ending

@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "relu", "identity"])
@pytest.mark.parametrize("M,N", [(1, 8), (37, 1000), (256, 14336)])
def test_swiglu_pointwise(cuda_lib, act, M, N):
    g, u = rand_bf16(M, (M, N), std=2.0), rand_bf16(M + 5, (M, N))
    C = rand_bf16(M + 9, (M, N))
    h = poison_bf16(M, N)
    cuda_lib.swiglu_pointwise(up(g), up(u), up(C), h, M, N, 0.75, 0.5, act)
    assert cuda_lib.gbf_check_device_error() == 0
    want = oracle.swiglu_pointwise(g, u, C, M=M, N=N, alpha=0.75, beta=0.5, act=act)
    assert_parity(down(h), want, f"swiglu_pointwise {act} {M}x{N}")

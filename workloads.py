"""Seeded synthetic inputs for the fused GEMM + epilogue path.

This module is the one piece shared by the CUDA side (tests, bench) and the
oracle side: it draws random inputs and holds none of the method's
arithmetic.  bf16 values are produced by drawing float32 samples with numpy's
PCG64 generator and converting them with torch's bf16 cast; they are returned
as numpy ``uint16`` bit patterns.  Packed int4 weights are uniform random
bytes (so both nibbles are uniform codes 0..15).

Workloads are the five configurations of the fused-GEMM study:
  tiny       M=64  K=256  N=128   A,B,C,bias ~N(0,1), out=silu(0.5AB+C+bias)
  prefill    M=N=K=4096           A~N(0,1), W (NxK)~N(0,1/64), bias~N(0,0.1),
                                  residual~N(0,1), out=AW^T+bias+residual
  swiglu     M=2048 N=14336 K=4096  x~N(0,1), Wg,Wu (NxK)~N(0,1/64)
  w4a16      M=16 K=8192 N=28672  A~N(0,1), codes uniform 0..15,
                                  scales uniform [0.005,0.02], group 128
  sweep      N=K=8192, M in {1,16,128,1024,8192}, A,B~N(0,1/sqrt(K)),
             C~N(0,1), bias~N(0,0.1), out=gelu_tanh(0.75AB+0.25C+bias)
  add_rmsnorm  M=N=4096 (the prefill projection's output), a,x~N(0,1),
               weight~N(1,0.01), eps=1e-5
  swiglu_pointwise  M=2048 N=14336 (the gate/up outputs), g,u~N(0,64)

N(0, x) is read as mean 0 and VARIANCE x (std = sqrt(x)); ``sigma_is_std``
switches to reading x as the standard deviation.
Seeds: 0x5EED0000 + 16*config_id + tensor_index.
"""
from __future__ import annotations

import math

import numpy as np
import torch

SEED_BASE = 0x5EED0000

SWEEP_M = (1, 16, 128, 1024, 8192)

CONFIGS = {
    "tiny": dict(id=1, op="gemm", M=64, N=128, K=256, layout="kn", alpha=0.5, beta=1.0,
                 act="silu", has_c=True, has_bias=True, has_res=False),
    "prefill": dict(id=2, op="gemm", M=4096, N=4096, K=4096, layout="nk", alpha=1.0,
                    beta=0.0, act="identity", has_c=False, has_bias=True, has_res=True),
    "swiglu": dict(id=3, op="swiglu", M=2048, N=14336, K=4096, layout="nk", alpha=1.0,
                   beta=0.0, act="silu", has_c=False),
    "w4a16": dict(id=4, op="w4a16", M=16, N=28672, K=8192, group=128, alpha=1.0,
                  beta=0.0, act="identity", has_c=False, has_bias=False, has_res=False),
    "sweep": dict(id=5, op="gemm", M=None, N=8192, K=8192, layout="kn", alpha=0.75,
                  beta=0.25, act="gelu_tanh", has_c=True, has_bias=True, has_res=False),
    # rows after the core path
    "add_rmsnorm": dict(id=6, op="add_rmsnorm", M=4096, N=4096, K=0, eps=1e-5, alpha=1.0,
                        beta=0.0, act="identity"),
    "swiglu_pointwise": dict(id=7, op="swiglu_pointwise", M=2048, N=14336, K=0, alpha=1.0,
                             beta=0.0, act="silu", has_c=False),
    # one gated MLP block with its residual at a decode step of 16 sequences:
    # x[16x4096], Wg, Wu [14336x4096], Wd [4096x14336]; out = M x D (N = D),
    # the input width K = D, the hidden width F.
    "mlp_decode": dict(id=8, op="mlp", M=16, N=4096, K=4096, D=4096, F=14336, alpha=1.0,
                       beta=0.0, act="silu"),
    # the W4A16 decode shape with FP8 (E4M3, bf16 group scales) and NVFP4
    # (E2M1, E4M3 scales per 16 along K, per-tensor factor as alpha) weights
    "w8a16_fp8": dict(id=9, op="w8a16_fp8", M=16, N=28672, K=8192, group=128, alpha=1.0,
                      beta=0.0, act="identity", has_c=False, has_bias=False, has_res=False),
    "w4a16_nvfp4": dict(id=10, op="w4a16_nvfp4", M=16, N=28672, K=8192, group=16,
                        alpha=1.0 / 256, beta=0.0, act="identity", has_c=False,
                        has_bias=False, has_res=False),
}


def rng_for(config_id: int, tensor_index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + 16 * config_id + tensor_index))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16) via torch's bf16 cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_normal(rng: np.random.Generator, shape, spread: float,
                sigma_is_std: bool = False) -> np.ndarray:
    std = spread if sigma_is_std else math.sqrt(spread)
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def bf16_uniform(rng: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return to_bf16_bits(rng.uniform(lo, hi, size=shape).astype(np.float32))


def int4_packed(rng: np.random.Generator, K: int, N: int) -> np.ndarray:
    """K x N/2 bytes, every nibble a uniform code in 0..15."""
    return rng.integers(0, 256, size=(K, N // 2), dtype=np.uint8)


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 values -> OCP E4M3 codes (uint8) via torch's float8 cast,
    clamped to the finite range +-448 first (no NaN codes)."""
    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, dtype=np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def make(name: str, M: int | None = None, sigma_is_std: bool = False,
         shape: dict | None = None) -> dict:
    """Inputs of one workload as numpy arrays plus its scalar parameters.

    ``shape`` overrides M/N/K (and group) to draw a smaller case with the same
    distributions; ``M`` picks the row count of the sweep."""
    cfg = dict(CONFIGS[name])
    if M is not None:
        cfg["M"] = M
    if shape:
        cfg.update(shape)
    if cfg["M"] is None:
        raise ValueError("the sweep workload needs M")
    cid, Mv, Nv, Kv = cfg["id"], cfg["M"], cfg["N"], cfg["K"]
    s = sigma_is_std
    out = dict(cfg)
    if name == "tiny":
        out["A"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), 1.0, s)
        out["B"] = bf16_normal(rng_for(cid, 1), (Kv, Nv), 1.0, s)
        out["C"] = bf16_normal(rng_for(cid, 2), (Mv, Nv), 1.0, s)
        out["bias"] = bf16_normal(rng_for(cid, 3), (Nv,), 1.0, s)
        out["residual"] = None
    elif name == "prefill":
        out["A"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), 1.0, s)
        out["B"] = bf16_normal(rng_for(cid, 1), (Nv, Kv), 1.0 / 64.0, s)
        out["C"] = None
        out["bias"] = bf16_normal(rng_for(cid, 3), (Nv,), 0.1, s)
        out["residual"] = bf16_normal(rng_for(cid, 4), (Mv, Nv), 1.0, s)
    elif name == "swiglu":
        out["x"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), 1.0, s)
        out["w_gate"] = bf16_normal(rng_for(cid, 1), (Nv, Kv), 1.0 / 64.0, s)
        out["w_up"] = bf16_normal(rng_for(cid, 2), (Nv, Kv), 1.0 / 64.0, s)
        out["C"] = None
    elif name == "w4a16":
        out["A"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), 1.0, s)
        out["Wq"] = int4_packed(rng_for(cid, 1), Kv, Nv)
        out["scales"] = bf16_uniform(rng_for(cid, 2), (Kv // cfg["group"], Nv), 0.005, 0.02)
        out["C"] = out["bias"] = out["residual"] = None
    elif name == "add_rmsnorm":
        out["a"] = bf16_normal(rng_for(cid, 0), (Mv, Nv), 1.0, s)
        out["x"] = bf16_normal(rng_for(cid, 1), (Mv, Nv), 1.0, s)
        out["weight"] = to_bf16_bits(rng_for(cid, 2).standard_normal(Nv).astype(np.float32)
                                     * np.float32(0.1) + np.float32(1.0))
    elif name == "swiglu_pointwise":
        out["g"] = bf16_normal(rng_for(cid, 0), (Mv, Nv), 64.0, s)
        out["u"] = bf16_normal(rng_for(cid, 1), (Mv, Nv), 64.0, s)
        out["C"] = None
    elif name == "w8a16_fp8":
        out["A"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), 1.0, s)
        # codes spread over the E4M3 range (N(0, 64^2), subnormals included)
        out["Wq"] = e4m3_codes(rng_for(cid, 1).standard_normal((Kv, Nv), dtype=np.float32) * 64)
        out["scales"] = bf16_uniform(rng_for(cid, 2), (Kv // cfg["group"], Nv), 1e-4, 4e-4)
        out["C"] = out["bias"] = out["residual"] = None
    elif name == "w4a16_nvfp4":
        out["A"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), 1.0, s)
        out["Wq"] = int4_packed(rng_for(cid, 1), Kv, Nv)  # all 16 E2M1 codes equally likely
        # block scales: E4M3 codes 0x30..0x3F (0.5 .. 1.875)
        out["scales"] = rng_for(cid, 2).integers(0x30, 0x40, size=(Kv // 16, Nv), dtype=np.uint8)
        out["C"] = out["bias"] = out["residual"] = None
    elif name == "mlp_decode":
        D, F = cfg["D"], cfg["F"]
        out["x"] = bf16_normal(rng_for(cid, 0), (Mv, D), 1.0, s)
        # fan-in scaled weights (variance 1/fan_in), so g, u ~ N(0, 1) and the
        # block output is of the same order as the residual it is added to
        out["w_gate"] = bf16_normal(rng_for(cid, 1), (F, D), 1.0 / D, s)
        out["w_up"] = bf16_normal(rng_for(cid, 2), (F, D), 1.0 / D, s)
        out["w_down"] = bf16_normal(rng_for(cid, 3), (D, F), 1.0 / F, s)
        out["residual"] = bf16_normal(rng_for(cid, 4), (Mv, D), 1.0, s)
    elif name == "sweep":
        var = 1.0 / math.sqrt(Kv)
        out["A"] = bf16_normal(rng_for(cid, 0), (Mv, Kv), var, s)
        out["B"] = bf16_normal(rng_for(cid, 1), (Kv, Nv), var, s)
        out["C"] = bf16_normal(rng_for(cid, 2), (Mv, Nv), 1.0, s)
        out["bias"] = bf16_normal(rng_for(cid, 3), (Nv,), 0.1, s)
        out["residual"] = None
    else:
        raise KeyError(name)
    return out


def sample_indices(M: int, N: int, count: int = 4096, seed: int = 0xC0FFEE,
                   edge: int = 128):
    """A seeded sample of (row, col) output positions for large outputs: the
    four corners, the rows and columns on both sides of every `edge`
    boundary (sampled along the other axis), the ragged last row/column,
    and uniform positions for the rest."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rows, cols = [], []
    for r in (0, M - 1):
        for c in (0, N - 1):
            rows.append(r)
            cols.append(c)
    b_rows = sorted({x for b in range(0, M, edge) for x in (b - 1, b) if 0 <= x < M} | {M - 1})
    b_cols = sorted({x for b in range(0, N, edge) for x in (b - 1, b) if 0 <= x < N} | {N - 1})
    budget = max(0, count // 4)
    for r in b_rows[:budget // 2 or 1]:
        rows.append(r)
        cols.append(int(rng.integers(0, N)))
    for c in b_cols[:budget // 2 or 1]:
        rows.append(int(rng.integers(0, M)))
        cols.append(c)
    while len(rows) < count:
        rows.append(int(rng.integers(0, M)))
        cols.append(int(rng.integers(0, N)))
    return np.asarray(rows[:count], dtype=np.int64), np.asarray(cols[:count], dtype=np.int64)

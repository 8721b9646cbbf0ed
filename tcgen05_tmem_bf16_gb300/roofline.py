"""Algorithmic FLOP and byte counts of the fused path and its unfused
composition, and the roofline time they imply.

FLOPs: 2*M*N*K per product (two products for the gate/up GEMM); the
epilogue's few operations per output are not counted.  Fusion does not
change this number ("Kernel fusion" guide, "Check yourself": fusion cuts
HBM trips and launches, not the FLOP count of the matmul).

Bytes: every tensor crossing HBM exactly once -- inputs read once, the
output written once -- with no credit or charge for re-reads caused by
tiling.  Unfused adds the intermediate's write and read-back ("kernel
fusion" wiki: unfused, the product writes its output and a second kernel
reads it and writes again), and for the gate/up pair the second read of x
by the second GEMM.  For W4A16 the weight bytes are the packed int4 bytes
plus the bf16 scales ("Fusion Thinking", Pattern 3: W_int4 is a quarter of
the bf16 bytes); its unfused form writes and reads back the bf16 weight.
"""
from __future__ import annotations

from dataclasses import dataclass

BF16 = 2


@dataclass
class Counts:
    flops: float
    fused_bytes: float
    unfused_bytes: float


def gemm_counts(M, N, K, has_c=False, has_bias=False, has_res=False) -> Counts:
    io = M * K * BF16 + K * N * BF16 + M * N * BF16
    io += (M * N * BF16 if has_c else 0) + (N * BF16 if has_bias else 0)
    io += M * N * BF16 if has_res else 0
    return Counts(2.0 * M * N * K, io, io + 2 * M * N * BF16)


def swiglu_counts(M, N, K, has_c=False) -> Counts:
    fused = M * K * BF16 + 2 * N * K * BF16 + M * N * BF16 + (M * N * BF16 if has_c else 0)
    # unfused: the second GEMM reads x again; g and u are written, then read
    # back by the pointwise pass.
    unfused = fused + M * K * BF16 + 2 * (2 * M * N * BF16)
    return Counts(4.0 * M * N * K, fused, unfused)


def swiglu_unfused_pointwise_read_bytes_per_token(N: int) -> int:
    """Bytes the separate silu(gate)*up pass reads per token (row)."""
    return 2 * N * BF16


def w4a16_counts(M, N, K, group, has_c=False, has_bias=False, has_res=False) -> Counts:
    wbytes = K * N // 2 + (K // group) * N * BF16
    io = M * K * BF16 + wbytes + M * N * BF16
    io += (M * N * BF16 if has_c else 0) + (N * BF16 if has_bias else 0)
    io += M * N * BF16 if has_res else 0
    return Counts(2.0 * M * N * K, io, io + 2 * K * N * BF16)


def wq_counts(fmt, M, N, K, group, has_c=False, has_bias=False, has_res=False) -> Counts:
    """Weight-only GEMM with FP8 (1 byte per weight, bf16 group scales) or
    NVFP4 (half a byte per weight, one E4M3 byte per 16 along K) weights."""
    if fmt == "w8a16_fp8":
        wbytes = K * N + (K // group) * N * BF16
    else:
        wbytes = K * N // 2 + (K // 16) * N
    io = M * K * BF16 + wbytes + M * N * BF16
    io += (M * N * BF16 if has_c else 0) + (N * BF16 if has_bias else 0)
    io += M * N * BF16 if has_res else 0
    return Counts(2.0 * M * N * K, io, io + 2 * K * N * BF16)


def int4_weight_bytes(K, N) -> int:
    return K * N // 2


def bf16_weight_bytes(K, N) -> int:
    return K * N * BF16


def add_rmsnorm_counts(M, N) -> Counts:
    """Fused: read a and x, write the residual and the norm (4 passes of
    M*N bf16) plus the weight row.  Unfused: the add kernel reads a, x and
    writes r; the RMSNorm kernel reads r back and writes the norm (5 passes)."""
    t = M * N * BF16
    return Counts(5.0 * M * N, 4 * t + N * BF16, 5 * t + N * BF16)


def swiglu_pointwise_counts(M, N) -> Counts:
    """Fused: read g and u, write h (3 passes).  Eager (sigmoid, mul, mul):
    s = sigmoid(g) reads g writes s; t = g*s reads g, s writes t; h = t*u reads
    t, u writes h (8 passes)."""
    t = M * N * BF16
    return Counts(6.0 * M * N, 3 * t, 8 * t)


def mlp_counts(M, D, F) -> Counts:
    """One gated MLP block with its residual.  FLOPs: the gate and up products
    (2*M*F*D each) and the down product (2*M*D*F).  Fused chain: x, the three
    weights, the residual and out cross HBM once, and h (M x F bf16) is
    written by the gate/up GEMM and read back by the down GEMM.  Unfused: x is
    read twice, g and u are written and read back, h likewise, and the down
    product D is written and read back by the residual-add pass."""
    x = M * D * BF16
    w = 3 * F * D * BF16
    h = M * F * BF16
    fused = x + w + 2 * h + 2 * x  # + residual read, out written
    unfused = fused + x + 2 * (2 * h) + 2 * x
    return Counts(6.0 * M * D * F, fused, unfused)


def roofline_seconds(c: Counts, peak_tflops: float, peak_gbs: float, fused=True) -> float:
    b = c.fused_bytes if fused else c.unfused_bytes
    return max(c.flops / (peak_tflops * 1e12), b / (peak_gbs * 1e9))


def bound(c: Counts, peak_tflops: float, peak_gbs: float) -> str:
    t_tc = c.flops / (peak_tflops * 1e12)
    t_hbm = c.fused_bytes / (peak_gbs * 1e9)
    return "tensor" if t_tc >= t_hbm else "hbm"


def counts_for(cfg: dict) -> Counts:
    op = cfg["op"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    if op == "gemm":
        return gemm_counts(M, N, K, cfg.get("has_c", False), cfg.get("has_bias", False),
                           cfg.get("has_res", False))
    if op == "swiglu":
        return swiglu_counts(M, N, K, cfg.get("has_c", False))
    if op == "w4a16":
        return w4a16_counts(M, N, K, cfg["group"], cfg.get("has_c", False),
                            cfg.get("has_bias", False), cfg.get("has_res", False))
    if op == "add_rmsnorm":
        return add_rmsnorm_counts(M, N)
    if op == "swiglu_pointwise":
        return swiglu_pointwise_counts(M, N)
    if op == "mlp":
        return mlp_counts(M, cfg["D"], cfg["F"])
    if op in ("w8a16_fp8", "w4a16_nvfp4"):
        return wq_counts(op, M, N, K, cfg.get("group", 16), cfg.get("has_c", False),
                         cfg.get("has_bias", False), cfg.get("has_res", False))
    raise KeyError(op)

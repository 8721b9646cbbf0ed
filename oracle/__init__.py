"""fp64 CPU oracle for the fused GEMM + epilogue path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``gbf_oracle.c`` (plain C,
fp64, one bf16 rounding at the end) through ctypes and shares no code with
the CUDA library in ``tcgen05_tmem_bf16_gb300``.

The C file is built twice: single-threaded (the default) and with OpenMP,
which shares the loop over output elements among the host's cores
(``set_parallel(True)`` or ``with all_cores():``).  Each element is computed
the same way by one thread in both builds, so their results are identical;
the parallel build serves the all-cores timing and the full-output checks of
the large workloads.

bf16 tensors are passed as numpy ``uint16`` arrays holding the raw bits;
packed int4 weights as ``uint8`` arrays (K x N/2, high nibble = even column).

Every function here follows the passage cited in ``gbf_oracle.c``:
  * gemm_epilogue  -- "Fusion and Epilogues", epilogue-fusion bullet;
                      "Kernel fusion" guide, Concept.
  * swiglu         -- "Fusion Thinking", Pattern 2 (Fused SwiGLU).
  * w4a16 / dequant_int4 -- "Fusion Thinking", Pattern 3 (Dequant + GEMM).
  * wq_gemm / dequant_wq -- the same with int4, FP8 (E4M3) or NVFP4 (E2M1 with
                      E4M3 scales per 16 along K) weights; Pattern 3 names
                      NVFP4 weight-only quantisation with BF16 activations.
  * add_rmsnorm    -- "Fusion Thinking", Pattern 1 (Fused RMSNorm + residual).
  * mlp_swiglu_down -- "Fusion Thinking", Pattern 2 (out = W_down h) with
                      Pattern 1's residual add after the MLP: the two calls
                      above composed, h rounded to bf16 in between.
  * unfused modes  -- "kernel fusion" wiki, the activation-after-matmul case.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gbf_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgbf_oracle.so")
_OMP_LIB_PATH = os.path.join(_BUILD, "libgbf_oracle_omp.so")

ACT = {"identity": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}
LAYOUT = {"kn": 0, "nk": 1}

_lock = threading.Lock()
_libs = {}
_parallel = False


def _compile(path: str, extra) -> str:
    if os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", *extra, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def build(force: bool = False) -> str:
    """Compile gbf_oracle.c with gcc (no fast-math, no FMA contraction so
    x86 and Arm hosts give the same fp64 results), once single-threaded and
    once with OpenMP."""
    os.makedirs(_BUILD, exist_ok=True)
    if force:
        for p in (_LIB_PATH, _OMP_LIB_PATH):
            if os.path.exists(p):
                os.unlink(p)
    _compile(_OMP_LIB_PATH, ["-fopenmp"])
    return _compile(_LIB_PATH, [])


def set_parallel(on: bool) -> bool:
    """Use the OpenMP build (all host cores) for later calls; returns the
    previous setting."""
    global _parallel
    prev, _parallel = _parallel, bool(on)
    return prev


class all_cores:
    """``with all_cores(): ...`` runs the enclosed oracle calls on the OpenMP
    build."""

    def __enter__(self):
        self._prev = set_parallel(True)
        return self

    def __exit__(self, *exc):
        set_parallel(self._prev)
        return False


def threads() -> int:
    """Threads the oracle calls use (the OpenMP build's count when it is on)."""
    return int(_load().oracle_threads())


def _load():
    key = "omp" if _parallel else "serial"
    with _lock:
        lib = _libs.get(key)
        if lib is not None:
            return lib
        build()
        lib = ctypes.CDLL(_OMP_LIB_PATH if _parallel else _LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        D = ctypes.c_double
        I = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = D
        lib.oracle_bf16_from_f64.argtypes = [D]
        lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
        lib.oracle_act.argtypes = [I, D]
        lib.oracle_act.restype = D
        lib.oracle_gemm_epilogue.argtypes = [P, P, I, P, P, P, I64, I64, I64, D, D, I, I,
                                             P, P, I64, P, P]
        lib.oracle_gemm_epilogue.restype = I
        lib.oracle_swiglu.argtypes = [P, P, P, I, P, I64, I64, I64, D, D, I, I,
                                      P, P, I64, P, P]
        lib.oracle_swiglu.restype = I
        lib.oracle_w4a16.argtypes = [P, P, P, I64, P, P, P, I64, I64, I64, D, D, I,
                                     P, P, I64, P, P]
        lib.oracle_w4a16.restype = I
        lib.oracle_dequant_int4.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_dequant_int4.restype = I
        lib.oracle_wq_gemm.argtypes = [I, P, P, P, I64, P, P, P, I64, I64, I64, D, D, I,
                                       P, P, I64, P, P]
        lib.oracle_wq_gemm.restype = I
        lib.oracle_wq_dequant.argtypes = [I, P, P, I64, I64, I64, P]
        lib.oracle_wq_dequant.restype = I
        lib.oracle_fp8_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_fp8_e4m3_to_f64.restype = D
        lib.oracle_fp4_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_fp4_e2m1_to_f64.restype = D
        lib.oracle_pointwise_epilogue.argtypes = [P, P, P, P, I64, I64, D, D, I, P]
        lib.oracle_pointwise_epilogue.restype = I
        lib.oracle_swiglu_pointwise.argtypes = [P, P, P, I64, I64, D, D, I, P]
        lib.oracle_swiglu_pointwise.restype = I
        lib.oracle_add_rmsnorm.argtypes = [P, P, P, I64, I64, D, I, P, P]
        lib.oracle_add_rmsnorm.restype = I
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = I
        _libs[key] = lib
        return lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 bits expected as uint16, got {a.dtype}"
    return a


def _idx(M, N, rows, cols):
    if rows is None:
        return None, None, M * N
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    assert rows.shape == cols.shape
    return rows, cols, rows.size


def _outputs(count, want_f64):
    ob = np.empty(count, dtype=np.uint16)
    of = np.empty(count, dtype=np.float64) if want_f64 else None
    return ob, of


def _finish(rc, ob, of, M, N, rows, want_f64):
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    if rows is None:
        ob = ob.reshape(M, N)
        of = of.reshape(M, N) if of is not None else None
    return (ob, of) if want_f64 else ob


# ---- scalar helpers ---------------------------------------------------------

def bf16_from_f64(v: float) -> int:
    return int(_load().oracle_bf16_from_f64(float(v)))


def bf16_to_f64(h: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(h) & 0xFFFF))


def act(name: str, v: float) -> float:
    return float(_load().oracle_act(ACT[name], float(v)))


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits (uint16) to float64 (no arithmetic)."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- the path ---------------------------------------------------------------

def gemm_epilogue(A, B, layout, C=None, bias=None, residual=None, *, M, N, K,
                  alpha=1.0, beta=0.0, act="identity", unfused=False,
                  rows=None, cols=None, want_f64=False):
    """out = bf16(act(alpha*A*B~ + beta*C + bias) + residual); B~ = B (KxN
    layout "kn") or W^T (W is NxK, layout "nk").  With rows/cols given, only
    those (m, n) elements are computed (1-D results)."""
    lib = _load()
    A, B, C, bias, residual = map(_u16, (A, B, C, bias, residual))
    r, c, count = _idx(M, N, rows, cols)
    ob, of = _outputs(count, want_f64)
    rc = lib.oracle_gemm_epilogue(_ptr(A), _ptr(B), LAYOUT[layout], _ptr(C), _ptr(bias),
                                  _ptr(residual), M, N, K, float(alpha), float(beta),
                                  ACT[act], int(bool(unfused)), _ptr(r), _ptr(c), count,
                                  _ptr(ob), _ptr(of))
    return _finish(rc, ob, of, M, N, rows, want_f64)


def swiglu(x, w_gate, w_up, layout, C=None, *, M, N, K, alpha=1.0, beta=0.0,
           act="silu", unfused=False, rows=None, cols=None, want_f64=False):
    """h = bf16(act(alpha*g)*(alpha*u) + beta*C), g = x*Wg~, u = x*Wu~."""
    lib = _load()
    x, w_gate, w_up, C = map(_u16, (x, w_gate, w_up, C))
    r, c, count = _idx(M, N, rows, cols)
    ob, of = _outputs(count, want_f64)
    rc = lib.oracle_swiglu(_ptr(x), _ptr(w_gate), _ptr(w_up), LAYOUT[layout], _ptr(C),
                           M, N, K, float(alpha), float(beta), ACT[act],
                           int(bool(unfused)), _ptr(r), _ptr(c), count, _ptr(ob), _ptr(of))
    return _finish(rc, ob, of, M, N, rows, want_f64)


def w4a16(A, Wq, scales, group_size, C=None, bias=None, residual=None, *, M, N, K,
          alpha=1.0, beta=0.0, act="identity", rows=None, cols=None, want_f64=False):
    """gemm_epilogue with B~[k][n] = bf16((q[k][n]-8)*s[k/G][n])."""
    lib = _load()
    A, scales, C, bias, residual = map(_u16, (A, scales, C, bias, residual))
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    r, c, count = _idx(M, N, rows, cols)
    ob, of = _outputs(count, want_f64)
    rc = lib.oracle_w4a16(_ptr(A), _ptr(Wq), _ptr(scales), int(group_size), _ptr(C),
                          _ptr(bias), _ptr(residual), M, N, K, float(alpha), float(beta),
                          ACT[act], _ptr(r), _ptr(c), count, _ptr(ob), _ptr(of))
    return _finish(rc, ob, of, M, N, rows, want_f64)


WQ_KIND = {"int4": 0, "fp8": 1, "nvfp4": 2}


def fp8_e4m3_to_f64(b: int) -> float:
    return float(_load().oracle_fp8_e4m3_to_f64(int(b) & 0xFF))


def fp4_e2m1_to_f64(b: int) -> float:
    return float(_load().oracle_fp4_e2m1_to_f64(int(b) & 0xF))


def _scales(kind, scales):
    if scales is None:
        return None
    if kind == "nvfp4":
        return np.ascontiguousarray(scales, dtype=np.uint8)
    return _u16(scales)


def wq_gemm(kind, A, Wq, scales, group_size=16, C=None, bias=None, residual=None, *, M, N, K,
            alpha=1.0, beta=0.0, act="identity", rows=None, cols=None, want_f64=False):
    """Weight-only GEMM: gemm_epilogue with B~ the dequantised weight of
    format ``kind`` ("int4", "fp8" or "nvfp4"; see gbf_oracle.c).  For nvfp4
    ``scales`` are E4M3 bytes [K/16][N] and alpha carries the per-tensor
    factor; group_size is ignored."""
    lib = _load()
    A, C, bias, residual = map(_u16, (A, C, bias, residual))
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    sc = _scales(kind, scales)
    r, c, count = _idx(M, N, rows, cols)
    ob, of = _outputs(count, want_f64)
    rc = lib.oracle_wq_gemm(WQ_KIND[kind], _ptr(A), _ptr(Wq), _ptr(sc), int(group_size),
                            _ptr(C), _ptr(bias), _ptr(residual), M, N, K, float(alpha),
                            float(beta), ACT[act], _ptr(r), _ptr(c), count, _ptr(ob), _ptr(of))
    return _finish(rc, ob, of, M, N, rows, want_f64)


def dequant_wq(kind, Wq, scales, group_size=16, *, K, N):
    """The dequantised K x N bf16 weight of format ``kind``."""
    lib = _load()
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    sc = _scales(kind, scales)
    out = np.empty((K, N), dtype=np.uint16)
    if lib.oracle_wq_dequant(WQ_KIND[kind], _ptr(Wq), _ptr(sc), int(group_size), K, N,
                             _ptr(out)) != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def dequant_int4(Wq, scales, group_size, *, K, N):
    lib = _load()
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    scales = _u16(scales)
    out = np.empty((K, N), dtype=np.uint16)
    if lib.oracle_dequant_int4(_ptr(Wq), _ptr(scales), int(group_size), K, N, _ptr(out)) != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def pointwise_epilogue(D, C=None, bias=None, residual=None, *, M, N, alpha=1.0,
                       beta=0.0, act="identity"):
    lib = _load()
    D, C, bias, residual = map(_u16, (D, C, bias, residual))
    out = np.empty((M, N), dtype=np.uint16)
    if lib.oracle_pointwise_epilogue(_ptr(D), _ptr(C), _ptr(bias), _ptr(residual), M, N,
                                     float(alpha), float(beta), ACT[act], _ptr(out)) != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def swiglu_pointwise(g, u, C=None, *, M, N, alpha=1.0, beta=0.0, act="silu"):
    lib = _load()
    g, u, C = map(_u16, (g, u, C))
    out = np.empty((M, N), dtype=np.uint16)
    if lib.oracle_swiglu_pointwise(_ptr(g), _ptr(u), _ptr(C), M, N, float(alpha),
                                   float(beta), ACT[act], _ptr(out)) != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def mlp_swiglu_down(x, w_gate, w_up, w_down, residual=None, *, M, D, F, unfused=False,
                    rows=None, want_f64=False):
    """(out, h) of one gated MLP block with its residual add:
    h = swiglu(x, Wg, Wu) rounded to bf16 ([M][F]), out = bf16(h*Wd^T +
    residual) ([M][D]).  x [M][D]; w_gate, w_up [F][D]; w_down [D][F].
    With ``rows`` only those rows are computed (h rows depend on x rows
    alone).  ``unfused`` rounds g, u and the down product to bf16 first."""
    x = _u16(x)
    residual = _u16(residual)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        x = np.ascontiguousarray(x.reshape(M, D)[rows])
        if residual is not None:
            residual = np.ascontiguousarray(residual.reshape(M, D)[rows])
        M = int(rows.size)
    h = swiglu(x, w_gate, w_up, "nk", M=M, N=F, K=D, act="silu", unfused=unfused)
    out = gemm_epilogue(h, w_down, "nk", residual=residual, M=M, N=D, K=F, unfused=unfused,
                        want_f64=want_f64)
    return out, h


def add_rmsnorm(a, x, w, *, M, N, eps=1e-5, unfused=False):
    """(norm, resid): resid = bf16(a + x); norm = bf16((a + x) * rsqrt(mean((a + x)^2) + eps) * w)
    per row (unfused: the norm is taken of the bf16-rounded residual)."""
    lib = _load()
    a, x, w = map(_u16, (a, x, w))
    norm = np.empty((M, N), dtype=np.uint16)
    resid = np.empty((M, N), dtype=np.uint16)
    if lib.oracle_add_rmsnorm(_ptr(a), _ptr(x), _ptr(w), M, N, float(eps), int(bool(unfused)),
                              _ptr(norm), _ptr(resid)) != 0:
        raise ValueError("oracle rejected its arguments")
    return norm, resid

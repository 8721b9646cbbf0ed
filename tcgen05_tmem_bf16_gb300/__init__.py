"""tcgen05_tmem_bf16_gb300 -- fused bf16 GEMM + epilogue for GB300 (sm_103a).

A thin ctypes binding of the C ABI in ``include/gbfuse.h``: every function
here has the C entry point's name and arguments and only marshals them (torch
tensors or integer device addresses for pointers, the current torch stream by
default).  All arithmetic runs in the CUDA kernels of ``_build/libgbfuse.so``;
there is no CPU fallback, and a missing library is an error.

  gemm_epilogue      out = act(alpha*A*B + beta*C + bias) + residual
  swiglu_dual_gemm   h = act(alpha*x*Wg) * (alpha*x*Wu) + beta*C
  w4a16_gemm         gemm_epilogue with int4 weights dequantised on-chip
  w8a16_fp8_gemm     the same with FP8 (E4M3) weights and bf16 group scales
  w4a16_nvfp4_gemm   the same with NVFP4 (E2M1 + E4M3 block scales) weights
  mlp_swiglu_down    gate/up GEMM -> bf16 h -> down GEMM + residual
  add_rmsnorm        fused residual add + RMSNorm
  *_unfused          the same results as GEMM -> HBM -> pointwise kernel
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

ACT = {"identity": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}
LAYOUT = {"kn": 0, "nk": 1}
OP = {"gemm_epilogue": 0, "swiglu": 1, "w4a16": 2, "mlp": 3, "w8a16_fp8": 4, "w4a16_nvfp4": 5}
STATUS = {0: "GBF_OK", 1: "GBF_ERR_INVALID_ARG", 2: "GBF_ERR_MISALIGNED",
          3: "GBF_ERR_UNSUPPORTED_SHAPE", 4: "GBF_ERR_WORKSPACE", 5: "GBF_ERR_CUDA",
          6: "GBF_ERR_TIMEOUT", 7: "GBF_ERR_NO_DEVICE"}
PATH = {0: "none", 1: "persistent", 2: "swap_splitk", 3: "w4a16", 4: "pair",
        5: "persistent_splitk", 6: "pair_1stream", 7: "pair_splitk"}

EXPORTS = ("gemm_epilogue", "swiglu_dual_gemm", "w4a16_gemm", "gemm_epilogue_unfused",
           "swiglu_dual_gemm_unfused", "w4a16_gemm_unfused", "gbf_workspace_size",
           "gbf_check_device_error", "gbf_status_string", "gbf_set_wait_timeout_ns",
           "gbf_debug_inject_timeout", "gbf_kernel_path", "gbf_version",
           "gemm_epilogue_unfused_noalloc", "gbf_debug_force_splits", "gbf_debug_force_path", "gbf_debug_set_profile",
           "swiglu_pointwise", "add_rmsnorm", "add_rmsnorm_unfused", "mlp_swiglu_down",
           "mlp_swiglu_down_unfused", "w8a16_fp8_gemm", "w8a16_fp8_gemm_unfused",
           "w4a16_nvfp4_gemm", "w4a16_nvfp4_gemm_unfused")

_lock = threading.Lock()
_lib = None


class GbfError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the shared library (build it first with ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise FileNotFoundError(
                f"{p} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        V, I64, F, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
        gemm_args = [V, V, I, V, V, V, V, I64, I64, I64, F, F, I, V, SZ, V]
        swiglu_args = [V, V, V, I, V, I64, I64, I64, F, F, V, I, V, SZ, V]
        w4_args = [V, V, V, I, V, V, V, V, I64, I64, I64, F, F, I, V, SZ, V]
        for name, args in (("gemm_epilogue", gemm_args), ("gemm_epilogue_unfused", gemm_args),
                           ("swiglu_dual_gemm", swiglu_args),
                           ("swiglu_dual_gemm_unfused", swiglu_args),
                           ("w4a16_gemm", w4_args), ("w4a16_gemm_unfused", w4_args),
                           ("w8a16_fp8_gemm", w4_args), ("w8a16_fp8_gemm_unfused", w4_args),
                           ("w4a16_nvfp4_gemm", w4_args[:3] + w4_args[4:]),
                           ("w4a16_nvfp4_gemm_unfused", w4_args[:3] + w4_args[4:])):
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        for name in ("mlp_swiglu_down", "mlp_swiglu_down_unfused"):
            fn = getattr(lib, name)
            fn.argtypes = [V, V, V, V, V, V, I64, I64, I64, V, SZ, V]
            fn.restype = I
        for name in ("add_rmsnorm", "add_rmsnorm_unfused"):
            fn = getattr(lib, name)
            fn.argtypes = [V, V, V, V, V, I64, I64, F, V]
            fn.restype = I
        lib.swiglu_pointwise.argtypes = [V, V, V, V, I64, I64, F, F, I, V]
        lib.swiglu_pointwise.restype = I
        lib.gemm_epilogue_unfused_noalloc.argtypes = [V, V, I, V, V, V, V, I64, I64, I64, F, F,
                                                      I, V]
        lib.gemm_epilogue_unfused_noalloc.restype = I
        lib.gbf_workspace_size.argtypes = [I, I64, I64, I64, I]
        lib.gbf_workspace_size.restype = SZ
        lib.gbf_check_device_error.argtypes = [V]
        lib.gbf_check_device_error.restype = I
        lib.gbf_status_string.argtypes = [I]
        lib.gbf_status_string.restype = ctypes.c_char_p
        lib.gbf_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.gbf_set_wait_timeout_ns.restype = I
        lib.gbf_debug_inject_timeout.argtypes = [I]
        lib.gbf_debug_inject_timeout.restype = I
        lib.gbf_debug_set_profile.argtypes = [V, SZ]
        lib.gbf_debug_set_profile.restype = I
        lib.gbf_debug_force_splits.argtypes = [I]
        lib.gbf_debug_force_splits.restype = I
        lib.gbf_debug_force_path.argtypes = [I]
        lib.gbf_debug_force_path.restype = I
        lib.gbf_kernel_path.argtypes = [I, I64, I64, I64, I, ctypes.POINTER(I)]
        lib.gbf_kernel_path.restype = I
        lib.gbf_version.argtypes = []
        lib.gbf_version.restype = I
        _lib = lib
        return lib


def _p(x):
    """A device address from a torch tensor, an int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _code(v, table):
    return table[v] if isinstance(v, str) else int(v)


def _check(status: int, where: str, raise_on_error: bool) -> int:
    if status != 0 and raise_on_error:
        raise GbfError(status, where)
    return status


def gemm_epilogue(A, B, b_layout, C, bias, residual, out, M, N, K, alpha=1.0, beta=0.0,
                  act="identity", workspace=None, workspace_bytes=0, stream=None,
                  raise_on_error=True):
    st = load().gemm_epilogue(_p(A), _p(B), _code(b_layout, LAYOUT), _p(C), _p(bias),
                              _p(residual), _p(out), M, N, K, alpha, beta, _code(act, ACT),
                              _p(workspace), workspace_bytes, _s(stream))
    return _check(st, "gemm_epilogue", raise_on_error)


def gemm_epilogue_unfused(A, B, b_layout, C, bias, residual, out, M, N, K, alpha=1.0, beta=0.0,
                          act="identity", workspace=None, workspace_bytes=0, stream=None,
                          raise_on_error=True):
    st = load().gemm_epilogue_unfused(_p(A), _p(B), _code(b_layout, LAYOUT), _p(C), _p(bias),
                                      _p(residual), _p(out), M, N, K, alpha, beta,
                                      _code(act, ACT), _p(workspace), workspace_bytes,
                                      _s(stream))
    return _check(st, "gemm_epilogue_unfused", raise_on_error)


def gemm_epilogue_unfused_noalloc(A, B, b_layout, C, bias, residual, out, M, N, K, alpha=1.0,
                                  beta=0.0, act="identity", stream=None, raise_on_error=True):
    """gemm_epilogue_unfused for callers that cannot allocate device memory:
    the intermediate lives in the library's built-in scratch array
    (M*N <= 4194304); no workspace argument."""
    st = load().gemm_epilogue_unfused_noalloc(_p(A), _p(B), _code(b_layout, LAYOUT), _p(C),
                                              _p(bias), _p(residual), _p(out), M, N, K, alpha,
                                              beta, _code(act, ACT), _s(stream))
    return _check(st, "gemm_epilogue_unfused_noalloc", raise_on_error)


def swiglu_dual_gemm(x, w_gate, w_up, w_layout, h, M, N, K, alpha=1.0, beta=0.0, C=None,
                     act="silu", workspace=None, workspace_bytes=0, stream=None,
                     raise_on_error=True):
    st = load().swiglu_dual_gemm(_p(x), _p(w_gate), _p(w_up), _code(w_layout, LAYOUT), _p(h),
                                 M, N, K, alpha, beta, _p(C), _code(act, ACT), _p(workspace),
                                 workspace_bytes, _s(stream))
    return _check(st, "swiglu_dual_gemm", raise_on_error)


def swiglu_dual_gemm_unfused(x, w_gate, w_up, w_layout, h, M, N, K, alpha=1.0, beta=0.0,
                             C=None, act="silu", workspace=None, workspace_bytes=0, stream=None,
                             raise_on_error=True):
    st = load().swiglu_dual_gemm_unfused(_p(x), _p(w_gate), _p(w_up), _code(w_layout, LAYOUT),
                                         _p(h), M, N, K, alpha, beta, _p(C), _code(act, ACT),
                                         _p(workspace), workspace_bytes, _s(stream))
    return _check(st, "swiglu_dual_gemm_unfused", raise_on_error)


def swiglu_pointwise(g, u, C, h, M, N, alpha=1.0, beta=0.0, act="silu", stream=None,
                     raise_on_error=True):
    st = load().swiglu_pointwise(_p(g), _p(u), _p(C), _p(h), M, N, alpha, beta,
                                 _code(act, ACT), _s(stream))
    return _check(st, "swiglu_pointwise", raise_on_error)


def add_rmsnorm(a, x, weight, out_norm, out_resid, M, N, eps=1e-5, stream=None,
                raise_on_error=True):
    st = load().add_rmsnorm(_p(a), _p(x), _p(weight), _p(out_norm), _p(out_resid), M, N, eps,
                            _s(stream))
    return _check(st, "add_rmsnorm", raise_on_error)


def add_rmsnorm_unfused(a, x, weight, out_norm, out_resid, M, N, eps=1e-5, stream=None,
                        raise_on_error=True):
    st = load().add_rmsnorm_unfused(_p(a), _p(x), _p(weight), _p(out_norm), _p(out_resid), M, N,
                                    eps, _s(stream))
    return _check(st, "add_rmsnorm_unfused", raise_on_error)


def mlp_swiglu_down(x, w_gate, w_up, w_down, residual, out, M, D, F, workspace=None,
                    workspace_bytes=0, stream=None, raise_on_error=True):
    st = load().mlp_swiglu_down(_p(x), _p(w_gate), _p(w_up), _p(w_down), _p(residual), _p(out),
                                M, D, F, _p(workspace), workspace_bytes, _s(stream))
    return _check(st, "mlp_swiglu_down", raise_on_error)


def mlp_swiglu_down_unfused(x, w_gate, w_up, w_down, residual, out, M, D, F, workspace=None,
                            workspace_bytes=0, stream=None, raise_on_error=True):
    st = load().mlp_swiglu_down_unfused(_p(x), _p(w_gate), _p(w_up), _p(w_down), _p(residual),
                                        _p(out), M, D, F, _p(workspace), workspace_bytes,
                                        _s(stream))
    return _check(st, "mlp_swiglu_down_unfused", raise_on_error)


def w4a16_gemm(A, Wq, scales, group_size, C, bias, residual, out, M, N, K, alpha=1.0,
               beta=0.0, act="identity", workspace=None, workspace_bytes=0, stream=None,
               raise_on_error=True):
    st = load().w4a16_gemm(_p(A), _p(Wq), _p(scales), group_size, _p(C), _p(bias),
                           _p(residual), _p(out), M, N, K, alpha, beta, _code(act, ACT),
                           _p(workspace), workspace_bytes, _s(stream))
    return _check(st, "w4a16_gemm", raise_on_error)


def w4a16_gemm_unfused(A, Wq, scales, group_size, C, bias, residual, out, M, N, K, alpha=1.0,
                       beta=0.0, act="identity", workspace=None, workspace_bytes=0,
                       stream=None, raise_on_error=True):
    st = load().w4a16_gemm_unfused(_p(A), _p(Wq), _p(scales), group_size, _p(C), _p(bias),
                                   _p(residual), _p(out), M, N, K, alpha, beta,
                                   _code(act, ACT), _p(workspace), workspace_bytes, _s(stream))
    return _check(st, "w4a16_gemm_unfused", raise_on_error)


def w8a16_fp8_gemm(A, Wq, scales, group_size, C, bias, residual, out, M, N, K, alpha=1.0,
                   beta=0.0, act="identity", workspace=None, workspace_bytes=0, stream=None,
                   raise_on_error=True):
    st = load().w8a16_fp8_gemm(_p(A), _p(Wq), _p(scales), group_size, _p(C), _p(bias),
                               _p(residual), _p(out), M, N, K, alpha, beta, _code(act, ACT),
                               _p(workspace), workspace_bytes, _s(stream))
    return _check(st, "w8a16_fp8_gemm", raise_on_error)


def w8a16_fp8_gemm_unfused(A, Wq, scales, group_size, C, bias, residual, out, M, N, K,
                           alpha=1.0, beta=0.0, act="identity", workspace=None,
                           workspace_bytes=0, stream=None, raise_on_error=True):
    st = load().w8a16_fp8_gemm_unfused(_p(A), _p(Wq), _p(scales), group_size, _p(C), _p(bias),
                                       _p(residual), _p(out), M, N, K, alpha, beta,
                                       _code(act, ACT), _p(workspace), workspace_bytes,
                                       _s(stream))
    return _check(st, "w8a16_fp8_gemm_unfused", raise_on_error)


def w4a16_nvfp4_gemm(A, Wq, scales, C, bias, residual, out, M, N, K, alpha=1.0, beta=0.0,
                     act="identity", workspace=None, workspace_bytes=0, stream=None,
                     raise_on_error=True):
    st = load().w4a16_nvfp4_gemm(_p(A), _p(Wq), _p(scales), _p(C), _p(bias), _p(residual),
                                 _p(out), M, N, K, alpha, beta, _code(act, ACT), _p(workspace),
                                 workspace_bytes, _s(stream))
    return _check(st, "w4a16_nvfp4_gemm", raise_on_error)


def w4a16_nvfp4_gemm_unfused(A, Wq, scales, C, bias, residual, out, M, N, K, alpha=1.0,
                             beta=0.0, act="identity", workspace=None, workspace_bytes=0,
                             stream=None, raise_on_error=True):
    st = load().w4a16_nvfp4_gemm_unfused(_p(A), _p(Wq), _p(scales), _p(C), _p(bias),
                                         _p(residual), _p(out), M, N, K, alpha, beta,
                                         _code(act, ACT), _p(workspace), workspace_bytes,
                                         _s(stream))
    return _check(st, "w4a16_nvfp4_gemm_unfused", raise_on_error)


def gbf_workspace_size(op, M, N, K, fused) -> int:
    return int(load().gbf_workspace_size(_code(op, OP), M, N, K, int(bool(fused))))


def gbf_check_device_error(stream=None) -> int:
    return int(load().gbf_check_device_error(_s(stream)))


def gbf_status_string(status: int) -> str:
    return load().gbf_status_string(int(status)).decode()


def gbf_set_wait_timeout_ns(ns: int) -> int:
    return int(load().gbf_set_wait_timeout_ns(int(ns)))


def gbf_debug_inject_timeout(on: bool) -> int:
    return int(load().gbf_debug_inject_timeout(int(bool(on))))


def gbf_debug_set_profile(counters, nbytes: int = 0) -> int:
    """Register a zeroed device buffer for per-CTA wait-time counters (None: off)."""
    if counters is not None and not nbytes:
        nbytes = counters.numel() * counters.element_size()
    return int(load().gbf_debug_set_profile(_p(counters), int(nbytes)))


def gbf_debug_force_splits(splits: int) -> int:
    return int(load().gbf_debug_force_splits(int(splits)))


def gbf_debug_force_path(path) -> int:
    """Force the dense kernel above the swapped range: "persistent",
    "persistent_splitk", "pair", "pair_1stream", "pair_splitk", or None /
    "auto" for the automatic choice."""
    code = {None: 0, "auto": 0, "persistent": 1, "pair": 4,
            "persistent_splitk": 5, "pair_1stream": 6, "pair_splitk": 7}.get(path, path)
    return int(load().gbf_debug_force_path(int(code)))


def gbf_kernel_path(op, M, N, K, b_layout="nk"):
    """(path name, split-K cluster size) the library picks for these sizes."""
    splits = ctypes.c_int(0)
    code = load().gbf_kernel_path(_code(op, OP), M, N, K, _code(b_layout, LAYOUT),
                                  ctypes.byref(splits))
    return PATH.get(code, "rejected"), splits.value


def gbf_version() -> int:
    return int(load().gbf_version())

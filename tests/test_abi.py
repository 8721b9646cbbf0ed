"""The C-ABI library loads and exports every symbol include/gbfuse.h declares;
argument validation runs on the host and needs no GPU (no compute call is
made here)."""
import ctypes
import os
import re

import pytest

import tcgen05_tmem_bf16_gb300 as gbf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbfuse.h")
DEBUG_HEADER = os.path.join(ROOT, "include", "gbfuse_debug.h")


def declared_symbols(path=HEADER):
    text = open(path).read()
    if "#define GBF_API" in text:
        text = text.split("#define GBF_API")[-1].split("\n", 1)[1]
    return sorted(set(re.findall(r"^GBF_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    from tcgen05_tmem_bf16_gb300 import build
    build.build()
    return gbf.load()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("gemm_epilogue", "swiglu_dual_gemm", "w4a16_gemm", "gemm_epilogue_unfused",
                 "swiglu_dual_gemm_unfused", "w4a16_gemm_unfused", "gbf_workspace_size",
                 "gbf_check_device_error", "gbf_status_string"):
        assert name in syms
    hooks = declared_symbols(DEBUG_HEADER)
    # the product boundary holds no test or tuning hook; the hooks live in
    # their own header, and the binding names exactly the union of the two
    assert not any(n.startswith("gbf_debug_") for n in syms)
    assert hooks and all(n.startswith("gbf_debug_") for n in hooks)
    assert not set(syms) & set(hooks)
    assert set(syms) | set(hooks) == set(gbf.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols() + declared_symbols(DEBUG_HEADER):
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_library_exports_nothing_undeclared(lib):
    import subprocess
    from tcgen05_tmem_bf16_gb300 import build
    r = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm unavailable")
    exported = {line.split()[-1] for line in r.stdout.splitlines()
                if len(line.split()) == 3 and line.split()[1] == "T"}
    ours = {n for n in exported if n.startswith(("gbf_", "gemm_", "swiglu_", "w4a16_",
                                                  "w8a16_", "add_rmsnorm", "mlp_"))}
    assert ours == set(declared_symbols()) | set(declared_symbols(DEBUG_HEADER))


def test_status_strings_and_version(lib):
    assert gbf.gbf_status_string(0) == "ok"
    assert "aligned" in gbf.gbf_status_string(2)
    assert "bounded wait" in gbf.gbf_status_string(6)
    assert gbf.gbf_status_string(99) == "unknown status"
    assert gbf.gbf_version() == 100


def test_workspace_sizes(lib):
    assert gbf.gbf_workspace_size("gemm_epilogue", 4096, 4096, 4096, True) == 0
    assert gbf.gbf_workspace_size("gemm_epilogue", 3, 8, 8, False) == 256
    assert gbf.gbf_workspace_size("gemm_epilogue", 4096, 4096, 16, False) == 4096 * 4096 * 2
    assert gbf.gbf_workspace_size("swiglu", 2048, 14336, 4096, False) == 2 * 2048 * 14336 * 2
    assert gbf.gbf_workspace_size("w4a16", 16, 28672, 8192, False) == 8192 * 28672 * 2
    assert gbf.gbf_workspace_size("w8a16_fp8", 16, 28672, 8192, False) == 8192 * 28672 * 2
    assert gbf.gbf_workspace_size("mlp", 16, 4096, 14336, True) == 16 * 14336 * 2
    assert gbf.gbf_workspace_size("mlp", 16, 4096, 14336, False) == 4 * 16 * 14336 * 2 + \
        16 * 4096 * 2


def test_kernel_path_planning(lib):
    assert gbf.gbf_kernel_path("gemm_epilogue", 4096, 4096, 4096) == ("pair", 1)
    # mid-size M: the pair kernel's 512 x 256 units would leave most SMs idle,
    # and the 256 x 256 tiles fit one round of clusters of two CTA pairs:
    # each pair over half of K (split K)
    assert gbf.gbf_kernel_path("gemm_epilogue", 300, 4096, 4096) == ("pair_splitk", 2)
    assert gbf.gbf_kernel_path("gemm_epilogue", 512, 4096, 4096) == ("pair_splitk", 2)
    assert gbf.gbf_kernel_path("gemm_epilogue", 1024, 4096, 4096)[0] == "pair_1stream"
    # 37 tiles of 256 x 256: one more than the 36 clusters of two pairs that
    # fit at once, so the one-SM kernel's split-K form (74 tiles, 148 CTAs)
    assert gbf.gbf_kernel_path("gemm_epilogue", 256, 256 * 37, 4096) == ("persistent_splitk", 2)
    # too little K to pay for the exchange of the partial sums
    assert gbf.gbf_kernel_path("gemm_epilogue", 300, 4096, 256)[0] not in ("pair_splitk",
                                                                          "persistent_splitk")
    assert gbf.gbf_kernel_path("gemm_epilogue", 1024, 8192, 8192, "kn") == ("pair", 1)
    path, splits = gbf.gbf_kernel_path("gemm_epilogue", 16, 8192, 8192, "kn")
    assert path == "swap_splitk" and 1 <= splits <= 8
    assert gbf.gbf_kernel_path("swiglu", 2048, 14336, 4096)[0] == "pair"
    assert gbf.gbf_kernel_path("swiglu", 200, 14336, 4096)[0] == "persistent"
    assert gbf.gbf_kernel_path("swiglu", 33, 14336, 4096)[0] == "persistent"
    path, splits = gbf.gbf_kernel_path("swiglu", 16, 14336, 4096)
    assert path == "swap_splitk" and 1 <= splits <= 8
    for op in ("w8a16_fp8", "w4a16_nvfp4"):
        assert gbf.gbf_kernel_path(op, 16, 28672, 8192)[0] == "w4a16"
    assert gbf.gbf_kernel_path("w4a16_nvfp4", 16, 64, 48)[0] == "w4a16"
    assert gbf.gbf_kernel_path("w8a16_fp8", 16, 64, 48)[0] == "rejected"
    path, splits = gbf.gbf_kernel_path("w4a16", 16, 28672, 8192)
    assert path == "w4a16" and 1 <= splits <= 8
    assert gbf.gbf_kernel_path("gemm_epilogue", 0, 8, 8)[0] == "none"
    assert gbf.gbf_kernel_path("gemm_epilogue", 8, 12, 8)[0] == "rejected"
    assert gbf.gbf_kernel_path("w4a16", 8, 48, 128)[0] == "rejected"   # N % 32


def _bad(status):
    return status not in (0, 7)  # validation errors come before the device check


def test_validation_errors_are_returned_before_any_launch(lib):
    a = 0x10000  # never dereferenced: every call below fails validation first
    f = lambda **kw: gbf.gemm_epilogue(**{**dict(A=a, B=a, b_layout=1, C=None, bias=None,
                                                 residual=None, out=a, M=8, N=8, K=8),
                                          **kw}, stream=0, raise_on_error=False)
    assert f(A=None) == 1
    assert f(out=None) == 1
    assert f(b_layout=2) == 1
    assert f(act=4) == 1
    assert f(M=-1) == 1
    assert f(N=12) == 3
    assert f(K=20) == 3
    assert f(A=a + 8) == 2
    assert f(bias=a + 2) == 2
    s = gbf.w4a16_gemm(a, a, a, 100, None, None, None, a, 8, 64, 200, stream=0, raise_on_error=False)
    assert s == 3  # group size not a multiple of 64
    s = gbf.w4a16_gemm(a, a, a, 0, None, None, None, a, 8, 64, 128, stream=0, raise_on_error=False)
    assert s == 1
    s = gbf.w4a16_gemm(a, a, a, 128, None, None, None, a, 8, 48, 128, stream=0, raise_on_error=False)
    assert s == 3  # N % 32
    s = gbf.gemm_epilogue_unfused(a, a, 1, None, None, None, a, 8, 8, 8, workspace=None,
                                  workspace_bytes=0, stream=0, raise_on_error=False)
    assert s == 4
    s = gbf.swiglu_dual_gemm(a, a, None, 1, a, 8, 8, 8, stream=0, raise_on_error=False)
    assert s == 1
    # the NVFP4 kernel restores its 2^-19 operand scale through alpha
    nv = lambda alpha: gbf.w4a16_nvfp4_gemm(a, a, a, None, None, None, a, 8, 64, 64, alpha,
                                            stream=0, raise_on_error=False)
    assert nv(2.0 ** 100) == 1 and nv(-(2.0 ** 101)) == 1 and nv(3e38) == 1


def test_timeout_setting_is_clamped(lib):
    assert gbf.gbf_set_wait_timeout_ns(1) == 0
    assert gbf.gbf_set_wait_timeout_ns(2_000_000_000) == 0


def test_force_path_hook(lib):
    try:
        assert gbf.gbf_debug_force_path("persistent") == 0
        assert gbf.gbf_kernel_path("gemm_epilogue", 4096, 4096, 4096)[0] == "persistent"
        assert gbf.gbf_kernel_path("gemm_epilogue", 16, 4096, 4096)[0] == "swap_splitk"
        assert gbf.gbf_debug_force_path("pair") == 0
        assert gbf.gbf_kernel_path("gemm_epilogue", 300, 4096, 4096)[0] == "pair"
        assert gbf.gbf_kernel_path("swiglu", 200, 14336, 4096)[0] == "pair"
        assert gbf.gbf_debug_force_path("pair_splitk") == 0
        assert gbf.gbf_kernel_path("gemm_epilogue", 512, 4096, 4096) == ("pair_splitk", 2)
        # one K block cannot be split over two pairs
        assert gbf.gbf_kernel_path("gemm_epilogue", 512, 4096, 64)[0] != "pair_splitk"
        assert gbf.gbf_kernel_path("swiglu", 512, 4096, 4096)[0] != "pair_splitk"
        assert gbf.gbf_debug_force_path(2) == 1  # GBF_ERR_INVALID_ARG
        assert gbf.gbf_debug_force_path(8) == 1
    finally:
        gbf.gbf_debug_force_path(None)
    assert gbf.gbf_kernel_path("gemm_epilogue", 4096, 4096, 4096)[0] == "pair"


@pytest.mark.parametrize("op,M,N,K,layout,want", [
    # measured on one GB300 with every kernel forced, TFLOP/s
    # (CTA pair / one-SM / one-SM split-K / CTA pair with one stream /
    # its split-K form over two pairs per tile):
    ("gemm_epilogue", 256, 4096, 4096, "nk", "pair_splitk"),         # 209 / 265 / 379 / 322 / 450
    ("gemm_epilogue", 384, 4096, 4096, "nk", "pair_splitk"),         # 314 / 399 / 565 / 482 / 646
    ("gemm_epilogue", 512, 4096, 4096, "nk", "pair_splitk"),         # 410 / 527 / 720 / 641 / 850
    ("gemm_epilogue", 512, 2048, 2048, "nk", "pair_splitk"),         # 159 / 209 / 261 / 249 / 308
    ("gemm_epilogue", 640, 4096, 4096, "nk", "pair_1stream"),        # 508 / 654 / 544 / 815 / 572
    ("gemm_epilogue", 768, 4096, 4096, "nk", "pair_1stream"),        # 610 / 784 / 624 / 969 / 682
    ("gemm_epilogue", 1024, 4096, 4096, "nk", "pair_1stream"),       # 810 / 1044 / 802 / 1274 / 883
    ("gemm_epilogue", 1536, 4096, 4096, "nk", "pair"),               # 1185 / 927 / 838 / 1049
    ("gemm_epilogue", 2048, 4096, 4096, "nk", "pair"),               # 1564 / 1218 / 862 / 1395
    ("gemm_epilogue", 256, 8192, 8192, "kn", "pair_splitk"),         # 486 / 620 / 925 / 738 / 1077
    ("gemm_epilogue", 512, 8192, 8192, "kn", "pair_1stream"),        # 951 / 1205 / 1048 / 1456 / 1179
    ("gemm_epilogue", 768, 8192, 8192, "kn", "pair"),                # 1240 / 1014 / 1095 / 1179
    ("gemm_epilogue", 1536, 8192, 8192, "kn", "pair_1stream"),       # 1283 / 1360 / 1185 / 1587
    ("gemm_epilogue", 384, 14336, 4096, "nk", "pair"),               # 1021 / 737 / 708 / 931 / 594
    ("gemm_epilogue", 640, 14336, 4096, "nk", "persistent"),         # 925 / 1274 / 899 / 1070
    ("gemm_epilogue", 1024, 14336, 4096, "nk", "pair_1stream"),      # 1453 / 1434 / 985 / 1590
    # earlier measurements (pair / one-SM), still the planner's choice:
    ("gemm_epilogue", 4096, 4096, 4096, "nk", "pair"),               # 1595 / 1354
    ("gemm_epilogue", 3072, 8192, 8192, "kn", "pair"),               # 1648 / 1447
    ("gemm_epilogue", 4096, 14336, 4096, "nk", "pair"),              # 1633 / 1489
    ("swiglu", 512, 14336, 4096, "nk", "persistent"),                # 1347 / 1456
    ("swiglu", 1024, 14336, 4096, "nk", "pair"),                     # 1790 / 1581
])
def test_planner_picks_the_measured_faster_kernel(lib, op, M, N, K, layout, want):
    assert gbf.gbf_kernel_path(op, M, N, K, layout)[0] == want

"""GPU parity of the gated MLP block chain ("Fusion Thinking", Pattern 2 with
the down projection, and Pattern 1's residual add after the MLP): the fused
gate/up GEMM writes bf16 h, the down GEMM adds the residual in its ending.
Checked stage by stage against the oracle: h against the oracle's h from x,
then out against the oracle's down projection of the h the GPU produced.
Also the unfused composition, and the CUDA-graph replay ("Fusion Thinking",
CUDA Graphs section), which must give the same bits as direct launches."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import assert_parity, down, poison_bf16, up

pytestmark = pytest.mark.gpu


def block_inputs(M, D, F, seed=0):
    w = workloads.make("mlp_decode", shape=dict(M=M, D=D, F=F, N=D, K=D))
    if seed:
        rng = np.random.Generator(np.random.PCG64(seed))
        w["x"] = workloads.to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
        w["residual"] = workloads.to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
    return w


def check_stagewise(w, h_gpu, out_gpu, M, D, F, residual=True, what=""):
    _, h_want = oracle.mlp_swiglu_down(w["x"], w["w_gate"], w["w_up"], w["w_down"], None,
                                       M=M, D=D, F=F)
    assert_parity(h_gpu, h_want, f"{what} h")
    out_want = oracle.gemm_epilogue(h_gpu, w["w_down"], "nk",
                                    residual=w["residual"] if residual else None,
                                    M=M, N=D, K=F)
    assert_parity(out_gpu, out_want, f"{what} out")


def check_unfused_stagewise(w, ws, out_gpu, M, D, F, what=""):
    """The unfused chain stores g, u, h and the down product D in bf16; each
    stored tensor is a rounding decision, so every kernel is checked on the
    GPU's own inputs: g, u against the oracle's products of x, h against the
    oracle's GLU of the GPU's g and u, D against the oracle's product of the
    GPU's h, out against the oracle's residual add of the GPU's D."""
    hb = (M * F * 2 + 255) // 256 * 256

    def sect(off, rows, cols):
        return down(ws[off:off + rows * cols * 2].view(torch.bfloat16).view(rows, cols))

    g, u, h, d = sect(0, M, F), sect(hb, M, F), sect(2 * hb, M, F), sect(3 * hb, M, D)
    for name, wt, got in (("g", w["w_gate"], g), ("u", w["w_up"], u)):
        assert_parity(got, oracle.gemm_epilogue(w["x"], wt, "nk", M=M, N=F, K=D),
                      f"{what} {name}")
    assert_parity(h, oracle.swiglu_pointwise(g, u, M=M, N=F), f"{what} h")
    assert_parity(d, oracle.gemm_epilogue(h, w["w_down"], "nk", M=M, N=D, K=F), f"{what} D")
    assert_parity(out_gpu, oracle.pointwise_epilogue(d, residual=w["residual"], M=M, N=D),
                  f"{what} out")


def run_block(cuda_lib, w, M, D, F, fused=True, residual=True, inplace=False, keep_ws=False):
    ws_bytes = cuda_lib.gbf_workspace_size("mlp", M, D, F, fused)
    ws = torch.full((max(ws_bytes, 256),), 0xFF, dtype=torch.uint8, device="cuda")
    r = up(w["residual"]) if residual else None
    out = r if inplace else poison_bf16(M, D)
    fn = cuda_lib.mlp_swiglu_down if fused else cuda_lib.mlp_swiglu_down_unfused
    fn(up(w["x"]), up(w["w_gate"]), up(w["w_up"]), up(w["w_down"]), r, out, M, D, F, ws,
       ws_bytes)
    assert cuda_lib.gbf_check_device_error() == 0
    hb = (M * F * 2 + 255) // 256 * 256
    off = 0 if fused else 2 * hb
    h = down(ws[off:off + M * F * 2].view(torch.bfloat16).view(M, F))
    if keep_ws:
        return ws, down(out)
    return h, down(out)


@pytest.mark.parametrize("M,D,F", [(1, 256, 512), (16, 1024, 2816), (37, 512, 1376),
                                   (300, 1024, 2048), (640, 512, 1024)])
def test_mlp_chain_fused(cuda_lib, M, D, F):
    w = block_inputs(M, D, F)
    h, out = run_block(cuda_lib, w, M, D, F)
    check_stagewise(w, h, out, M, D, F, what=f"fused {M}x{D}x{F}")


@pytest.mark.parametrize("M,D,F", [(16, 1024, 2816), (300, 512, 1024)])
def test_mlp_chain_unfused(cuda_lib, M, D, F):
    w = block_inputs(M, D, F)
    ws, out = run_block(cuda_lib, w, M, D, F, fused=False, keep_ws=True)
    check_unfused_stagewise(w, ws, out, M, D, F, what=f"unfused {M}x{D}x{F}")


def test_mlp_chain_decode_workload_full_output(cuda_lib):
    w = workloads.make("mlp_decode")
    M, D, F = w["M"], w["D"], w["F"]
    h, out = run_block(cuda_lib, w, M, D, F)
    check_stagewise(w, h, out, M, D, F, what="decode workload")


def test_mlp_chain_in_place_residual_and_no_residual(cuda_lib):
    M, D, F = 16, 512, 1024
    w = block_inputs(M, D, F, seed=5)
    h, out = run_block(cuda_lib, w, M, D, F, inplace=True)
    check_stagewise(w, h, out, M, D, F, what="in place")
    h, out = run_block(cuda_lib, w, M, D, F, residual=False)
    check_stagewise(w, h, out, M, D, F, residual=False, what="no residual")


def test_mlp_chain_degenerate_sizes(cuda_lib):
    w = block_inputs(4, 64, 128, seed=3)
    x, wg, wu, wd = (up(w[k]) for k in ("x", "w_gate", "w_up", "w_down"))
    r = up(w["residual"])
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    out = poison_bf16(4, 64)
    # F = 0: the down product is empty and the block returns the residual
    assert cuda_lib.mlp_swiglu_down(x, wg, wu, wd, r, out, 4, 64, 0, ws, ws.numel()) == 0
    assert cuda_lib.gbf_check_device_error() == 0
    assert np.array_equal(down(out), w["residual"])
    # M = 0: nothing to do, nothing written
    out2 = poison_bf16(4, 64)
    assert cuda_lib.mlp_swiglu_down(x, wg, wu, wd, r, out2, 0, 64, 128, ws, ws.numel()) == 0
    assert torch.isnan(out2.float()).all()


def test_mlp_chain_validation(cuda_lib):
    t = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    f = lambda fn=cuda_lib.mlp_swiglu_down, **kw: fn(**{**dict(
        x=t, w_gate=t, w_up=t, w_down=t, residual=None, out=t, M=16, D=64, F=128,
        workspace=ws, workspace_bytes=ws.numel()), **kw}, raise_on_error=False)
    assert f() == 0
    assert f(F=12) == 3
    assert f(D=60) == 3
    assert f(M=-1) == 1
    assert f(x=None) == 1
    assert f(workspace=None, workspace_bytes=0) == 4
    assert f(workspace_bytes=16 * 128 * 2 - 2) == 4
    assert f(fn=cuda_lib.mlp_swiglu_down_unfused, workspace_bytes=16 * 128 * 2) == 4
    assert f(out=t[1:]) == 2
    torch.cuda.synchronize()


def test_graph_replay_matches_direct_launches(cuda_lib):
    from tcgen05_tmem_bf16_gb300.graphs import MLPBlock
    M, D, F = 16, 1024, 2816
    w = block_inputs(M, D, F)
    wg, wu, wd = (up(w[k]) for k in ("w_gate", "w_up", "w_down"))
    direct = MLPBlock(wg, wu, wd, M, graph=False)
    graphed = MLPBlock(wg, wu, wd, M, graph=True)
    for seed in (0, 9, 10):
        wi = block_inputs(M, D, F, seed=seed)
        x, r = up(wi["x"]), up(wi["residual"])
        a = down(direct.run(x, r))
        b = down(graphed.run(x, r))
        assert cuda_lib.gbf_check_device_error() == 0
        assert np.array_equal(a, b), f"graph replay differs from direct launches (seed {seed})"
        check_stagewise(wi, down(graphed.h), b, M, D, F, what=f"graph seed {seed}")


def test_graph_replay_of_unfused_chain(cuda_lib):
    from tcgen05_tmem_bf16_gb300.graphs import MLPBlock
    M, D, F = 8, 512, 1024
    w = block_inputs(M, D, F, seed=4)
    blk = MLPBlock(up(w["w_gate"]), up(w["w_up"]), up(w["w_down"]), M, fused=False)
    out = down(blk.run(up(w["x"]), up(w["residual"])))
    assert cuda_lib.gbf_check_device_error() == 0
    check_unfused_stagewise(w, blk.workspace, out, M, D, F, what="unfused graph")


def test_graph_buckets_pad_rows(cuda_lib):
    from tcgen05_tmem_bf16_gb300.graphs import MLPBlockBuckets
    D, F = 512, 1024
    w = block_inputs(16, D, F, seed=6)
    buckets = MLPBlockBuckets(up(w["w_gate"]), up(w["w_up"]), up(w["w_down"]),
                              buckets=(1, 8, 16))
    for rows in (1, 5, 16):
        x, r = w["x"][:rows], w["residual"][:rows]
        out = down(buckets.run(up(x), up(r)))
        assert cuda_lib.gbf_check_device_error() == 0
        blk = next(b for m, b in buckets.blocks.items() if rows <= m)
        wi = dict(w, x=x, residual=r)
        check_stagewise(wi, down(blk.h)[:rows], out, rows, D, F, what=f"bucket rows {rows}")
    with pytest.raises(ValueError):
        buckets.run(up(w["x"][:1]).repeat(17, 1), up(w["residual"][:1]).repeat(17, 1))

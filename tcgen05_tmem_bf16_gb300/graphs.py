"""CUDA-graph capture of a fixed chain of library calls, and the gated MLP
block (gate/up GEMM -> bf16 h -> down GEMM + residual) replayed from one.

A graph records the launches of a chain once and replays them as a single
submission, so a decode step pays one launch instead of the per-call host
work (argument checks, tensor-map encoding, kernel launch) of every call in
the chain ("Fusion Thinking", CUDA Graphs section: capture once, replay with
new inputs copied in place; one graph per input shape, several shape buckets
captured up front).

Everything here is host plumbing around the C ABI: the launches inside the
graph are the library's own kernels.  The caller's buffers are baked into the
graph by address, so inputs change by copying into the static tensors.
"""
from __future__ import annotations

import torch

from . import gbf_workspace_size, mlp_swiglu_down, mlp_swiglu_down_unfused


class CapturedChain:
    """``chain(stream)`` issues a fixed sequence of launches on ``stream``.
    The chain runs ``warmup`` times on a side stream first (which also lets
    the library set up its per-device state, which a capture must not do),
    then once under capture; ``replay()`` re-issues the recorded launches on
    the current stream."""

    def __init__(self, chain, warmup: int = 3):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                chain(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            chain(torch.cuda.current_stream())

    def replay(self):
        self.graph.replay()


class MLPBlock:
    """One gated MLP block with its residual, ``out = W_down(silu(W_gate x) *
    (W_up x)) + residual``, for a fixed number of rows M.

    Weights: w_gate, w_up [F][D], w_down [D][F], bf16 on the device.  The
    block owns static x / residual / out tensors and the workspace holding h;
    ``run(x, residual)`` copies the inputs in and replays the captured graph
    (``graph=False`` issues the two launches directly instead).  ``fused=False``
    runs the unfused composition (g, u, h and the down product all stored in
    HBM between kernels)."""

    def __init__(self, w_gate, w_up, w_down, M: int, fused: bool = True, graph: bool = True):
        F, D = w_gate.shape
        if tuple(w_up.shape) != (F, D) or tuple(w_down.shape) != (D, F):
            raise ValueError("w_gate, w_up must be [F][D] and w_down [D][F]")
        dev = w_gate.device
        self.M, self.D, self.F, self.fused = M, D, F, fused
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.x = torch.zeros(M, D, dtype=torch.bfloat16, device=dev)
        self.residual = torch.zeros(M, D, dtype=torch.bfloat16, device=dev)
        self.out = torch.empty(M, D, dtype=torch.bfloat16, device=dev)
        self.ws_bytes = gbf_workspace_size("mlp", M, D, F, fused)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.graph = CapturedChain(self.launch) if graph else None

    @property
    def h(self):
        """The block's bf16 h [M][F] as left in the workspace (fused form) or
        its h section (unfused form: after g and u)."""
        off = 0 if self.fused else 2 * self._h_bytes()
        n = self.M * self.F
        return self.workspace[off:off + 2 * n].view(torch.bfloat16).view(self.M, self.F)

    def _h_bytes(self):
        return (self.M * self.F * 2 + 255) // 256 * 256

    def launch(self, stream=None):
        fn = mlp_swiglu_down if self.fused else mlp_swiglu_down_unfused
        fn(self.x, self.w_gate, self.w_up, self.w_down, self.residual, self.out, self.M,
           self.D, self.F, self.workspace, self.ws_bytes, stream=stream)

    def run(self, x=None, residual=None):
        if x is not None:
            self.x.copy_(x)
        if residual is not None:
            self.residual.copy_(residual)
        if self.graph is not None:
            self.graph.replay()
        else:
            self.launch()
        return self.out


class MLPBlockBuckets:
    """One captured MLPBlock per row count; ``run`` pads a batch of rows up
    to the smallest bucket that holds it and returns its rows of the
    output."""

    def __init__(self, w_gate, w_up, w_down, buckets=(1, 8, 16, 32, 64)):
        self.blocks = {m: MLPBlock(w_gate, w_up, w_down, m) for m in sorted(buckets)}

    def run(self, x, residual):
        rows = x.shape[0]
        for m, blk in self.blocks.items():
            if rows <= m:
                blk.x.zero_()
                blk.residual.zero_()
                blk.x[:rows].copy_(x)
                blk.residual[:rows].copy_(residual)
                return blk.run()[:rows]
        raise ValueError(f"{rows} rows exceed the largest bucket {max(self.blocks)}")

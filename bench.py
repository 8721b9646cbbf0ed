#!/usr/bin/env python3
"""Benchmark of the fused GEMM + epilogue path on GB300.

One step = one pass of the hot path over one batch of synthetic input: a
single fused call (TMA staging -> tcgen05 main loop -> fused epilogue ->
one store).  The default run (--workload all) measures every workload: the
JSON line's headline (value, roofline, e2e, cpu_baseline) is the largest one,
the epilogue sweep at M = 8192 (out = gelu_tanh(0.75*A*B + 0.25*C + bias),
A[8192x8192], B[8192x8192], bf16 in, fp32 accumulate, bf16 out), and the key
"configs" holds one record per other workload (the tiny case, the prefill
projection, the gate/up SwiGLU GEMM, the W4A16 decode GEMM, the sweep at
M = 1, 16, 128 and 1024, and the FP8 / NVFP4 weight-only GEMMs, fused
add + RMSNorm, the level-1 SwiGLU ending and the MLP block at decode), each
with its value, roofline fractions against both the tensor and the HBM peak,
recorded DRAM traffic and fused-vs-unfused speedup.  --workload NAME runs one
workload alone.

Prints ONE JSON line.  ``value`` is whole-job throughput (the workload's
metric: TFLOP/s when tensor-bound, GB/s of algorithmic bytes when HBM-bound,
summed over ranks / max over ranks of the timed region).  Inputs are
resident in HBM; rotating input sets (>= 2x L2 in total) keep consecutive
steps from reading each other's data out of L2.  CUDA events on the launching
stream bracket the timed region; a step is one kernel launch, so region /
steps is the kernel's average launch duration used for the roofline
fraction.  Extra keys: roofline, cpu_baseline (the fp64 oracle timed on a
bounded sample on all host cores, with the single-threaded build beside it),
e2e (the same metric with host buffers and host<->device copies inside the
timed region), clocks (nvidia-smi samples taken during the timed region),
the unfused composition's time and the fused-vs-unfused speedup.

--impl reference times the fp64 CPU oracle (the only reference this path
has) on the same workload, each step a bounded sample of output elements.

Multi-GPU: the path shards with no exchange step, so N GPUs run N
independent replicas (launched by torchrun); the timed region is bracketed by
barriers and its maximum over ranks is used.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+epilogue TFLOP/s or GB/s as % of roofline; fused vs unfused speedup"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024

HEADLINE = "sweep-8192"
SUB_WORKLOADS = ("tiny", "prefill", "swiglu", "w4a16", "sweep-1", "sweep-16", "sweep-128",
                 "sweep-1024", "w8a16_fp8", "w4a16_nvfp4", "add_rmsnorm", "swiglu_pointwise",
                 "mlp_decode")

WORKLOAD_TEXT = {
    "add_rmsnorm": "fused residual add + RMSNorm, a,x[4096x4096] bf16, eps 1e-5",
    "swiglu_pointwise": "level-1 fused SwiGLU ending, g,u[2048x14336] bf16 (vs eager sigmoid/mul/mul)",
    "prefill": "prefill projection A[4096x4096] x W[4096x4096]^T + bias + residual, bf16",
    "swiglu": "gate/up SwiGLU dual GEMM x[2048x4096], Wg,Wu[14336x4096], bf16",
    "w4a16": "W4A16 decode GEMM A[16x8192] x int4 W[8192x28672], group 128",
    "w8a16_fp8": "FP8-weight decode GEMM A[16x8192] x E4M3 W[8192x28672], bf16 scales per 128",
    "w4a16_nvfp4": "NVFP4-weight decode GEMM A[16x8192] x E2M1 W[8192x28672], E4M3 scales "
                   "per 16, per-tensor factor 1/256",
    "tiny": "tiny fused GEMM 64x256x128, SiLU(0.5AB + C + bias)",
    "mlp_decode": "gated MLP block + residual at decode, x[16x4096], Wg,Wu[14336x4096], "
                  "Wd[4096x14336], bf16, replayed from one CUDA graph",
}


# ---------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCE = {"gemm_pair_kernel": "gemm_pair.cu", "gemm_persistent_kernel": "gemm_tc.cu",
                 "gemm_swap_kernel": "gemm_tc.cu", "wq_gemm_kernel": "wq_gemm.cu",
                 "add_rmsnorm_kernel": "rmsnorm.cu", "swiglu_pointwise_kernel": "pointwise.cu"}


def _code_only(src: str) -> str:
    """C++/CUDA source without its comments and with every run of white
    space reduced to one blank (the sources hold no comment markers inside
    string literals)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return re.sub(r"\s+", " ", src).strip()


def kernel_source_sha(kernel: str) -> str:
    """Hash of the code a kernel is built from (comments left out): its own
    .cu file, the shared headers and the launch planner."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tcgen05_tmem_bf16_gb300", "csrc")
    own = KERNEL_SOURCE.get(kernel)
    for name in sorted(os.listdir(csrc)):
        if name.endswith(".cu") and name not in (own, "api.cu"):
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    capture, if it was taken on the kernel's current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel") != kernel or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(seconds: float, units: float, world: int):
    """(max seconds over ranks, sum of units over ranks)."""
    if world <= 1:
        return seconds, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen([exe, "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=self.fh, stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return math.nan
        loaded = [r for r in rows if num(r[4]) >= 50] or rows
        sm = [num(r[1]) for r in loaded if not math.isnan(num(r[1]))]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in loaded:
            for name, v in zip(names, r[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]),
                "power_w_max": max(num(r[3]) for r in loaded),
                "samples": len(rows), "samples_under_load": len(loaded),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workloads

def describe(w: dict) -> dict:
    if w["op"] == "mlp":
        return {"M": w["M"], "D": w["D"], "F": w["F"], "op": "mlp", "act": "silu"}
    d = {"M": w["M"], "N": w["N"], "K": w["K"], "op": w["op"]}
    if "eps" in w:
        d["eps"] = w["eps"]
    if "layout" in w:
        d["b_layout"] = w["layout"]
    if w["op"] in ("w4a16", "w8a16_fp8", "w4a16_nvfp4"):
        d["group_size"] = w["group"]
    d.update(alpha=w["alpha"], beta=w["beta"], act=w["act"])
    return d


def workload_text(name: str) -> str:
    if name.startswith("sweep-"):
        M = int(name.split("-")[1])
        return (f"epilogue sweep M={M}: gelu_tanh(0.75*A*B + 0.25*C + bias), A[{M}x8192], "
                f"B[8192x8192] (K x N), C[{M}x8192], bf16")
    return WORKLOAD_TEXT.get(name, name)


def config_of(name: str, w: dict, world: int) -> dict:
    return {"workload": workload_text(name), "name": name, **describe(w),
            "parallelism": f"replicas x{world}"}


class Workload:
    """Device inputs (several rotating sets), host copies for e2e, and the
    fused/unfused calls of one workload."""

    def __init__(self, name: str, dev):
        import numpy as np
        import torch

        import tcgen05_tmem_bf16_gb300 as gbf
        import workloads
        from tcgen05_tmem_bf16_gb300 import roofline

        self.gbf, self.np, self.torch = gbf, np, torch
        self.name = name
        if name.startswith("sweep-"):
            M = int(name.split("-")[1])
            w = workloads.make("sweep", M=M)
        else:
            w = workloads.make(name)
        self.w = w
        self.op = w["op"]
        self.M, self.N, self.K = w["M"], w["N"], w["K"]
        self.counts = roofline.counts_for(w)
        host = {}
        for key in ("A", "B", "C", "bias", "residual", "x", "w_gate", "w_up", "w_down", "Wq",
                    "scales", "a", "weight", "g", "u"):
            if w.get(key) is not None:
                host[key] = w[key]
        self.host_np = host
        set_bytes = sum(v.nbytes for v in host.values()) + self.M * self.N * 2
        self.n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes))
        self.set_bytes = set_bytes

        def up(a):
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            t = t.to(dev)
            return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

        self.sets = []
        for _ in range(self.n_sets):
            d = {k: up(v) for k, v in host.items()}
            d["out"] = torch.empty(self.M, self.N, dtype=torch.bfloat16, device=dev)
            if self.op == "add_rmsnorm":
                d["resid"] = torch.empty(self.M, self.N, dtype=torch.bfloat16, device=dev)
            self.sets.append(d)
        gemm_op = {"gemm": "gemm_epilogue", "swiglu": "swiglu", "w4a16": "w4a16",
                   "mlp": "mlp", "w8a16_fp8": "w8a16_fp8",
                   "w4a16_nvfp4": "w4a16_nvfp4"}.get(self.op)
        wK = w["F"] if self.op == "mlp" else self.K
        ws = gbf.gbf_workspace_size(gemm_op, self.M, self.N, wK, False) if gemm_op else 0
        self.ws_bytes = ws
        self.ws_fused_bytes = gbf.gbf_workspace_size(gemm_op, self.M, self.N, wK, True) \
            if gemm_op else 0
        self.ws = torch.empty(max(ws, self.ws_fused_bytes, 16), dtype=torch.uint8, device=dev)
        # pinned host buffers for the end-to-end leg: every operand, except for
        # the MLP block, whose per-step inputs are its activations (x and the
        # residual) while its weights stay resident like a model's parameters
        step_keys = ("x", "residual") if self.op == "mlp" else tuple(host)
        self.pinned = {k: torch.from_numpy(host[k].copy()).pin_memory() for k in step_keys}
        self.pinned_out = [torch.empty(self.M * self.N * 2, dtype=torch.uint8).pin_memory()
                           for _ in range(2)]
        self.h2d_bytes = sum(host[k].nbytes for k in step_keys)
        self.d2h_bytes = self.M * self.N * 2
        self.graphs = None
        if self.op == "mlp":
            self.path, self.splits = gbf.gbf_kernel_path("swiglu", self.M, w["F"], w["D"], "nk")
        elif gemm_op:
            self.path, self.splits = gbf.gbf_kernel_path(gemm_op, self.M, self.N, self.K,
                                                         w.get("layout", "kn"))
        else:
            self.path, self.splits = self.op, 1

    def describe(self) -> dict:
        return describe(self.w)

    def mlp_direct(self, i: int, stream=None, fused: bool = True):
        s = self.sets[i % self.n_sets]
        w, gbf = self.w, self.gbf
        fn = gbf.mlp_swiglu_down if fused else gbf.mlp_swiglu_down_unfused
        fn(s["x"], s["w_gate"], s["w_up"], s["w_down"], s["residual"], s["out"], self.M, w["D"],
           w["F"], self.ws, self.ws_fused_bytes if fused else self.ws_bytes, stream=stream)

    def capture(self):
        """MLP block: one CUDA graph per input set, fused and unfused chains."""
        from tcgen05_tmem_bf16_gb300.graphs import CapturedChain
        self.graphs = [CapturedChain(lambda st, i=i: self.mlp_direct(i, st))
                       for i in range(self.n_sets)]
        self.graphs_unfused = [CapturedChain(lambda st, i=i: self.mlp_direct(i, st, False))
                               for i in range(self.n_sets)]

    def launches_per_step(self) -> int:
        return 2 if self.op == "mlp" else 1

    def fused(self, i: int, stream=None):
        s = self.sets[i % self.n_sets]
        w, gbf = self.w, self.gbf
        if self.op == "mlp":
            if self.graphs is None:
                self.mlp_direct(i, stream)
            else:
                self.graphs[i % self.n_sets].replay()
        elif self.op == "gemm":
            gbf.gemm_epilogue(s["A"], s["B"], w["layout"], s.get("C"), s.get("bias"),
                              s.get("residual"), s["out"], self.M, self.N, self.K, w["alpha"],
                              w["beta"], w["act"], stream=stream)
        elif self.op == "swiglu":
            gbf.swiglu_dual_gemm(s["x"], s["w_gate"], s["w_up"], w["layout"], s["out"], self.M,
                                 self.N, self.K, w["alpha"], w["beta"], s.get("C"), w["act"],
                                 stream=stream)
        elif self.op == "w4a16":
            gbf.w4a16_gemm(s["A"], s["Wq"], s["scales"], w["group"], s.get("C"), s.get("bias"),
                           s.get("residual"), s["out"], self.M, self.N, self.K, w["alpha"],
                           w["beta"], w["act"], stream=stream)
        elif self.op == "w8a16_fp8":
            gbf.w8a16_fp8_gemm(s["A"], s["Wq"], s["scales"], w["group"], None, None, None,
                               s["out"], self.M, self.N, self.K, w["alpha"], w["beta"],
                               w["act"], stream=stream)
        elif self.op == "w4a16_nvfp4":
            gbf.w4a16_nvfp4_gemm(s["A"], s["Wq"], s["scales"], None, None, None, s["out"],
                                 self.M, self.N, self.K, w["alpha"], w["beta"], w["act"],
                                 stream=stream)
        elif self.op == "add_rmsnorm":
            gbf.add_rmsnorm(s["a"], s["x"], s["weight"], s["out"], s["resid"], self.M, self.N,
                            w["eps"], stream=stream)
        else:
            gbf.swiglu_pointwise(s["g"], s["u"], None, s["out"], self.M, self.N, w["alpha"],
                                 w["beta"], w["act"], stream=stream)

    def unfused(self, i: int, stream=None):
        s = self.sets[i % self.n_sets]
        w, gbf = self.w, self.gbf
        kw = dict(workspace=self.ws, workspace_bytes=self.ws_bytes, stream=stream)
        if self.op == "mlp":
            if self.graphs is None:
                self.mlp_direct(i, stream, fused=False)
            else:
                self.graphs_unfused[i % self.n_sets].replay()
        elif self.op == "gemm":
            gbf.gemm_epilogue_unfused(s["A"], s["B"], w["layout"], s.get("C"), s.get("bias"),
                                      s.get("residual"), s["out"], self.M, self.N, self.K,
                                      w["alpha"], w["beta"], w["act"], **kw)
        elif self.op == "swiglu":
            gbf.swiglu_dual_gemm_unfused(s["x"], s["w_gate"], s["w_up"], w["layout"], s["out"],
                                         self.M, self.N, self.K, w["alpha"], w["beta"],
                                         s.get("C"), w["act"], **kw)
        elif self.op == "w4a16":
            gbf.w4a16_gemm_unfused(s["A"], s["Wq"], s["scales"], w["group"], s.get("C"),
                                   s.get("bias"), s.get("residual"), s["out"], self.M, self.N,
                                   self.K, w["alpha"], w["beta"], w["act"], **kw)
        elif self.op == "w8a16_fp8":
            gbf.w8a16_fp8_gemm_unfused(s["A"], s["Wq"], s["scales"], w["group"], None, None,
                                       None, s["out"], self.M, self.N, self.K, w["alpha"],
                                       w["beta"], w["act"], **kw)
        elif self.op == "w4a16_nvfp4":
            gbf.w4a16_nvfp4_gemm_unfused(s["A"], s["Wq"], s["scales"], None, None, None,
                                         s["out"], self.M, self.N, self.K, w["alpha"],
                                         w["beta"], w["act"], **kw)
        elif self.op == "add_rmsnorm":
            gbf.add_rmsnorm_unfused(s["a"], s["x"], s["weight"], s["out"], s["resid"], self.M,
                                    self.N, w["eps"], stream=stream)
        else:
            # the eager composition the level-1 kernel replaces: sigmoid, mul, mul
            g, u = s["g"], s["u"]
            torch = self.torch
            torch.mul(torch.mul(g, torch.sigmoid(g)), u, out=s["out"])

    def unfused_kind(self) -> str:
        if self.op == "swiglu_pointwise":
            return "eager torch: sigmoid, mul, mul (3 kernels)"
        if self.op == "mlp":
            return ("two GEMMs -> bf16 g, u -> GLU pointwise -> bf16 h -> GEMM -> bf16 D -> "
                    "residual-add pass (5 kernels, one CUDA graph)")
        return {"gemm": "GEMM -> bf16 D in HBM -> pointwise kernel",
                "swiglu": "two GEMMs -> bf16 g, u in HBM -> GLU pointwise kernel",
                "w4a16": "dequantise kernel -> bf16 W in HBM -> bf16 GEMM",
                "w8a16_fp8": "dequantise kernel -> bf16 W in HBM -> bf16 GEMM",
                "w4a16_nvfp4": "dequantise kernel -> bf16 W in HBM -> bf16 GEMM",
                "add_rmsnorm": "residual-add kernel -> bf16 r in HBM -> RMSNorm kernel"}[self.op]

    def copy_in(self, b: int):
        """Host->device copy of a step's inputs into input set b (current stream)."""
        s = self.sets[b]
        for k, v in self.pinned.items():
            dst = s[k]
            dst_raw = dst.view(self.torch.int16) if dst.dtype == self.torch.bfloat16 else dst
            src = v if v.dtype != self.torch.uint16 else v.view(self.torch.int16)
            dst_raw.copy_(src.view(dst_raw.dtype), non_blocking=True)

    def e2e_run(self, steps: int, stream) -> float:
        """`steps` end-to-end steps through the public API, timed on the device:
        each step copies its inputs from pinned host memory into one of two
        device input sets, makes the call, and copies its result back to pinned
        host memory.  The copies run on their own streams, so a step's input
        copy overlaps the previous step's call and result copy (as a serving
        loop would); events order every copy against the calls that use its
        buffers.  Returns the region in seconds."""
        torch = self.torch
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(steps)]
        ev_call = [torch.cuda.Event() for _ in range(steps)]
        ev_out = [torch.cuda.Event() for _ in range(steps)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_call[i - 2])  # set b is no longer read
                self.copy_in(b)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # set b's result has been read back
            self.fused(b, stream=stream)
            ev_call[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_call[i])
                self.pinned_out[b].copy_(self.sets[b]["out"].view(torch.uint8).reshape(-1),
                                         non_blocking=True)
                ev_out[i].record(s_out)
        stream.wait_event(ev_out[-1])
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / 1e3


def time_loop(fn, steps: int, stream, per_launch: bool):
    """Run fn(i) `steps` times on `stream`; returns (region seconds, mean
    per-launch seconds or None)."""
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    evs = []
    if per_launch:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    start.record(stream)
    for i in range(steps):
        if per_launch:
            evs[i][0].record(stream)
        fn(i)
        if per_launch:
            evs[i][1].record(stream)
    end.record(stream)
    end.synchronize()
    region = start.elapsed_time(end) / 1e3
    per = None
    if per_launch:
        per = sum(a.elapsed_time(b) for a, b in evs) / len(evs) / 1e3
    return region, per


# ---------------------------------------------------------------- CPU (oracle) legs

def oracle_elements(w: dict, rows, cols):
    """The oracle on the given output positions (row-wise ops: on the rows
    they belong to).  Returns the number of output elements computed."""
    import numpy as np
    import oracle
    op = w["op"]
    M, N, K = w["M"], w["N"], w["K"]
    if op in ("add_rmsnorm", "swiglu_pointwise", "mlp"):
        r = np.unique(np.asarray(rows) % M)
        if op == "mlp":
            oracle.mlp_swiglu_down(w["x"], w["w_gate"], w["w_up"], w["w_down"], w["residual"],
                                   M=M, D=w["D"], F=w["F"], rows=r)
        elif op == "add_rmsnorm":
            oracle.add_rmsnorm(w["a"][r], w["x"][r], w["weight"], M=r.size, N=N, eps=w["eps"])
        else:
            oracle.swiglu_pointwise(w["g"][r], w["u"][r], M=r.size, N=N, alpha=w["alpha"],
                                    beta=w["beta"], act=w["act"])
        return r.size * N
    if op == "gemm":
        oracle.gemm_epilogue(w["A"], w["B"], w["layout"], w.get("C"), w.get("bias"),
                             w.get("residual"), M=M, N=N, K=K, alpha=w["alpha"],
                             beta=w["beta"], act=w["act"], rows=rows, cols=cols)
    elif op == "swiglu":
        oracle.swiglu(w["x"], w["w_gate"], w["w_up"], w["layout"], w.get("C"), M=M, N=N,
                      K=K, alpha=w["alpha"], beta=w["beta"], act=w["act"], rows=rows,
                      cols=cols)
    elif op in ("w8a16_fp8", "w4a16_nvfp4"):
        oracle.wq_gemm("fp8" if op == "w8a16_fp8" else "nvfp4", w["A"], w["Wq"], w["scales"],
                       w["group"], M=M, N=N, K=K, alpha=w["alpha"], beta=w["beta"],
                       act=w["act"], rows=rows, cols=cols)
    else:
        oracle.w4a16(w["A"], w["Wq"], w["scales"], w["group"], w.get("C"), w.get("bias"),
                     w.get("residual"), M=M, N=N, K=K, alpha=w["alpha"], beta=w["beta"],
                     act=w["act"], rows=rows, cols=cols)
    return len(rows)


def metric_per_element(w: dict):
    """(units of the workload's metric per output element, unit): algorithmic
    FLOPs (TFLOP/s) for tensor-bound workloads, algorithmic bytes (GB/s) for
    HBM-bound ones, spread evenly over the M*N outputs."""
    from tcgen05_tmem_bf16_gb300 import roofline as rf
    peaks, _ = load_peaks()
    c = rf.counts_for(w)
    per = 1.0 / (w["M"] * w["N"])
    if rf.bound(c, peaks["bf16_tflops"], peaks["hbm_gbs"]) == "tensor":
        return c.flops * per / 1e12, "TFLOP/s"
    return c.fused_bytes * per / 1e9, "GB/s"


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_sample(w: dict, seconds: float, parallel: bool):
    """(output elements, seconds, threads) of the oracle on seeded positions
    of the workload for about `seconds`."""
    import oracle
    import workloads
    rows, cols = workloads.sample_indices(w["M"], w["N"], 1 << 21, seed=0xBEEF)
    prev = oracle.set_parallel(parallel)
    try:
        threads = oracle.threads()
        pos, done, t0, batch = 0, 0, time.perf_counter(), 64
        cap = 4096 * max(1, threads)
        while True:
            done += oracle_elements(w, rows[pos:pos + batch], cols[pos:pos + batch])
            pos += batch
            el = time.perf_counter() - t0
            if el >= seconds or pos + batch > rows.size:
                break
            batch = min(batch * 2, cap)
    finally:
        oracle.set_parallel(prev)
    return done, el, threads


def cpu_baseline(w: dict, seconds: float = 10.0) -> dict:
    """The oracle as it stands (fp64 C) on seeded output elements of the same
    workload, for about `seconds` each: the OpenMP build on all host cores
    (the record's value) and the single-threaded build beside it."""
    per, unit = metric_per_element(w)
    shape = (f"{w['M']}x{w['D']}x{w['F']}" if w["op"] == "mlp"
             else f"{w['M']}x{w['N']}x{w['K']}")
    n1, t1, _ = _oracle_sample(w, seconds, parallel=False)
    nn, tn, threads = _oracle_sample(w, seconds, parallel=True)
    return {"value": nn * per / tn, "unit": unit, "cores": threads, "kind": "oracle",
            "cpu": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"{nn} output elements of the {shape} workload at seeded positions "
                      f"({tn:.1f} s, OpenMP build of the fp64 C oracle, {threads} threads)",
            "single_thread": {"value": n1 * per / t1, "unit": unit, "cores": 1,
                              "kind": "oracle",
                              "sample": f"{n1} output elements, same positions ({t1:.1f} s, "
                                        f"single-threaded build)"}}


def run_reference(args, workload_name):
    """--impl reference: the fp64 CPU oracle on the same workload; each step
    computes a bounded sample of output elements."""
    import numpy as np
    import workloads
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if workload_name == "all":
        workload_name = HEADLINE
    w = (workloads.make("sweep", M=int(workload_name.split("-")[1]))
         if workload_name.startswith("sweep-") else workloads.make(workload_name))
    rows, cols = workloads.sample_indices(w["M"], w["N"], 1 << 20, seed=0xFACE)
    oracle.set_parallel(True)  # the OpenMP build: every host core
    threads = oracle.threads()
    oracle_elements(w, rows[:threads], cols[:threads])  # thread pool start-up
    t0 = time.perf_counter()
    n0 = oracle_elements(w, rows[:32 * threads], cols[:32 * threads])
    per_elem = max((time.perf_counter() - t0) / n0, 1e-9)
    budget = 90.0 / max(1, args.steps + args.warmup)
    per_step = int(max(1, min(rows.size // 2, budget / per_elem)))
    if w["op"] in ("add_rmsnorm", "swiglu_pointwise", "mlp"):
        per_step = max(1, per_step // w["N"])  # rows per step
    pos, done = 0, 0

    def step():
        nonlocal pos, done
        if pos + per_step > rows.size:
            pos = 0
        done += oracle_elements(w, rows[pos:pos + per_step], cols[pos:pos + per_step])
        pos += per_step

    for _ in range(args.warmup):
        step()
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    per, unit = metric_per_element(w)
    value = done * per / el
    shape = (f"{w['M']}x{w['D']}x{w['F']}" if w["op"] == "mlp"
             else f"{w['M']}x{w['N']}x{w['K']}")
    sample = (f"{done // args.steps} output elements per step at seeded positions of the "
              f"{shape} workload, fp64 C oracle (OpenMP build, {threads} threads)")
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": config_of(workload_name, w, max(1, args.gpus)),
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                             "cpu": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- MLP block legs

def mlp_latency(wl, stream, reps: int = 200) -> dict:
    """Median host wall time (us) of one synchronous MLP block step -- issue,
    then wait for it -- for each way of issuing it: fused chain replayed from
    a CUDA graph, fused chain launched directly (two C-ABI launches), the
    unfused composition (graph and direct), and PyTorch eager (cuBLAS GEMMs
    plus elementwise kernels) as the outside point of comparison."""
    import torch
    import torch.nn.functional as Fn

    def eager(i):
        s = wl.sets[i % wl.n_sets]
        g = Fn.linear(s["x"], s["w_gate"])
        u = Fn.linear(s["x"], s["w_up"])
        torch.add(Fn.linear(Fn.silu(g) * u, s["w_down"]), s["residual"], out=s["out"])

    legs = {
        "fused_graph": lambda i: wl.graphs[i % wl.n_sets].replay(),
        "fused_direct": lambda i: wl.mlp_direct(i, stream),
        "unfused_graph": lambda i: wl.graphs_unfused[i % wl.n_sets].replay(),
        "unfused_direct": lambda i: wl.mlp_direct(i, stream, fused=False),
        "torch_eager": eager,
    }
    out = {}
    for name, fn in legs.items():
        for i in range(5):
            fn(i)
        torch.cuda.synchronize()
        t = []
        for i in range(reps):
            t0 = time.perf_counter()
            fn(i)
            stream.synchronize()
            t.append(time.perf_counter() - t0)
        out[name] = statistics.median(t) * 1e6
    out["note"] = ("median host wall time of one step issued and synchronised alone, weights "
                   "cold in L2 (two rotating weight sets of 352 MB)")
    return out


def mlp_gate_up_kernel_time(wl, stream, steps: int):
    """Average launch duration of the block's gate/up GEMM alone (CUDA events
    around a back-to-back loop on the launching stream), and its counts."""
    from tcgen05_tmem_bf16_gb300 import roofline as rf
    w, gbf = wl.w, wl.gbf
    M, D, F = w["M"], w["D"], w["F"]

    def gate_up(i):
        s = wl.sets[i % wl.n_sets]
        gbf.swiglu_dual_gemm(s["x"], s["w_gate"], s["w_up"], "nk", wl.ws, M, F, D, 1.0, 0.0,
                             None, "silu", stream=stream)

    for i in range(5):
        gate_up(i)
    region, _ = time_loop(gate_up, steps, stream, per_launch=False)
    return region / steps, rf.swiglu_counts(M, F, D)


# ---------------------------------------------------------------- main



def measure(name: str, args, dev, stream, peaks, peak_src, world: int, headline: bool) -> dict:
    """Time one workload: the fused call (value and roofline of its dominant
    kernel), the unfused composition (speedup), and the end-to-end call with
    host buffers.  Returns the workload's record; frees its device memory."""
    import torch

    import tcgen05_tmem_bf16_gb300 as gbf
    from tcgen05_tmem_bf16_gb300 import roofline as rf

    wl = Workload(name, dev)
    # warm-up (also checks the launch works)
    for i in range(args.warmup):
        wl.fused(i)
    torch.cuda.synchronize()
    if wl.op == "mlp":
        wl.capture()  # the block is replayed from CUDA graphs from here on
        for i in range(args.warmup):
            wl.fused(i)
        torch.cuda.synchronize()
    steps = args.steps
    if steps is None or not headline:
        t_cal, _ = time_loop(wl.fused, 20, stream, per_launch=False)
        if steps is None:
            steps = int(min(50000, max(200, 1.5 / max(t_cal / 20, 1e-6))))
        else:
            # the other workloads' records: at least ~30 ms of timed work, so
            # that the average per launch of a short kernel is well formed
            steps = int(min(5000, max(steps, 0.03 / max(t_cal / 20, 1e-6))))
        if world > 1:
            import torch.distributed as dist
            k = torch.tensor([steps], dtype=torch.int64, device=dev)
            dist.all_reduce(k, op=dist.ReduceOp.MIN)
            steps = int(k.item())
    if gbf.gbf_check_device_error() != 0:
        raise SystemExit(f"{name}: kernel reported a timeout during warm-up")

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    # One event pair around the region; a step is exactly one kernel launch
    # (two for the MLP block), so the kernel's average launch duration is
    # region / steps (conservative: gaps between launches count against it).
    region, _ = time_loop(wl.fused, steps, stream, per_launch=False)
    per_launch = region / steps
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    bnd = rf.bound(wl.counts, peaks["bf16_tflops"], peaks["hbm_gbs"])
    # the workload's metric: TFLOP/s when tensor-bound, GB/s of algorithmic
    # bytes when HBM-bound
    per_step, vscale, vunit = ((wl.counts.flops, 1e12, "TFLOP/s") if bnd == "tensor"
                               else (wl.counts.fused_bytes, 1e9, "GB/s"))
    max_region, total_units = aggregate(region, per_step * steps, world)
    if gbf.gbf_check_device_error() != 0:
        raise SystemExit(f"{name}: kernel reported a timeout in the timed region")
    value = total_units / max_region / vscale

    # unfused composition, same workload, same rotation of input sets.  The
    # speedup is taken from alternating blocks of fused and unfused steps of
    # equal length (about 0.1 s each), so that both see the same clock and
    # power-cap state; the median block ratio is reported.
    for i in range(3):
        wl.unfused(i)
    torch.cuda.synchronize()
    block = max(3, min(args.unfused_steps, int(0.1 / max(per_launch, 1e-6))))
    ratios, un_times, fu_times = [], [], []
    for _ in range(args.speedup_rounds):
        f_reg, _ = time_loop(wl.fused, block, stream, per_launch=False)
        u_reg, _ = time_loop(wl.unfused, block, stream, per_launch=False)
        ratios.append(u_reg / f_reg)
        un_times.append(u_reg / block * 1e3)
        fu_times.append(f_reg / block * 1e3)

    # end to end through the public API with host buffers
    wl.e2e_run(2, stream)
    torch.cuda.synchronize()
    e2e_region = wl.e2e_run(args.e2e_steps, stream)
    e2e_max, e2e_units = aggregate(e2e_region, per_step * args.e2e_steps, world)

    # MLP block: per-step latency of each way of issuing it, and the
    # dominant kernel (the gate/up GEMM) timed on its own
    extra = {}
    per_launch_dom = per_launch
    dom_counts = wl.counts
    if wl.op == "mlp":
        extra["latency_us"] = mlp_latency(wl, stream)
        per_launch_dom, dom_counts = mlp_gate_up_kernel_time(wl, stream, steps)

    # roofline of the dominant kernel of the step, against both peaks
    long_loop = region > 0.5
    tpeak = peaks["bf16_tflops_sustained"] if long_loop else peaks["bf16_tflops"]
    ach_tf = dom_counts.flops / per_launch_dom / 1e12
    ach_gb = dom_counts.fused_bytes / per_launch_dom / 1e9
    if bnd == "tensor":
        achieved, peak, unit = ach_tf, tpeak, "TFLOP/s"
    else:
        achieved, peak, unit = ach_gb, peaks["hbm_gbs"], "GB/s"
    kname = {"persistent": "gemm_persistent_kernel", "persistent_splitk": "gemm_persistent_kernel",
             "swap_splitk": "gemm_swap_kernel",
             "w4a16": "wq_gemm_kernel", "pair": "gemm_pair_kernel",
             "pair_1stream": "gemm_pair_kernel", "pair_splitk": "gemm_pair_kernel",
             "add_rmsnorm": "add_rmsnorm_kernel",
             "swiglu_pointwise": "swiglu_pointwise_kernel"}.get(wl.path, wl.path)
    tpeak_name = ("bf16_tflops_sustained (back-to-back loop)" if long_loop
                  else "bf16_tflops (burst)")
    roof = {"bound": bnd, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": recorded_traffic(name, kname),
            "peak_source": f"{peak_src}: " + (tpeak_name if bnd == "tensor" else "hbm_gbs"),
            "kernel": kname,
            "splits": wl.splits,
            "kernel_ms": per_launch_dom * 1e3,
            "algorithmic_flops": dom_counts.flops, "algorithmic_bytes": dom_counts.fused_bytes,
            # both sides of the roofline (the slower of the two is the bound)
            "achieved_tflops": ach_tf, "achieved_gbs": ach_gb,
            "frac_tensor": ach_tf / tpeak, "frac_hbm": ach_gb / peaks["hbm_gbs"],
            "tensor_peak": tpeak, "tensor_peak_source": f"{peak_src}: {tpeak_name}",
            "hbm_peak": peaks["hbm_gbs"],
            "roofline_ms": rf.roofline_seconds(dom_counts, peaks["bf16_tflops"],
                                               peaks["hbm_gbs"]) * 1e3}
    roof["frac_of_roofline"] = roof["roofline_ms"] / roof["kernel_ms"]
    if bnd == "tensor":
        roof["frac_of_burst_peak"] = ach_tf / peaks["bf16_tflops"]
    if wl.op == "mlp":
        chain_gbs = wl.counts.fused_bytes / per_launch / 1e9
        roof["kernel"] = f"{roof['kernel']} (gate/up GEMM, the larger of the block's two)"
        roof["chain"] = {"achieved": chain_gbs, "unit": "GB/s",
                         "frac": chain_gbs / peaks["hbm_gbs"],
                         "ms": per_launch * 1e3, "algorithmic_bytes": wl.counts.fused_bytes}
    rec = {
        "value": value, "unit": vunit, "steps": steps, "ms_per_step": max_region / steps * 1e3,
        "config": config_of(name, wl.w, world),
        "l2": f"{wl.n_sets} rotating input sets of {wl.set_bytes / 2**20:.0f} MiB (> 2x L2)",
        "roofline": roof,
        "unfused_ms_per_step": statistics.median(un_times),
        "unfused_kind": wl.unfused_kind(),
        "speedup_vs_unfused": statistics.median(ratios),
        "speedup_method": (f"median over {args.speedup_rounds} alternating blocks of {block} "
                           f"fused and {block} unfused steps (fused block "
                           f"{statistics.median(fu_times):.4f} ms/step)"),
        "e2e": {"value": e2e_units / e2e_max / vscale, "unit": vunit,
                "h2d_bytes_per_step": wl.h2d_bytes, "d2h_bytes_per_step": wl.d2h_bytes,
                "method": (f"{args.e2e_steps} steps: inputs copied from pinned host memory "
                           "into one of two device sets, the call, the result copied back; "
                           "copies on their own streams overlap the neighbouring steps")},
        "gpu_launches": steps * wl.launches_per_step(),
        "clocks": clocks,
        **extra,
    }
    w = wl.w
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec, w


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps per workload (default: enough for about 1.5 s of work)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    help="all (default: every workload, headline sweep-8192) | prefill | "
                         "swiglu | w4a16 | tiny | sweep-<M> | w8a16_fp8 | w4a16_nvfp4 | "
                         "add_rmsnorm | swiglu_pointwise | mlp_decode")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--unfused-steps", type=int, default=200,
                    help="upper bound on the steps of one block of the fused/unfused comparison")
    ap.add_argument("--speedup-rounds", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        return run_reference(args, args.workload)

    import torch
    world, rank, local = dist_env()
    if args.gpus > 1 and world == 1:
        print("bench.py --gpus N>1 must be launched by torchrun (one rank per GPU)",
              file=sys.stderr)
        return 2
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from __graft_entry__ import build
    build()
    import tcgen05_tmem_bf16_gb300 as gbf
    gbf.load()

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    head_name = HEADLINE if args.workload == "all" else args.workload
    head, head_w = measure(head_name, args, dev, stream, peaks, peak_src, world, headline=True)
    configs = {}
    if args.workload == "all":
        for name in SUB_WORKLOADS:
            rec, _ = measure(name, args, dev, stream, peaks, peak_src, world, headline=False)
            configs[name] = rec

    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
        "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": head["config"],
        "l2": head["l2"],
        "impl": "gbfuse",
        "roofline": head["roofline"],
        "unfused_ms_per_step": head["unfused_ms_per_step"],
        "unfused_kind": head["unfused_kind"],
        "speedup_vs_unfused": head["speedup_vs_unfused"],
        "speedup_method": head["speedup_method"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        **{k: v for k, v in head.items() if k == "latency_us"},
    }
    if configs:
        line["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(head_w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

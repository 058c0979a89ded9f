#!/usr/bin/env python3
"""Benchmark of the small-M NVFP4 W4A4 decode linear on GB300.

Workload (one "step"): one decode step of an 8B-shaped model at M = 1 -- the
four decode linears (qkv 4096->6144, o 4096->4096, gate_up 4096->24576,
down 12288->4096) of each of 36 layers with distinct seeded weights, each
call an on-the-fly activation quantisation followed by the small-M GEMM, all
replayed as one CUDA graph.  The packed weights (3.9 GB) are far larger than
L2, so every step streams them from HBM.

Printed: one JSON line (rank 0).  ``value`` is the achieved HBM throughput of
the whole step over its algorithmic bytes (GB/s, higher is better);
``detail.per_linear`` has the microseconds per call of each linear shape.

``--impl reference`` times the CPU oracle instead (the only reference that
exists for this method here), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import queue
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "NVFP4 W4A4 small-M linear µs/call and HBM GB/s (% of roofline), M=1..8"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # the nominal GB300 HBM3e figure the workload's target is quoted against
WORKLOAD = ("8B-shaped decode linears qkv/o/gate_up/down (K->N 4096->6144, 4096->4096, "
            "4096->24576, 12288->4096), M=1, act-quantize + GEMM per call, 36 layers of "
            "distinct weights per step under one CUDA graph")


def algorithmic_bytes(m: int, n: int, k: int, x_bytes: int = 4, y_bytes: int = 4) -> dict:
    """Bytes a call must move at minimum: packed weights and scales once,
    packed activations, both tensor scales, the output (FP32 or BF16); and the
    activation quantiser's read of X (FP32 or BF16) plus packed write."""
    wbytes = n * k // 2 + n * k // 16
    gemm = wbytes + m * k // 2 + m * k // 16 + 8 + y_bytes * m * n
    quant = x_bytes * m * k + m * k // 2 + m * k // 16 + 4
    return {"weights": wbytes, "gemm": gemm, "quant": quant}


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
            if hbm:
                return {"hbm_gbs": float(hbm), "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw",
                "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [s.strip() for s in line.split(",")]
                if len(p) < len(CLOCK_FIELDS):
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, val in zip(names, p[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs its own copy of the step)
# ---------------------------------------------------------------------------

def dist_setup(gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float, world: int, device: str = "cuda") -> float:
    """Max of v over the ranks (the slowest rank's time sets the job's)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, ms_step_max: float, world: int) -> float:
    """Whole-job GB/s: every rank moves its own bytes per step (replicas, weak
    scaling); the step time is the maximum over ranks."""
    return world * bytes_per_rank_step / (ms_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class DecodeStack:
    """36 layers x 4 linears of packed weights resident in HBM, per-call
    activation buffers, and the graphs that replay them.

    Two ways to run a step:
    * ``launches``: every linear is its own nvfp4_linear call (quantiser +
      GEMM, programmatic dependent launch between them), one (x_q, x_s) pair
      per linear shape shared by all layers and one workspace shared by all
      calls -- the form a model whose linears depend on each other needs;
    * ``chain``: the step's 144 independent linears as one nvfp4_linear_chain
      call (one quantiser launch for all of them, one persistent GEMM launch),
      each linear with its own (x_q, x_s) -- the synthetic step's inputs are
      all known when it starts.  Any M up to 32 on the tensor cores (M <= 2 on
      the CUDA-core stream)."""

    def __init__(self, nv, torch, m: int, layers: int, seed: int = 1234, pdl: bool = True,
                 fused: bool = True, kernel: int = 0, bf16: bool = False, mode: str = "launches",
                 chain_kernel: int = 0, chain_workspace: bool = True, tiled: bool = False):
        self.nv, self.torch = nv, torch
        self.m = m
        self.bf16 = bf16   # BF16 activations in and BF16 outputs out
        io = torch.bfloat16 if bf16 else torch.float32
        self.pdl = pdl
        self.fused = fused
        self.kernel = kernel
        self.layers = layers
        self.seed = seed
        self.chain_kernel = chain_kernel   # the chain's engine (0: the library's choice)
        self.lins = synthetic.LINEARS_8B
        if mode not in ("launches", "chain"):
            raise ValueError(f"unknown mode {mode}")
        self.has_chain = all(nv.chain_supported(m, lin.n, lin.k) for lin in self.lins)
        if mode == "chain" and not self.has_chain:
            raise ValueError(f"the chain does not take M = {m}")
        self.mode = mode
        # one workspace for every call of the step (calls run one after another)
        wsz = max(nv.gemm_workspace_size(m, lin.n, lin.k, kernel) for lin in self.lins) \
            if m <= 8 else 0
        self.workspace = (torch.zeros(wsz, dtype=torch.uint8, device="cuda") if wsz else None)
        dev = torch.device("cuda")
        self.w = []          # [layer][j] -> (wq, ws, wg)
        for l in range(layers):
            row = []
            for j, lin in enumerate(self.lins):
                wf = self.weight_fp32(l, j)
                row.append(nv.pack_weight(wf))
                del wf
            self.w.append(row)
        torch.cuda.synchronize()
        # activations: X ~ N(0,1) with 0.5 % x20 outlier channels, per call;
        # all calls' X (and Y) are views of one flat buffer, so a step's inputs
        # and outputs move between host and device in one copy each
        xsz = sum(m * lin.k for lin in self.lins) * layers
        ysz = sum(m * lin.n for lin in self.lins) * layers
        self.x_flat = torch.empty(xsz, dtype=io, device=dev)
        self.y_flat = torch.empty(ysz, dtype=io, device=dev)
        self.x, self.xg, self.y = [], [], []
        xo = yo = 0
        for l in range(layers):
            xr, gr, yr = [], [], []
            for j, lin in enumerate(self.lins):
                xa = synthetic.activations(m, lin.k, seed=synthetic.weight_seed(seed + 7, l, j))
                xd = self.x_flat[xo:xo + m * lin.k].view(m, lin.k)
                xd.copy_(torch.from_numpy(xa))     # rounded to BF16 when the I/O is BF16
                xo += m * lin.k
                xr.append(xd)
                # static calibration, not timed (from the FP32 values of X)
                gr.append(nv.global_scale(xd.float().contiguous()))
                yr.append(self.y_flat[yo:yo + m * lin.n].view(m, lin.n))
                yo += m * lin.n
            self.x.append(xr)
            self.xg.append(gr)
            self.y.append(yr)
        # launches: one activation-code buffer pair per linear shape, shared by
        # the layers
        self.xq = [(torch.empty((m, lin.k // 2), dtype=torch.uint8, device=dev),
                    torch.empty((m, lin.k // 16), dtype=torch.uint8, device=dev)) for lin in self.lins]
        self.chain = None
        # the tensor-core chain streams tile-major weights (an offline repack
        # of the same bytes: contiguous 16 KB stages, and at M <= 2 the CUDA-core
        # stream warps take the last tiles of every linear); row-major on request
        self.tiled = bool(tiled) and self.has_chain and chain_kernel in (0, nv.KERNEL_TC)
        self.wt = None
        if self.tiled:
            self.wt = [[nv.tile_weight(*self.w[l][j]) for j in range(4)] for l in range(layers)]
            torch.cuda.synchronize()
        if self.has_chain:
            # chain: one pair per linear (every linear of the step is in flight)
            self.xq_item = [[(torch.empty((m, lin.k // 2), dtype=torch.uint8, device=dev),
                              torch.empty((m, lin.k // 16), dtype=torch.uint8, device=dev))
                             for lin in self.lins] for _ in range(layers)]
            self.chain = nv.Chain([self._chain_entry(l, j) for l in range(layers)
                                   for j in range(4)], kernel=chain_kernel,
                                  workspace=chain_workspace)
            self.chain_j = [nv.Chain([self._chain_entry(l, j) for l in range(layers)],
                                     kernel=chain_kernel, workspace=chain_workspace)
                            for j in range(4)]
        torch.cuda.synchronize()

    def _chain_entry(self, l: int, j: int, x=None, y=None):
        wts = self.wt[l][j] if self.tiled else self.w[l][j]
        return ((x or self.x)[l][j], self.xg[l][j], self.xq_item[l][j], wts, (y or self.y)[l][j])

    def second_buffers(self):
        """A second X / Y buffer set and the step over it as a chain on the same
        weights and activation-code buffers (consecutive steps' kernels stay
        ordered on the compute stream): (x_flat, y_flat, chain)."""
        torch = self.torch
        x2 = torch.empty_like(self.x_flat)
        y2 = torch.empty_like(self.y_flat)
        x2.copy_(self.x_flat)
        xs, ys = [], []
        xo = yo = 0
        for l in range(self.layers):
            xr, yr = [], []
            for lin in self.lins:
                xr.append(x2[xo:xo + self.m * lin.k].view(self.m, lin.k))
                yr.append(y2[yo:yo + self.m * lin.n].view(self.m, lin.n))
                xo += self.m * lin.k
                yo += self.m * lin.n
            xs.append(xr)
            ys.append(yr)
        ch = self.nv.Chain([self._chain_entry(l, j, xs, ys) for l in range(self.layers)
                            for j in range(4)], kernel=self.chain_kernel,
                           workspace=self.chain.workspace is not None)
        return x2, y2, ch

    def weight_fp32(self, l: int, j: int):
        """FP32 weights of linear j of layer l, drawn on the device: N(0, 0.02^2),
        torch's generator seeded per linear (the packed copy is made from
        exactly this tensor)."""
        torch = self.torch
        lin = self.lins[j]
        gen = torch.Generator(device="cuda")
        gen.manual_seed(synthetic.weight_seed(self.seed, l, j))
        wf = torch.randn((lin.n, lin.k), generator=gen, device="cuda", dtype=torch.float32)
        wf.mul_(synthetic.WEIGHT_STD_8B)
        return wf

    def codes(self, l: int, j: int):
        """The (x_q, x_s) buffers the step's linear j of layer l writes."""
        return self.xq_item[l][j] if self.mode == "chain" else self.xq[j]

    def chosen(self, lin) -> int:
        """Kernel id the step's calls of this linear run."""
        if self.mode == "chain":
            return self.chain.engine
        wsz = self.workspace.numel() if self.workspace is not None else 0
        return self.nv.gemm_select(self.m, lin.n, lin.k, self.kernel, wsz)

    def launches_per_step(self) -> int:
        if self.mode == "chain":
            return self.chain.launches()
        return sum(1 if (self.fused and self.chosen(lin) == self.nv.KERNEL_GEMV) else 2
                   for lin in self.lins) * self.layers

    def gemm_launches_per_step(self) -> int:
        if self.mode == "chain":
            return self.chain.launches(quantize=False)
        return 4 * self.layers

    def step(self):
        if self.mode == "chain":
            self.chain.run(pdl=self.pdl)
            return
        nv = self.nv
        for l in range(self.layers):
            for j in range(4):
                wq, ws, wg = self.w[l][j]
                nv.linear(self.x[l][j], self.xg[l][j], wq, ws, wg, out=self.y[l][j],
                          x_out=self.xq[j], kernel=self.kernel, pdl=self.pdl, fused=self.fused,
                          workspace=self.workspace)

    def linear_only(self, j: int):
        """The step's calls of linear j only (quantise + GEMM each)."""
        if self.mode == "chain":
            self.chain_j[j].run(pdl=self.pdl)
            return
        nv = self.nv
        for l in range(self.layers):
            wq, ws, wg = self.w[l][j]
            nv.linear(self.x[l][j], self.xg[l][j], wq, ws, wg, out=self.y[l][j],
                      x_out=self.xq[j], kernel=self.kernel, pdl=self.pdl, fused=self.fused,
                      workspace=self.workspace)

    def quantize_only(self, j: int):
        """The step's activation quantisations of linear j only."""
        for l in range(self.layers):
            self.nv.quantize_act(self.x[l][j], self.xg[l][j], out=self.codes(l, j), pdl=self.pdl)

    def quantize_all(self):
        """Fill the activation-code buffers (before GEMM-only timing)."""
        for l in range(self.layers):
            for j in range(4):
                self.nv.quantize_act(self.x[l][j], self.xg[l][j], out=self.codes(l, j))

    def gemm_only(self, j=None):
        if self.mode == "chain":
            (self.chain if j is None else self.chain_j[j]).gemm_only(pdl=self.pdl)
            return
        nv = self.nv
        for l in range(self.layers):
            for jj in (range(4) if j is None else (j,)):
                xq, xs = self.xq[jj]
                wq, ws, wg = self.w[l][jj]
                nv.gemm_smallm(xq, xs, self.xg[l][jj], wq, ws, wg, out=self.y[l][jj],
                               kernel=self.kernel, pdl=self.pdl, workspace=self.workspace)

    def capture(self, fn):
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()                       # warm (module load, first-launch costs)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    def bytes_per_step(self):
        tot = {"weights": 0, "gemm": 0, "quant": 0}
        io = 2 if self.bf16 else 4
        for lin in self.lins:
            b = algorithmic_bytes(self.m, lin.n, lin.k, io, io)
            for key in tot:
                tot[key] += self.layers * b[key]
        return tot


def time_graph(torch, g, reps: int, warm: int = 3) -> float:
    """Average ms per replay, CUDA events on the replay stream."""
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        g.replay()
    b.record(st)
    b.synchronize()
    return a.elapsed_time(b) / reps


def read_probe_gbs(nv, torch, nbytes: int = 2 << 30, calls: int = 4) -> float:
    """GB/s of the library's read-only streaming probe over a buffer of
    `nbytes` (16x the L2): a CUDA graph of `calls` probes, timed with CUDA
    events, best of three replays."""
    buf = torch.ones(nbytes // 8, dtype=torch.int64, device="cuda")
    sink = torch.empty(1, dtype=torch.int64, device="cuda")
    nv.read_probe(buf, sink=sink)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(calls):
            nv.read_probe(buf, sink=sink)
    best = min(time_graph(torch, g, reps=1) for _ in range(3))
    del g, buf
    torch.cuda.empty_cache()
    return nbytes * calls / (best * 1e-3) / 1e9


def make_weights(nv, torch, lin, std, copies, seed):
    gen = torch.Generator(device="cuda")
    out = []
    for c in range(copies):
        gen.manual_seed(seed + c)
        wf = torch.randn((lin.n, lin.k), generator=gen, device="cuda", dtype=torch.float32)
        wf.mul_(std)
        out.append(nv.pack_weight(wf))
        del wf
    return out


def time_linear(nv, torch, weights, lin, m, kernel, pdl, reps, seed=5, workspace=True):
    """µs per call of one linear shape at this M: a graph of len(weights) GEMMs
    over distinct weight copies (larger than L2 together), replayed; with the
    workspace the kernel asks for, or (``workspace=False``) none, as the plain
    boundary call offers."""
    xa = synthetic.activations(m, lin.k, seed=seed)
    xd = torch.from_numpy(xa).cuda()
    xg = nv.global_scale(xd)
    xq, xs = nv.quantize_act(xd, xg)
    y = torch.empty((m, lin.n), device="cuda")
    wsp = nv.workspace(m, lin.n, lin.k, kernel) if workspace else False

    def calls():
        for wq, ws, wg in weights:
            nv.gemm_smallm(xq, xs, xg, wq, ws, wg, out=y, kernel=kernel, pdl=pdl, workspace=wsp)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    ms = time_graph(torch, g, reps=reps)
    us = ms * 1e3 / len(weights)
    b = algorithmic_bytes(m, lin.n, lin.k)["gemm"]
    return {"us_per_call": round(us, 3), "GBps": round(b / (us * 1e-6) / 1e9, 1)}


def takes(nv, m, lin, kid) -> bool:
    """Whether kernel `kid` runs this shape when given the workspace it asks for."""
    wsz = nv.library().nvfp4_gemm_workspace_size(m, lin.n, lin.k, kid)
    return wsz >= 0 and nv.gemm_select(m, lin.n, lin.k, kid, wsz) == kid


def auto_choice(nv, m, lin) -> int:
    """The library's kernel for this shape, offered the workspace it asks for."""
    return nv.gemm_select(m, lin.n, lin.k, nv.KERNEL_AUTO,
                          nv.gemm_workspace_size(m, lin.n, lin.k))


def tiny_latency(nv, torch, kernels: dict, pdl: bool, calls: int = 50) -> dict:
    """The single 256 x 512 GEMV at M = 1 (75 KB: latency, not bandwidth):
    µs per call of a CUDA graph of `calls` back-to-back calls on the same
    seeded operands (L2-resident), for the library's choice and every kernel
    that takes the shape, GEMM alone and quantise + GEMM (nvfp4_linear)."""
    lin = synthetic.TINY
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    w = torch.randn((lin.n, lin.k), generator=gen, device="cuda") * synthetic.WEIGHT_STD_8B
    wq, ws, wg = nv.pack_weight(w)
    x = torch.from_numpy(synthetic.activations(1, lin.k, seed=0, outliers=False)).cuda()
    xg = nv.global_scale(x)
    xq, xs = nv.quantize_act(x, xg)
    y = torch.empty((1, lin.n), device="cuda")

    def timed(fn):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                fn()
        return round(min(time_graph(torch, g, reps=5) for _ in range(3)) * 1e3 / calls, 3)

    res = {"n": lin.n, "k": lin.k, "m": 1,
           "kernel": nv.KERNEL_NAMES.get(auto_choice(nv, 1, lin))}
    for name, kid in kernels.items():
        if not takes(nv, 1, lin, kid):
            continue
        wsp = nv.workspace(1, lin.n, lin.k, kid)
        res[name] = {
            "gemm_us_per_call": timed(lambda: nv.gemm_smallm(xq, xs, xg, wq, ws, wg, out=y,
                                                             kernel=kid, pdl=pdl, workspace=wsp)),
            "quantize_plus_gemm_us_per_call": timed(
                lambda: nv.linear(x, xg, wq, ws, wg, out=y, x_out=(xq, xs), kernel=kid, pdl=pdl,
                                  workspace=wsp))}
    return res


def time_chain_linear(nv, torch, weights, lin, m, kernel, pdl, reps, seed=5):
    """µs per linear of one shape when len(weights) distinct copies of it run
    as one multi-linear GEMM call (nvfp4_gemm_chain on pre-quantised codes):
    the rate of the shape inside a long chain, graph-replayed."""
    xa = synthetic.activations(m, lin.k, seed=seed)
    xd = torch.from_numpy(xa).cuda()
    xg = nv.global_scale(xd)
    entries = []
    for wts in weights:                 # (w_q, w_s, w_g) triples or TiledWeight
        codes = nv.quantize_act(xd, xg)
        entries.append((xd, xg, codes, wts, torch.empty((m, lin.n), device="cuda")))
    ch = nv.Chain(entries, kernel=kernel)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ch.gemm_only(pdl=pdl)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ch.gemm_only(pdl=pdl)
    ms = time_graph(torch, g, reps=reps)
    us = ms * 1e3 / len(weights)
    b = algorithmic_bytes(m, lin.n, lin.k)["gemm"]
    return {"us_per_call": round(us, 3), "GBps": round(b / (us * 1e-6) / 1e9, 1)}


def sweep(nv, torch, stack, peaks, args) -> dict:
    """µs/call and GB/s of every linear shape for every M of the sweep: each
    kernel that takes the shape as a lone call (graph of calls over rotating
    weight copies, L2-cold), the library's choice marked, and the shape
    inside a multi-linear call on the tensor cores (``tc_chain``); at
    M = 2..8 also the plain boundary call without a workspace (``plain``).
    Beyond M = 8 (tensor-core kernel only) the 8B shapes at M = 12..32."""
    kernels = {"gemv": nv.KERNEL_GEMV, "mma": nv.KERNEL_MMA, "tma": nv.KERNEL_TMA,
               "splitk": nv.KERNEL_SPLITK, "tc": nv.KERNEL_TC, "generic": nv.KERNEL_GENERIC}
    out = {"8B": {}, "32B": {}, "C1": tiny_latency(nv, torch, kernels, stack.pdl)}
    reps = 5

    def entry(m, lin, ws, wt=None):
        auto = auto_choice(nv, m, lin) if m <= 8 else nv.KERNEL_TC
        ent = {"kernel": nv.KERNEL_NAMES.get(auto)}
        for name, kid in kernels.items():
            if name == "generic" and not args.sweep_generic:
                continue
            if m > 8 and kid != nv.KERNEL_TC:
                continue
            if not takes(nv, m, lin, kid):
                continue
            ent[name] = time_linear(nv, torch, ws, lin, m, kid, stack.pdl, reps)
        ent["frac_of_peak"] = round(ent[ent["kernel"]]["GBps"] / peaks["hbm_gbs"], 4)
        if 2 <= m <= 8:
            # the plain boundary call: the library's choice with no workspace
            # (the split-K kernel's cluster form where K takes several chunks)
            plain = nv.gemm_select(m, lin.n, lin.k)
            ent["plain"] = time_linear(nv, torch, ws, lin, m, nv.KERNEL_AUTO, stack.pdl, reps,
                                       workspace=False)
            ent["plain"]["kernel"] = nv.KERNEL_NAMES.get(plain)
        # inside a chain: the tile-major weights the decode step uses
        ent["tc_chain"] = time_chain_linear(nv, torch, wt if wt is not None else ws, lin, m,
                                            nv.KERNEL_TC, stack.pdl, reps)
        ent["tc_chain"]["frac_of_peak"] = round(ent["tc_chain"]["GBps"] / peaks["hbm_gbs"], 4)
        return ent

    w8 = {j: [stack.w[l][j] for l in range(stack.layers)] for j in range(4)}
    w8t = {j: ([stack.wt[l][j] for l in range(stack.layers)] if stack.tiled else None)
           for j in range(4)}
    for m in tuple(synthetic.M_SWEEP_8B) + tuple(synthetic.M_SWEEP_WIDE):
        out["8B"][f"M={m}"] = {lin.name: entry(m, lin, w8[j], w8t[j])
                               for j, lin in enumerate(synthetic.LINEARS_8B)}
    for j, lin in enumerate(synthetic.LINEARS_32B):
        per_copy = lin.n * lin.k * 9 // 16
        copies = max(3, -(-400_000_000 // per_copy))
        ws = make_weights(nv, torch, lin, synthetic.WEIGHT_STD_32B, copies, seed=4000 + 100 * j)
        wt = [nv.tile_weight(*w) for w in ws] if stack.tiled else None
        for m in synthetic.M_SWEEP_32B:
            out["32B"].setdefault(f"M={m}", {})[lin.name] = entry(m, lin, ws, wt)
        del ws, wt
        torch.cuda.empty_cache()
    return out


def run_ours(args) -> dict:
    import torch

    import nvfp4_w4a4_decode_gb300 as nv
    from nvfp4_w4a4_decode_gb300 import build as nvbuild

    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    nvbuild.build()
    nv.library()
    peaks = load_peaks()

    mode = args.mode
    if mode == "auto":
        chain_ok = not args.fused and args.kernel == "auto" and all(
            nv.chain_supported(args.m, lin.n, lin.k) for lin in synthetic.LINEARS_8B)
        mode = "chain" if chain_ok else "launches"
    stack = DecodeStack(nv, torch, m=args.m, layers=args.layers, pdl=not args.no_pdl,
                        fused=args.fused, kernel=KERNELS[args.kernel](nv), bf16=args.bf16,
                        mode=mode, chain_kernel=KERNELS[args.chain_kernel](nv),
                        chain_workspace=not args.no_chain_workspace,
                        tiled=not args.row_major_weights)
    step_graph = stack.capture(stack.step)
    if args.profile_step:
        # only the step graph, replayed: a clean launch list for the profiler
        for _ in range(args.warmup + args.steps):
            step_graph.replay()
        torch.cuda.synchronize()
        return None
    launches_per_step = stack.launches_per_step()
    bytes_step = stack.bytes_per_step()
    alg_step = bytes_step["gemm"] + bytes_step["quant"]

    # ---- the timed steps: W warm-up replays, then K timed, barrier+sync around
    for _ in range(args.warmup):
        step_graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        ev0.record(st)
        for _ in range(args.steps):
            step_graph.replay()
        ev1.record(st)
        ev1.synchronize()
        wall = time.perf_counter() - t0
    torch.cuda.synchronize()
    barrier(world)
    ms_step = ev0.elapsed_time(ev1) / args.steps
    ms_step_max = reduce_max(ms_step, world)
    value = job_throughput(alg_step, ms_step_max, world)

    # ---- dominant kernel: the GEMM alone, same calls, same graph discipline
    stack.quantize_all()
    gemm_graph = stack.capture(stack.gemm_only)
    ms_gemm = time_graph(torch, gemm_graph, reps=max(3, args.steps // 2))
    del gemm_graph
    gemm_launches = stack.gemm_launches_per_step()
    gemm_avg_us = ms_gemm * 1e3 / gemm_launches
    gemm_bytes_per_launch = bytes_step["gemm"] / gemm_launches
    achieved = gemm_bytes_per_launch / (gemm_avg_us * 1e-6) / 1e9

    per_linear = {}
    io = 2 if stack.bf16 else 4
    for j, lin in enumerate(stack.lins):
        g = stack.capture(lambda j=j: stack.gemm_only(j))
        ms = time_graph(torch, g, reps=max(3, args.steps // 2))
        us = ms * 1e3 / stack.layers
        b = algorithmic_bytes(args.m, lin.n, lin.k, io, io)["gemm"]
        gbs = b / (us * 1e-6) / 1e9
        gq = stack.capture(lambda j=j: stack.quantize_only(j))
        us_q = time_graph(torch, gq, reps=max(3, args.steps // 2)) * 1e3 / stack.layers
        gp = stack.capture(lambda j=j: stack.linear_only(j))
        us_p = time_graph(torch, gp, reps=max(3, args.steps // 2)) * 1e3 / stack.layers
        per_linear[lin.name] = {"n": lin.n, "k": lin.k, "us_per_call": round(us, 3),
                                "kernel": nv.KERNEL_NAMES.get(stack.chosen(lin)),
                                "GBps": round(gbs, 1),
                                "frac_of_peak": round(gbs / peaks["hbm_gbs"], 4),
                                "quantize_us_per_call": round(us_q, 3),
                                "quantize_plus_gemm_us_per_call": round(us_p, 3)}
        del g, gq, gp
    # the other way of running the same step, on the same weights
    other = None
    # (one call per linear takes M up to 8)
    alt = ("launches" if args.m <= 8 else None) if mode == "chain" else \
        ("chain" if stack.has_chain else None)
    if alt is not None:
        stack.mode = alt
        g_alt = stack.capture(stack.step)
        ms_alt = time_graph(torch, g_alt, reps=max(3, args.steps // 2))
        stack.quantize_all()
        g_alt_gemm = stack.capture(stack.gemm_only)
        ms_alt_gemm = time_graph(torch, g_alt_gemm, reps=max(3, args.steps // 2))
        other = {"mode": alt, "ms_per_step": round(ms_alt, 4),
                 "GBps": round(alg_step / (ms_alt * 1e-3) / 1e9, 1),
                 "gemm_only_ms_per_step": round(ms_alt_gemm, 4),
                 "launches_per_step": stack.launches_per_step()}
        del g_alt, g_alt_gemm
        stack.mode = mode
    probe_gbs = read_probe_gbs(nv, torch)

    # ---- end to end: pinned host X in, host Y out, through the public API
    e2e = run_e2e(torch, stack, step_graph, args, world)
    sweep_detail = None if args.no_sweep else sweep(nv, torch, stack, peaks, args)

    # the committed traffic capture is of the default step's GEMM kernel
    default_step = args.m == 1 and not args.bf16 and not args.fused and args.kernel == "auto"
    traffic_name = ("gemm_chain" if stack.chosen(stack.lins[0]) == nv.KERNEL_GEMV else
                    ("gemm_tc_tiled" if stack.tiled else "gemm_tc")) if mode == "chain" else \
        "gemm_smallm"
    traffic = profile_traffic(traffic_name) if default_step else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic (seeded Gaussian weights std 0.02, Gaussian activations with "
                "0.5% x20 outlier channels)",
        "config": {"workload": WORKLOAD, "m": args.m, "layers": stack.layers,
                   "weight_bytes_per_step": bytes_step["weights"],
                   "algorithmic_bytes_per_step": alg_step,
                   "l2": "inputs larger than L2: 3.9 GB of packed weights per step",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "graph": "one CUDA graph per step",
                   "mode": mode,
                   "weights": "tile-major" if stack.tiled else "row-major",
                   "pdl": not args.no_pdl,
                   "fused_quantize": args.fused,
                   "io": "bf16 X in, bf16 Y out" if args.bf16 else "fp32 X in, fp32 Y out"},
        "roofline": {"bound": "hbm",
                     "kernel": (f"nvfp4_gemm_chain ({nv.KERNEL_NAMES[stack.chain.engine]})"
                                if mode == "chain" else "nvfp4_gemm_smallm"),
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "peak_source": peaks["source"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic,
                     "bytes_per_launch": round(gemm_bytes_per_launch),
                     "avg_launch_us": round(gemm_avg_us, 3),
                     "launches_per_step": gemm_launches,
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "read_probe_gbs": round(probe_gbs, 1),
                     "frac_of_read_probe": round(achieved / probe_gbs, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "wall_s_timed": round(wall, 4),
        "detail": {"per_linear_m1" if args.m == 1 else f"per_linear_m{args.m}": per_linear,
                   "step_frac_of_peak": round(value / world / peaks["hbm_gbs"], 4),
                   "step_frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
                   "other_mode": other,
                   "sweep": sweep_detail},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # rank 0 at N = 1 only
        # the oracle on the host: the timed baseline, then a check of sampled
        # outputs of the timed step against it (outside every timed region)
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
        line["parity"] = step_parity(stack)
        if not line["parity"]["ok"]:
            print(json.dumps(line), flush=True)
            raise SystemExit("the decode step's outputs disagree with the oracle")
    return line if rank == 0 else None


def run_e2e(torch, stack, step_graph, args, world: int = 1) -> dict:
    """End to end through the public API: every step copies all of its
    activations from pinned host memory to the device, replays the step (the
    same graph of C-ABI calls) and reads all of its outputs back to pinned host
    memory -- both copies inside the timed region.  With several ranks: a
    barrier on both sides, the slowest rank's time, all ranks' bytes.

    In chain mode the steps alternate between two device buffer sets (two
    graphs of the same chain call over the same weights), so that a step's
    input copy (its own stream) runs while the previous step computes and its
    output copy (another stream) while the next one does; every step still
    copies all of its inputs in and all of its outputs out."""
    if stack.mode == "chain":
        return run_e2e_overlapped(torch, stack, step_graph, args, world)
    x_host = stack.x_flat.cpu().pin_memory()
    y_host = torch.empty(stack.y_flat.shape, dtype=stack.y_flat.dtype).pin_memory()
    h2d = x_host.numel() * x_host.element_size()
    d2h = y_host.numel() * y_host.element_size()

    def one_step():
        stack.x_flat.copy_(x_host, non_blocking=True)
        step_graph.replay()
        y_host.copy_(stack.y_flat, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    reps = max(10, args.steps // 3)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(reps):
        one_step()
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / reps
    barrier(world)
    sec = reduce_max(sec, world)
    b = stack.bytes_per_step()
    v = world * (b["gemm"] + b["quant"]) / sec / 1e9
    return {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(sec * 1e3, 3),
            "path": "per step: pinned H2D of all activations, the step's CUDA graph of "
                    "nvfp4_linear calls, D2H of all outputs; wall clock"}


def run_e2e_overlapped(torch, stack, step_graph, args, world: int = 1) -> dict:
    x2, y2, chain2 = stack.second_buffers()
    graph2 = stack.capture(lambda: chain2.run(pdl=stack.pdl))
    xs, ys, graphs = (stack.x_flat, x2), (stack.y_flat, y2), (step_graph, graph2)
    x_host = [stack.x_flat.cpu().pin_memory(), x2.cpu().pin_memory()]
    y_host = [torch.empty(stack.y_flat.shape, dtype=stack.y_flat.dtype).pin_memory()
              for _ in range(2)]
    h2d = x_host[0].numel() * x_host[0].element_size()
    d2h = y_host[0].numel() * y_host[0].element_size()
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {key: [torch.cuda.Event(), torch.cuda.Event()] for key in ("in", "comp", "out")}
    used = [False, False]

    def one_step(i):
        b = i & 1
        with torch.cuda.stream(cin):
            if used[b]:
                cin.wait_event(ev["comp"][b])     # the step that last read this X is done
            xs[b].copy_(x_host[b], non_blocking=True)
            ev["in"][b].record(cin)
        comp.wait_event(ev["in"][b])
        if used[b]:
            comp.wait_event(ev["out"][b])         # this Y has been read back
        graphs[b].replay()
        ev["comp"][b].record(comp)
        with torch.cuda.stream(cout):
            cout.wait_event(ev["comp"][b])
            y_host[b].copy_(ys[b], non_blocking=True)
            ev["out"][b].record(cout)
        used[b] = True

    for i in range(max(4, args.warmup)):
        one_step(i)
    torch.cuda.synchronize()
    reps = max(10, args.steps // 3)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(reps):
        one_step(i)
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / reps
    barrier(world)
    sec = reduce_max(sec, world)
    b = stack.bytes_per_step()
    v = world * (b["gemm"] + b["quant"]) / sec / 1e9
    return {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(sec * 1e3, 3),
            "path": "per step: pinned H2D of all activations (own stream), the step's CUDA "
                    "graph of the nvfp4_linear_chain call, D2H of all outputs (own stream); "
                    "two device buffer sets alternate so that the copies overlap the "
                    "neighbouring steps' kernels; wall clock"}


def profile_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    only if the summary was taken from the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_hash") != kernel_source_hash(kernel):
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


# the sources each measured kernel (with the activation quantiser before it)
# and its launch path are built from
TRAFFIC_SOURCES = {
    "gemm_smallm": ("api.cu", "formats.cuh", "gemm_gemv.cu", "kernels.cuh", "launch_cache.cuh",
                    "quantize.cu", "stream_core.cuh"),
    "gemm_chain": ("api.cu", "formats.cuh", "gemm_chain.cu", "kernels.cuh", "launch_cache.cuh",
                   "stream_core.cuh"),
    "gemm_tc": ("api.cu", "formats.cuh", "gemm_tc.cu", "kernels.cuh", "launch_cache.cuh",
                "mma_frag.cuh"),
    "gemm_tc_tiled": ("api.cu", "formats.cuh", "gemm_tc.cu", "kernels.cuh", "launch_cache.cuh",
                      "mma_frag.cuh"),
}


def kernel_source_hash(kernel: str = "gemm_smallm") -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_w4a4_decode_gb300", "csrc")
    for name in TRAFFIC_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def step_parity(stack, layers=None, rows: int = 16, seed: int = 5) -> dict:
    """Sampled outputs of the decode step the GPU just ran, against the oracle
    (host side, after every timed region): for the first and last layer, all
    four linears -- the oracle's tensor scales and activation codes compared
    bit for bit with the GPU's (the step's x_q / x_s buffers), and ``rows``
    output rows of every Y (rows 0 and n - 1 among them) with the FP64 result
    the oracle computes from its own quantisation of X and of those weight
    rows.  Error metric: max |y - ref| / max(|ref|, rms of the row of ref)."""
    import oracle
    torch = stack.torch
    torch.cuda.synchronize()
    if layers is None:
        layers = sorted({0, stack.layers - 1})
    rng = np.random.default_rng(seed)
    tol = 1e-3 + (2.0 ** -8) * (1 + 1e-3) if stack.bf16 else 1e-3
    worst, codes_ok, checked = 0.0, True, 0

    def host_f32(t):
        if t.dtype == torch.bfloat16:
            return oracle.bf16_to_f32(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
        return t.cpu().numpy()

    for l in layers:
        for j, lin in enumerate(stack.lins):
            x = host_f32(stack.x[l][j])
            gx = oracle.global_scale(x)
            codes_ok &= bool(np.float32(stack.xg[l][j].cpu().numpy()[0]) == gx)
            oxq, oxs = oracle.quantize(x, gx)
            if stack.mode == "chain" or l == stack.layers - 1:   # shared buffers: last layer's
                xq, xs = stack.codes(l, j)
                codes_ok &= bool(np.array_equal(xq.cpu().numpy(), oxq) and
                                 np.array_equal(xs.cpu().numpy(), oxs))
            wf = stack.weight_fp32(l, j)
            w = wf.cpu().numpy()
            del wf
            gw = oracle.global_scale(w)
            codes_ok &= bool(np.float32(stack.w[l][j][2].cpu().numpy()[0]) == gw)
            sel = np.unique(np.concatenate([[0, lin.n - 1], rng.integers(0, lin.n, rows - 2)]))
            owq, ows = oracle.quantize(w[sel], gw)
            del w
            ref = oracle.gemm(oxq, oxs, gx, owq, ows, gw)
            y = host_f32(stack.y[l][j])[:, sel].astype(np.float64)
            rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
            den = np.maximum(np.abs(ref), rms)
            den = np.where(den > 0, den, 1.0)
            worst = max(worst, float(np.max(np.abs(y - ref) / den)))
            checked += 1
    return {"ok": bool(codes_ok and worst <= tol), "max_err": worst, "tol": tol,
            "codes_bit_exact": codes_ok, "layers": layers, "rows_per_linear": rows,
            "linears_checked": checked, "mode": stack.mode,
            "metric": "max |y - ref| / max(|ref|, row rms of ref), ref = oracle FP64"}


def oracle_sample(rows_per_linear: int, seed: int = 99, layers: int = 1, first_layer: int = 0):
    """Packed operands for a bounded sample of the workload: the four linears
    of ``layers`` layers from ``first_layer`` on (distinct seeded weights),
    ``rows_per_linear`` output rows each (packing not timed)."""
    import oracle
    items = []
    for l in range(first_layer, first_layer + layers):
        for j, lin in enumerate(synthetic.LINEARS_8B):
            rows = min(rows_per_linear, lin.n)
            s = synthetic.weight_seed(seed, l, j)
            w = synthetic.weights(rows, lin.k, synthetic.WEIGHT_STD_8B, seed=s)
            x = synthetic.activations(1, lin.k, seed=s + 1)
            wq, ws, gw = oracle.pack_weight(w)
            del w
            gx = oracle.global_scale(x)
            items.append((x, gx, wq, ws, gw, rows, lin.k))
    return items


def oracle_pass(items):
    """One pass of the hot path on the CPU: quantise X, GEMM from packed bytes."""
    import oracle
    for x, gx, wq, ws, gw, rows, k in items:
        xq, xs = oracle.quantize(x, gx)
        oracle.gemm(xq, xs, gx, wq, ws, gw)


def sample_bytes(items):
    tot = 0
    for x, gx, wq, ws, gw, rows, k in items:
        tot += algorithmic_bytes(1, rows, k)["gemm"] + algorithmic_bytes(1, rows, k)["quant"]
    return tot


def calibrate_sample(budget_s: float):
    """(rows per linear, layers) of an oracle sample that takes about
    ``budget_s`` seconds on this host: a probe of 8 rows per linear sets the
    cost per row; below one whole layer the rows are cut, above it whole
    layers are added (at most the 36 of the step)."""
    probe = oracle_sample(8)
    t0 = time.perf_counter()
    oracle_pass(probe)
    dt = max(time.perf_counter() - t0, 1e-4)
    per_elem = dt / sum(8 * lin.k for lin in synthetic.LINEARS_8B)
    full_layer = per_elem * sum(lin.n * lin.k for lin in synthetic.LINEARS_8B)
    if full_layer >= budget_s:
        rows = int(budget_s / per_elem / sum(lin.k for lin in synthetic.LINEARS_8B))
        return max(8, rows), 1
    return max(lin.n for lin in synthetic.LINEARS_8B), int(min(36, max(1, round(budget_s / full_layer))))


def cpu_baseline(budget_s: float = 12.0, all_cores: bool = True) -> dict:
    """The oracle on the host: a bounded sample of the step sized to about
    ``budget_s`` seconds.  When whole layers fit, one layer is timed first
    (untimed warm-up of the sample) to fix how many layers the budget holds.
    With ``all_cores`` (and more than one core) the reported line is the
    all-cores run, the single-thread one nested in it."""
    rows, layers = calibrate_sample(budget_s)
    items = oracle_sample(rows, layers=1)
    if rows >= max(lin.n for lin in synthetic.LINEARS_8B):
        t0 = time.perf_counter()
        oracle_pass(items)
        one = max(time.perf_counter() - t0, 1e-3)
        layers = int(min(36, max(1, round(budget_s / one))))
        if layers > 1:
            items += oracle_sample(rows, layers=layers - 1, first_layer=1)
    t0 = time.perf_counter()
    oracle_pass(items)
    sec = time.perf_counter() - t0
    v = sample_bytes(items) / sec / 1e9
    what = (f"{layers} whole layers (all output rows)" if layers > 1 or rows >= 24576
            else f"one layer, {rows} output rows per linear")
    single = {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
              "sample": f"the four 8B-shaped linears at M=1 of {what}: quantise X + FP64 GEMM "
                        f"from packed bytes, {sec:.1f} s, single thread",
              "seconds": round(sec, 2)}
    if not all_cores or len(os.sched_getaffinity(0)) < 2:
        return single
    # whole layers are what the all-cores run gives out: time one when the
    # single-thread sample had only part of one
    layer_s = sec / layers if rows >= max(lin.n for lin in synthetic.LINEARS_8B) else \
        sec * sum(lin.n * lin.k for lin in synthetic.LINEARS_8B) / \
        sum(min(rows, lin.n) * lin.k for lin in synthetic.LINEARS_8B)
    try:
        line = cpu_baseline_all_cores(layer_s, budget_s)
    except Exception as e:  # the single-thread line still stands
        single["all_cores_error"] = f"{type(e).__name__}: {e}"[:200]
        return single
    line["single_thread"] = single
    return line


def _oracle_worker(layers: int, first_layer: int, barrier, out) -> None:
    """One host process of the all-cores baseline: build its whole layers of
    the sample (untimed), wait for the others, time one oracle pass."""
    items = oracle_sample(max(lin.n for lin in synthetic.LINEARS_8B), layers=layers,
                          first_layer=first_layer)
    barrier.wait(timeout=900)
    t0 = time.perf_counter()
    oracle_pass(items)
    t1 = time.perf_counter()
    out.put((t0, t1, sample_bytes(items)))


def cpu_baseline_all_cores(layer_seconds: float, budget_s: float = 12.0) -> dict:
    """The same oracle on every core of this process's affinity mask: one
    single-threaded process per core (started with spawn), each with its own
    whole layers of the step (at most the step's 36 in total, about
    ``budget_s`` seconds each), all timed together: the wall time from the
    first start to the last finish."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    per_worker = max(1, int(budget_s / max(layer_seconds, 1e-3)))
    total = min(synthetic.DECODE_LAYERS_8B, per_worker * cores)
    workers = min(cores, total)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(workers)
    out = ctx.Queue()
    procs, first = [], 0
    for i in range(workers):
        n = total // workers + (1 if i < total % workers else 0)
        procs.append(ctx.Process(target=_oracle_worker, args=(n, first, barrier, out)))
        first += n
    for p in procs:
        p.start()
    res, deadline = [], time.time() + 1800
    while len(res) < len(procs):
        try:
            res.append(out.get(timeout=2))
        except queue.Empty:
            if time.time() > deadline or any(p.exitcode not in (None, 0) for p in procs):
                for p in procs:      # the processes started here, by handle
                    p.terminate()
                raise RuntimeError("an all-cores oracle process failed or ran out of time")
    for p in procs:
        p.join()
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    v = sum(r[2] for r in res) / wall / 1e9
    return {"value": round(v, 4), "unit": UNIT, "cores": workers, "kind": "oracle",
            "sample": f"{total} whole layers of the step (the four 8B-shaped linears at M=1, all "
                      f"output rows), spread over {workers} single-threaded processes: quantise X "
                      f"+ FP64 GEMM from packed bytes, {wall:.1f} s wall",
            "seconds": round(wall, 2)}


KERNELS = {"auto": lambda nv: nv.KERNEL_AUTO, "generic": lambda nv: nv.KERNEL_GENERIC,
           "gemv": lambda nv: nv.KERNEL_GEMV, "mma": lambda nv: nv.KERNEL_MMA,
           "tma": lambda nv: nv.KERNEL_TMA, "splitk": lambda nv: nv.KERNEL_SPLITK,
           "tc": lambda nv: nv.KERNEL_TC}


def run_single(args) -> None:
    """One linear shape, repeated: the case the kernel-level ncu captures run.
    Seeded N(0, 0.02^2) weights packed on the device, one seeded activation
    batch quantised once, then the GEMM with the chosen kernel `reps` times, then
    a CUDA graph of 20 calls timed with CUDA events (printed: µs per call, GB/s;
    the same weights every call, so shapes below L2 read from L2)."""
    import torch

    import nvfp4_w4a4_decode_gb300 as nv
    from nvfp4_w4a4_decode_gb300 import build as nvbuild
    m, n, k = args.single
    kernel = KERNELS[args.kernel](nv)
    nvbuild.build()
    nv.library()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    w = torch.randn((n, k), generator=gen, device="cuda") * synthetic.WEIGHT_STD_8B
    wq, ws, wg = nv.pack_weight(w)
    del w
    x = torch.from_numpy(synthetic.activations(m, k, seed=1)).cuda()
    xg = nv.global_scale(x)
    xq, xs = nv.quantize_act(x, xg)
    torch.cuda.synchronize()
    y = torch.empty((m, n), device="cuda")
    wsp = nv.workspace(m, n, k, kernel)
    for _ in range(args.reps):
        nv.gemm_smallm(xq, xs, xg, wq, ws, wg, out=y, kernel=kernel, workspace=wsp)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(20):
            nv.gemm_smallm(xq, xs, xg, wq, ws, wg, out=y, kernel=kernel, workspace=wsp)
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    b.synchronize()
    us = a.elapsed_time(b) * 1e3 / 20
    byt = algorithmic_bytes(m, n, k)["gemm"]
    print(json.dumps({"single": [m, n, k], "kernel": args.kernel, "us_per_call": round(us, 3),
                      "GBps": round(byt / (us * 1e-6) / 1e9, 1), "y00": float(y[0, 0])}))


def run_profile_shapes(args) -> None:
    """Every linear shape of the workloads once, with the library's kernel
    choice (workspace offered): the 256 x 512 single GEMV at M = 1, the four
    8B linears at M = 1, 2, 4, 8 and the four 32B linears at M = 1, 4.  One
    weight matrix at a time on the device (at most 148 MB), `reps` GEMM launches
    each; prints the kernel per shape.  The case the per-shape counter capture
    runs."""
    import torch

    import nvfp4_w4a4_decode_gb300 as nv
    from nvfp4_w4a4_decode_gb300 import build as nvbuild
    nvbuild.build()
    nv.library()
    cases = [(synthetic.TINY, 1, synthetic.WEIGHT_STD_8B, "C1")]
    cases += [(lin, m, synthetic.WEIGHT_STD_8B, "8B") for m in synthetic.M_SWEEP_8B
              for lin in synthetic.LINEARS_8B]
    cases += [(lin, m, synthetic.WEIGHT_STD_32B, "32B") for m in synthetic.M_SWEEP_32B
              for lin in synthetic.LINEARS_32B]
    gen = torch.Generator(device="cuda")
    for i, (lin, m, std, fam) in enumerate(cases):
        gen.manual_seed(7000 + i)
        w = torch.randn((lin.n, lin.k), generator=gen, device="cuda") * std
        wq, ws, wg = nv.pack_weight(w)
        del w
        x = torch.from_numpy(synthetic.activations(m, lin.k, seed=7100 + i)).cuda()
        xg = nv.global_scale(x)
        xq, xs = nv.quantize_act(x, xg)
        y = torch.empty((m, lin.n), device="cuda")
        wsp = nv.workspace(m, lin.n, lin.k)
        kid = nv.gemm_select(m, lin.n, lin.k, nv.KERNEL_AUTO, wsp.numel() if wsp is not None else 0)
        for _ in range(args.reps):
            nv.gemm_smallm(xq, xs, xg, wq, ws, wg, out=y, workspace=wsp)
        torch.cuda.synchronize()
        print(json.dumps({"case": i, "family": fam, "linear": lin.name, "m": m, "n": lin.n,
                          "k": lin.k, "kernel": nv.KERNEL_NAMES.get(kid),
                          "gemm_bytes": algorithmic_bytes(m, lin.n, lin.k)["gemm"]}), flush=True)
        del wq, ws, wg, x, xq, xs, y, wsp
        torch.cuda.empty_cache()


def run_reference(args) -> dict | None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    oracle.build()
    # each step a bounded sample, sized so that the whole run (warm-up and
    # timed steps) takes about two and a half minutes of host time
    budget = args.ref_step_seconds or max(0.05, 150.0 / (args.steps + args.warmup))
    rows, layers = calibrate_sample(budget)
    items = oracle_sample(rows, layers=layers)
    for _ in range(args.warmup):
        oracle_pass(items)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_pass(items)
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    v = sample_bytes(items) / sec / 1e9
    what = (f"{layers} whole layers" if layers > 1 or rows >= 24576
            else f"one layer, {rows} output rows per linear")
    sample = (f"per step: the four 8B-shaped linears at M=1 of {what} (quantise X + FP64 GEMM "
              f"from packed bytes), {sec:.2f} s, single thread")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "m": 1, "sample_rows_per_linear": rows,
                       "sample_layers": layers},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--layers", type=int, default=synthetic.DECODE_LAYERS_8B)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.0,
                    help="host seconds per reference step (default: ~150 s over the run)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16", action="store_true",
                    help="BF16 activations in and BF16 outputs out (FP32 otherwise)")
    ap.add_argument("--fused", action="store_true",
                    help="one kernel per linear (quantisation in the GEMM prologue) instead of "
                         "quantiser + GEMM")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-shape M sweep (8B M=1,2,4,8; 32B M=1,4)")
    ap.add_argument("--sweep-generic", action="store_true",
                    help="also time the shape-general kernel in the sweep")
    ap.add_argument("--single", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="time one linear shape (for kernel-level profiling) and exit")
    ap.add_argument("--mode", default="auto", choices=["auto", "chain", "launches"],
                    help="the step as one multi-linear call (chain, M <= 2) or one call per "
                         "linear (launches); auto: chain where it applies")
    ap.add_argument("--chain-kernel", default="auto", choices=["auto", "gemv", "tc"],
                    help="engine of the chain step (auto: the library's choice, the tensor "
                         "cores at every M; gemv: the CUDA-core stream, M <= 2)")
    ap.add_argument("--row-major-weights", action="store_true",
                    help="the tensor-core chain reads the row-major packed weights (TMA with a "
                         "tensor map, no stream warps) instead of the tile-major repack "
                         "(nvfp4_tile_weight: one bulk copy a stage)")
    ap.add_argument("--no-chain-workspace", action="store_true",
                    help="run the tensor-core chain without its workspace (CTA shares end on "
                         "tile boundaries)")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNELS),
                    help="GEMM kernel for the decode step (and for --single)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--profile-shapes", action="store_true",
                    help="run every workload shape once per rep with the library's kernel "
                         "choice (for a per-shape counter capture) and exit")
    ap.add_argument("--profile-step", action="store_true",
                    help="replay only the step graph (warmup + steps times) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.single:
        run_single(args)
        return
    if args.profile_shapes:
        run_profile_shapes(args)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the FP4 quantized linear layer (forward + backward).

One step = one pass of the whole hot path over one batch of synthetic input:
for every distinct activation (linears that share an input share this phase)
  quantile threshold + clamp + CSR of dA + row codes of A_clamped (fp4_quantize_rows_outliers)
and for every linear of the workload
  column quantization of W                               (fp4_quantize_cols)
  FP4 GEMM + scales + dA*W compensation -> BF16 Y       (fp4_linear_fwd; fp4_linear_fwd_dense
                                                          when dA averages >= 28 entries per row)
  BF16 weight-gradient GEMM x DGE factor -> fp32 dW     (fp4_linear_wgrad_dge)
  BF16 input-gradient GEMM dY W^T -> BF16 dX             (fp4_linear_dgrad)

Metric: fwd + bwd TFLOP/s = sum over linears of 6 M K N / step time, with
inputs resident in HBM and L2 flushed (256 MiB write) before every step.
`e2e` is the same metric through the C ABI from pinned HOST buffers: the
host->device copy of A, W, dY and the device->host copy of Y, dW and dX are inside
the timed region, on their own streams so that they overlap the kernels (the
phases wait, by events, for their inputs to land; linear by linear, so one
linear's outputs go back while the next one's inputs come in).  `e2e.link`
times the same copies alone.  `--impl reference` times the CPU oracle instead (bounded
sample, single thread).  Under torchrun each rank runs an independent replica
on its own GPU (the layer has no data-path exchange on one GPU's batch);
value = work of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "c4_llama13b_layer_16384tok"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_PER_BF16 = 13.5 / 2.25      # nominal dense FP4 : BF16 tensor rate
L2_FLUSH_BYTES = 256 << 20
HEAD_START_CYCLES = 400_000     # ~0.2 ms GPU spin so the step's launches are all queued
DGE_K, DGE_CLIP = 5.0, 3.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

_REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
                0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 3:
                try:
                    self.samples.append((float(parts[0]), float(parts[1]), int(parts[2], 16)))
                except ValueError:
                    pass
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        busy = [s for s in self.samples if not (s[2] & 0x1)] or self.samples
        reasons = sorted({name for s in busy for bit, name in _REASON_BITS.items() if s[2] & bit and bit != 0x1})
        return {"sm_mhz": statistics.median(s[0] for s in busy), "sm_max_mhz": max(s[1] for s in busy),
                "reasons": reasons, "samples": len(busy)}


# ------------------------------------------------------------------ the GPU arm

class ActStep:
    """One distinct activation (and clamp quantile): threshold, clamp, CSR of dA
    and the row codes / scales of A_clamped, all in fp4_quantize_rows_outliers."""

    PHASE = "fp4_quantize_rows_outliers"
    LAUNCHES = 1   # one cooperative kernel (threshold, clamp, CSR, row codes)

    def __init__(self, fp4, A, q, label=""):
        import torch
        self.fp4, self.A, self.q, self.label = fp4, A, q, label
        M, K = A.shape
        cap = fp4.outlier_max_nnz(M, K, q)
        dev = A.device
        self.out = {
            "t": torch.empty(1, dtype=torch.float32, device=dev),
            "row_ptr": torch.empty(M + 1, dtype=torch.int32, device=dev),
            "col_idx": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
            "vals": torch.empty(max(cap, 1), dtype=torch.float32, device=dev),
            "nnz": torch.empty(1, dtype=torch.int64, device=dev),
            "codes": torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
            "scales": torch.empty(M, dtype=torch.float32, device=dev),
        }
        self.out["workspace"] = torch.empty(fp4.outlier_clamp_quantile_workspace(M, K, max(cap, 1)),
                                            dtype=torch.uint8, device=dev)

    def fn(self):
        return lambda: self.fp4.fp4_quantize_rows_outliers(self.A, self.q, out=self.out)

    def algorithmic_bytes(self) -> float:
        """Two reads of A (the exact global quantile must be known before any
        element is clamped), codes 0.5 B/elem, scales 4 B/row, CSR 8 B/entry + row_ptr."""
        M, K = self.A.shape
        nnz = int(self.out["nnz"].item())
        return 4.0 * M * K + 0.5 * M * K + 4 * M + 8 * nnz + 4 * (M + 1)


class LinStep:
    """One linear: column quantization of W, FP4 GEMM, DGE weight gradient, input gradient."""

    PHASES = ("fp4_quantize_cols", "fp4_linear_fwd", "fp4_linear_wgrad_dge", "fp4_linear_dgrad")

    def launches(self) -> int:
        """Kernels one step of this linear launches: column maxima + codes;
        the forward's 2 compensation prep kernels and the GEMM (K >= 4096: the
        wide GEMM and its many-column fallback), or, for a dense dA, the FP4
        GEMM, the split of dA, W^T and the BF16 product; wgrad; dgrad."""
        if self.dense:
            fwd = 4
        else:
            fwd = 2 + (2 if self.lin.K >= 4096 else 1)
        return 2 + fwd + 1 + 1

    def __init__(self, fp4, lin, act: ActStep, W, dY):
        import torch
        self.fp4, self.lin, self.act = fp4, lin, act
        K, N = lin.K, lin.N
        dev = W.device
        self.W, self.dY = W, dY
        self.w_codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
        self.s_w = torch.empty(N, dtype=torch.float32, device=dev)
        self.ws_cols = torch.empty(max(fp4.fp4_quantize_cols_workspace(N), 16), dtype=torch.uint8, device=dev)
        self.Y = torch.empty((lin.M, N), dtype=torch.bfloat16, device=dev)
        # a dense dA (a low clamp quantile) is multiplied on the BF16 tensor cores
        self.dense = fp4.use_dense_compensation(lin.M, K, lin.q)
        self.ws_fwd = torch.empty((fp4.fp4_linear_fwd_dense_workspace if self.dense else fp4.fp4_linear_fwd_workspace)(
            lin.M, N, K), dtype=torch.uint8, device=dev)
        self.dW = torch.empty((K, N), dtype=torch.float32, device=dev)
        self.dX = torch.empty((lin.M, K), dtype=torch.bfloat16, device=dev)
        # split-tail workspaces of the backward GEMMs (None when the shapes never split)
        wb, db = fp4.fp4_linear_wgrad_dge_workspace(lin.M, N, K), fp4.fp4_linear_dgrad_workspace(lin.M, N, K)
        self.ws_wgrad = torch.empty(wb, dtype=torch.uint8, device=dev) if wb else None
        self.ws_dgrad = torch.empty(db, dtype=torch.uint8, device=dev) if db else None

    def fns(self):
        fp4, lin, a = self.fp4, self.lin, self.act
        return [
            lambda: fp4.fp4_quantize_cols(self.W, codes_t=self.w_codes, scales=self.s_w, workspace=self.ws_cols),
            (lambda: fp4.fp4_linear_fwd_dense(a.out["codes"], a.out["scales"], self.w_codes, self.s_w, lin.K,
                                              csr=a.out, W=self.W, out_type="bf16", Y=self.Y,
                                              workspace=self.ws_fwd)) if self.dense else
            (lambda: fp4.fp4_linear_fwd(a.out["codes"], a.out["scales"], self.w_codes, self.s_w, lin.K, csr=a.out,
                                        W=self.W, out_type="bf16", Y=self.Y, workspace=self.ws_fwd)),
            lambda: fp4.fp4_linear_wgrad_dge(a.A, self.dY, self.W, self.s_w, DGE_K, DGE_CLIP, dW=self.dW,
                                             workspace=self.ws_wgrad),
            lambda: fp4.fp4_linear_dgrad(self.dY, self.W, dX=self.dX, workspace=self.ws_dgrad),
        ]

    def algorithmic(self):
        M, K, N = self.lin.M, self.lin.K, self.lin.N
        return {
            "fp4_quantize_cols": (2.5 * K * N + 4 * N, "B", "hbm"),
            "fp4_linear_fwd": (2 * M * K * N, "FLOP", "tensor_fp4"),
            "fp4_linear_wgrad_dge": (2 * M * K * N, "FLOP", "tensor_bf16"),
            "fp4_linear_dgrad": (2 * M * K * N, "FLOP", "tensor_bf16"),
        }


class StepPlan:
    """All launches of one step: each distinct (activation, q) once, then every linear."""

    def __init__(self, fp4, work, device_inputs):
        self.acts = {}
        self.lins = []
        for lin, (A, W, dY) in zip(work.linears, device_inputs):
            key = (lin.act, lin.q)
            if key not in self.acts:
                self.acts[key] = ActStep(fp4, A, lin.q, lin.act)
            self.lins.append(LinStep(fp4, lin, self.acts[key], W, dY))
        # (phase name, callable) in launch order, and what each call works on
        self.calls = [(ActStep.PHASE, a.fn()) for a in self.acts.values()]
        self.labels = [a.label for a in self.acts.values()]
        for l in self.lins:
            self.calls += list(zip(LinStep.PHASES, l.fns()))
            self.labels += [l.lin.name] * len(LinStep.PHASES)

    def run(self):
        for _, fn in self.calls:
            fn()

    def capture(self):
        import torch
        self.graphs = []
        for _, fn in self.calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            self.graphs.append(g)

    def replay(self, events=None):
        for i, g in enumerate(self.graphs):
            if events is not None:
                events[i].record()
            g.replay()
        if events is not None:
            events[len(self.graphs)].record()

    def step(self, side):
        """One step as a user of the layer runs it: the column quantization of
        every W on the `side` stream while the row pipelines of the activations
        run on the current one; then the forwards; then every dgrad on `side`
        while the weight gradients run on the current stream."""
        import torch
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            for l in self.lins:
                l.fns()[0]()
        for a in self.acts.values():
            a.fn()()
        main.wait_stream(side)
        for l in self.lins:
            l.fns()[1]()
        fork2 = torch.cuda.Event()
        fork2.record(main)
        side.wait_event(fork2)
        with torch.cuda.stream(side):
            for l in self.lins:
                l.fns()[3]()
        for l in self.lins:
            l.fns()[2]()
        main.wait_stream(side)

    def capture_step(self):
        import torch
        self.side = torch.cuda.Stream()
        for _ in range(2):
            self.step(self.side)
        torch.cuda.synchronize()
        self.step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.step_graph):
            self.step(self.side)

    def launches(self):
        return ActStep.LAUNCHES * len(self.acts) + sum(l.launches() for l in self.lins)


def _src_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "precision_gemm_row_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "fp4_linear_wgrad_dge": ["gemm_wgrad.cu", "bwd_gemm.cuh", "common.cuh"],
    "fp4_linear_dgrad": ["gemm_dgrad.cu", "bwd_gemm.cuh", "common.cuh"],
    "fp4_linear_fwd": ["gemm_fwd.cu", "gemm_fwd_dense.cu", "bwd_gemm.cuh", "common.cuh"],
    "fp4_quantize_cols": ["quantize.cu", "common.cuh"],
    "fp4_quantize_rows_outliers": ["outlier.cu", "common.cuh"],
}


def dram_traffic(phase: str, workload: str, launch: str):
    """Per-launch DRAM bytes of `phase` on `launch` (a linear or activation of the
    workload) from the committed ncu summary, or None if the kernel source
    changed since the capture (or none was taken)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(f"{phase}[{launch}]")
    if not e or e.get("source_hash") != _src_hash(KERNEL_SOURCES[phase]):
        return None
    return e.get("bytes_per_launch")


def select_linears(wl, args):
    """The workload, with shared-input linears fused (--fuse-shared-input) and
    restricted to the linears named by --linear (all when none is named)."""
    import types
    work = wl.WORKLOADS[args.workload]
    if args.fuse_shared_input:
        work = wl.fuse_shared_inputs(work)
    if args.linear:
        names = {l.name for l in work.linears}
        unknown = [n for n in args.linear if n not in names]
        if unknown:
            raise SystemExit(f"--linear {unknown}: not in {sorted(names)}")
        keep = tuple(l for l in work.linears if l.name in args.linear)
        work = types.SimpleNamespace(key=work.key, seed=work.seed, linears=keep, activation=work.activation,
                                     weight=work.weight, grad=work.grad)
    return work


def arm_config(args, work, world: int):
    """The workload as both arms report it."""
    return {"workload": args.workload, "linears": [[l.name, l.M, l.K, l.N, l.q] for l in work.linears],
            "fused_shared_input": bool(args.fuse_shared_input), "only_linears": args.linear or None,
            "bwd": "weight gradient with DGE + input gradient dY W^T (BF16; the pages give no dgrad)",
            "l2": "flushed before every step (256 MiB write); the inputs are larger than L2 as well",
            "launch": "one CUDA graph per step (column quantization alongside the row pipeline, dgrad "
                      "alongside wgrad, on two streams), replayed after a 0.2 ms GPU head start; kernel "
                      "times from a second pass of one graph per phase",
            "parallelism": f"replicas x{world}"}


# ------------------------------------------------------------------ replicas

def max_over_ranks(values, device):
    """Element-wise maximum of `values` over the ranks of the default process
    group (the slowest replica sets the time); the values unchanged on one rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(world: int, flops_per_replica: float, ms_max: float) -> float:
    """Whole-job TFLOP/s: every replica does the same work, the slowest sets the time."""
    return world * flops_per_replica / (ms_max * 1e-3) / 1e12


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from precision_gemm_row_gb300 import build as fp4build
    from precision_gemm_row_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    if local == 0 or world == 1:
        fp4build.build()
    if world > 1:
        dist.barrier()
    from precision_gemm_row_gb300 import fp4lin as fp4

    work = select_linears(wl, args)
    host = []
    dev_inputs = []
    pinned_cache = {}
    to_pinned = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    for lin in work.linears:
        akey = (lin.act,)
        if akey not in pinned_cache:
            pinned_cache[akey] = to_pinned(work.activation(lin))
        hA = pinned_cache[akey]
        hW, hG = to_pinned(work.weight(lin)), to_pinned(work.grad(lin))
        host.append((hA, hW, hG))
    dev_cache = {}
    for lin, (hA, hW, hG) in zip(work.linears, host):
        if id(hA) not in dev_cache:
            dev_cache[id(hA)] = hA.cuda()
        dev_inputs.append((dev_cache[id(hA)], hW.cuda(), hG.cuda()))
    plan = StepPlan(fp4, work, dev_inputs)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flops = sum(6 * l.M * l.K * l.N for l in work.linears)

    for _ in range(args.warmup):
        plan.run()
    torch.cuda.synchronize()
    plan.capture()
    plan.capture_step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        plan.replay()
        plan.step_graph.replay()
    st, fl = fp4.fp4_device_status()
    if st != "FP4_OK":
        raise RuntimeError(f"device status after warm-up: {st} flags={fl}")

    # ---- device-resident timed region: L2 flush, then a short GPU-side head start
    # so the step is queued before the first event fires.  The step is one CUDA
    # graph (independent phases on two streams, see StepPlan.step).
    ev_step = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            flush.fill_(float(k))
            torch.cuda._sleep(HEAD_START_CYCLES)
            ev_step[k][0].record()
            plan.step_graph.replay()
            ev_step[k][1].record()
        torch.cuda.synchronize()
        # ---- per-phase pass (the roofline's kernel times): the same phases one
        # after another, one graph per phase, events between them on the stream
        # that launches them
        ncalls = len(plan.calls)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ncalls + 1)] for _ in range(args.steps)]
        for k in range(args.steps):
            flush.fill_(float(k))
            torch.cuda._sleep(HEAD_START_CYCLES)
            plan.replay(ev[k])
        torch.cuda.synchronize()
    st, fl = fp4.fp4_device_status()
    if st != "FP4_OK":
        raise RuntimeError(f"device status after timed steps: {st} flags={fl}")
    step_ms = [ev_step[k][0].elapsed_time(ev_step[k][1]) for k in range(args.steps)]
    ms_per_step = sum(step_ms) / len(step_ms)
    seq_ms = sum(ev[k][0].elapsed_time(ev[k][ncalls]) for k in range(args.steps)) / args.steps
    phase_ms, call_ms = {}, []
    for i, (name, _) in enumerate(plan.calls):
        t = sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)) / args.steps
        call_ms.append(t)
        phase_ms[name] = phase_ms.get(name, 0.0) + t

    # ---- end to end through the C ABI from pinned host buffers
    hY = [torch.empty(l.Y.shape, dtype=l.Y.dtype).pin_memory() for l in plan.lins]
    hdW = [torch.empty(l.dW.shape, dtype=l.dW.dtype).pin_memory() for l in plan.lins]
    hdX = [torch.empty(l.dX.shape, dtype=l.dX.dtype).pin_memory() for l in plan.lins]
    uniq_hA = {id(h[0]): h[0] for h in host}
    bi = sum(h.numel() * 2 for h in uniq_hA.values()) + sum(h[1].numel() * 2 + h[2].numel() * 2 for h in host)
    bo = sum(y.numel() * 2 + d.numel() * 4 + x.numel() * 2 for y, d, x in zip(hY, hdW, hdX))
    e2e_ms = []
    # Copies overlap the kernels: host to device on one stream, linear by linear
    # (its activation if new, W, then dY), the phases on the current stream as
    # their inputs land (an activation's row call before its first linear,
    # dgrad before wgrad), device to host on a third stream as each output is
    # done, so the outputs of one linear go back while the next one's inputs
    # come in.  Like the device step, the whole of it is one CUDA graph.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_ops():
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        ev_a, ev_w, ev_g = {}, [], []
        with torch.cuda.stream(s_in):
            for i, l in enumerate(plan.lins):
                if id(l.act) not in ev_a:
                    l.act.A.copy_(host[i][0], non_blocking=True)
                    ev_a[id(l.act)] = torch.cuda.Event()
                    ev_a[id(l.act)].record(s_in)
                l.W.copy_(host[i][1], non_blocking=True)
                ev_w.append(torch.cuda.Event())
                ev_w[-1].record(s_in)
                l.dY.copy_(host[i][2], non_blocking=True)
                ev_g.append(torch.cuda.Event())
                ev_g[-1].record(s_in)
        done_acts = set()
        for i, l in enumerate(plan.lins):
            if id(l.act) not in done_acts:
                main.wait_event(ev_a[id(l.act)])
                l.act.fn()()
                done_acts.add(id(l.act))
            fns = dict(zip(LinStep.PHASES, l.fns()))
            main.wait_event(ev_w[i])
            fns["fp4_quantize_cols"]()
            fns["fp4_linear_fwd"]()
            ev_y = torch.cuda.Event()
            ev_y.record(main)
            main.wait_event(ev_g[i])
            fns["fp4_linear_dgrad"]()
            ev_x = torch.cuda.Event()
            ev_x.record(main)
            fns["fp4_linear_wgrad_dge"]()
            ev_w2 = torch.cuda.Event()
            ev_w2.record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_y)
                hY[i].copy_(l.Y, non_blocking=True)
                s_out.wait_event(ev_x)
                hdX[i].copy_(l.dX, non_blocking=True)
                s_out.wait_event(ev_w2)
                hdW[i].copy_(l.dW, non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    for _ in range(2):
        e2e_ops()
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        e2e_ops()
    s_c = torch.cuda.current_stream()
    e2e_ms = []
    for k in range(args.warmup + args.steps):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_c)
        e2e_graph.replay()
        e1.record(s_c)
        e1.synchronize()
        if k >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_ms_mean = sum(e2e_ms) / len(e2e_ms)

    # ---- the same copies alone, on the same streams, with no kernels: the
    # link's rate for these bytes, which bounds e2e from below
    def copies_only(h2d: bool, d2h: bool) -> float:
        ts = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_c)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
            if h2d:
                with torch.cuda.stream(s_in):
                    seen = set()
                    for i, l in enumerate(plan.lins):
                        if id(l.act) not in seen:
                            l.act.A.copy_(host[i][0], non_blocking=True)
                            seen.add(id(l.act))
                        l.W.copy_(host[i][1], non_blocking=True)
                        l.dY.copy_(host[i][2], non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    for i, l in enumerate(plan.lins):
                        hY[i].copy_(l.Y, non_blocking=True)
                        hdX[i].copy_(l.dX, non_blocking=True)
                        hdW[i].copy_(l.dW, non_blocking=True)
            s_c.wait_stream(s_in)
            s_c.wait_stream(s_out)
            e1.record(s_c)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    t_in, t_out, t_both = copies_only(True, False), copies_only(False, True), copies_only(True, True)
    link = {"h2d_gbs": round(bi / t_in / 1e6, 1), "d2h_gbs": round(bo / t_out / 1e6, 1),
            "copies_only_ms": round(t_both, 3), "e2e_over_copies_only": round(e2e_ms_mean / t_both, 3)}

    # ---- max over ranks
    ms_max, e2e_max = max_over_ranks([ms_per_step, e2e_ms_mean], "cuda")

    peaks, peak_src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_PER_BF16
    nnz = sum(int(a.out["nnz"].item()) for a in plan.acts.values())
    amounts = {ActStep.PHASE: (sum(a.algorithmic_bytes() for a in plan.acts.values()), "B", "hbm")}
    for l in plan.lins:
        for name, (amt, unit, bound) in l.algorithmic().items():
            prev = amounts.get(name, (0.0, unit, bound))
            amounts[name] = (prev[0] + amt, unit, bound)
    kernels = {}
    for name, (amount, unit, bound) in amounts.items():
        per_s = amount / (phase_ms[name] * 1e-3)
        if unit == "B":
            ach, u, pk = per_s / 1e9, "GB/s", peaks["hbm_gbs"]
        elif bound == "tensor_fp4":
            ach, u, pk = per_s / 1e12, "TFLOP/s", fp4_peak
        else:
            ach, u, pk = per_s / 1e12, "TFLOP/s", peaks["bf16_tflops"]
        kernels[name] = {"ms": round(phase_ms[name], 5), "achieved": round(ach, 2), "unit": u, "peak": pk,
                         "frac": round(ach / pk, 4), "bound": "hbm" if unit == "B" else "tensor"}
    # roofline: the single launch (phase of one linear, or one activation's row
    # call) with the longest time, its algorithmic work per launch / its time
    per_call = []
    for i, (name, _) in enumerate(plan.calls):
        if name == ActStep.PHASE:
            act = list(plan.acts.values())[i]
            amount, unit, bound = act.algorithmic_bytes(), "B", "hbm"
        else:
            lin = plan.lins[(i - len(plan.acts)) // len(LinStep.PHASES)]
            amount, unit, bound = lin.algorithmic()[name]
        per_call.append((call_ms[i], name, plan.labels[i], amount, unit, bound))
    ms_d, dom, dom_label, amount, unit, bound = max(per_call, key=lambda c: c[0])
    per_s = amount / (ms_d * 1e-3)
    if unit == "B":
        ach, u, pk = per_s / 1e9, "GB/s", peaks["hbm_gbs"]
    elif bound == "tensor_fp4":
        ach, u, pk = per_s / 1e12, "TFLOP/s", fp4_peak
    else:
        ach, u, pk = per_s / 1e12, "TFLOP/s", peaks["bf16_tflops"]
    tr = dram_traffic(dom, args.workload, dom_label)
    roofline = {"bound": "hbm" if unit == "B" else "tensor", "kernel": dom, "launch": dom_label,
                "achieved": round(ach, 2), "peak": pk,
                "peak_source": f"{peak_src}" + (" x nominal FP4/BF16 ratio 6" if dom == "fp4_linear_fwd" else ""),
                "unit": u, "frac": round(ach / pk, 4), "traffic": tr, "launch_ms": round(ms_d, 5),
                "work_per_launch": amount, "work_unit": "B" if unit == "B" else "FLOP"}
    qnames = (ActStep.PHASE, "fp4_quantize_cols")
    quant_bytes = sum(amounts[n][0] for n in qnames)
    quant_ms = sum(kernels[n]["ms"] for n in qnames)
    value = job_throughput(world, flops, ms_max)
    e2e_value = job_throughput(world, flops, e2e_max)
    line = {
        "metric": "FP4 linear fwd+bwd TFLOPS on 1 GB300, % of dense FP4 peak; quantize GB/s vs HBM",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp4_e2m1 fwd / bf16 wgrad + dgrad, fp32 accumulate", "data": "synthetic (seeded, LLaMA-shaped)",
        "config": arm_config(args, work, world),
        "fp4_peak_frac": round(value / world / fp4_peak, 4),
        "quantize": {"gbs": round(quant_bytes / (quant_ms * 1e-3) / 1e9, 1), "frac_of_hbm": round(
            quant_bytes / (quant_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
        "kernels": kernels, "phases_one_after_another_ms": round(seq_ms, 5), "nnz": nnz,
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "ms_per_step": round(e2e_max, 5), "link": link},
        "gpu_launches": args.steps * plan.launches(),
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # the CPU baseline is a single-GPU figure
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_sample)   # two measured steps
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return line if rank == 0 else None


# ------------------------------------------------------------------ the CPU oracle

_ORACLE_SAMPLE = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
from oracle import fp4_linear as orc
from precision_gemm_row_gb300 import workloads as wl
work = wl.WORKLOADS[sys.argv[2]]
S = int(sys.argv[3])
nsteps = int(sys.argv[4])
# the sub-problem of every linear: its first S tokens and first S output
# columns, with the whole reduction length K (drawn once, outside the timing)
inputs = []
for lin in work.linears:
    ms, ns = min(S, lin.M), min(S, lin.N)
    A = work.activation(lin, rows=ms)
    W = np.ascontiguousarray(work.weight(lin)[:, :ns])
    dY = np.ascontiguousarray(work.grad(lin, rows=ms)[:, :ns])
    inputs.append((lin, A, W, dY))
flops = sum(6 * A.shape[0] * A.shape[1] * W.shape[1] for _, A, W, _ in inputs)
steps = []
for _ in range(nsteps):
    t0 = time.perf_counter()
    for lin, A, W, dY in inputs:
        t, _, _ = orc.quantile_threshold(A, lin.q)
        A_c, rp, ci, cv = orc.clamp_and_compensation(A, t)
        a_codes, s_a = orc.quantize_rows(A_c)
        w_codes, s_w = orc.quantize_cols(orc.bf16_to_f32(W))
        orc.f64_to_bf16(orc.linear_fwd(a_codes, s_a, w_codes, s_w, rp, ci, cv, W))
        orc.wgrad_dge(A, dY, W, s_w, 5.0, 3.0)
        orc.f64_to_bf16(orc.linear_dgrad(dY, W))
    steps.append(time.perf_counter() - t0)
print(json.dumps(dict(steps=steps, flops=flops)))
"""

ORACLE_SAMPLE = 256     # tokens x output columns of every linear's sub-problem


FULL_PROBLEM_MAX = 1024   # a workload whose linears all have M, N <= this is timed in full


def effective_sample(workload: str, sample: int) -> int:
    """The sub-problem size: the whole problem when it is small (every token and
    output column), else `sample`."""
    from precision_gemm_row_gb300 import workloads as wl
    lins = wl.WORKLOADS[workload].linears
    if all(l.M <= FULL_PROBLEM_MAX and l.N <= FULL_PROBLEM_MAX for l in lins):
        return max(max(l.M, l.N) for l in lins)
    return sample


def _oracle_steps(workload: str, sample: int, nsteps: int):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _ORACLE_SAMPLE, ROOT, workload, str(sample), str(nsteps)],
                       env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle baseline failed: " + r.stderr[-800:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def _sample_text(sample: int, workload: str) -> str:
    from precision_gemm_row_gb300 import workloads as wl
    lins = wl.WORKLOADS[workload].linears
    if all(l.M <= sample and l.N <= sample for l in lins):
        return ("the whole problem: every linear of the workload on all its tokens and output columns (quantile + "
                "clamp + CSR + row codes, column codes, FP4 GEMM + epilogue, DGE weight gradient, input gradient), "
                "all measured; value = 6 M K N summed over the linears / measured time; one thread "
                "(OPENBLAS/OMP threads = 1)")
    return (f"every linear of the workload on its first {sample} tokens x first {sample} output columns (the whole "
            f"reduction length K): quantile + clamp + CSR + row codes of that activation slice, column codes of that "
            f"weight slice, FP4 GEMM + epilogue, DGE weight gradient and input gradient, all measured (nothing "
            f"extrapolated); value = 6 m K n summed over the sub-problems / measured time; one thread "
            f"(OPENBLAS/OMP threads = 1)")


def cpu_baseline(workload: str, sample: int = ORACLE_SAMPLE, nsteps: int = 2):
    """The oracle, as it stands, timed in a fresh single-thread interpreter on a
    bounded sub-problem of every linear of the workload (see _sample_text)."""
    t0 = time.time()
    sample = effective_sample(workload, sample)
    d = _oracle_steps(workload, sample, nsteps)
    step_s = statistics.median(d["steps"])
    return {"value": round(d["flops"] / step_s / 1e12, 8), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": _sample_text(sample, workload), "sample_flops_per_step": d["flops"], "step_s": round(step_s, 6),
            "steps": nsteps, "wall_s": round(time.time() - t0, 1)}


def run_reference(args):
    """`--impl reference`: the oracle on the host cores, W + K steps of the
    bounded sub-problem in one process (inputs drawn once), each step measured;
    ms_per_step is the median measured step time of what it ran."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from precision_gemm_row_gb300 import workloads as wl
    t0 = time.time()
    sample = effective_sample(args.workload, args.cpu_sample)
    d = _oracle_steps(args.workload, sample, args.warmup + args.steps)
    step_s = statistics.median(d["steps"][args.warmup:])
    v = round(d["flops"] / step_s / 1e12, 8)
    cb = {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": _sample_text(sample, args.workload),
          "sample_flops_per_step": d["flops"], "step_s": round(step_s, 6), "steps": args.steps,
          "wall_s": round(time.time() - t0, 1)}
    return {"impl": "reference", "metric": "FP4 linear fwd+bwd TFLOPS on 1 GB300, % of dense FP4 peak; quantize GB/s "
            "vs HBM", "value": v, "unit": "TFLOP/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_s * 1e3, 3), "extrapolated": False, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (oracle)", "data": "synthetic (seeded, LLaMA-shaped)",
            "config": arm_config(args, select_linears(wl, args), 1), "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=ORACLE_SAMPLE,
                    help="tokens and output columns of every linear in the oracle's sub-problem")
    ap.add_argument("--fuse-shared-input", action="store_true",
                    help="linears reading the same activation run as one GEMM over their concatenated weights")
    ap.add_argument("--linear", action="append", default=[],
                    help="run only this linear of the workload (repeatable; default: all)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

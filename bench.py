#!/usr/bin/env python3
"""Benchmark of the Q8_0 GEMV library on its decode-step workload; prints one JSON line.

Workload (one step): the projection chain of a 32-layer 7B-class decode step over Q8_0 weights -- per layer q, k, v, o
(4096 x 4096), gate and up (4096 x 14336) and down (14336 x 4096) -- then the tied head (4096 x 128256) with the
arg-max over its fp32 logits fused.  Per layer q/k/v read one activation and gate/up another, as in a transformer
layer, so each pair or triple is one q8_gemv_parts call; o and down are q8_gemv calls: 128 layer calls and one
q8_gemv_argmax, m activation rows each (m = 1 and 16 by default), 9.36 GB of weights per step at m = 1: every step
reads far more than the 129 MB L2, so no flush is needed.  The planner runs some calls as two launches
(q8_plan_launches; the gate/up pairs and the head on 152 SMs), which gpu_launches counts.
Weights: q uniform int8 in [-127, 127] with a +-127 per block, s = 2^u/127, u ~ U[-8, -2], drawn on the device from a
seed; activations bf16 N(0,1), drawn per layer.

value = algorithmic bytes per step (K * N * 1.125 per weight and m * N * 4 per output, m * K * 2 per activation read
by a call; the head writes m * 8 index bytes instead of logits) / device time per step, summed over ranks (replicas:
every rank runs the whole step on its own GPU).

Arms:
  --impl ours       (default) the CUDA library, the chain captured as CUDA graphs and replayed per step;
  --impl reference  the fp64 CPU oracle on the host cores, a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q8_0 GEMV achieved HBM GB/s (% of GB300 peak) and µs/call at m=1..16"
LAYERS = 32
HIDDEN, FFN, VOCAB = 4096, 14336, 128256
WORKLOAD = (f"decode-step Q8_0 projection chain: {LAYERS} layers x (q,k,v,o 4096x4096; gate,up 4096x14336; "
            f"down 14336x4096) + tied head 4096x128256 with fused arg-max; per layer q/k/v share one activation and "
            f"gate/up another (one multi-projection call each), o and down their own")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
FUSED_NOTE = ("; --fused: q/k/v read the previous layer's normed output, o and down add into the fp32 residual "
              "stream in place and write the next RMS norm (q8_gemv_residual_norm), gate/up is the gated pair")
GLU_NOTE = ("; --ffn glu: gate and up as one gated-pair launch (q8_gemv_glu, SwiGLU) writing bf16 silu(gate) * up, "
            "which the down projection reads")
Q8ACT_NOTE = ("; --act q8: every launch's activation quantized on the device first (q8_quantize_act: int8 codes and "
              "an fp32 scale per 32 values), the products under the quantized numerics (Q8_FLAG_Q8_ACT)")


def act_read_bytes(m, K, q8act=False):
    """Bytes of an activation one launch reads: bf16, or the quantized form (1 byte a value + 4 bytes a 32)."""
    return m * K * (1.125 if q8act else 2)


def quantize_bytes(m, K):
    """Bytes of one q8_quantize_act: the bf16 values read, the quantized form written."""
    return m * K * (2 + 1.125)


def layer_shapes():
    return [(HIDDEN, HIDDEN)] * 4 + [(HIDDEN, FFN)] * 2 + [(FFN, HIDDEN)]


def chain_shapes():
    return [shape for _ in range(LAYERS) for shape in layer_shapes()]


def padded(n):
    return -(-n // 32) * 32


def gemv_bytes(m, K, N, argmax=False):
    """Algorithmic bytes of one call: the Q8_0 weight (1 byte a value + 4 bytes a 32-value block: 1.125 a weight,
    "from_q8.rs" module doc), the bf16 activations and the fp32 outputs (the arg-max's int64 indices instead), over
    the N real columns: the zero-padded last tile's columns are not counted."""
    return K * N * 1.125 + m * K * 2 + (m * 8 if argmax else m * N * 4)


def padded_gemv_bytes(m, K, N):
    """The same over the Np = N rounded up to 32 columns that the row-major storage holds (pads included)."""
    Np = padded(N)
    return K * Np * 1.125 + m * K * 2 + m * Np * 4


def step_bytes(m):
    return sum(gemv_bytes(m, K, N) for K, N in chain_shapes()) + gemv_bytes(m, HIDDEN, VOCAB, argmax=True)


STREAM_SOURCES = ("q8_stream.cu", "q8_device.cuh")  # the sources of the kernels the traffic record covers


def strip_comments(src: str) -> str:
    """C++ source without its comments and with whitespace runs collapsed: what the compiler sees of it (the kernel
    sources hold no comment markers inside string literals)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def source_hash():
    """Hash of the stream kernels' sources as compiled (comments and layout ignored), the key of the traffic record."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "q8_block_quantized_gemv_gb300", "csrc")
    for name in STREAM_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs (one every 100 ms, each stamped
    with its host arrival time so that the summary keeps those of the region: mark() at its start and end)."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch
        self.index = str(device)
        try:
            self.index = f"GPU-{torch.cuda.get_device_properties(device).uuid}"
        except Exception:
            pass
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.marks = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        """Median SM clock, its maximum and the throttle reasons seen over the samples that arrived between the first
        and last mark (plus 0.2 s for nvidia-smi's delivery); all samples when fewer than two of those exist."""
        mhz, maxmhz, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if len(self.marks) >= 2:
            inside = [(t, l) for t, l in self.lines if self.marks[0] <= t <= self.marks[-1] + 0.2]
            if len(inside) >= 2:
                lines = inside
        for _, line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                mhz.append(float(parts[0]))
                maxmhz.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxmhz), "reasons": sorted(reasons),
                "samples": len(mhz), "in_timed_region": lines is not self.lines,
                "timed_region_s": (self.marks[-1] - self.marks[0]) if len(self.marks) >= 2 else None}


# ---------------------------------------------------------------------------------------------------------------------
# the reference arm and the CPU baseline: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------------------------------------------------

def oracle_sample(m, budget_s, weights=None, q8act=False):
    """Time the oracle on the chain's GEMVs in step order until `budget_s` seconds of oracle time have run.

    weights: optional callable i -> (x, q, s) host arrays for GEMV i of the chain (the device's inputs copied
    back); host draws from the seeded generator otherwise.  q8act: each activation quantized first and the product
    taken under the quantized numerics.  Returns (GB/s, description, threads)."""
    import oracle
    import synth_inputs as si
    shapes = chain_shapes() + [(HIDDEN, VOCAB)]
    spent, nbytes, done = 0.0, 0.0, 0
    for i, (K, N) in enumerate(shapes):
        if weights is not None:
            x, q, s = weights(i)
        else:
            x, q, s = si.case(m, K, N, si.case_seed(4, m, i))
        t0 = time.perf_counter()
        if q8act:
            xq, xd = oracle.quantize_act(x)
            y, _ = oracle.gemv_q8act(xq, xd, q, s)
        else:
            y, _ = oracle.gemv(x, q, s)
        if i == len(shapes) - 1:
            oracle.argmax(y, N)
        spent += time.perf_counter() - t0
        nbytes += gemv_bytes(m, K, N, argmax=(i == len(shapes) - 1))
        if q8act:
            nbytes += act_read_bytes(m, K, True) - act_read_bytes(m, K) + quantize_bytes(m, K)
        done += 1
        if spent >= budget_s:
            break
    desc = f"first {done} of {len(shapes)} GEMVs of one step in chain order (m={m}), {spent:.1f} s of oracle time"
    return nbytes / spent / 1e9, desc, oracle.threads(), spent


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    import synth_inputs as si
    # one bounded sample per step: the first layer's seven GEMVs (host draws, prepared before the clock)
    shapes = layer_shapes()
    m = args.m[0]
    cases = [si.case(m, K, N, si.case_seed(4, m, i)) for i, (K, N) in enumerate(shapes)]
    per_step = sum(gemv_bytes(m, K, N) for K, N in shapes)

    def one_step():
        for x, q, s in cases:
            oracle.gemv(x, q, s)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = (time.perf_counter() - t0) / args.steps
    value = per_step / dt / 1e9
    sample = f"one layer's 7 GEMVs (4 x 4096x4096, 2 x 4096x14336, 14336x4096) per step, m={m}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": m, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------------------------------

def reduce_max(v: float, world: int, device: str) -> float:
    """The largest of every rank's v (the step time a replicated run reports: its slowest rank)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job GB/s of N replicas: every rank runs the whole step, the step time is the slowest rank's."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9

class ChainWeights:
    """The decode step's Q8_0 weights, drawn on the device once and shared by the row counts the bench times: the
    row-major tensors as drawn (the CPU baseline reads them back) and the tiled storage the library streams, made
    once as a model would make it at load time."""

    def __init__(self, seed=4000):
        import synth_inputs as si
        import q8_block_quantized_gemv_gb300 as q8
        self.shapes = chain_shapes()
        self.w = [si.device_weight(K, N, seed + i) for i, (K, N) in enumerate(self.shapes)]
        self.head = si.device_weight(HIDDEN, VOCAB, seed + len(self.shapes))
        self.wt = [q8.tile_device(q, s, N) for (q, s), (_, N) in zip(self.w, self.shapes)]
        self.head_t = q8.tile_device(self.head[0], self.head[1], VOCAB)


class Chain:
    """Device-resident activations and outputs of one decode step at m rows over shared weights, and its CUDA graphs.

    The step's data flow is a transformer layer's: q, k and v multiply one activation (one q8_gemv_parts launch),
    o its own, gate and up one more (one q8_gemv_parts launch), down its own; then the tied head with its arg-max.
    Weights are stored tiled (q8_tile_device), as a model would store them once at load time."""

    def __init__(self, torch, m, weights, seed=4000, glu=False, fused=False, q8act=False):
        import q8_block_quantized_gemv_gb300 as q8
        self.torch, self.m, self.glu, self.fused, self.q8act = torch, m, glu or fused, fused, q8act
        self.shapes = weights.shapes
        self.w, self.head, self.wt, self.head_t = weights.w, weights.head, weights.wt, weights.head_t
        # activations: per layer one for q/k/v, one for o, one for gate/up, one for down; then the head's
        self.x_shapes = [K for _ in range(LAYERS) for K in (HIDDEN, HIDDEN, HIDDEN, FFN)] + [HIDDEN]
        sizes = [m * K for K in self.x_shapes]
        self.x_all = torch.empty(sum(sizes), dtype=torch.bfloat16, device="cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 99991)
        self.x_all.copy_(torch.randn(sum(sizes), generator=g, device="cuda", dtype=torch.float32))
        self.x, off = [], 0
        for K in self.x_shapes:
            self.x.append(self.x_all[off:off + m * K].view(m, K))
            off += m * K
        self.y = [torch.empty((m, padded(N)), dtype=torch.float32, device="cuda") for _, N in self.shapes]
        # gated-pair FFN: the gate/up launch writes silu(gate) * up as bf16, which the down projection reads
        self.h = torch.empty((m, padded(FFN)), dtype=torch.bfloat16, device="cuda") if self.glu else None
        # fused layers: the residual stream (fp32, updated in place by o and down), the norms' weights, and the
        # normed activations o and down write for the next launch
        if fused:
            g = torch.Generator(device="cuda")
            g.manual_seed(seed + 7)
            self.res = torch.randn((m, HIDDEN), generator=g, device="cuda", dtype=torch.float32)
            self.gammas = [0.5 + torch.rand(HIDDEN, generator=g, device="cuda") for _ in range(2 * LAYERS)]
            self.xn = [torch.empty((m, HIDDEN), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        self.idx = torch.empty((m,), dtype=torch.int64, device="cuda")
        # quantized activations: one buffer per width, rewritten before each launch that reads it (stream order)
        self.xa = {K: q8.QuantAct(torch.empty((q8.act_bytes(m, K),), dtype=torch.uint8, device="cuda"), m, K)
                   for K in (HIDDEN, FFN)} if q8act else None
        # fused layers under --act q8: the norms and the gated pair write the quantized form the next launch reads
        if fused and q8act:
            def qa(K):
                return q8.QuantAct(torch.empty((q8.act_bytes(m, K),), dtype=torch.uint8, device="cuda"), m, K)
            self.xnq, self.hq = [qa(HIDDEN), qa(HIDDEN)], qa(padded(FFN))
        self.quant_widths = []  # widths of the quantizer launches of one pass of the layers
        self.g_layers = self.g_head = None
        torch.cuda.synchronize()

    def a(self, x):
        """The activation a launch reads: x itself, or (--act q8) its quantized form, quantized now."""
        if not self.q8act:
            return x
        import q8_block_quantized_gemv_gb300 as q8
        self.quant_widths.append(x.shape[1])
        return q8.quantize_act(x, out=self.xa[x.shape[1]])

    def layer_calls(self):
        """(activation index, [GEMV indices]) of every launch of the layers, in order."""
        calls = []
        for layer in range(LAYERS):
            base, xb = 7 * layer, 4 * layer
            calls += [(xb, [base, base + 1, base + 2]), (xb + 1, [base + 3]), (xb + 2, [base + 4, base + 5]),
                      (xb + 3, [base + 6])]
        return calls

    def run_layers(self):
        import q8_block_quantized_gemv_gb300 as q8
        self.quant_widths = []
        if self.fused:
            return self.run_fused_layers()
        for xi, gis in self.layer_calls():
            if self.glu and len(gis) == 2:  # gate, up -> h
                q8.gemv_glu(self.a(self.x[xi]), self.wt[gis[0]], self.wt[gis[1]], FFN, out_bf16=self.h, want=(),
                            constant_weights=True)
            elif self.glu and self.shapes[gis[0]] == (FFN, HIDDEN):  # down reads h
                q8.gemv_parts(self.a(self.h), [(self.wt[gis[0]][0], self.wt[gis[0]][1], HIDDEN)],
                              ys=[self.y[gis[0]]], constant_weights=True, tiled=True)
            else:
                q8.gemv_parts(self.a(self.x[xi]), [(self.wt[i][0], self.wt[i][1], self.shapes[i][1]) for i in gis],
                              ys=[self.y[i] for i in gis], constant_weights=True, tiled=True)

    def run_fused_layers(self):
        """A decode layer's data flow with every fusion: q/k/v read the previous layer's normed output (the first
        layer its drawn activation); o (over a drawn attention output) adds into the residual stream in place and
        writes the norm the FFN reads; gate/up is the gated pair; down adds into the residual stream and writes the
        norm the next layer reads."""
        import q8_block_quantized_gemv_gb300 as q8
        if self.q8act:
            # the producers write the quantized form (no quantizer launch); the drawn inputs are quantized first
            for layer in range(LAYERS):
                base, xb = 7 * layer, 4 * layer
                x_in = self.a(self.x[xb]) if layer == 0 else self.xnq[1]
                q8.gemv_parts(x_in, [(self.wt[i][0], self.wt[i][1], HIDDEN) for i in (base, base + 1, base + 2)],
                              ys=[self.y[base], self.y[base + 1], self.y[base + 2]], constant_weights=True,
                              tiled=True)
                q8.gemv_residual_norm(self.a(self.x[xb + 1]), self.wt[base + 3][0], self.wt[base + 3][1], HIDDEN,
                                      self.res, self.gammas[2 * layer], 1e-6, h=self.res, want=(),
                                      out_q8=self.xnq[0], constant_weights=True)
                q8.gemv_glu(self.xnq[0], self.wt[base + 4], self.wt[base + 5], FFN, want=(), out_q8=self.hq,
                            constant_weights=True)
                q8.gemv_residual_norm(self.hq, self.wt[base + 6][0], self.wt[base + 6][1], HIDDEN, self.res,
                                      self.gammas[2 * layer + 1], 1e-6, h=self.res, want=(), out_q8=self.xnq[1],
                                      constant_weights=True)
            return
        for layer in range(LAYERS):
            base, xb = 7 * layer, 4 * layer
            x_in = self.x[xb] if layer == 0 else self.xn[1]
            q8.gemv_parts(x_in, [(self.wt[i][0], self.wt[i][1], HIDDEN) for i in (base, base + 1, base + 2)],
                          ys=[self.y[base], self.y[base + 1], self.y[base + 2]], constant_weights=True, tiled=True)
            q8.gemv_residual_norm(self.x[xb + 1], self.wt[base + 3][0], self.wt[base + 3][1], HIDDEN,
                                  self.res, self.gammas[2 * layer], 1e-6, h=self.res, out_bf16=self.xn[0],
                                  constant_weights=True)
            q8.gemv_glu(self.xn[0], self.wt[base + 4], self.wt[base + 5], FFN, out_bf16=self.h, want=(),
                        constant_weights=True)
            q8.gemv_residual_norm(self.h, self.wt[base + 6][0], self.wt[base + 6][1], HIDDEN, self.res,
                                  self.gammas[2 * layer + 1], 1e-6, h=self.res, out_bf16=self.xn[1],
                                  constant_weights=True)

    def run_head(self):
        import q8_block_quantized_gemv_gb300 as q8
        q, s = self.head_t
        layer_quants = len(self.quant_widths)
        q8.gemv_argmax(self.a(self.x[-1]), q, s, VOCAB, idx=self.idx, constant_weights=True, tiled=True)
        del self.quant_widths[layer_quants:]  # the head's quantizer is counted with the head

    def capture(self):
        torch = self.torch
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            self.run_layers()
            self.run_head()
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        self.g_layers, self.g_head = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_layers):
            self.run_layers()
        with torch.cuda.graph(self.g_head):
            self.run_head()
        torch.cuda.synchronize()

    def capture_second_buffer(self):
        """A second set of the step's graphs over a second activation buffer (x_all2), so that the end-to-end loop can
        copy step s + 1's inputs from the host while step s runs on the other buffer."""
        torch = self.torch
        first = (self.x_all, self.x)
        self.x_all2 = torch.empty_like(self.x_all)
        self.x_all2.copy_(self.x_all)
        off, self.x = 0, []
        for xv in first[1]:
            self.x.append(self.x_all2[off:off + xv.numel()].view(xv.shape))
            off += xv.numel()
        try:
            self.g_layers2, self.g_head2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_layers2):
                self.run_layers()
            with torch.cuda.graph(self.g_head2):
                self.run_head()
            torch.cuda.synchronize()
        finally:
            self.x_all, self.x = first
        self.x_all_bufs = (self.x_all, self.x_all2)

    def layer_launches(self):
        """Kernel launches of the layers: each product call's (q8_plan_launches, q8_plan_glu_launches: 1, or 2 when
        the planner splits a launch in two); under --fused, o and down as residual norms (the product, then the norm's
        own launch unless the one-launch fold is selected)."""
        import q8_block_quantized_gemv_gb300 as q8
        n = 0
        for _, gis in self.layer_calls():
            if self.glu and len(gis) == 2:
                n += q8.plan_glu_launches(self.m, self.shapes[gis[0]][0], FFN, q8_act=self.q8act)
            elif self.fused and len(gis) == 1:
                n += q8.residual_norm_launches()
            else:
                n += q8.plan_launches(self.m, self.shapes[gis[0]][0], [self.shapes[i][1] for i in gis],
                                      q8_act=self.q8act)
        return n

    def launches_per_step(self):
        """The layers' launches, the head's product launch(es) and its index decode, and (--act q8) the quantizer
        launches."""
        import q8_block_quantized_gemv_gb300 as q8
        n = self.layer_launches() + q8.plan_launches(self.m, HIDDEN, (VOCAB,), q8_act=self.q8act) + 1
        return n + (len(self.quant_widths) + 1 if self.q8act else 0)

    def head_bytes(self):
        m = self.m
        return (gemv_bytes(m, HIDDEN, VOCAB, argmax=True) + (act_read_bytes(m, HIDDEN, True) - act_read_bytes(m, HIDDEN)
                + quantize_bytes(m, HIDDEN) if self.q8act else 0.0))

    def layer_bytes(self):
        """Algorithmic bytes of the layers' launches: weights, each activation once, outputs."""
        m = self.m
        total = 0.0
        # an activation output (the gated pair's, a norm's): bf16, or its quantized form under --act q8
        out_act = 1.125 if self.q8act else 2
        for xi, gis in self.layer_calls():
            total += act_read_bytes(m, self.x_shapes[xi], self.q8act)
            for i in gis:
                K, N = self.shapes[i]
                total += K * N * 1.125 + m * N * 4
            if self.glu and len(gis) == 2:  # one activation output instead of two fp32 ones
                total -= 2 * m * FFN * 4 - m * FFN * out_act
            if self.fused and self.shapes[gis[0]][1] == HIDDEN and len(gis) == 1:
                # o and down: the residual read, h written over it, the normed row and the norm's weight
                total += m * HIDDEN * 4 + m * HIDDEN * out_act + HIDDEN * 4
        # the quantizer launches of one pass (counted as the layers were captured)
        total += sum(quantize_bytes(m, K) for K in self.quant_widths)
        return total


def traffic_record(m, default_step):
    """ncu DRAM bytes per layer call at m rows (the sum over its launches; profiles/traffic.json), while the kernel
    sources match the capture and the step is the one captured (bf16 activations, two-output gate/up, no fused
    epilogues); else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
        if rec.get("source_hash") == source_hash() and default_step:
            return rec.get("by_m", {}).get(str(m), {}).get("traffic_bytes_per_call")
    except (OSError, ValueError):
        pass
    return None


def measure_chain(args, torch, weights, m, world, local_rank, barrier, max_over_ranks):
    """Time one row count's step: W warm-up replays, then exactly K timed steps (CUDA events on the launching
    stream, nvidia-smi clocks sampled meanwhile), then the same K steps end to end (the step's activations copied in
    from pinned host memory and its tokens copied back, every step).  Returns (chain, result dict)."""
    chain = Chain(torch, m, weights, glu=args.ffn == "glu", fused=args.fused, q8act=args.act == "q8")
    chain.capture()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        chain.g_layers.replay()
        chain.g_head.replay()
    torch.cuda.synchronize()

    # ---- device-timed region: inputs resident, K steps of graph replay ----
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local_rank) as clocks:
        barrier()
        torch.cuda.synchronize()
        clocks.mark()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            chain.g_layers.replay()
            ev[i][1].record(stream)
            chain.g_head.replay()
            ev[i][2].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        clocks.mark()
        barrier()
    ms = start.elapsed_time(end) / args.steps
    layers_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    head_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms = max_over_ranks(ms)
    bytes_step = chain.layer_bytes() + chain.head_bytes()

    # ---- end-to-end: host activations in, the step's tokens out, every step.  Two activation buffers, each with its
    # own graphs: a copy stream brings step s + 1's inputs from pinned host memory into one while step s runs on the
    # other (the copy waits for the step that last read that buffer; the step waits for its copy). ----
    x_host = torch.empty(chain.x_all.shape, dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(chain.x_all.cpu())
    idx_host = torch.empty((m,), dtype=torch.int64, pin_memory=True)
    chain.capture_second_buffer()
    graphs = ((chain.g_layers, chain.g_head), (chain.g_layers2, chain.g_head2))
    side = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_steps(k):
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            side.wait_event(used[0])
            chain.x_all_bufs[0].copy_(x_host, non_blocking=True)
            copied[0].record(side)
        for i in range(k):
            b = i % 2
            stream.wait_event(copied[b])
            graphs[b][0].replay()
            graphs[b][1].replay()
            idx_host.copy_(chain.idx, non_blocking=True)
            used[b].record(stream)
            if i + 1 < k:
                with torch.cuda.stream(side):
                    side.wait_event(used[1 - b])
                    chain.x_all_bufs[1 - b].copy_(x_host, non_blocking=True)
                    copied[1 - b].record(side)

    e2e_steps(2)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    barrier()

    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    layer_bytes = chain.layer_bytes()
    achieved = layer_bytes / (layers_ms * 1e-3) / 1e9
    traffic = traffic_record(m, not (chain.q8act or chain.glu or chain.fused))
    n_layer_calls = len(chain.layer_calls())
    res = {
        "m": m,
        "value": job_throughput(bytes_step, ms, world), "unit": "GB/s", "ms_per_step": ms,
        "us_per_gemv": ms * 1e3 / (len(chain.shapes) + 1),
        "pct_of_8TBps": 100.0 * bytes_step / (ms * 1e-3) / 8e12,
        "bytes_per_step": bytes_step, "layers_ms": layers_ms, "head_ms": head_ms,
        "launches_per_step": chain.launches_per_step(),
        "roofline": {"bound": "hbm", "kernel": f"q8 stream kernels (the {n_layer_calls} layer calls of a step, "
                     f"{chain.layer_launches()} launches, back to back"
                     + (", with their activation quantizer launches" if chain.q8act else "") + ")",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "traffic_unit": "DRAM bytes per layer call",
                     "algorithmic_bytes_per_call": layer_bytes / n_layer_calls,
                     "call_us": layers_ms * 1e3 / n_layer_calls},
        "e2e": {"value": world * bytes_step / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": chain.x_all.numel() * 2, "d2h_bytes_per_step": m * 8},
        "gpu_launches": chain.launches_per_step() * args.steps,
        "clocks": clocks.summary(),
    }
    return chain, res


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    torch.cuda.set_device(local_rank)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        return reduce_max(v, world, "cuda")

    weights = ChainWeights()
    torch.cuda.synchronize()
    results, first = [], None
    for m in args.m:
        chain, res = measure_chain(args, torch, weights, m, world, local_rank, barrier, max_over_ranks)
        results.append(res)
        if first is None:
            first = chain  # the headline chain; the CPU baseline reads its inputs back
        else:
            del chain
            torch.cuda.empty_cache()
    head, chain = results[0], first
    m = head["m"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD + (FUSED_NOTE if args.fused else GLU_NOTE if args.ffn == "glu" else "")
                   + (Q8ACT_NOTE if chain.q8act else ""), "m": m,
                   "m_timed": [r["m"] for r in results],
                   "gemvs_per_step": len(chain.shapes) + 1,
                   "launches_per_step": head["launches_per_step"],
                   "bytes_per_step": head["bytes_per_step"], "us_per_gemv": head["us_per_gemv"],
                   "pct_of_8TBps": head["pct_of_8TBps"],
                   "layers_ms": head["layers_ms"], "head_ms": head["head_ms"],
                   "operands": ("x int8 + fp32 scale per 32 values (quantized on the device), W Q8_0 (int8 + fp32 "
                                "scale per 32 rows), exact integer block sums, fp32 fold" if chain.q8act else
                                "x bf16, W Q8_0 (int8 + fp32 scale per 32 rows), fp32 accumulation"),
                   "l2": "inputs larger than L2 (9.4 GB of weights per step against 129 MB)",
                   "parallelism": f"replicas x{world}", **({"tuning": args.tune} if args.tune else {})},
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "per_m": {str(r["m"]): {k: v for k, v in r.items() if k != "m"} for r in results},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def host_case(i):
            if i < len(chain.shapes):
                q, s = chain.w[i]
                xi = [c[0] for c in chain.layer_calls() for _ in c[1]][i]
            else:
                q, s = chain.head
                xi = len(chain.x) - 1
            return (chain.x[xi].view(torch.int16).cpu().numpy().view("uint16"), q.cpu().numpy(), s.cpu().numpy())
        gbs, desc, cores, _ = oracle_sample(m, args.cpu_budget, host_case, q8act=chain.q8act)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------------------------------
# single launch shapes: the per-call sweep and the profiling case
# ---------------------------------------------------------------------------------------------------------------------

# One launch of each kind of the chain: (K, [N of each projection]) -- a multi-projection launch for q/k/v and gate/up.
LAUNCHES = {"qkv": (HIDDEN, [HIDDEN] * 3), "o": (HIDDEN, [HIDDEN]), "gateup": (HIDDEN, [FFN] * 2),
            "down": (FFN, [HIDDEN]), "head": (HIDDEN, [VOCAB])}
# The single-GEMV workloads: the attention projection, the FFN projections and the ragged tensor-parallel shapes.
SWEEP_SHAPES = [(4096, 4096), (4096, 14336), (14336, 4096), (5120, 40), (5120, 3000), (5120, 6144)]


def _weights(K, Ns, copies, seed, layout="tiled"):
    """copies x [(q, s, N) per projection]: drawn on the device, tiled unless layout is "rowmajor"."""
    import synth_inputs as si
    import q8_block_quantized_gemv_gb300 as q8
    out = []
    for c in range(copies):
        row = []
        for i, N in enumerate(Ns):
            q, s = si.device_weight(K, N, seed + 10 * c + i)
            if layout == "tiled":
                q, s = q8.tile_device(q, s, N)
            row.append((q, s, N))
        out.append(row)
    return out


def run_profile_case(args):
    """Four calls of one launch kind (constant-weights flag, as in the chain; tiled unless --layout rowmajor), for a
    profiler to capture the last.  A call the planner splits is two launches (gate/up and the head at every m), so
    `ncu ... -k regex:stream -s 6 -c 2 python bench.py --profile-case gateup --m 16` takes the fourth call's pair;
    `-s 3 -c 1` the fourth call of an unsplit kind."""
    import torch
    import synth_inputs as si
    import q8_block_quantized_gemv_gb300 as q8
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    K, Ns = LAUNCHES[args.profile_case]
    tiled = args.layout == "tiled"
    w = _weights(K, Ns, 1, 21, args.layout)[0]
    x = si.device_activations(args.m[0], K, 3)
    for _ in range(4):
        if args.profile_case == "head":
            q8.gemv_argmax(x, w[0][0], w[0][1], VOCAB, constant_weights=True, tiled=tiled)
        else:
            q8.gemv_parts(x, w, tiled=tiled, constant_weights=True)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "m": args.m[0], "layout": args.layout,
                      "device_fault": q8.device_fault()}))


def run_sweep(args):
    """µs per call and GB/s of the single-GEMV workloads at each m: every call reads its own weight copy (copies
    totalling over 4 x L2, so each call streams from HBM), calls back to back in a CUDA graph with the
    constant-weights flag, CUDA events around 5 replays after 3 warm-up replays.  One JSON line per (shape, m).
    --layout rowmajor: the weights as q8_gemv takes them ([K][Np] int8, [K/32][Np] fp32), no tiling step."""
    import torch
    import synth_inputs as si
    import q8_block_quantized_gemv_gb300 as q8
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    ms = [int(v) for v in args.sweep_m.split(",")]
    tiled = args.layout == "tiled"
    shapes = SWEEP_SHAPES
    if args.sweep_shapes:
        shapes = [tuple(int(v) for v in kn.split("x")) for kn in args.sweep_shapes.split(",")]
    for K, N in shapes:
        wb = K * padded(N) * 1.125
        copies = max(2, int(4 * l2 // wb) + 1)
        ws = _weights(K, [N], copies, 7, args.layout)
        for m in ms:
            x = si.device_activations(m, K, 3)
            y = torch.empty((m, padded(N)), dtype=torch.float32, device="cuda")
            per = max(copies, 32)

            def calls():
                for i in range(per):
                    q, s, _ = ws[i % copies][0]
                    q8.gemv(x, q, s, N, y=y, tiled=tiled, constant_weights=True)
            calls()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                calls()
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (5 * per)
            gbs = gemv_bytes(m, K, N) / (us * 1e-6) / 1e9
            print(json.dumps({"sweep": f"single GEMV, {args.layout}, back to back", "K": K, "N": N, "m": m,
                              **({"tuning": args.tune} if args.tune else {}),
                              "tflops": 2.0 * m * K * N / (us * 1e-6) / 1e12,
                              "us_per_call": us, "gbs": gbs, "frac_of_peak": gbs / peak, "peak": peak,
                              "peak_kind": peak_kind, "pct_of_8TBps": 100.0 * gbs / 8000.0,
                              "padded_gbs": padded_gemv_bytes(m, K, N) / (us * 1e-6) / 1e9}), flush=True)
            del g
        del ws
        torch.cuda.empty_cache()


def run_sweep_launches(args):
    """µs per call and GB/s of each launch kind of the decode chain (q/k/v and gate/up as multi-projection calls, o,
    down, the head with its arg-max) at each m of --sweep-m, in the chain's configuration: tiled weights, the
    constant-weights flag, calls back to back in a CUDA graph, each call on its own weight copy (copies totalling over
    4 x L2).  One JSON line per (launch, m)."""
    import torch
    import synth_inputs as si
    import q8_block_quantized_gemv_gb300 as q8
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    ms = [int(v) for v in args.sweep_m.split(",")]
    for name, (K, Ns) in LAUNCHES.items():
        wb = sum(K * padded(N) * 1.125 for N in Ns)
        copies = max(2, int(4 * l2 // wb) + 1)
        ws = _weights(K, Ns, copies, 11, "tiled")
        for m in ms:
            x = si.device_activations(m, K, 3)
            ys = [torch.empty((m, padded(N)), dtype=torch.float32, device="cuda") for N in Ns]
            idx = torch.empty((m,), dtype=torch.int64, device="cuda")
            per = max(copies, 16)

            def calls():
                for i in range(per):
                    w = ws[i % copies]
                    if name == "head":
                        q8.gemv_argmax(x, w[0][0], w[0][1], VOCAB, idx=idx, constant_weights=True, tiled=True)
                    else:
                        q8.gemv_parts(x, w, ys=ys, constant_weights=True, tiled=True)
            calls()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                calls()
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (5 * per)
            nbytes = sum(gemv_bytes(m, K, N, argmax=(name == "head")) for N in Ns) - (len(Ns) - 1) * m * K * 2
            print(json.dumps({"sweep": "chain launch kind, tiled, back to back", "launch": name, "K": K, "N": Ns,
                              "m": m, "us_per_call": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                              "frac_of_peak": nbytes / (us * 1e-6) / 1e9 / peak, "peak_kind": peak_kind,
                              **({"tuning": args.tune} if args.tune else {})}), flush=True)
            del g
        del ws
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)  # about 1 s of timed steps at m = 1, 1.3 s at m = 16
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--m", default="1,16",
                    help="activation rows per call (1..512), a comma list: the first is the headline value, every "
                         "one is timed and reported under per_m (default 1,16: the decode step's two row counts)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--ffn", choices=["parts", "glu"], default="parts",
                    help="the layers' gate/up launch: two fp32 outputs (default) or the fused gated pair")
    ap.add_argument("--fused", action="store_true",
                    help="the layers with every fusion: residual add + RMS norm after o and down, the gated pair")
    ap.add_argument("--act", choices=["bf16", "q8"], default="bf16",
                    help="activations as bf16 (default) or quantized on the device before each launch (int8 + scale "
                         "per 32, the quantized numerics)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the step: µs/call of the single-GEMV workloads, one JSON line each")
    ap.add_argument("--sweep-m", default="1,2,4,8,16", help="row counts of --sweep")
    ap.add_argument("--sweep-launches", action="store_true",
                    help="instead of the step: µs/call of each launch kind of the chain (q/k/v, o, gate/up, down, "
                         "head), one JSON line each")
    ap.add_argument("--sweep-shapes", default="",
                    help="shapes of --sweep as KxN,KxN,... (default: the attention, FFN and ragged workloads)")
    ap.add_argument("--layout", choices=["tiled", "rowmajor"], default="tiled",
                    help="weights of --sweep: the tiled storage (q8_tile_device, Q8_FLAG_TILED) or row-major as "
                         "q8_gemv takes them with no tiling step")
    ap.add_argument("--tune", default="",
                    help="planner overrides as name=value,... (q8_set_tuning: ksplit, gemm, norm_fold, split)")
    ap.add_argument("--profile-case", choices=sorted(LAUNCHES),
                    help="instead of the step: four calls of one launch kind of the step, for a profiler")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    try:
        args.m = [int(v) for v in str(args.m).split(",") if v.strip()]
    except ValueError:
        ap.error("--m takes a comma list of row counts")
    if not args.m or not all(1 <= m <= 512 for m in args.m):
        ap.error("m must be in 1..512 (more than 16 rows: the tiled storage's row groups or prefill GEMM)")
    if args.layout == "rowmajor" and args.sweep and any(int(v) > 16 for v in args.sweep_m.split(",")):
        ap.error("the row-major kernels take at most 16 rows")
    tune = {}
    for item in filter(None, args.tune.split(",")):
        name, _, value = item.partition("=")
        try:
            tune[name.strip()] = int(value)
        except ValueError:
            ap.error(f"--tune: {item!r} is not name=integer")
    args.tune = tune
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.tune:
        import q8_block_quantized_gemv_gb300 as q8
        from q8_block_quantized_gemv_gb300 import build
        build.build()
        for name, value in args.tune.items():
            q8.set_tuning(name, value)
    if args.profile_case:
        run_profile_case(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.sweep_launches:
        run_sweep_launches(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

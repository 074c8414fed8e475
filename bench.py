"""Benchmark of the NVFP4 FP4-explore hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic input of a
rollout linear (default: the FLUX.1-shaped MLP up-projection, M = 8 images x 4608
tokens = 36864, K = 3072, N = 12288), all calls through the library's C ABI:
  1. nvfp4_requant       LoRA (r = 32) merge of W [N, K] bf16 + per-tensor NVFP4
  2. nvfp4_act_quant     per-row NVFP4 of X [M, K] bf16
  3. nvfp4_gemm          Y = X W'^T + bias, block-scaled FP4 on the tensor cores
  4. bf16_gemm           the BF16 counterpart (Stage 2), for the FP4 / BF16 ratio
  5. select_contrastive  32 prompts x 96 proxy rewards -> top/bottom 12 + reward transform

Prints one JSON line.  `value` is the NVFP4 GEMM throughput in TFLOP/s (2MNK per
launch / mean CUDA-event duration of the launch over the timed steps, summed over
ranks); the re-quantization GB/s and every other kernel's roofline are reported
beside it.  Outside the timed steps it also measures, on rank 0: the same calls on
the SANA- and SD3.5-L-shaped linears (`per_config`), the iteration-shaped batch
(57 weight re-quantizations and the 442368-row 3072 -> 12288 -> 3072 chain,
`iteration`), cuBLAS's NVFP4 GEMM at 8192^3 as a reference point for the FP4 peak,
and the spread of the selected rewards against N (`evt_spread`).  `--impl reference`
times the CPU oracle on a bounded sample of the same workload instead (no GPU work).
`--gpus N` without a launcher starts N local replicas itself (torchrun).
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "flux_up"
SWEEP_CONFIGS = ["sana", "sd35_qkv", "sd35_mlp"]
REWARD_CFG = "iter"
ITER_MATRICES = 57          # weights re-quantized per iteration, alternating up / down
EVT_DELTA = 0.1             # bounded proxy perturbation used by the EVT spread report
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25  # dense NVFP4 / dense BF16 tensor rates, GB300 nominal
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20  # written between timed repetitions of the sweeps (L2 is 129 MB)


# ----------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "nvfp4_gemm": ["nvfp4_quantized_dit_gb300/csrc/gemm.cu", "nvfp4_quantized_dit_gb300/csrc/common.cuh",
                   "nvfp4_quantized_dit_gb300/csrc/gemm_epilogue.cuh"],
    "bf16_gemm": ["nvfp4_quantized_dit_gb300/csrc/gemm.cu", "nvfp4_quantized_dit_gb300/csrc/common.cuh",
                  "nvfp4_quantized_dit_gb300/csrc/gemm_epilogue.cuh"],
    "nvfp4_act_quant": ["nvfp4_quantized_dit_gb300/csrc/quant.cu", "nvfp4_quantized_dit_gb300/csrc/common.cuh"],
    "nvfp4_act_quant_prescaled": ["nvfp4_quantized_dit_gb300/csrc/quant.cu",
                                  "nvfp4_quantized_dit_gb300/csrc/common.cuh"],
    "nvfp4_requant": ["nvfp4_quantized_dit_gb300/csrc/merge_tc.cu", "nvfp4_quantized_dit_gb300/csrc/common.cuh"],
}


def dram_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since it was captured (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = source_hash(*KERNEL_SOURCES[kernel])
    with open(path) as f:
        for ln in f:
            parts = ln.split()
            if len(parts) >= 4 and not ln.startswith("#") and parts[0] == kernel and parts[1] == workload:
                return float(parts[3]) if parts[2] == cur else None
    return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region.

    The sampler runs from before the region (start() returns once the first sample has
    arrived, or after a bounded wait), begin() and end() bracket the region on the
    host clock, and stop() summarises the samples that arrived inside the bracket (or
    within one interval after it, for the query's own latency); a region shorter than
    the interval falls back to the first sample that arrived after its start (stop()
    waits for it, bounded)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (host monotonic time of arrival, CSV line)
        self.thread = None
        self.t_begin = None
        self.t_end = None
        self.interval_ms = self.INTERVAL_MS

    def start(self, wait_s: float = 5.0):
        # The recipe's 200 ms interval is the fallback should this nvidia-smi refuse a
        # shorter one (it then exits without a sample).
        for interval in (self.INTERVAL_MS, 200):
            self.interval_ms = interval
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", str(interval)],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
                return
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.monotonic() + wait_s
            while not self.lines and self.proc.poll() is None and time.monotonic() < deadline:
                time.sleep(0.01)
            if self.lines or self.proc.poll() is None:
                return
            self.thread.join(timeout=5)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.monotonic(), ln.strip()))

    def begin(self):
        self.t_begin = time.monotonic()

    def end(self):
        self.t_end = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        # A region shorter than the interval may end before its first sample: wait
        # (bounded) for one that arrives after the region's start.
        deadline = time.monotonic() + 2 * self.interval_ms / 1000.0 + 0.5
        while (self.t_begin is not None and not any(t >= self.t_begin for t, _ in self.lines)
               and self.proc.poll() is None and time.monotonic() < deadline):
            time.sleep(0.01)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        return self.summarize(self.in_region(self.lines, self.t_begin, self.t_end, self.interval_ms / 1000.0))

    @staticmethod
    def in_region(stamped, t_begin, t_end, interval_s):
        """The CSV lines of (arrival time, line) pairs that belong to the region
        [t_begin, t_end]: those that arrived from its start to one interval after its end,
        else the first one that arrived after its start.  Without a bracket, all lines."""
        if t_begin is None or t_end is None:
            return [ln for _, ln in stamped]
        inside = [ln for t, ln in stamped if t_begin <= t <= t_end + interval_s]
        if inside:
            return inside
        after = [ln for t, ln in stamped if t >= t_begin]
        return after[:1]

    @staticmethod
    def summarize(lines):
        """Median SM clock, the maximum, and the throttle reasons seen as Active, from
        nvidia-smi's CSV lines (FIELDS order, no header, no units)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def replica_command(n: int, argv) -> list:
    """The command that runs this script as n local replicas, one process per GPU
    (torchrun on this node, rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
            os.path.abspath(__file__), *argv]


# ----------------------------------------------------------------------------- workload

def algorithmic_bytes(cfg):
    M, K, N = cfg.M, cfg.K, cfg.N
    sf_w = (N + 127) // 128 * 128 * (K // 16)
    sf_a = (M + 127) // 128 * 128 * (K // 16)
    return {
        # single read of W, A, B; write of codes, scales and s_t
        "nvfp4_requant": N * K * 2 + 32 * K * 4 + N * 32 * 4 + N * K // 2 + sf_w + 4,
        # read X once; write codes, scales, one fp32 per row
        "nvfp4_act_quant": M * K * 2 + M * K // 2 + sf_a + 4 * M,
        # the same with one per-tensor scale
        "act_quant_per_tensor": M * K * 2 + M * K // 2 + sf_a + 4,
        # the same with the row amax read instead of found
        "act_quant_prescaled": M * K * 2 + M * K // 2 + sf_a + 8 * M,
    }


def host_inputs(name, seed=0, rows=None):
    import dataclasses
    import workloads
    cfg = workloads.LINEARS[name]
    if rows:
        cfg = dataclasses.replace(cfg, M=int(rows))
    host = {"X": workloads.activations(cfg, seed), "W": workloads.weight(cfg, seed),
            "bias": workloads.bias(cfg, seed)}
    host["A"], host["B"] = workloads.lora(cfg, seed)
    return cfg, host


class L2Flush:
    """Writes a buffer larger than L2 between timed repetitions."""

    def __init__(self, device):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.fill_(1.0)


def time_call(fn, reps, flush, warm=3):
    """Median CUDA-event duration (ms) of fn() on the current stream, L2 flushed
    before every repetition (outside the events)."""
    import torch
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def linear_sweep(name, device, flush, pk, fp4_peak, reps=10):
    """requant, act_quant, nvfp4_gemm and bf16_gemm of one configuration, each timed
    alone (median of `reps`, L2 flushed before each)."""
    import torch
    import nvfp4_quantized_dit_gb300 as nv
    import workloads
    cfg, host = host_inputs(name)
    d = {k: v.to(device) for k, v in host.items()}
    M, K, N = cfg.M, cfg.K, cfg.N
    wq = (torch.empty(N, K // 2, dtype=torch.uint8, device=device),
          torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device=device),
          torch.empty(1, dtype=torch.float32, device=device))
    aq = (torch.empty(M, K // 2, dtype=torch.uint8, device=device),
          torch.empty(nv.sf_bytes(M, K), dtype=torch.uint8, device=device),
          torch.empty(M, dtype=torch.float32, device=device))
    ws = torch.empty(max(nv.requant_workspace_bytes(nv.W_BF16, 32, N, K), 1), dtype=torch.uint8, device=device)
    y4 = torch.empty(M, N, dtype=torch.bfloat16, device=device)
    y16 = torch.empty(M, N, dtype=torch.bfloat16, device=device)
    ms = {
        "nvfp4_requant": time_call(lambda: nv.nvfp4_requant(d["W"], d["A"], d["B"], workloads.LORA_ALPHA,
                                                            *wq, workspace=ws), reps, flush),
        "nvfp4_act_quant": time_call(lambda: nv.nvfp4_act_quant(d["X"], *aq), reps, flush),
        "nvfp4_gemm": time_call(lambda: nv.nvfp4_gemm(aq, wq, d["bias"], out=y4), reps, flush),
        "bf16_gemm": time_call(lambda: nv.bf16_gemm(d["X"], d["W"], d["bias"], out=y16), reps, flush),
    }
    ab = algorithmic_bytes(cfg)
    flop = 2.0 * M * N * K
    t4 = flop / (ms["nvfp4_gemm"] * 1e-3) / 1e12
    t16 = flop / (ms["bf16_gemm"] * 1e-3) / 1e12
    rq = ab["nvfp4_requant"] / (ms["nvfp4_requant"] * 1e-3) / 1e9
    aqg = ab["nvfp4_act_quant"] / (ms["nvfp4_act_quant"] * 1e-3) / 1e9
    out = {"workload": cfg.description, "M": M, "K": K, "N": N,
           "kernel_ms": {k: round(v, 4) for k, v in ms.items()},
           "nvfp4_gemm_tflops": round(t4, 1), "nvfp4_gemm_frac": round(t4 / fp4_peak, 4),
           "bf16_gemm_tflops": round(t16, 1), "bf16_gemm_frac": round(t16 / pk["bf16_tflops"], 4),
           "fp4_over_bf16": round(t4 / t16, 3),
           "requant_gbs": round(rq, 1), "requant_frac": round(rq / pk["hbm_gbs"], 4),
           "act_quant_gbs": round(aqg, 1), "act_quant_frac": round(aqg / pk["hbm_gbs"], 4)}
    del d, wq, aq, ws, y4, y16
    torch.cuda.empty_cache()
    return out


def iteration_sweep(device, pk, fp4_peak, reps=3):
    """The iteration-shaped batch: ITER_MATRICES LoRA merges + re-quantizations of
    [12288, 3072] / [3072, 12288] weights back to back (each its own buffer in HBM,
    4.3 GB in all, so nothing is served from L2), then the 442368-row chain
    act_quant -> nvfp4_gemm -> act_quant -> nvfp4_gemm (3072 -> 12288 -> 3072)."""
    import torch
    import nvfp4_quantized_dit_gb300 as nv
    import workloads
    up, dn = workloads.LINEARS["iter_up"], workloads.LINEARS["iter_down"]
    shapes = [up, dn]
    base = [workloads.weight(c, 0).to(device) for c in shapes]
    lora = [tuple(t.to(device) for t in workloads.lora(c, 0)) for c in shapes]
    Ws = [base[i % 2].clone() for i in range(ITER_MATRICES)]
    outs = []
    for i in range(ITER_MATRICES):
        c = shapes[i % 2]
        outs.append((torch.empty(c.N, c.K // 2, dtype=torch.uint8, device=device),
                     torch.empty(nv.sf_bytes(c.N, c.K), dtype=torch.uint8, device=device),
                     torch.empty(1, dtype=torch.float32, device=device)))
    wss = [torch.empty(nv.requant_workspace_bytes(nv.W_BF16, 32, c.N, c.K), dtype=torch.uint8, device=device)
           for c in shapes]

    def sweep():
        for i in range(ITER_MATRICES):
            A, B = lora[i % 2]
            nv.nvfp4_requant(Ws[i], A, B, workloads.LORA_ALPHA, *outs[i], workspace=wss[i % 2])

    sweep()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        sweep()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    sweep_ms = statistics.median(ts)
    rq_bytes = sum(algorithmic_bytes(shapes[i % 2])["nvfp4_requant"] for i in range(ITER_MATRICES))
    rq_gbs = rq_bytes / (sweep_ms * 1e-3) / 1e9
    requant = {"matrices": ITER_MATRICES, "ms": round(sweep_ms, 4),
               "us_per_matrix": round(sweep_ms * 1e3 / ITER_MATRICES, 2), "gbs": round(rq_gbs, 1),
               "frac": round(rq_gbs / pk["hbm_gbs"], 4),
               "floor_ms": round(rq_bytes / (pk["hbm_gbs"] * 1e9) * 1e3, 4)}
    w_up, w_dn = outs[0], outs[1]
    del Ws, wss
    torch.cuda.empty_cache()

    # the chain over the whole batch (inputs drawn on the device: timing only)
    M = up.M
    X = workloads.activations_on_device(up, device, 0)
    bias_up, bias_dn = workloads.bias(up, 0).to(device), workloads.bias(dn, 0).to(device)
    xq = (torch.empty(M, up.K // 2, dtype=torch.uint8, device=device),
          torch.empty(nv.sf_bytes(M, up.K), dtype=torch.uint8, device=device),
          torch.empty(M, dtype=torch.float32, device=device))
    H = torch.empty(M, up.N, dtype=torch.bfloat16, device=device)
    hq = (torch.empty(M, dn.K // 2, dtype=torch.uint8, device=device),
          torch.empty(nv.sf_bytes(M, dn.K), dtype=torch.uint8, device=device),
          torch.empty(M, dtype=torch.float32, device=device))
    Y = torch.empty(M, dn.N, dtype=torch.bfloat16, device=device)
    h_amax = torch.empty(M, dtype=torch.float32, device=device)
    # The up-projection hands its output's row amax to the hidden state's quantization,
    # which then streams H once (nvfp4_gemm_rowamax -> nvfp4_act_quant_prescaled).
    calls = [("act_quant_x", lambda: nv.nvfp4_act_quant(X, *xq)),
             ("gemm_up", lambda: nv.nvfp4_gemm_rowamax(xq, w_up, bias_up, out=H, row_amax=h_amax)),
             ("act_quant_hidden", lambda: nv.nvfp4_act_quant_prescaled(H, h_amax, *hq)),
             ("gemm_down", lambda: nv.nvfp4_gemm(hq, w_dn, bias_dn, out=Y))]
    for _, fn in calls:
        fn()
    torch.cuda.synchronize()
    per = {n: [] for n, _ in calls}
    total = []
    for _ in range(reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        ev[0].record()
        for i, (_, fn) in enumerate(calls):
            fn()
            ev[i + 1].record()
        ev[-1].synchronize()
        for i, (n, _) in enumerate(calls):
            per[n].append(ev[i].elapsed_time(ev[i + 1]))
        total.append(ev[0].elapsed_time(ev[-1]))
    per = {n: statistics.median(v) for n, v in per.items()}
    chain_ms = statistics.median(total)
    # For comparison: the hidden state's quantization without the handed-over row amax
    # (nvfp4_act_quant, which finds each row's amax itself), and the up-projection
    # without the row-amax epilogue.
    alt = {"act_quant_hidden_row_buffered": lambda: nv.nvfp4_act_quant(H, *hq),
           "gemm_up_plain": lambda: nv.nvfp4_gemm(xq, w_up, bias_up, out=H)}
    alt_ms = {}
    for n, fn in alt.items():
        fn()
        vs = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            vs.append(a.elapsed_time(b))
        alt_ms[n] = statistics.median(vs)
    flop = 2.0 * M * up.N * up.K
    by_x = algorithmic_bytes(up)["nvfp4_act_quant"]
    by_h = algorithmic_bytes(dn)["nvfp4_act_quant"]
    chain = {"rows": M, "kernel_ms": {n: round(v, 4) for n, v in per.items()}, "ms": round(chain_ms, 4),
             "gemm_up_tflops": round(flop / (per["gemm_up"] * 1e-3) / 1e12, 1),
             "gemm_down_tflops": round(flop / (per["gemm_down"] * 1e-3) / 1e12, 1),
             "gemm_frac": round(2 * flop / ((per["gemm_up"] + per["gemm_down"]) * 1e-3) / 1e12 / fp4_peak, 4),
             "act_quant_hidden_gbs": round(by_h / (per["act_quant_hidden"] * 1e-3) / 1e9, 1),
             "act_quant_hidden_frac": round(by_h / (per["act_quant_hidden"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
             "act_quant_hidden_calls": "nvfp4_gemm_rowamax (up) -> nvfp4_act_quant_prescaled",
             "compare_ms": {n: round(v, 4) for n, v in alt_ms.items()},
             "act_quant_x_gbs": round(by_x / (per["act_quant_x"] * 1e-3) / 1e9, 1),
             "chain_tflops": round(2 * flop / (chain_ms * 1e-3) / 1e12, 1)}
    del X, xq, H, hq, Y, h_amax
    torch.cuda.empty_cache()
    return {"requant_sweep": requant, "chain": chain}


def cublas_nvfp4_peak(device, size=8192, reps=10):
    """cuBLAS's NVFP4 GEMM (torch._scaled_mm) at size^3 on random operand bytes, best of
    `reps`: a measured reference point for the FP4 tensor rate.  None if torch cannot
    run it."""
    import torch
    try:
        g = torch.Generator(device=device)
        g.manual_seed(0)
        a = torch.randint(0, 256, (size, size // 2), dtype=torch.uint8, device=device, generator=g)
        w = torch.randint(0, 256, (size, size // 2), dtype=torch.uint8, device=device, generator=g)
        nsf = size * size // 16
        sa = torch.randint(0x30, 0x40, (nsf,), dtype=torch.uint8, device=device, generator=g)
        sw = torch.randint(0x30, 0x40, (nsf,), dtype=torch.uint8, device=device, generator=g)
        A4, W4 = a.view(torch.float4_e2m1fn_x2), w.view(torch.float4_e2m1fn_x2)
        SA, SW = sa.view(torch.float8_e4m3fn), sw.view(torch.float8_e4m3fn)

        def fn():
            return torch._scaled_mm(A4, W4.t(), SA, SW, out_dtype=torch.bfloat16)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        # This library's nvfp4_gemm on the same operand bytes (the scale bytes taken as its
        # blocked layout; per-row and per-tensor scales 1), timed the same way.
        import nvfp4_quantized_dit_gb300 as nv
        ones = torch.ones(size, dtype=torch.float32, device=device)
        y = torch.empty(size, size, dtype=torch.bfloat16, device=device)

        def ours():
            nv.nvfp4_gemm((a, sa, ones), (w, sw, ones[:1]), out=y)
        for _ in range(3):
            ours()
        torch.cuda.synchronize()
        best_ours = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ours()
            e1.record()
            e1.synchronize()
            best_ours = min(best_ours, e0.elapsed_time(e1))
        return {"tflops": round(2.0 * size ** 3 / (best * 1e-3) / 1e12, 1), "size": size, "reps": reps,
                "ours_tflops": round(2.0 * size ** 3 / (best_ours * 1e-3) / 1e12, 1),
                "how": "torch._scaled_mm float4_e2m1fn_x2 x float4_e2m1fn_x2, float8_e4m3fn block scales, "
                       "bf16 out, best of reps (CUDA events); ours_tflops: nvfp4_gemm on the same bytes"}
    except Exception as e:  # noqa: BLE001 - a reference point only
        return {"tflops": None, "unavailable": repr(e)[:200]}


def evt_report(device, P=2048, K=24, delta=EVT_DELTA, seed=0):
    """Spread of the selected rewards against N (AI Trends summary, the paragraph on
    extreme value theory: the expected reward range W of the explored group grows like
    2 sigma sqrt(2 log N), less 4 Delta for a perturbation bounded by Delta).  True
    rewards ~ N(0, 1) for P prompts x N seeds; the proxy (standing in for the FP4
    rollout's reward) adds noise uniform in [-Delta, Delta]; select_contrastive picks
    on the proxy.  Reported per N: the mean true-reward gap between the best and worst
    proxy-selected seeds, the mean true range max - min, and the page's expression."""
    import torch
    import nvfp4_quantized_dit_gb300 as nv
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    rows = []
    for N in (24, 48, 96, 192, 384, 768, 1024):
        r = torch.randn(P, N, generator=g, device=device)
        proxy = r + (torch.rand(P, N, generator=g, device=device) * 2 - 1) * delta
        idx, _ = nv.select_contrastive(proxy, K, with_transform=False)
        top, bot = idx[:, 0].long(), idx[:, K // 2].long()
        ar = torch.arange(P, device=device)
        gap = (r[ar, top] - r[ar, bot]).mean().item()
        rng = (r.max(dim=1).values - r.min(dim=1).values).mean().item()
        rows.append({"N": N, "selected_gap": round(gap, 4), "true_range": round(rng, 4),
                     "page_expression": round(2 * math.sqrt(2 * math.log(N)) - 4 * delta, 4)})
    return {"prompts": P, "K": K, "delta": delta, "rows": rows}


# ----------------------------------------------------------------------------- our arm

def dit_block_report(device, pk, fp4_peak, reps=5, images=None):
    """The FLUX.1-shaped synthetic DiT block (8 images x 4608 tokens, D 3072, 24 heads):
    one nvfp4_dit_block call on resident inputs, median of `reps` (CUDA events on the
    launching stream; the activations, 226 MB, exceed L2), and its attention alone.
    FLOPs: the four linears 24 T D^2 (NVFP4), the attention 4 B S^2 D (bf16).  `frac` is
    the time both would take at the measured peaks (FP4 = bf16 x the nominal ratio) over
    the measured time."""
    import torch
    import nvfp4_quantized_dit_gb300 as nv
    import workloads
    cfg = workloads.BLOCKS["flux"]
    if images is not None:
        cfg = dataclasses.replace(cfg, B=images, description=f"{cfg.description}; {images} image(s)")
    B, S, D, H = cfg.B, cfg.S, cfg.D, cfg.H
    T = B * S
    x = workloads.block_input(cfg, seed=0).to(device)
    wts = workloads.block_weights(cfg, seed=0)
    weights = []
    for name in workloads.BLOCK_LINEARS:
        W, b = wts[name]
        weights.append((*nv.nvfp4_requant(W.to(device)), b.to(device)))
    out = torch.empty_like(x)
    ws = torch.empty(nv.dit_block_workspace_bytes(B, S, D, H), dtype=torch.uint8, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(1)
    qkv = torch.randn(T, 3 * D, generator=g, device=device).to(torch.bfloat16)
    o = torch.empty(T, D, dtype=torch.bfloat16, device=device)
    wsa = torch.empty(nv.dit_attention_workspace_bytes(B, S, D, H), dtype=torch.uint8, device=device)

    def med(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        vs = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            vs.append(e0.elapsed_time(e1))
        return statistics.median(vs)
    block_ms = med(lambda: nv.nvfp4_dit_block(x, B, S, H, weights, out=out, workspace=ws))
    attn_ms = med(lambda: nv.nvfp4_dit_attention(qkv, B, S, H, o=o, workspace=wsa))
    lin_flop = 24.0 * T * D * D
    attn_flop = 4.0 * B * S * S * D
    ideal_ms = (lin_flop / (fp4_peak * 1e12) + attn_flop / (pk["bf16_tflops"] * 1e12)) * 1e3
    res = {"workload": cfg.description, "ms": round(block_ms, 3),
           "tflops": round((lin_flop + attn_flop) / (block_ms * 1e-3) / 1e12, 1),
           "attention_ms": round(attn_ms, 3),
           "attention_tflops": round(attn_flop / (attn_ms * 1e-3) / 1e12, 1),
           "rest_ms": round(block_ms - attn_ms, 3),
           "rest_linear_tflops": round(lin_flop / ((block_ms - attn_ms) * 1e-3) / 1e12, 1),
           "flop": {"linears_nvfp4": lin_flop, "attention_bf16": attn_flop},
           "frac": round(ideal_ms / block_ms, 4), "reps": reps,
           "device_status": nv.nvfp4_device_status()}
    del x, weights, out, ws, qkv, o, wsa
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    import nvfp4_quantized_dit_gb300 as nv
    import workloads

    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    nv.library()

    cfg, host = host_inputs(args.config, rows=args.rows)
    rcfg = workloads.REWARDS[REWARD_CFG]
    host["rewards"] = workloads.rewards(rcfg, 0)
    dev = {k: v.to(device) for k, v in host.items()}
    M, K, N = cfg.M, cfg.K, cfg.N
    Kr = rcfg.K
    # outputs, allocated once
    w_codes = torch.empty(N, K // 2, dtype=torch.uint8, device=device)
    w_sf = torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device=device)
    w_st = torch.empty(1, dtype=torch.float32, device=device)
    a_codes = torch.empty(M, K // 2, dtype=torch.uint8, device=device)
    a_sf = torch.empty(nv.sf_bytes(M, K), dtype=torch.uint8, device=device)
    a_s = torch.empty(M, dtype=torch.float32, device=device)
    Y4 = torch.empty(M, N, dtype=torch.bfloat16, device=device)
    Y16 = torch.empty(M, N, dtype=torch.bfloat16, device=device)
    idx = torch.empty(rcfg.P, Kr, dtype=torch.int32, device=device)
    rr = torch.empty(rcfg.P, Kr, dtype=torch.float32, device=device)
    # requant's scratch (the tensor-core merge's split operands and norms), allocated once
    ws_bytes = nv.requant_workspace_bytes(nv.W_BF16, 32, N, K)
    rq_ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
    names = ["nvfp4_requant", "nvfp4_act_quant", "nvfp4_gemm", "bf16_gemm", "select_contrastive"]
    # requant: split kernel, then the fused amax + quantize kernel (tensor-core merge)
    launches_per_step = {"nvfp4_requant": 2, "nvfp4_act_quant": 1, "nvfp4_gemm": 1, "bf16_gemm": 1,
                         "select_contrastive": 2}

    def step(d, events=None, y4=Y4, sel=(idx, rr)):
        def mark(i):
            if events is not None:
                events[i].record()
        mark(0)
        nv.nvfp4_requant(d["W"], d["A"], d["B"], workloads.LORA_ALPHA, w_codes, w_sf, w_st,
                         workspace=rq_ws)
        mark(1)
        nv.nvfp4_act_quant(d["X"], a_codes, a_sf, a_s)
        mark(2)
        nv.nvfp4_gemm((a_codes, a_sf, a_s), (w_codes, w_sf, w_st), d["bias"], out=y4)
        mark(3)
        nv.bf16_gemm(d["X"], d["W"], d["bias"], out=Y16)
        mark(4)
        nv.select_contrastive(d["rewards"], Kr, True, True, sel[0], sel[1])
        mark(5)

    # ---- device-resident timing
    for _ in range(args.warmup):
        step(dev)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(device.index)
    clocks.start()
    barrier(world, device)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks.begin()
    t0.record()
    for s in range(args.steps):
        step(dev, ev[s])
    t1.record()
    torch.cuda.synchronize()
    clocks.end()
    barrier(world, device)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, device)
    per = {n: statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps))
           for i, n in enumerate(names)}
    per = {n: max_over_ranks(v, world, device) for n, v in per.items()}

    # ---- a variant outside the step: NVFP4 of X with one per-tensor scale (two passes
    # over X)
    xq_codes = torch.empty_like(a_codes)
    xq_sf = torch.empty_like(a_sf)
    xq_st = torch.empty(1, dtype=torch.float32, device=device)

    def per_tensor():
        nv.nvfp4_act_quant_tensor(dev["X"], xq_codes, xq_sf, xq_st)

    for _ in range(3):
        per_tensor()
    torch.cuda.synchronize()
    vt = []
    for _ in range(10):
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        v0.record()
        per_tensor()
        v1.record()
        v1.synchronize()
        vt.append(v0.elapsed_time(v1))
    per_tensor_ms = max_over_ranks(statistics.median(vt), world, device)

    # ---- variants of the step's act_quant and GEMM with the row amax handed over: the
    # GEMM's epilogue reduces its output rows' amax (nvfp4_gemm_rowamax), and a
    # streaming quantizer takes it (nvfp4_act_quant_prescaled, here on X with its own
    # row amax, as if X came from such a GEMM)
    x_amax = dev["X"].float().abs().amax(dim=1)
    y_amax = torch.empty(M, dtype=torch.float32, device=device)
    variant_ms = {}
    for n, fn in {"act_quant_prescaled": lambda: nv.nvfp4_act_quant_prescaled(dev["X"], x_amax, xq_codes, xq_sf,
                                                                                a_s),
                  "nvfp4_gemm_rowamax": lambda: nv.nvfp4_gemm_rowamax((a_codes, a_sf, a_s),
                                                                      (w_codes, w_sf, w_st), dev["bias"],
                                                                      out=Y4, row_amax=y_amax)}.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        vt = []
        for _ in range(10):
            v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            v0.record()
            fn()
            v1.record()
            v1.synchronize()
            vt.append(v0.elapsed_time(v1))
        variant_ms[n] = max_over_ranks(statistics.median(vt), world, device)
    # a_s is act_quant's own output again (the prescaled call above rewrote it identically)
    del xq_codes, xq_sf, x_amax, y_amax

    # ---- end to end: pinned host inputs in, result out, every step
    extras = {}
    if args.no_e2e:
        e2e_ms = float("nan")
        h2d = d2h = 0
    else:
        e2e_ms, h2d, d2h, copy_rates = run_e2e(args, host, dev, step, Y4, idx, rr, M, N, rcfg, Kr, world, device)
        extras["copy_rates"] = copy_rates
    status = nv.nvfp4_device_status()

    # ---- measurements outside the step (rank 0)
    if rank == 0:
        pk, _ = peaks()
        fp4_peak = pk["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
        flush = L2Flush(device)
        if not args.no_per_config:
            extras["per_config"] = {n: linear_sweep(n, device, flush, pk, fp4_peak)
                                    for n in SWEEP_CONFIGS if n != args.config}
        if not args.no_iteration:
            extras["iteration"] = iteration_sweep(device, pk, fp4_peak)
        if not args.no_peak_probe:
            extras["cublas_nvfp4_8192"] = cublas_nvfp4_peak(device)
        extras["evt_spread"] = evt_report(device)
        if not args.no_block:
            extras["dit_block"] = dit_block_report(device, pk, fp4_peak)
        extras["device_status_after_extras"] = nv.nvfp4_device_status()
    return report(args, cfg, rcfg, host, per, elapsed_ms, e2e_ms, h2d, d2h, status, clk, world, rank,
                  launches_per_step, per_tensor_ms, extras, variant_ms)


def run_e2e(args, host, dev, step, Y4, idx, rr, M, N, rcfg, Kr, world, device):
    """End to end through the public calls with host buffers: every step copies its
    inputs from pinned host memory and its results (Y of the NVFP4 GEMM and the
    selection) back to pinned host memory, all inside the timed region.  The copies
    run on their own streams with two sets of device buffers, so step i's kernels
    overlap step i+1's input copy and step i-1's result copy, as a serving loop would
    run them."""
    import torch
    nbuf = 2
    pinned = {k: v.pin_memory() for k, v in host.items()}
    dev_in = [{k: torch.empty_like(v) for k, v in dev.items()} for _ in range(nbuf)]
    y_dev = [Y4] + [torch.empty_like(Y4) for _ in range(nbuf - 1)]
    sel_dev = [(idx, rr)] + [(torch.empty_like(idx), torch.empty_like(rr)) for _ in range(nbuf - 1)]
    y_host = [torch.empty(M, N, dtype=torch.bfloat16, pin_memory=True) for _ in range(nbuf)]
    sel_host = [(torch.empty(rcfg.P, Kr, dtype=torch.int32, pin_memory=True),
                 torch.empty(rcfg.P, Kr, dtype=torch.float32, pin_memory=True)) for _ in range(nbuf)]
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = y_host[0].numel() * 2 + sel_host[0][0].numel() * 4 + sel_host[0][1].numel() * 4
    s_in, s_run, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # inputs of buffer b landed
    ev_run = [torch.cuda.Event() for _ in range(nbuf)]   # kernels done with buffer b
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]   # results of buffer b copied out

    def e2e_step(i):
        b = i % nbuf
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_run[b])       # the step two back no longer reads these inputs
            for k, v in pinned.items():
                dev_in[b][k].copy_(v, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b])
            s_run.wait_event(ev_out[b])      # the step two back has been read out
            step(dev_in[b], y4=y_dev[b], sel=sel_dev[b])
            ev_run[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            y_host[b].copy_(y_dev[b], non_blocking=True)
            sel_host[b][0].copy_(sel_dev[b][0], non_blocking=True)
            sel_host[b][1].copy_(sel_dev[b][1], non_blocking=True)
            ev_out[b].record(s_out)

    def run(n):
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(cur)
        for s in (s_in, s_run, s_out):
            s.wait_event(start)
        for i in range(n):
            e2e_step(i)
        for s in (s_in, s_run, s_out):
            cur.wait_stream(s)
        stop.record(cur)
        return start, stop

    run(args.warmup)
    torch.cuda.synchronize()
    barrier(world, device)
    e0, e1 = run(args.steps)
    torch.cuda.synchronize()
    barrier(world, device)
    elapsed = max_over_ranks(e0.elapsed_time(e1), world, device)
    # The plain pinned-memory copy rates on this machine, for the same buffers, one copy at a
    # time on one stream (best of 3): what bounds the end-to-end step.
    def best_of(fn, nbytes, reps=3):
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        return round(nbytes / (best * 1e-3) / 1e9, 1)
    rates = {"d2h_gbs": best_of(lambda: y_host[0].copy_(y_dev[0], non_blocking=True), y_host[0].numel() * 2),
             "h2d_gbs": best_of(lambda: dev_in[0]["X"].copy_(pinned["X"], non_blocking=True),
                                pinned["X"].numel() * pinned["X"].element_size()),
             "how": "one pinned-host copy at a time (Y out, X in), best of 3, CUDA events"}
    return elapsed, h2d, d2h, rates


def workload_name(cfg, rcfg):
    return (f"{cfg.description}: M={cfg.M} K={cfg.K} N={cfg.N} + LoRA r=32 requant + "
            f"{rcfg.P}x{rcfg.N} reward selection (K={rcfg.K})")


def bench_config(cfg, rcfg, world):
    """The `config` object of the JSON line, the same for both arms."""
    x_mb = cfg.M * cfg.K * 2 / 1e6
    y_mb = cfg.M * cfg.N * 2 / 1e6
    return {"workload": workload_name(cfg, rcfg),
            "M": cfg.M, "K": cfg.K, "N": cfg.N, "lora_rank": 32, "prompts": rcfg.P, "seeds": rcfg.N,
            "selected": rcfg.K, "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2 within a step (X {x_mb:.0f} MB read, Y {y_mb:.0f} MB "
                  "written twice per step)"}


def report(args, cfg, rcfg, host, per, elapsed_ms, e2e_ms, h2d, d2h, status, clk, world, rank,
           launches_per_step, per_tensor_ms, extras, variant_ms):
    if rank != 0:
        return None
    M, K, N = cfg.M, cfg.K, cfg.N
    Kr = rcfg.K

    pk, pk_kind = peaks()
    fp4_peak = pk["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
    gemm_flops = 2.0 * M * N * K
    ab = algorithmic_bytes(cfg)
    tflops4 = gemm_flops / (per["nvfp4_gemm"] * 1e-3) / 1e12
    tflops16 = gemm_flops / (per["bf16_gemm"] * 1e-3) / 1e12
    rq_gbs = ab["nvfp4_requant"] / (per["nvfp4_requant"] * 1e-3) / 1e9
    aq_gbs = ab["nvfp4_act_quant"] / (per["nvfp4_act_quant"] * 1e-3) / 1e9
    aqp_gbs = ab["act_quant_prescaled"] / (variant_ms["act_quant_prescaled"] * 1e-3) / 1e9
    ms_per_step = elapsed_ms / args.steps
    e2e_ms_step = e2e_ms / args.steps

    # The captured traffic is of the full workload: a --rows run has none.
    workload = args.config if not args.rows else f"{args.config}@{args.rows}"

    def roof(bound, achieved, peak, unit, kernel):
        return {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": dram_traffic(kernel, workload)}

    cub = extras.get("cublas_nvfp4_8192") or {}
    out = {
        "metric": "NVFP4 GEMM TFLOP/s (FLUX.1-shaped linears) & re-quant GB/s, % of roofline",
        "value": round(tflops4 * world, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e4m3 block scale) -> fp32 accumulate -> bf16",
        "data": "synthetic (seeded; model-shaped weights, activations, LoRA r=32, rewards)",
        "config": bench_config(cfg, rcfg, world),
        "value_basis": "mean CUDA-event duration of the nvfp4_gemm launch inside the timed steps",
        "requant_gbs": round(rq_gbs, 1),
        "act_quant_gbs": round(aq_gbs, 1),
        "bf16_gemm_tflops": round(tflops16, 1),
        "fp4_over_bf16": round(tflops4 / tflops16, 3),
        "select_us": round(per["select_contrastive"] * 1e3, 2),
        "kernel_ms": {n: round(v, 4) for n, v in per.items()},
        "roofline": roof("tensor", tflops4, fp4_peak, "TFLOP/s", "nvfp4_gemm"),
        "rooflines": {
            "nvfp4_gemm": roof("tensor", tflops4, fp4_peak, "TFLOP/s", "nvfp4_gemm"),
            "bf16_gemm": roof("tensor", tflops16, pk["bf16_tflops"], "TFLOP/s", "bf16_gemm"),
            "nvfp4_requant": roof("hbm", rq_gbs, pk["hbm_gbs"], "GB/s", "nvfp4_requant"),
            "nvfp4_act_quant": roof("hbm", aq_gbs, pk["hbm_gbs"], "GB/s", "nvfp4_act_quant"),
        },
        "peak_source": f"{pk_kind}: bf16 {pk['bf16_tflops']} TFLOP/s x {NOMINAL_FP4_OVER_BF16:g} "
                       f"(nominal dense NVFP4/BF16) for NVFP4; HBM {pk['hbm_gbs']} GB/s",
        "nvfp4_vs_cublas_peak": None if not cub.get("tflops") else {
            "cublas_8192_tflops": cub["tflops"], "ours_8192_tflops": cub.get("ours_tflops"),
            "frac": round(tflops4 / cub["tflops"], 4), "how": cub["how"]},
        "e2e": None if args.no_e2e else {
            "value": round(gemm_flops / (e2e_ms_step * 1e-3) / 1e12 * world, 2), "unit": "TFLOP/s",
            "ms_per_step": round(e2e_ms_step, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copy_rates": extras.get("copy_rates")},
        "variants": {"act_quant_per_tensor": {
            "call": "nvfp4_act_quant_tensor (one per-tensor scale, two passes over X)",
            "ms": round(per_tensor_ms, 4),
            "gbs": round(ab["act_quant_per_tensor"] / (per_tensor_ms * 1e-3) / 1e9, 1),
            "frac": round(ab["act_quant_per_tensor"] / (per_tensor_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)},
            "act_quant_prescaled": {
                "call": "nvfp4_act_quant_prescaled (row amax handed over, e.g. by nvfp4_gemm_rowamax, "
                        "instead of reduced over the row)",
                "ms": round(variant_ms["act_quant_prescaled"], 4),
                "gbs": round(aqp_gbs, 1),
                "frac": round(aqp_gbs / pk["hbm_gbs"], 4),
                "roofline": roof("hbm", aqp_gbs, pk["hbm_gbs"], "GB/s", "nvfp4_act_quant_prescaled")},
            "nvfp4_gemm_rowamax": {
                "call": "nvfp4_gemm_rowamax (nvfp4_gemm plus the output rows' amax from the epilogue)",
                "ms": round(variant_ms["nvfp4_gemm_rowamax"], 4),
                "tflops": round(gemm_flops / (variant_ms["nvfp4_gemm_rowamax"] * 1e-3) / 1e12, 1)}},
        "gpu_launches": sum(launches_per_step.values()) * args.steps,
        "device_status": status,
        "clocks": clk,
    }
    for k in ("per_config", "iteration", "dit_block", "evt_spread", "device_status_after_extras"):
        if k in extras:
            out[k] = extras[k]
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, host, rcfg, budget_s=args.cpu_budget)
    return out


# ----------------------------------------------------------------------------- oracle legs

def _timed(fn):
    t = time.perf_counter()
    fn()
    return time.perf_counter() - t


def cpu_baseline(cfg, host, rcfg, budget_s=12.0):
    """The oracle, as it stands, on the host cores: NVFP4 GEMM over a row sample
    sized to about `budget_s` seconds (the weights quantized by the oracle), plus the
    quantizers (all cores and one core) and the selection (one core)."""
    import numpy as np
    import oracle
    import workloads
    oracle.build()
    cores = oracle.num_threads()
    wb = workloads.bf16_bits(host["W"])
    A, B = host["A"].numpy(), host["B"].numpy()
    ab = algorithmic_bytes(cfg)
    legs = {}
    t_all = _timed(lambda: oracle.requant(wb, A, B, workloads.LORA_ALPHA))
    oracle.set_num_threads(1)
    try:
        t_one = _timed(lambda: oracle.requant(wb, A, B, workloads.LORA_ALPHA))
        xs = workloads.bf16_bits(host["X"][:2048])
        aq_bytes = ab["nvfp4_act_quant"] * 2048 / cfg.M
        t_aq1 = _timed(lambda: oracle.act_quant(xs))
        rw = workloads.rewards(rcfg, 0).numpy()
        t_sel = min(_timed(lambda: oracle.select_contrastive(rw, rcfg.K)) for _ in range(5))
    finally:
        oracle.set_num_threads(cores)
    t_aqn = _timed(lambda: oracle.act_quant(xs))
    legs["requant_gbs"] = {"all_cores": round(ab["nvfp4_requant"] / t_all / 1e9, 4),
                           "one_core": round(ab["nvfp4_requant"] / t_one / 1e9, 4),
                           "sample": f"full weight [{cfg.N}, {cfg.K}], LoRA r=32 merge + quantize"}
    legs["act_quant_gbs"] = {"all_cores": round(aq_bytes / t_aqn / 1e9, 4),
                             "one_core": round(aq_bytes / t_aq1 / 1e9, 4),
                             "sample": f"2048 rows x K={cfg.K}"}
    legs["select_us_one_core"] = round(t_sel * 1e6, 1)

    wc, wsf, ws = oracle.requant(wb, A, B, workloads.LORA_ALPHA)
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(cfg.M, 16, replace=False))
    ac, asf, a_s = oracle.act_quant(workloads.bf16_bits(host["X"])[probe])
    t = time.perf_counter()
    oracle.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, workloads.bf16_bits(host["bias"]))
    per_row = (time.perf_counter() - t) / len(probe)
    nrows = int(max(16, min(4096, budget_s / max(per_row, 1e-6))))
    rows = np.sort(rng.choice(cfg.M, nrows, replace=False))
    ac, asf, a_s = oracle.act_quant(workloads.bf16_bits(host["X"])[rows])
    t = time.perf_counter()
    oracle.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, workloads.bf16_bits(host["bias"]))
    dt = time.perf_counter() - t
    flops = 2.0 * nrows * cfg.N * cfg.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"fp64 NVFP4 GEMM oracle on {nrows} sampled rows x N={cfg.N} x K={cfg.K} "
                      f"({dt:.1f} s), weights re-quantized by the oracle",
            "legs": legs}


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload (requant of the full weight, act_quant + GEMM of 32 rows, selection)."""
    import numpy as np
    import oracle
    import workloads
    world, rank, _ = dist_setup()
    if rank != 0:
        return None
    oracle.build()
    cfg, host = host_inputs(args.config, rows=args.rows)
    rcfg = workloads.REWARDS[REWARD_CFG]
    host["rewards"] = workloads.rewards(rcfg)
    wb = workloads.bf16_bits(host["W"])
    xb_all = workloads.bf16_bits(host["X"])
    bias = workloads.bf16_bits(host["bias"])
    rows_per_step = 32
    rng = np.random.default_rng(0)

    def step():
        wc, wsf, ws = oracle.requant(wb, host["A"].numpy(), host["B"].numpy(), workloads.LORA_ALPHA)
        rows = np.sort(rng.choice(cfg.M, rows_per_step, replace=False))
        ac, asf, a_s = oracle.act_quant(xb_all[rows])
        t = time.perf_counter()
        oracle.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, bias)
        g = time.perf_counter() - t
        oracle.select_contrastive(host["rewards"].numpy(), rcfg.K)
        return g

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    gemm_s = sum(step() for _ in range(args.steps))
    total = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * cfg.N * cfg.K * args.steps
    v = flops / gemm_s / 1e12
    return {
        "impl": "reference",
        "metric": "NVFP4 GEMM TFLOP/s (FLUX.1-shaped linears) & re-quant GB/s, % of roofline",
        "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp64 over NVFP4 values (oracle)", "data": "synthetic (seeded)",
        "config": bench_config(cfg, rcfg, world),
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"per step: full-weight requant, act_quant + fp64 GEMM of "
                                   f"{rows_per_step} sampled rows, selection"},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def parse_args(argv=None):
    import workloads
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=[HEADLINE, *SWEEP_CONFIGS], default=HEADLINE,
                    help="the rollout linear of the timed step (default: the FLUX.1 up-projection)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end phase")
    ap.add_argument("--no-per-config", action="store_true", help="skip the SANA / SD3.5-L sweeps")
    ap.add_argument("--no-iteration", action="store_true", help="skip the iteration-shaped batch")
    ap.add_argument("--no-peak-probe", action="store_true", help="skip cuBLAS's NVFP4 8192^3 reference")
    ap.add_argument("--no-block", action="store_true", help="skip the FLUX.1-shaped DiT block timing")
    ap.add_argument("--block-only", action="store_true",
                    help="time only the DiT block (one JSON object; for profiling the block's kernels)")
    ap.add_argument("--block-images", type=int, default=None,
                    help="images of the block-only run (default: the workload's 8)")
    ap.add_argument("--rows", type=int, default=None,
                    help="override M (a smaller case for profiling; the default is the config's)")
    args = ap.parse_args(argv)
    assert args.config in workloads.LINEARS
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    return args


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # no launcher: start the replicas here, one process per GPU, and pass on
        # their exit status (rank 0 prints the line)
        return subprocess.call(replica_command(args.gpus, argv))
    if args.block_only:
        import torch
        pk, _ = peaks()
        out = {"dit_block": dit_block_report(torch.device("cuda", 0), pk, pk["bf16_tflops"] * NOMINAL_FP4_OVER_BF16,
                                             images=args.block_images)}
        print(json.dumps(out), flush=True)
        return 0
    out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)
    world, _, _ = dist_setup()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

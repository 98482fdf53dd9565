"""Benchmark of the group-wise quantized linear layer on GB300.

Default run (one JSON line on stdout): every workload configuration of the
layer, the drafter layer as the headline and the others as keyed sub-records
under "configs":

  layer    one DFlash2 drafter layer's seven W8A8 GS128 projections (q
           5120->4096, k/v 5120->1024, o 4096->5120, gate/up 5120->17408,
           down 17408->5120) at M = 8*C tokens for C in {1, 8, 12}
           (M = 8, 64, 96)  [headline]
  single   one W8A8 GS128 linear 5120->1024 at M = 8
  drafter  the full drafter, 35 W8A8 GS128 linears + fc 25600->5120, M = 96
  w4a16    the same 36 shapes in W4A16 g128, M in {8, 64}
  prefill  W8A8 gate/up 5120->17408 and down 17408->5120 at M in {128, 512,
           2048, 8192} (tensor-bound at M >= 2048)
  vocab    the W8A8 GS128 vocabulary head 5120->248320 at M in {8, 96}

One step of a workload = dynamic INT8 quantization of its distinct inputs
(W8A8), then its GEMMs, replayed as one CUDA graph.  Metric: weight GB/s
(qweight + scale bytes streamed per step / step time), TOPS beside it; the
prefill record reports TOPS.  Each record carries its own roofline (the
GEMM launches alone), end-to-end rate through the binding with host copies,
and the oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|layer|single|drafter|w4a16|w8a16|prefill|
                                vocab|vocab_argmax|producers]

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (the layer has no exchange step on one GPU);
value = total over ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
LARGE_M = 2048          # prefill batches at and above this are tensor-bound


# ------------------------------------------------------------------ workloads

def workload_specs(name: str):
    """List of (linear name, K, N, activation kind, M, kind 'w8a8'|'w4a16'|...)."""
    from w4a16_linear_layers_gb300 import synth

    specs = []
    if name == "layer":
        for M in (8, 64, 96):
            for lname, K, N, kind in synth.DRAFTER_LAYER:
                specs.append((f"layers.0.{lname}", K, N, kind, M, "w8a8"))
    elif name == "single":
        specs.append(("single", 5120, 1024, "outliers", 8, "w8a8"))
    elif name == "drafter":
        for lname, K, N, kind in synth.drafter_linears():
            specs.append((lname, K, N, kind, 96, "w8a8"))
    elif name == "w4a16":
        for M in (8, 64):
            for lname, K, N, kind in synth.drafter_linears():
                specs.append((lname, K, N, "normal", M, "w4a16"))
    elif name == "w8a16":
        for M in (8, 64):
            for lname, K, N, kind in synth.DRAFTER_LAYER:
                specs.append((f"layers.0.{lname}", K, N, "normal", M, "w8a16"))
    elif name == "prefill":
        for M in (128, 512, 2048, 8192):
            specs.append(("layers.0.gate_proj", 5120, 17408, "outliers", M, "w8a8"))
            specs.append(("layers.0.up_proj", 5120, 17408, "outliers", M, "w8a8"))
            specs.append(("layers.0.down_proj", 17408, 5120, "silu_mul", M, "w8a8"))
    elif name == "vocab":
        for M in (8, 96):
            specs.append(("lm_head", 5120, 248320, "outliers", M, "w8a8"))
    elif name == "vocab_argmax":
        for M in (8, 96):
            specs.append(("lm_head", 5120, 248320, "outliers", M, "w8a8_argmax"))
    else:
        raise SystemExit(f"unknown workload {name}")
    return specs


WORKLOAD_DESC = {
    "layer": "drafter layer: 7 W8A8 GS128 linears x M in {8,64,96}",
    "single": "single W8A8 GS128 linear 5120->1024, M=8",
    "drafter": "full drafter: 35 W8A8 GS128 linears + fc 25600->5120, M=96",
    "w4a16": "full drafter in W4A16 g128 (36 linears), M in {8,64}",
    "w8a16": "drafter layer: 7 W8A16 group-32 linears x M in {8,64}",
    "prefill": "W8A8 GS128 gate/up 5120->17408 + down 17408->5120, M in {128,512,2048,8192}",
    "vocab": "W8A8 GS128 vocab head 5120->248320, M in {8,96}",
    "vocab_argmax": "W8A8 GS128 vocab head 5120->248320 with fused greedy argmax, M in {8,96}",
    "producers": "fused producers + per-token INT8 act-quant: RMSNorm over [M,5120] and "
                 "SiLU(gate)*up over [M,2x17408], M in {8,96,2048,8192}",
}

# the default run: the headline, then the sub-records (workload configurations)
HEADLINE = "layer"
SUB_RECORDS = ("single", "drafter", "w4a16", "prefill", "vocab")
METRIC = "W8A8-GS128 linear weight GB/s (TOPS beside it); % of HBM / tensor roofline"

W8A16_GROUP = 32   # the bench's W8A16 scale group (the DFlash2 recipe's group-32 int8)


def weight_bytes(K, N, kind):
    kind = kind.replace("_argmax", "")
    if kind == "w8a16":
        return K * N + 2 * (K // W8A16_GROUP) * N
    return (K * N if kind == "w8a8" else K * N // 2) + 2 * (K // 128) * N


def gemm_algo_bytes(M, K, N, kind):
    """Algorithmic bytes of one GEMM launch: weights + scales once, the
    activation operand once (int8 for W8A8, bf16 for W4A16), activation
    scales, and the output (bf16 y, or one int32 index per row for the
    greedy-argmax variant)."""
    out = 4 * M if kind.endswith("_argmax") else 2 * M * N
    kind = kind.replace("_argmax", "")
    act = M * K * (1 if kind == "w8a8" else 2) + (4 * M if kind == "w8a8" else 0)   # w4a16/w8a16: bf16 x
    return weight_bytes(K, N, kind) + act + out


def bound_of(name):
    return "tensor" if name == "prefill" else "hbm"


def workload_config(name, fused, world):
    """The static description of a workload (the same in both arms)."""
    specs = workload_specs(name)
    return {
        "workload": WORKLOAD_DESC[name],
        "linears_per_step": len(specs),
        "fused_projections": ("projections that read the same input (q/k/v, gate/up) run as one "
                              "GEMM over their weights concatenated along N: same bytes and outputs"
                              if fused else "off: one GEMM per linear"),
        "weight_bytes_per_step": sum(weight_bytes(K, N, wk) for _, K, N, _, _, wk in specs),
        "ops_per_step": sum(2 * M * K * N for _, K, N, _, M, _ in specs),
        "parallelism": f"replicas x{world}",
    }


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    """Roofline denominators: the measured copy bandwidth and bf16
    tensor rates of this GPU model (MEASURED_PEAKS.json), else fallbacks."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": FALLBACK_HBM_GBS, "bf16": FALLBACK_BF16_TFLOPS,
                "bf16_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


def source_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "w4a16_linear_layers_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ("gemm.cu", "qlin_device.cuh")


def profiled_traffic(key, sources=GEMM_SOURCES):
    """DRAM bytes per launch of a workload's dominant kernel, from the ncu
    counters recorded in profiles/traffic.json, or None when that kernel's
    sources changed since the capture (each entry records the sha256 prefix
    of the sources it measured)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not entry or entry.get("sources_sha16") != source_hash(sources):
        return None
    return int(entry["dram_bytes_per_launch"])


# ---------------------------------------------------------------- our arm

class LayerRunner:
    """Device-resident weights and inputs for a workload, and one step.

    With fuse, projections that read the same input (q/k/v, gate/up) run as
    one GEMM over their weights concatenated along N: the same bytes and
    outputs (output columns are independent), fewer launches.  The unfused
    call list is kept beside it so both can be timed.

    copies > 1 holds that many distinct copies of the weights, used in turn
    by consecutive steps, so that a workload whose weights fit in L2 still
    streams them from HBM every step."""

    def __init__(self, specs, device, seed=0, copies=1):
        import torch

        from w4a16_linear_layers_gb300 import qlin, synth

        self.torch, self.qlin = torch, qlin
        self.specs = specs
        self.device = device
        self.copies = copies
        self.ws = qlin.Workspace(device)
        weights = {}
        self.inputs = {}
        self.acts = {}
        # W8A8 inputs of more than 32 rows read only by plain W8A8 GEMMs take
        # their codes as fp16 (act_quant_c16 -> gemm_w8a8_gs128_c16): the
        # GEMM's tensor-core operand, with no int8 -> fp16 pass in between
        self.c16 = {}
        for spec in specs:
            ikey = self._ikey(spec)
            ok = spec[5] == "w8a8" and spec[4] > 32
            self.c16[ikey] = self.c16.get(ikey, True) and ok
        for name, K, N, kind, M, wk in specs:
            key = (name, wk)
            if key not in weights:
                weights[key] = self._weights(name, K, N, wk, seed)
            ikey = self._ikey((name, K, N, kind, M, wk))
            if ikey not in self.inputs:
                xb = synth.activations(seed, f"{ikey[0]}/M{M}", M, K, kind)
                self.inputs[ikey] = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(device)
                if wk.startswith("w8a8"):
                    cdt = torch.float16 if self.c16[ikey] else torch.int8
                    self.acts[ikey] = (torch.empty((M, K), dtype=cdt, device=device),
                                       torch.empty((M,), dtype=torch.float32, device=device))
        # calls[fused][copy]: unfused = one call per linear; fused = one call
        # per (input, format)
        self.calls = {False: [], True: []}
        groups = {}
        for spec in specs:
            groups.setdefault((self._ikey(spec), spec[5]), []).append(spec[0])
        for c in range(copies):
            self.calls[False].append([self._call(weights, wk, self._ikey(spec), [spec[0]], spec[4],
                                                 spec[1], c)
                                      for spec in specs for wk in [spec[5]]])
            self.calls[True].append([self._call(weights, wk, ikey, names, ikey[1], ikey[2], c)
                                     for (ikey, wk), names in groups.items()])
        del weights
        torch.cuda.synchronize()
        self.weight_bytes = sum(weight_bytes(K, N, wk) for _, K, N, _, _, wk in specs)
        self.ops = sum(2 * M * K * N for _, K, N, _, M, _ in specs)
        self.n_actq = len(self.acts)

    def _weights(self, name, K, N, wk, seed):
        """Packed weights and scales of one linear, drawn as synth's
        w8a8_weights / w4a16_weights / w8a16_weights draw them: the integer
        weights on the device (the same stream, bit for bit), the scales on
        the host."""
        torch, qlin = self.torch, self.qlin
        from w4a16_linear_layers_gb300 import synth

        if wk.startswith("w8a8"):
            q = synth.randint_device(seed, name + "/qw", (K, N), -127, 127, self.device)
            s = synth.f16_bits(synth.log_uniform(seed, name + "/sw", (K // 128, N), 1e-3, 1e-2))
            bits, sdt = 8, torch.float16
        elif wk == "w8a16":
            q = synth.randint_device(seed, name + "/w8a16/qw", (K, N), -127, 127, self.device)
            s = synth.bf16_bits(synth.log_uniform(seed, name + "/w8a16/sw", (K // W8A16_GROUP, N),
                                                  1e-3, 1e-2))
            bits, sdt = 8, torch.bfloat16
        else:
            q = synth.randint_device(seed, name + "/w4/qw", (K, N), -7, 7, self.device)
            s = synth.bf16_bits(synth.log_uniform(seed, name + "/w4/sw", (K // 128, N), 1e-3, 3e-2))
            bits, sdt = 4, torch.bfloat16
        qw, _ = qlin.pack_gptq(q, bits, with_qzeros=False)
        del q
        sd = torch.from_numpy(s.view(np.int16)).view(sdt).to(self.device)
        return qw, sd

    def _call(self, weights, wk, ikey, names, M, K, copy):
        torch = self.torch
        parts = [weights[(n, wk)] for n in names]
        if len(parts) == 1:
            qw, sc = parts[0]
            if copy > 0:
                qw, sc = qw.clone(), sc.clone()
        else:
            qw = torch.cat([p[0] for p in parts], dim=1).contiguous()
            sc = torch.cat([p[1] for p in parts], dim=1).contiguous()
        N = qw.shape[1]
        # two output buffers: the end-to-end leg overlaps one step's read-back
        # with the next step's compute
        if wk.endswith("_argmax"):     # greedy token per row
            ys = [torch.empty((M,), dtype=torch.int32, device=self.device) for _ in range(2)]
        else:
            ys = [torch.empty((M, N), dtype=torch.bfloat16, device=self.device) for _ in range(2)]
        self.ws.get(M, N, K)
        return {"wk": wk, "ikey": ikey, "qw": qw, "sc": sc, "ys": ys, "M": M, "N": N, "K": K,
                "names": names}

    def outputs(self, fused, buf=0, copy=0):
        return [c["ys"][buf] for c in self.calls[fused][copy]]

    def n_gemm(self, fused):
        return len(self.calls[fused][0])

    def gemm_bytes(self, fused, sel=None):
        return sum(gemm_algo_bytes(c["M"], c["K"], c["N"], c["wk"])
                   for c in self.calls[fused][0] if sel is None or sel(c))

    def gemm_ops(self, fused, sel=None):
        return sum(2 * c["M"] * c["K"] * c["N"] for c in self.calls[fused][0]
                   if sel is None or sel(c))

    def n_launches(self, fused):
        # one kernel per act-quant and per GEMM, plus the int8 -> fp16 operand
        # pass of W8A8 GEMMs with token tiles of 64 and more (M > 32) that
        # read int8 codes, plus the argmax decode
        return self.n_actq + sum(1 + (c["wk"].startswith("w8a8") and c["M"] > 32
                                      and not self.c16[c["ikey"]])
                                 + c["wk"].endswith("_argmax") for c in self.calls[fused][0])

    def _ikey(self, spec):
        from w4a16_linear_layers_gb300 import synth

        name, K, N, kind, M, wk = spec
        return (synth.shared_input_name(name), M, K, kind)

    def quantize(self):
        for ikey, (q, s) in self.acts.items():
            if self.c16[ikey]:
                self.qlin.act_quant_c16(self.inputs[ikey], q, s)
            else:
                self.qlin.act_quant_i8(self.inputs[ikey], q, s)

    def gemms(self, fused=False, buf=0, copy=0, sel=None):
        ws = self.ws.buf
        for c in self.calls[fused][copy]:
            if sel is not None and not sel(c):
                continue
            y = c["ys"][buf]
            if c["wk"] == "w8a8_argmax":
                q, s = self.acts[c["ikey"]]
                self.qlin.gemm_w8a8_gs128_argmax(q, s, c["qw"], c["sc"], y, workspace=ws)
            elif c["wk"] == "w8a8":
                q, s = self.acts[c["ikey"]]
                gemm = (self.qlin.gemm_w8a8_gs128_c16 if self.c16[c["ikey"]]
                        else self.qlin.gemm_w8a8_gs128)
                gemm(q, s, c["qw"], c["sc"], y, workspace=ws)
            elif c["wk"] == "w8a16":
                self.qlin.gemm_w8a16(self.inputs[c["ikey"]], c["qw"], c["sc"], W8A16_GROUP, y,
                                     workspace=ws)
            else:
                self.qlin.gemm_w4a16_g128(self.inputs[c["ikey"]], c["qw"], c["sc"], y,
                                          workspace=ws)

    def step(self, fused=False, buf=0, copy=0):
        self.quantize()
        self.gemms(fused, buf, copy)

    def all_copies(self, fn):
        for c in range(self.copies):
            fn(c)

    def capture(self, fn):
        torch = self.torch
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()              # warm the launch path (attributes, tensor maps)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank floats over all ranks (identity
    without a process group).  Every rank gets the result."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_step, steps, world, seconds):
    """Throughput of the whole job: every rank processed units_per_step per
    step (weak scaling), and the job took the slowest rank's time."""
    return units_per_step * steps * world / seconds


def time_graph(torch, graph, reps):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(reps):
        graph.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3  # seconds


def measure(name, args, device, world, steps, fused=True, with_alt=False, clocks=None):
    """Time one workload: its step graph (act-quants + GEMMs), its GEMM
    launches alone (the roofline kernel), the end-to-end leg through the
    binding with host copies, and, for the headline, the other call list.
    `clocks`, if given, samples the SM clocks from the soak to the end of the
    timed replays.  Returns (record without the oracle baseline, runner)."""
    import torch

    from w4a16_linear_layers_gb300 import qlin

    specs = workload_specs(name)
    wbytes = sum(weight_bytes(K, N, wk) for _, K, N, _, _, wk in specs)
    # weights that fit in L2 rotate through distinct copies, three L2s' worth
    copies = 1 if wbytes >= 2 * L2_BYTES else int(math.ceil(3 * L2_BYTES / wbytes))
    runner = LayerRunner(specs, device, copies=copies)
    # the roofline kernel: every GEMM of the step, or for the tensor-bound
    # prefill the batches of LARGE_M rows and more
    sel = (lambda c: c["M"] >= LARGE_M) if bound_of(name) == "tensor" else None
    step_graph = runner.capture(lambda: runner.all_copies(lambda c: runner.step(fused, 0, c)))
    gemm_graph = runner.capture(lambda: runner.all_copies(lambda c: runner.gemms(fused, 0, c, sel)))
    alt_graph = None
    if with_alt and runner.n_gemm(True) != runner.n_gemm(False):
        alt_graph = runner.capture(lambda: runner.all_copies(lambda c: runner.step(not fused, 0, c)))
    if clocks is not None:
        clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        step_graph.replay()
        torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        step_graph.replay()
    torch.cuda.synchronize()
    st, where, block = qlin.device_error_detail()
    if st != qlin.QLIN_OK:
        raise SystemExit(f"{name}: device status after warm-up: {qlin.status_string(st)} "
                         f"(wait {where}, block {block})")
    if steps is None:
        # sub-records: about a quarter of a second of timed replays
        one = time_graph(torch, step_graph, 1)
        steps = int(min(1000, max(5, round(0.25 / max(one, 1e-6)))))
    reps = steps           # graph replays; each replay runs `copies` steps
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_step = time_graph(torch, step_graph, reps)
    t_gemm = time_graph(torch, gemm_graph, reps)
    t_alt = time_graph(torch, alt_graph, reps) if alt_graph is not None else 0.0
    clock_info = clocks.stop() if clocks is not None else None
    t_step, t_gemm, t_alt = max_over_ranks([t_step, t_gemm, t_alt], device)
    n_steps = reps * copies

    # End to end through the binding, no graph: every step copies its inputs
    # from pinned host memory and reads its outputs back.  Two sets of device
    # inputs and outputs let the copies of one step overlap the compute of the
    # next, as a serving loop does: a copy stream uploads step i + 1's inputs
    # while step i computes, then reads step i's outputs back.
    inputs0 = runner.inputs
    in_sets = [inputs0, {k: torch.empty_like(v) for k, v in inputs0.items()}]
    host_in = {k: v.cpu().pin_memory() for k, v in inputs0.items()}
    host_out = [[torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
                 for y in runner.outputs(fused, b)] for b in range(2)]
    h2d = sum(v.numel() * 2 for v in host_in.values())
    d2h = sum(y.numel() * y.element_size() for y in runner.outputs(fused, 0))
    comp = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def upload(b):
        # the inputs of set b were last read by the step that computed on b
        copy_s.wait_event(comp_done[b])
        with torch.cuda.stream(copy_s):
            for k, v in host_in.items():
                in_sets[b][k].copy_(v, non_blocking=True)
        in_ready[b].record(copy_s)

    def run_steps(n):
        upload(0)
        for i in range(n):
            b = i & 1
            comp.wait_event(in_ready[b])
            comp.wait_event(out_read[b])      # outputs of set b read back
            runner.inputs = in_sets[b]
            runner.step(fused, b, i % copies)
            comp_done[b].record(comp)
            if i + 1 < n:
                upload(b ^ 1)
            copy_s.wait_event(comp_done[b])
            with torch.cuda.stream(copy_s):
                for h, y in zip(host_out[b], runner.outputs(fused, b, i % copies)):
                    h.copy_(y, non_blocking=True)
            out_read[b].record(copy_s)
        torch.cuda.synchronize()
        runner.inputs = inputs0

    run_steps(max(2, args.warmup))
    e2e_steps = max(3 * copies, min(n_steps, 100))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run_steps(e2e_steps)
    t_e2e = (time.perf_counter() - t0) / e2e_steps
    t_e2e, = max_over_ranks([t_e2e], device)
    st, where, block = qlin.device_error_detail()
    if st != qlin.QLIN_OK:
        raise SystemExit(f"{name}: device status after timing: {qlin.status_string(st)} "
                         f"(wait {where}, block {block})")

    peaks = measured_peaks()
    n_gemm_launch = sum(1 for c in runner.calls[fused][0] if sel is None or sel(c))
    gemm_avg_s = t_gemm / (reps * copies * n_gemm_launch)
    gbs = whole_job_rate(runner.weight_bytes, n_steps, world, t_step) / 1e9
    tops = whole_job_rate(runner.ops, n_steps, world, t_step) / 1e12
    if bound_of(name) == "tensor":
        ops_per_launch = runner.gemm_ops(fused, sel) / n_gemm_launch
        achieved = ops_per_launch / gemm_avg_s / 1e12
        roof = {"bound": "tensor", "kernel": "qlin_gemm_kernel (W8A8 GS128), M >= %d" % LARGE_M,
                "achieved": round(achieved, 1), "peak": peaks["bf16_sustained"],
                "peak_source": peaks["source"] + " (bf16 sustained: launches inside a long step)",
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_sustained"], 4),
                "frac_of_burst_peak": round(achieved / peaks["bf16"], 4),
                "traffic": profiled_traffic(name),
                "ops_per_launch": round(ops_per_launch), "avg_launch_us": round(gemm_avg_s * 1e6, 3)}
        value, unit = tops, "TOPS"
    else:
        bytes_per_launch = runner.gemm_bytes(fused) / n_gemm_launch
        achieved = bytes_per_launch / gemm_avg_s / 1e9
        roof = {"bound": "hbm", "kernel": "qlin_gemm_kernel (%s)" % (
                    "W4A16 g128" if name == "w4a16" else "W8A16" if name == "w8a16" else "W8A8 GS128"),
                "achieved": round(achieved, 1), "peak": peaks["hbm"],
                "peak_source": peaks["source"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm"], 4),
                "traffic": profiled_traffic(name),
                "bytes_per_launch": round(bytes_per_launch),
                "avg_launch_us": round(gemm_avg_s * 1e6, 3)}
        value, unit = gbs, "GB/s"
    e2e_gbs = runner.weight_bytes * world / t_e2e / 1e9
    e2e_tops = runner.ops * world / t_e2e / 1e12
    rec = {
        "value": round(value, 3 if unit == "TOPS" else 2),
        "unit": unit,
        "steps": n_steps,
        "ms_per_step": round(t_step / n_steps * 1e3, 4),
        "gbs": round(gbs, 2),
        "tops": round(tops, 3),
        "config": workload_config(name, fused, world),
        "gemm_launches_per_step": runner.n_gemm(fused),
        "act_quant_per_step": runner.n_actq,
        "gpu_launches": runner.n_launches(fused) * n_steps,
        "l2": ("inputs larger than L2: each step streams its weight bytes once; no matrix is "
               "re-read before the others have passed through" if copies == 1 else
               f"weights smaller than L2: {copies} distinct copies of the weights "
               f"({copies * runner.weight_bytes / 1e6:.0f} MB), used in turn by consecutive steps"),
        "timing": (f"CUDA graph of {copies} step(s), {reps} replays timed with CUDA events on the "
                   f"replay stream after {max(3, args.warmup)} warm-up replays"),
        "roofline": roof,
        "e2e": {"value": round(e2e_tops if unit == "TOPS" else e2e_gbs, 3 if unit == "TOPS" else 2),
                "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(t_e2e * 1e3, 4)},
        "clocks": clock_info,
    }
    if alt_graph is not None:
        alt_gbs = whole_job_rate(runner.weight_bytes, n_steps, world, t_alt) / 1e9
        alt_tops = whole_job_rate(runner.ops, n_steps, world, t_alt) / 1e12
        rec["other_call_list"] = {
            "fused_projections": not fused,
            "value": round(alt_tops, 3) if unit == "TOPS" else round(alt_gbs, 2),
            "unit": unit, "gbs": round(alt_gbs, 2), "tops": round(alt_tops, 3),
            "ms_per_step": round(t_alt / n_steps * 1e3, 4),
            "gemm_launches_per_step": runner.n_gemm(not fused)}
    return rec, runner


# ------------------------------------------- fused producers (RMSNorm, SiLU*up)

PRODUCER_MS = (8, 96, 2048, 8192)
PRODUCER_HIDDEN, PRODUCER_INTER, PRODUCER_EPS = 5120, 17408, 1e-6


def producer_specs():
    """(kind, M, K): K is the quantized row length (the hidden size for the
    norm, the intermediate size for SiLU(gate)*up)."""
    return [(kind, M, PRODUCER_HIDDEN if kind == "rmsnorm" else PRODUCER_INTER)
            for M in PRODUCER_MS for kind in ("rmsnorm", "silu_mul")]


def producer_bytes(kind, M, K):
    """Algorithmic bytes of one call: the bf16 input (and the norm weight),
    the int8 output and the fp32 scales."""
    read = 2 * M * K + 2 * K if kind == "rmsnorm" else 2 * M * 2 * K
    return read + M * K + 4 * M


_PRODUCER_INPUTS = {}


def producer_inputs(kind, M, K, seed=0):
    key = (kind, M, K, seed)
    if key not in _PRODUCER_INPUTS:
        _PRODUCER_INPUTS[key] = _make_producer_inputs(kind, M, K, seed)
    return _PRODUCER_INPUTS[key]


PRODUCER_DISTINCT_ROWS = 64   # rows repeat with this period (input generation time)


def _make_producer_inputs(kind, M, K, seed):
    from w4a16_linear_layers_gb300 import synth

    r = min(M, PRODUCER_DISTINCT_ROWS)
    reps = (M + r - 1) // r
    if kind == "rmsnorm":
        x = synth.activations(seed, f"producers/rms/M{M}", r, K, "outliers")
        g = synth.bf16_bits(1.0 + 0.1 * synth.normal(seed, "producers/rms/gamma", (K,)))
        return np.ascontiguousarray(np.tile(x, (reps, 1))[:M]), g
    x = synth.activations(seed, f"producers/silu/M{M}", r, 2 * K, "normal2")
    return np.ascontiguousarray(np.tile(x, (reps, 1))[:M]), None


def run_producers(args, rank, world, local_rank):
    import torch
    from w4a16_linear_layers_gb300 import build as qbuild
    from w4a16_linear_layers_gb300 import qlin

    qbuild.build()
    device = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(device)
    specs = producer_specs()
    calls = []
    for kind, M, K in specs:
        x, g = producer_inputs(kind, M, K)
        xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        gd = None if g is None else torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).to(device)
        q = torch.empty((M, K), dtype=torch.int8, device=device)
        sa = torch.empty((M,), dtype=torch.float32, device=device)
        calls.append((kind, M, K, xd, gd, q, sa))

    def one(c):
        kind, M, K, xd, gd, q, sa = c
        if kind == "rmsnorm":
            qlin.rmsnorm_act_quant_i8(xd, gd, PRODUCER_EPS, q=q, s_a=sa)
        else:
            qlin.silu_mul_act_quant_i8(xd, q=q, s_a=sa)

    def capture(cs):
        st = torch.cuda.Stream(device)
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            for c in cs:
                one(c)
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for c in cs:
                one(c)
        torch.cuda.synchronize()
        return gr

    step_graph = capture(calls)
    # the dominant launch: SiLU(gate)*up at the largest M
    top = max(calls, key=lambda c: producer_bytes(c[0], c[1], c[2]))
    top_graph = capture([top])
    for _ in range(args.warmup):
        step_graph.replay()
    torch.cuda.synchronize()
    if qlin.device_status() != qlin.QLIN_OK:
        raise SystemExit("device status after warm-up is not OK")
    clocks = ClockSampler(local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_step = time_graph(torch, step_graph, args.steps)
    t_top = time_graph(torch, top_graph, args.steps)
    clock_info = clocks.stop()
    t_step, t_top = max_over_ranks([t_step, t_top], device)

    host_in = [c[3].cpu().pin_memory() for c in calls]
    host_q = [torch.empty(c[5].shape, dtype=torch.int8, pin_memory=True) for c in calls]
    host_s = [torch.empty(c[6].shape, dtype=torch.float32, pin_memory=True) for c in calls]
    h2d = sum(h.numel() * 2 for h in host_in)
    d2h = sum(h.numel() for h in host_q) + sum(h.numel() * 4 for h in host_s)

    def e2e_step():
        for h, c in zip(host_in, calls):
            c[3].copy_(h, non_blocking=True)
        for c in calls:
            one(c)
        for hq, hs, c in zip(host_q, host_s, calls):
            hq.copy_(c[5], non_blocking=True)
            hs.copy_(c[6], non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(reps):
        e2e_step()
    torch.cuda.synchronize()
    t_e2e = (time.perf_counter() - t0) / reps
    t_e2e, = max_over_ranks([t_e2e], device)
    if qlin.device_status() != qlin.QLIN_OK:
        raise SystemExit("device status after timing is not OK")
    if rank != 0:
        return None
    step_bytes = sum(producer_bytes(k, M, K) for k, M, K in specs)
    top_bytes = producer_bytes(top[0], top[1], top[2])
    peaks = measured_peaks()
    hbm, peak_src = peaks["hbm"], peaks["source"]
    top_s = t_top / args.steps
    achieved = top_bytes / top_s / 1e9
    return {
        "metric": "fused producer + INT8 act-quant GB/s (algorithmic bytes); % of HBM roofline",
        "value": round(whole_job_rate(step_bytes, args.steps, world, t_step) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, fp32 producer arithmetic, int8 + fp32 scale out",
        "data": "synthetic (seeded splitmix64; N(0,1) rows with outlier channels, "
                "N(0,2) gate/up pre-activations, norm weight 1 + N(0, 0.01); "
                f"rows repeat with period {PRODUCER_DISTINCT_ROWS})",
        "config": {
            "workload": WORKLOAD_DESC["producers"],
            "calls_per_step": len(calls),
            "bytes_per_step": step_bytes,
            "l2": "inputs larger than L2: one step moves about 0.9 GB",
            "timing": "CUDA graph of one step, CUDA events on the replay stream",
            "parallelism": f"replicas x{world}",
        },
        "gpu_launches": len(calls) * args.steps,
        "roofline": {
            "bound": "hbm",
            "kernel": f"producer_quant_kernel<SiLU*up> (M={top[1]}, I={top[2]})",
            "achieved": round(achieved, 1),
            "peak": hbm,
            "peak_source": peak_src,
            "unit": "GB/s",
            "frac": round(achieved / hbm, 4),
            "traffic": profiled_traffic("producers", ("act_quant.cu",)),
            "bytes_per_launch": top_bytes,
            "avg_launch_us": round(top_s * 1e6, 3),
        },
        "e2e": {
            "value": round(step_bytes * world / t_e2e / 1e9, 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(t_e2e * 1e3, 4),
        },
        "clocks": clock_info,
    }


def producer_oracle_sample(budget_s, seed=0, rows=None):
    """The oracle on the first `rows` rows of every call of the step (the
    whole step when rows is None), repeated while the time stays under half
    the budget, on all host cores (one thread per row slice).
    Returns (algorithmic bytes covered, seconds, threads, text)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    nthreads = cores()
    specs = producer_specs()
    tasks, step_bytes = [], 0
    for kind, M, K in specs:
        x, g = producer_inputs(kind, M, K, seed)
        r = M if rows is None else min(rows, M)
        step_bytes += producer_bytes(kind, r, K)
        for sl in np.array_split(np.arange(r), min(nthreads, r)):
            if sl.size:
                tasks.append((kind, np.ascontiguousarray(x[sl]), g))

    def work(kind, x, g):
        if kind == "rmsnorm":
            oracle.rmsnorm_act_quant_i8(x, g, PRODUCER_EPS)
        else:
            oracle.silu_mul_act_quant_i8(x)

    reps, total = 0, 0.0
    while reps < 5 and (reps == 0 or total < 0.5 * budget_s):
        t0 = time.perf_counter()
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(lambda t: work(*t), tasks))
        total += time.perf_counter() - t0
        reps += 1
    what = "every row" if rows is None else f"the first {rows} rows"
    return step_bytes * reps, total, nthreads, (
        f"oracle on {what} of each of the {len(specs)} calls of the step, {reps} time(s), "
        f"{nthreads} threads")


# ------------------------------------------------------------ oracle (CPU)

def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_sample(specs, budget_s, seed=0, cache=None, frac=None):
    """Time the oracle on a bounded sample of the workload: for every linear
    of the step, the same fraction of its output columns (all rows), run on
    all host cores (one thread per column slice; the C oracle runs without the
    GIL).  The sampled columns' weights are drawn alone (the generator is
    counter-based).  The fraction is calibrated to the time budget unless
    given.  Returns (weight bytes covered, ops covered, seconds, threads,
    description, fraction)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from w4a16_linear_layers_gb300 import synth

    oracle.build()
    nthreads = cores()
    cache = {} if cache is None else cache

    def operands(name, K, N, kind, M, wk, nc):
        cols = np.arange(nc)
        if wk.startswith("w8a8"):
            q = synth.randint_at(seed, name + "/qw", N, np.arange(K), cols, -127, 127)
            s = synth.f16_bits(synth.log_uniform_at(seed, name + "/sw", N, np.arange(K // 128),
                                                    cols, 1e-3, 1e-2))
        elif wk == "w8a16":
            q = synth.randint_at(seed, name + "/w8a16/qw", N, np.arange(K), cols, -127, 127)
            s = synth.bf16_bits(synth.log_uniform_at(seed, name + "/w8a16/sw", N,
                                                     np.arange(K // W8A16_GROUP), cols, 1e-3, 1e-2))
        else:
            q = synth.randint_at(seed, name + "/w4/qw", N, np.arange(K), cols, -7, 7)
            s = synth.bf16_bits(synth.log_uniform_at(seed, name + "/w4/sw", N, np.arange(K // 128),
                                                     cols, 1e-3, 3e-2))
        q, s = np.ascontiguousarray(q), np.ascontiguousarray(s)
        xb = synth.activations(seed, f"{synth.shared_input_name(name)}/M{M}", M, K, kind)
        if wk.startswith("w8a8"):
            qw, _, _ = oracle.pack_gptq(q, 8)
            qa, sa = oracle.act_quant_i8(xb)
            return (lambda ch, a=(qa, sa, qw, s, K): oracle.gemm_w8a8_gs128(*a, cols=ch))
        if wk == "w8a16":
            qw, _, _ = oracle.pack_gptq(q, 8)
            return (lambda ch, a=(xb, qw, s, K): oracle.gemm_w8a16(*a, W8A16_GROUP, cols=ch))
        qw, _, _ = oracle.pack_gptq(q, 4)
        return (lambda ch, a=(xb, qw, s, K): oracle.gemm_w4a16_g128(*a, cols=ch))

    def run(frac):
        total_bytes, total_ops = 0, 0
        tasks = []
        for name, K, N, kind, M, wk in specs:
            nc = max(1, int(round(N * frac)))
            total_bytes += weight_bytes(K, nc, wk)
            total_ops += 2 * M * K * nc
            key = ("operands", name, K, N, kind, M, wk, nc)
            if key not in cache:
                cache[key] = operands(name, K, N, kind, M, wk.replace("_argmax", ""), nc)
            fn = cache[key]
            for ch in np.array_split(np.arange(nc), min(nthreads, nc)):
                if ch.size:
                    tasks.append((fn, ch))
        t0 = time.perf_counter()
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(lambda t: t[0](t[1]), tasks))
        return total_bytes, total_ops, time.perf_counter() - t0

    if frac is None:
        frac = 1e-4
        while True:                       # calibrate the sample size on this host
            _, _, t = run(frac)
            if t >= 0.2 * budget_s or frac >= 1.0:
                break
            frac = min(1.0, frac * min(16.0, max(2.0, 0.3 * budget_s / max(t, 1e-3))))
        frac = min(1.0, frac * budget_s / max(t, 1e-3))
    b, ops, t = run(frac)
    desc = (f"oracle on {frac * 100:.3f}% of the output columns of every linear of the step "
            f"(all rows), {nthreads} threads")
    return b, ops, t, nthreads, desc, frac


def cpu_baseline_record(name, specs, budget_s):
    b, ops, t, thr, desc, _ = oracle_sample(specs, budget_s)
    if bound_of(name) == "tensor":
        return {"value": round(ops / t / 1e12, 6), "unit": "TOPS", "cores": thr, "kind": "oracle",
                "sample": desc}
    return {"value": round(b / t / 1e9, 6), "unit": "GB/s", "cores": thr, "kind": "oracle",
            "sample": desc}


def run_reference_producers(args):
    # about a minute of oracle work over all steps: rows per call calibrated
    # once so that one step takes the per-step budget
    budget = max(0.02, 60.0 / max(1, args.steps + args.warmup))
    rows = 1
    while rows < 8192:
        _, t, _, _ = producer_oracle_sample(0.0, rows=rows)
        if t >= budget:
            break
        rows *= 2
    for _ in range(args.warmup):
        producer_oracle_sample(0.0, rows=rows)
    tot_b, tot_t, thr, desc = 0, 0.0, 1, ""
    for _ in range(args.steps):
        b, t, thr, desc = producer_oracle_sample(0.0, rows=rows)
        tot_b += b
        tot_t += t
    value = tot_b / tot_t / 1e9
    return {
        "impl": "reference",
        "metric": "fused producer + INT8 act-quant GB/s (algorithmic bytes); % of HBM roofline",
        "value": round(value, 6), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp64 producer arithmetic, fp32 act-quant (CPU oracle)",
        "data": "synthetic (seeded splitmix64)",
        "config": {"workload": WORKLOAD_DESC["producers"]},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": thr,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    if args.workload == "producers":
        return run_reference_producers(args)
    name = HEADLINE if args.workload == "all" else args.workload
    specs = workload_specs(name)
    # about a minute of oracle work over all warm-up and timed steps: the
    # sample fraction is calibrated once, then every step runs that sample
    per_step_budget = max(0.02, 60.0 / max(1, args.steps + args.warmup))
    cache = {}
    frac = oracle_sample(specs, per_step_budget, cache=cache)[5]
    for _ in range(args.warmup):
        oracle_sample(specs, per_step_budget, cache=cache, frac=frac)
    tot_b, tot_ops, tot_t = 0, 0, 0.0
    desc, thr = "", 1
    for _ in range(args.steps):
        b, ops, t, thr, desc, _ = oracle_sample(specs, per_step_budget, cache=cache, frac=frac)
        tot_b += b
        tot_ops += ops
        tot_t += t
    if bound_of(name) == "tensor":
        value, unit = tot_ops / tot_t / 1e12, "TOPS"
    else:
        value, unit = tot_b / tot_t / 1e9, "GB/s"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8xint8->int64 exact, fp32 rescale chain (CPU oracle)",
        "data": "synthetic (seeded splitmix64)",
        "config": workload_config(name, not args.no_fuse, world),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": thr,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--soak", type=float, default=0.5,
                    help="seconds of untimed replays before the warm-up (clock ramp)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(WORKLOAD_DESC),
                    help="all: the headline drafter layer plus every other configuration as "
                         "sub-records")
    ap.add_argument("--no-fuse", action="store_true",
                    help="one GEMM per linear (default: projections sharing an input run as one GEMM)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the headline's cpu_baseline sample "
                         "(a third of it for each sub-record)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    from w4a16_linear_layers_gb300 import build as qbuild

    qbuild.build()
    device = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(device)
    if args.workload == "producers":
        line = run_producers(args, rank, world, local_rank)
        if line is not None:
            b, t, thr, desc = producer_oracle_sample(args.cpu_budget)
            line["cpu_baseline"] = {"value": round(b / t / 1e9, 6), "unit": "GB/s", "cores": thr,
                                    "kind": "oracle", "sample": desc}
            print(json.dumps(line), flush=True)
    else:
        fused = not args.no_fuse
        name = HEADLINE if args.workload == "all" else args.workload
        clocks = ClockSampler(local_rank)
        rec, runner = measure(name, args, device, world, args.steps, fused, with_alt=True,
                              clocks=clocks)
        specs = runner.specs
        del runner
        subs = {}
        if args.workload == "all":
            for sub in SUB_RECORDS:
                torch.cuda.empty_cache()
                r, sub_runner = measure(sub, args, device, world, None, fused)
                subs[sub] = (r, sub_runner.specs)
                del sub_runner
        if rank == 0:
            line = {
                "metric": METRIC,
                "value": rec["value"],
                "unit": rec["unit"],
                "n_gpus": world,
                "steps": rec["steps"],
                "warmup": args.warmup,
                "ms_per_step": rec["ms_per_step"],
                "higher_is_better": True,
                "scaling": "weak",
                "vs_baseline": None,
                "dtype": "int8xint8->fp32 (exact on fp16 tcgen05), bf16 out"
                         if name not in ("w4a16", "w8a16") else "bf16 x int weights -> fp32, bf16 out",
                "data": "synthetic (seeded splitmix64; weights uniform int8/int4, log-uniform "
                        "group scales; activations N(0,1) with outlier channels)",
                "config": rec["config"],
                "tops": rec["tops"],
                "gemm_launches_per_step": rec["gemm_launches_per_step"],
                "act_quant_per_step": rec["act_quant_per_step"],
                "l2": rec["l2"],
                "timing": rec["timing"],
                "gpu_launches": rec["gpu_launches"],
                "roofline": rec["roofline"],
                "e2e": rec["e2e"],
                "clocks": rec["clocks"],
            }
            if "other_call_list" in rec:
                line["other_call_list"] = rec["other_call_list"]
            line["cpu_baseline"] = cpu_baseline_record(name, specs, args.cpu_budget)
            if subs:
                line["configs"] = {}
                for sub, (r, sub_specs) in subs.items():
                    r["cpu_baseline"] = cpu_baseline_record(sub, sub_specs, args.cpu_budget / 3)
                    line["configs"][sub] = r
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of one MoE layer between DP attention and EP on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode|prefill|...]
    python bench.py --impl reference ...      # the CPU oracle, timed on host cores

A step is one pass of the whole hot path over one batch: DP gather (hidden
states and router logits), top-k routing, dispatch, grouped SwiGLU expert FFN
on the tensor cores, combine and DP scatter.  The default workload is the
DeepSeek-V3-shaped prefill layer, the largest single-GPU workload: T = 8192
tokens of one request on one replica, hidden 7168, 256 experts with uniform
popularity, top-8, expert intermediate 2048, bf16 weights/activations with
fp32 accumulation.  `--config decode` runs the 8-replica decode layer (seeded
token counts in [0, 64], one idle, MAX padding).

Printed: one JSON line (rank 0).  `value` is tokens/s with inputs resident in
HBM; `e2e` is the same metric through the same C-ABI calls with the step's
inputs copied from pinned host buffers and its outputs copied back inside the
timed region.  `roofline` reports the grouped FFN (the dominant call: tcgen05
kernels that stream the expert weights) against the measured bf16 tensor peak
(burst and sustained) and against the HBM roofline at its arithmetic
intensity, and, under `permutes`, the gather, dispatch and combine + scatter
stages as algorithmic bytes over their live stage time against the measured
HBM copy bandwidth.  N > 1 runs independent replicas, one per GPU (the layer
has no cross-GPU exchange on this path), and reports the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from combine_dp_gather_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300"
UNIT = "tokens/s"
L2_NOTE = "inputs larger than L2: every step streams the touched experts' weights from HBM"

def launches_per_step(rows: int, k: int, E: int, P: int, cap: int, align: int,
                      fp8: bool = False, router_gemm: bool = False, sms: int = 152,
                      fused_combine: bool = False, ffn_split: bool = False,
                      fp8_pair: bool = False, fp8_split: bool = False) -> int:
    """Kernel launches of one layer step: gather (with given logits it routes the rows
    in the same launch, the fused add + RMSNorm included), dispatch (one CTA-wide kernel for <= 8192 routed pairs whose tables
    fit 48 KB, else histogram + scan + rank; then the row copy; + the alignment pad
    kernel when align > 1, plus the FP8 rows' pad kernel on the FP8 path), grouped FFN
    (MM1+SwiGLU and MM2; one persistent launch for both on FP8 with few rows per
    slot, MM1 + the quantisation of h + MM2 with many), combine with the DP
    scatter (none when the down projection's epilogue combines).  With the router gate
    GEMM the logits gather goes and routing is one fused kernel (>= sms/4 row tiles and
    k <= 8) or split GEMM + sum + top-k."""
    small = rows * k <= 8192 and 4 * (33 * E + 3 * P + 1) <= 48 * 1024
    dispatch = (1 if small else 3) + 1 + (1 + (1 if fp8 else 0) if align > 1 else 0)
    gather, route = 1, 0
    if router_gemm:
        gather = 1
        route = 1 if (k <= 8 and 4 * ((rows + 127) // 128) >= sms) else 3
    ffn = ((3 if fp8_pair else (4 if fp8_split else 1)) if fp8
           else (4 if ffn_split else 2))   # bf16 split: 2 per stream
    return gather + route + dispatch + ffn + (0 if fused_combine else 1)


def fp8_pair(cap: int, P: int, H: int, I: int) -> bool:
    """True if the FP8 grouped FFN runs on SM pairs with block-scaled MMAs (192 or
    more sorted rows per slot on average, H and I multiples of 512)."""
    return cap // max(P, 1) >= 192 and H % 512 == 0 and I % 512 == 0


def fp8_split(cap: int, P: int, H: int, I: int) -> bool:
    """True if the FP8 grouped FFN sends its slots of 192 or more rows to the pair
    kernel and the rest to the one-launch kernel (32-191 rows per slot on average)."""
    return (32 <= cap // max(P, 1) < 192 and cap >= 192 and H % 512 == 0
            and I % 512 == 0)


def ffn_kernel(cap: int, P: int, fp8: bool = False, H: int = 0, I: int = 0) -> str:
    """The grouped-FFN kernel the library picks: on FP8 operands the block-scaled
    pair kernel with many rows per slot, else the weights-as-M single-SM kernel; in
    bf16 weights as M on SM pairs from 192 sorted rows per slot on average, else
    tokens as M on single SMs."""
    if fp8:
        if fp8_split(cap, P, H, I):
            return "ffn_f8swap_kernel for slots of >= 192 rows, ffn_fp8_kernel for the rest"
        return "ffn_f8swap_kernel" if fp8_pair(cap, P, H, I) else "ffn_fp8_kernel"
    return "ffn_swap_kernel" if cap // max(P, 1) >= 192 else "ffn_tc_kernel"

# dram__bytes_read.sum + dram__bytes_write.sum of the grouped-FFN launches (two in bf16; on
# FP8 one with few rows per slot, three with many: MM1, the quantisation of h, MM2) of one step
# of the workload (ncu, --clock-control none), valid while the kernel's sources hash to the
# recorded SHA-256 prefix; any other source reports traffic null.  The records come from shrunk
# cases of the same kernels (32-expert prefill, 64-expert decode) and are scaled to the workload
# by the units processed (traffic per slot and per routed row is the same).
FFN_TRAFFIC = {
    "prefill": {"sources": ["ffn_tc_swap.cu", "tc_ptx.cuh"], "sha256_16": "2e18b47c963aca57",
                "bytes": 25088589824},
    "decode": {"sources": ["ffn_tc.cu", "tc_ptx.cuh"], "sha256_16": "ec94ad3d0984b261",
               "bytes": 5580442771},
    "decode_fp8": {"sources": ["ffn_fp8.cu", "tc_ptx.cuh", "fp8.cuh"],
                   "sha256_16": "1c554e5f6c0387c9", "bytes": 2790912240},
    "prefill_fp8": {"sources": ["ffn_fp8_swap.cu", "ffn_fp8.cu", "fp8.cu", "tc_ptx.cuh"],
                    "sha256_16": "de840ae3f400969f", "bytes": 13571117056},
}


def sources_sha(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "combine_dp_gather_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="prefill",
                    help="decode | prefill | eplb | tiny | pad_sweep[:mix:tokens_per_req:mode]")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--experts", type=int, default=None,
                    help="shrink the layer to this many experts at the same rows per expert "
                         "(small cases for profiling)")
    ap.add_argument("--shared", type=int, default=0,
                    help="shared experts, always selected with weight 1 (0 = none)")
    ap.add_argument("--boundary", default="plain", choices=["plain", "addnorm"],
                    help="addnorm: residual add + RMSNorm fused into the hidden-state gather")
    ap.add_argument("--router", default="logits", choices=["logits", "gemm"],
                    help="gemm: router logits from the gate GEMM (W_r N(0, 1/H) plus the "
                         "workload's Zipf bias) fused ahead of top-k instead of given logits")
    ap.add_argument("--stage-every", type=int, default=None,
                    help="record the per-stage CUDA events on every n-th timed step (default: "
                         "every step up to 50 steps, else enough steps for 50 samples; the "
                         "events themselves cost ~2 us each on the device)")
    ap.add_argument("--exec", default="graph", choices=["graph", "eager"],
                    help="graph: each step is a replay of a CUDA graph of the layer (all its "
                         "kernels; captured before the timed region); eager: stream launches")
    ap.add_argument("--combine", default="separate", choices=["fused", "separate"],
                    help="fused: combine + DP scatter through moe_grouped_ffn_combine (in the "
                         "down projection's epilogue with few rows per slot, else its own "
                         "launch inside the call); separate: moe_grouped_ffn, then "
                         "moe_combine_scatter")
    ap.add_argument("--ffn-split", default=None,
                    help="HOT_ROWS:HOT_SMS: the grouped FFN split by slot over two streams "
                         "(slots with >= HOT_ROWS rows on the pair kernel on HOT_SMS SMs, the "
                         "rest on the single-SM kernel beside it); 'none' for one kernel")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 dispatch and grouped FFN (e4m3, UE8M0 scales per 128-token group "
                         "and 128x128 weight block); layer input and output stay bf16")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads of the timed oracle (cpu_baseline and --impl reference); "
                         "0 = every core")
    ap.add_argument("--tokens", type=int, default=None,
                    help="prefill token count (with --experts: many rows, few weights)")
    return ap.parse_args()


def make_spec(name: str, seed: int, experts=None, tokens=None):
    if name == "prefill" and (experts or tokens):
        E = experts or 256
        return synth.spec_prefill(T=tokens or 8192 * E // 256, E=E)
    if name == "decode":
        spec = synth.spec_decode(seed=seed)
        if experts:
            spec.E = experts
        return spec
    if name == "prefill":
        return synth.spec_prefill()
    if name.startswith("pad_sweep"):
        # pad_sweep[:mix:tokens_per_req:mode], e.g. pad_sweep:mix0:4:static
        parts = name.split(":")
        mix = parts[1] if len(parts) > 1 else "mix1"
        tpr = int(parts[2]) if len(parts) > 2 else 4
        mode = {"sum": synth.PAD_SUM, "max": synth.PAD_MAX, "static": synth.PAD_STATIC}[
            parts[3] if len(parts) > 3 else "max"]
        return synth.spec_pad_sweep(mix, tpr, mode)
    if name == "eplb":
        return synth.spec_eplb()
    return synth.spec_tiny()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
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

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        busy = [s for s in sms if mx and s > 0.5 * mx] or sms
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------------------ native arm
class StepEvents:
    """CUDA events recorded on the launching stream at each stage boundary."""

    def __init__(self, external: bool = False):
        self.marks = []
        self.external = external

    def mark(self, name):
        # external: recorded as a node when the step is captured into a CUDA graph
        e = torch.cuda.Event(enable_timing=True, external=self.external)
        e.record()
        self.marks.append((name, e))

    def durations(self):
        out = {}
        for (a, ea), (b, eb) in zip(self.marks, self.marks[1:]):
            out[b] = ea.elapsed_time(eb)
        return out


def ffn_traffic(args):
    if args.experts is not None or args.tokens is not None or args.seed != 0:
        return None  # recorded for the default workload only
    if args.combine == "fused" or ffn_split_of(args):
        return None  # recorded for the grouped FFN's own launches
    rec = FFN_TRAFFIC.get(args.config + ("_fp8" if args.fp8 else ""))
    if not rec or rec["bytes"] is None:
        return None
    return rec["bytes"] if sources_sha(rec["sources"]) == rec["sha256_16"] else None


def run_native(args, rank, world, local_rank):
    from combine_dp_gather_gb300 import build as cbuild
    from combine_dp_gather_gb300 import moe_dp as md
    if rank == 0 or not os.path.exists(cbuild.LIB):
        cbuild.build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    spec = make_spec(args.config, args.seed, args.experts, args.tokens)
    if args.shared:
        if spec.P is not None and spec.P != spec.E:
            raise SystemExit("--shared is not combined with an expert map")
        spec.n_shared = args.shared
    l2p_np, nrep_np, p2l = synth.make_map(spec)
    x_loc = synth.hidden_states(spec, dev)
    lg_loc = synth.router_logits(spec, dev)
    wgu, wd = synth.expert_weights(spec, p2l, dev)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode, spec.static_bound, spec.tokens_per_req)
    gate_w = gate_b = gate_np = None
    if args.router == "gemm":
        gate_w, gate_b = synth.router_gate(spec, dev)
        gate_np = gate_to_host(gate_w, gate_b)
    layer = md.MoeLayer(
        R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu, w_down=wd,
        max_rows=max(rows, 1), mode=spec.mode, static_bound=spec.static_bound,
        tokens_per_req=spec.tokens_per_req, renormalize=spec.renormalize, align=spec.align,
        l2p=None if l2p_np is None else torch.from_numpy(l2p_np).to(dev),
        nrep=None if nrep_np is None else torch.from_numpy(nrep_np).to(dev),
        n_shared=spec.n_shared, fp8=args.fp8, router_weight=gate_w, router_bias=gate_b,
        fused_combine=(args.combine == "fused" and not args.fp8),
        ffn_split=ffn_split_of(args))
    out = [torch.empty(c, spec.H, device=dev, dtype=wgu.dtype) for c in spec.counts]
    res_loc = None
    if args.boundary == "addnorm":
        gen = torch.Generator(device=dev)
        gen.manual_seed(spec.seed * 1000 + 5)
        res_loc = [torch.randn(c, spec.H, generator=gen, device=dev).to(wgu.dtype)
                   for c in spec.counts]
        layer.norm_gamma = torch.ones(spec.H, device=dev, dtype=wgu.dtype)
    layer.set_counts(spec.counts)
    for _ in range(args.warmup):
        layer.forward(x_loc, lg_loc, out, local_residual=res_loc)
    torch.cuda.synchronize()
    if int(layer.status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.status.item()):#x} after warm-up")

    # ---- timed region: K steps, inputs resident in HBM
    every = stage_every(args)
    use_graph = args.exec == "graph"
    evs = [StepEvents(external=use_graph) if i % every == 0 else None
           for i in range(args.steps)]
    graphs = None
    if use_graph:
        graphs = [layer.capture(x_loc, lg_loc, out, local_residual=res_loc, timings=evs[i])
                  for i in range(args.steps)]
        for g in graphs:       # a graph's first launch also uploads it: keep that untimed
            g.replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.steps):
            if graphs is not None:
                graphs[i].replay()
            else:
                layer.forward(x_loc, lg_loc, out, timings=evs[i], local_residual=res_loc)
        t1.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_total = t0.elapsed_time(t1)
    clocks = clk.summary()
    stage = {}
    for e in evs:
        if e is None:
            continue
        for k, v in e.durations().items():
            stage.setdefault(k, []).append(v)
    stage_ms = {k: statistics.mean(v) for k, v in stage.items()}

    counts_P = layer.counts_P.cpu().numpy()
    touched = int((counts_P > 0).sum())
    routed = int(layer.offsets_P[-1].item())
    T = spec.T
    b = 2 if spec.dtype == "bf16" else 4
    if args.fp8:
        # e4m3 weights + one scale byte per 128x128 block; per routed row: FP8 input row
        # and scales, h written and read back (codes + scales), bf16 output row
        ffn_bytes = touched * 3 * spec.I * spec.H * (1 + 1 / 16384) + routed * (
            spec.H * (1 + 1 / 128) + 2 * spec.I * (1 + 1 / 128) + 2 * spec.H)
        if fp8_pair(layer.cap, layer.P, spec.H, spec.I):
            # h also goes through HBM in fp32: written by MM1, read by its quantisation
            ffn_bytes += routed * 8 * spec.I
    else:
        ffn_bytes = touched * 3 * spec.I * spec.H * b + routed * (2 * spec.H + 2 * spec.I) * b
        if layer.fused_combine:
            # the call's combine: the routed rows read back, T rows written, inv and w
            kk = spec.k + spec.n_shared
            ffn_bytes += T * kk * spec.H * b + T * spec.H * b + T * kk * 8
    # the combine runs inside the grouped-FFN call's down projection (no launch of its own)
    in_epi = layer.fused_combine and md.moe_grouped_ffn_combine_in_epilogue(
        layer.cap, layer.P, layer.dtype)
    ffn_flops = synth.flops_ffn(T, spec.k + spec.n_shared, spec.H, spec.I)
    ffn_ms = stage_ms["ffn"]
    pk = peaks()
    # an FP8 contraction takes the bf16 measured peak x 2 (the nominal fp8:bf16 ratio)
    tc_peak = pk["bf16_tflops"] * (2 if args.fp8 else 1)
    intensity = ffn_flops / ffn_bytes
    hbm_bound = intensity < (tc_peak * 1e12) / (pk["hbm_gbs"] * 1e9)
    if hbm_bound:
        achieved = ffn_bytes / (ffn_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4)}
    else:
        achieved = ffn_flops / (ffn_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(achieved / tc_peak, 4)}
    tflops = ffn_flops / (ffn_ms * 1e-3) / 1e12
    # attainable at this intensity: min(tensor peak, intensity x HBM bandwidth)
    attainable = min(tc_peak, intensity * pk["hbm_gbs"] / 1e3)
    roof.update({"traffic": ffn_traffic(args),
                 "kernel": ((f"moe_grouped_ffn_fp8 ({ffn_kernel(layer.cap, layer.P, True, spec.H, spec.I)} "
                             "MM1+SwiGLU and MM2 launches with block-scaled MMAs, h quantised "
                             "by its own launch between them)"
                             if fp8_pair(layer.cap, layer.P, spec.H, spec.I) else
                             (f"moe_grouped_ffn_fp8 ({ffn_kernel(layer.cap, layer.P, True, spec.H, spec.I)}: "
                              "pair launches with h quantised between them, then one launch)")
                             if fp8_split(layer.cap, layer.P, spec.H, spec.I) else
                             f"moe_grouped_ffn_fp8 ({ffn_kernel(layer.cap, layer.P, True)}: "
                             "MM1+SwiGLU and MM2 in one persistent launch)") if args.fp8 else
                            f"moe_grouped_ffn_combine ({ffn_kernel(layer.cap, layer.P)} "
                            "MM1+SwiGLU and MM2 launches; combine + DP scatter in MM2's "
                            "epilogue)" if layer.fused_combine and in_epi else
                            f"moe_grouped_ffn_combine ({ffn_kernel(layer.cap, layer.P)} "
                            "MM1+SwiGLU and MM2 launches, then the combine + DP scatter "
                            "launch)" if layer.fused_combine else
                            "moe_grouped_ffn_split (slots with >= {} rows: ffn_swap_kernel on "
                            "{} SMs of a second stream; the rest: ffn_tc_kernel beside it; "
                            "MM1+SwiGLU and MM2 launches each)".format(*layer.ffn_split)
                            if layer.ffn_split else
                            f"moe_grouped_ffn ({ffn_kernel(layer.cap, layer.P)} MM1+SwiGLU "
                            "and MM2 launches)"),
                 "tflops": round(tflops, 1),
                 "frac_of_bf16_peak": round(tflops / pk["bf16_tflops"], 4),
                 "frac_of_bf16_sustained": (round(tflops / pk["bf16_tflops_sustained"], 4)
                                            if pk.get("bf16_tflops_sustained") else None),
                 "frac_of_hbm_roofline": round(tflops / attainable, 4),
                 "intensity_flop_per_byte": round(intensity, 1),
                 "target_frac_of_bf16_peak": None if args.fp8 else 0.60,
                 "peak_source": pk["source"],
                 "algorithmic_bytes": int(ffn_bytes), "algorithmic_flops": int(ffn_flops),
                 "touched_slots": touched, "ffn_ms_per_step": round(ffn_ms, 4),
                 "ffn_samples": len(stage.get("ffn", [])),
                 "permutes": permute_fractions(spec, rows, stage_ms, pk["hbm_gbs"], args.fp8,
                                               layer.fused_combine)})

    # ---- e2e: same calls, inputs from pinned host memory, outputs back to host
    e2e = None
    if not args.no_e2e:
        # Serving-loop form of the same C-ABI calls: every step copies its inputs from
        # pinned host memory and reads its result back; double-buffered device inputs
        # and outputs let the next step's host->device copy and the previous step's
        # device->host read run on copy streams while this step computes.
        hx = [t.cpu().pin_memory() for t in x_loc]
        # with the gate GEMM the logits are computed on the device, not an input
        hl = [t.cpu().pin_memory() for t in lg_loc] if args.router == "logits" else []
        ho = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in out] for _ in range(2)]
        dx = [[torch.empty_like(t) for t in x_loc] for _ in range(2)]
        dl = [[torch.empty_like(t) for t in lg_loc] if args.router == "logits" else lg_loc
              for _ in range(2)]
        dout = [[torch.empty_like(t) for t in out] for _ in range(2)]
        comp = torch.cuda.current_stream()
        s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        fwd_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]

        def h2d(b):
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(fwd_done[b])  # the last step on buffer b read its inputs
                for a, h in zip(dx[b], hx):
                    a.copy_(h, non_blocking=True)
                for a, h in zip(dl[b], hl):
                    a.copy_(h, non_blocking=True)
                if e2e_graphs is not None:  # the step's counts travel with its inputs
                    e2e_graphs[b].stage(spec.counts, stream=s_h2d)
                h2d_done[b].record(s_h2d)

        # graph execution: one graph per buffer set, each with its own counts/offsets
        # buffer that the copy stream fills together with the step's inputs
        for b in range(2):  # capture warms up on these buffers: give them real rows
            for a, t in zip(dx[b] + (dl[b] if args.router == "logits" else []),
                            x_loc + (lg_loc if args.router == "logits" else [])):
                a.copy_(t)
        e2e_graphs = ([layer.capture(dx[b], dl[b], dout[b], local_residual=res_loc)
                       for b in range(2)] if use_graph else None)

        def step(i, n):
            b = i % 2
            comp.wait_event(h2d_done[b])
            comp.wait_event(d2h_done[b])  # dout[b] was read back
            if e2e_graphs is not None:
                e2e_graphs[b].replay()
            else:
                layer.forward(dx[b], dl[b], dout[b], counts=spec.counts, local_residual=res_loc)
            fwd_done[b].record(comp)
            if i + 1 < n:
                h2d(1 - b)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(fwd_done[b])
                for h, a in zip(ho[b], dout[b]):
                    h.copy_(a, non_blocking=True)
                d2h_done[b].record(s_d2h)

        def run(n):
            h2d(0)
            for i in range(n):
                step(i, n)
            comp.wait_event(d2h_done[(n - 1) % 2])

        for ev in fwd_done + d2h_done:
            ev.record(comp)
        run(3)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        run(args.e2e_steps)
        e1.record(comp)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        for a, b in zip(ho[(args.e2e_steps - 1) % 2], out if res_loc is None else []):
            if not torch.equal(a.to(b.device).view(torch.int16) if a.dtype == torch.bfloat16
                               else a.to(b.device), b.view(torch.int16)
                               if b.dtype == torch.bfloat16 else b):
                raise RuntimeError("end-to-end output differs from the device-resident run")
        h2d_b = sum(t.numel() * t.element_size() for t in hx + hl) + 4 * (2 * spec.R + 1)
        d2h_b = sum(t.numel() * t.element_size() for t in ho[0])
        e2e = {"ms_total": e2e_ms, "steps": args.e2e_steps, "h2d": h2d_b, "d2h": d2h_b}
    if int(layer.status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.status.item()):#x}")
    extra = {}
    if spec.mode != synth.PAD_SUM or args.config.startswith("pad_sweep"):
        # padding overhead: rows the global buffer carries that hold no token
        extra["wasted_row_fraction"] = round((rows - spec.T) / max(rows, 1), 4)
    if spec.P is not None and spec.P != spec.E:
        loads = md.moe_range_loads(counts_P.tolist(), spec.n_ranges)
        # the same routing on the trivial layout (slot = logical id, E slots in
        # n_ranges equal ranges): the per-slot counts summed over each logical
        # expert's replicas
        logical = md.moe_logical_counts(counts_P.tolist(), p2l.tolist(), spec.E)
        triv = md.moe_range_loads(logical, spec.n_ranges)
        extra["range_loads"] = loads
        extra["balancedness"] = round(md.moe_balancedness(loads), 4)
        extra["balancedness_trivial_layout"] = round(md.moe_balancedness(triv), 4)
    return dict(spec=spec, ms_total=ms_total, clocks=clocks, stage_ms=stage_ms, roof=roof,
                extra=extra,
                e2e=e2e, rows=rows, touched=touched,
                launches=launches_per_step(max(rows, 1), spec.k + spec.n_shared,
                                           spec.E + spec.n_shared, layer.P, layer.cap,
                                           spec.align, args.fp8, args.router == "gemm",
                                           torch.cuda.get_device_properties(dev).multi_processor_count,
                                           bool(in_epi), bool(layer.ffn_split),
                                           fp8_pair(layer.cap, layer.P, spec.H, spec.I),
                                           fp8_split(layer.cap, layer.P, spec.H, spec.I)),
                inputs=(x_loc, lg_loc, wgu, wd, l2p_np, nrep_np), gate=gate_np)


def ffn_split_of(args):
    """(hot_rows, hot_sms) of --ffn-split, or None."""
    if not args.ffn_split or args.ffn_split == "none" or args.fp8:
        return None
    a, b = args.ffn_split.split(":")
    return int(a), int(b)


def stage_every(args) -> int:
    """Timed steps between two recordings of the stage events: every step up to 50
    steps, else enough steps for 50 samples."""
    if args.stage_every is not None:
        return max(1, args.stage_every)
    return max(1, args.steps // 50)


def permute_fractions(spec, rows: int, stage_ms: dict, hbm_gbs: float, fp8: bool = False,
                      fused_combine: bool = False):
    """Algorithmic bytes of the layer's row-moving stages over their live stage time
    (CUDA events on the launching stream, launch gaps included), against the measured
    HBM copy bandwidth.  T real tokens, `rows` global rows, kk routed slots per token,
    b bytes per element:
      gather (+ routing of every row): read T rows and write `rows` rows of H, read the
        T rows' logits (E x 4 B), write ids and weights (kk x 8 B per row);
      dispatch (stable sort + row copy): read T rows, write their T x kk copies, read
        ids and write perm and inv (12 B per routed pair); on FP8 the copies are e4m3
        codes plus one scale byte per 128 values;
      combine + scatter: read the T x kk expert rows, write T rows, read inv and w
        (8 B per routed pair)."""
    b = 2 if spec.dtype == "bf16" else 4
    kk, T, H, E = spec.k + spec.n_shared, spec.T, spec.H, spec.E
    copy_row = H * (1 + 1 / 128) if fp8 else H * b
    algo = {
        "gather": T * H * b + rows * H * b + T * E * 4 + rows * kk * 8,
        "dispatch": T * H * b + T * kk * copy_row + T * kk * 12,
        "combine_scatter": T * kk * H * b + T * H * b + T * kk * 8,
    }
    out = {}
    for name, nbytes in algo.items():
        ms = stage_ms.get(name)
        if not ms:
            continue
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                     "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_gbs, 4)}
    if fused_combine:
        out["combine_scatter"] = ("inside the moe_grouped_ffn_combine call (its bytes are "
                                  "counted in the FFN's)")
    out["target_frac_of_hbm"] = 0.70
    out["peak_gbs"] = hbm_gbs
    return out


# ------------------------------------------------------------------ oracle (CPU)
def oracle_sample_step(spec, n_tokens, x_loc, lg_loc, wgu, wd, l2p, nrep, fp8=False, gate=None):
    """One oracle pass over the first n_tokens tokens of the workload (replica
    order, MAX/SUM/static layout of the truncated counts).  With fp8 the permuted
    rows are quantised (timed) and the experts run on FP8 operands (weight
    quantisation is preparation, not timed).  With gate = (W_r, bias) the router
    logits come from the oracle's gate projection (timed) instead of the given
    logits.  Returns (seconds of oracle compute, cpu seconds)."""
    import oracle
    counts, left = [], n_tokens
    for c in spec.counts:
        counts.append(min(c, left))
        left -= counts[-1]

    def bits(t):
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    to32 = (lambda t: oracle.bf16_bits_to_f32(bits(t))) if spec.dtype == "bf16" else (
        lambda t: t.detach().cpu().numpy())
    xs = [to32(x[:c]) for x, c in zip(x_loc, counts)]
    lgs = [lg[:c].detach().cpu().numpy() for lg, c in zip(lg_loc, counts)]
    w0, c0 = time.perf_counter(), time.process_time()
    offs, rows = oracle.dp_layout(counts, spec.mode, spec.static_bound, spec.tokens_per_req)
    valid = oracle.valid_rows(counts, offs, rows)
    xg = oracle.dp_gather(xs, counts, offs, rows)
    if gate is None:
        lg = oracle.dp_gather(lgs, counts, offs, rows)
    else:
        lg = oracle.router_logits(xg, gate[0], gate[1])
    ids, w = oracle.route_topk(lg, spec.k, spec.renormalize, valid, spec.n_shared)
    cnt, o, perm, inv = oracle.dispatch(ids, spec.E + spec.n_shared, spec.slots, l2p, nrep,
                                        spec.align)
    xsrt = oracle.permute_rows(xg, perm[: o[-1]])
    if fp8:
        xq, xe = oracle.quant_groups(xsrt)
    wall = time.perf_counter() - w0
    cpu = time.process_time() - c0
    ys = np.zeros(xsrt.shape, np.float64)
    for s in range(spec.slots):
        a, b_ = int(o[s]), int(o[s + 1])
        if b_ == a:
            continue
        wg_s, wd_s = to32(wgu[s]), to32(wd[s])        # input conversion, not timed
        if fp8:
            wq = (*oracle.quant_blocks(wg_s), *oracle.quant_blocks(wd_s))
        w0, c0 = time.perf_counter(), time.process_time()
        if fp8:
            ys[a:b_] = oracle.expert_ffn_fp8(xq[a:b_], xe[a:b_], *wq)
        else:
            ys[a:b_] = oracle.expert_ffn(xsrt[a:b_], wg_s, wd_s)
        wall += time.perf_counter() - w0
        cpu += time.process_time() - c0
    w0, c0 = time.perf_counter(), time.process_time()
    yg = oracle.combine(ys, inv, w)
    oracle.dp_scatter(yg, counts, offs)
    wall += time.perf_counter() - w0
    cpu += time.process_time() - c0
    return wall, cpu


def oracle_inputs(spec):
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    l2p, nrep, p2l = synth.make_map(spec)
    x_loc = synth.hidden_states(spec, dev)
    lg_loc = synth.router_logits(spec, dev)
    wgu, wd = synth.expert_weights(spec, p2l, dev)
    return x_loc, lg_loc, wgu, wd, l2p, nrep


def gate_to_host(w, b):
    """Gate weights as exact float32 host arrays for the oracle (bias may be None)."""
    import oracle
    wb = w.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return oracle.bf16_bits_to_f32(wb), (None if b is None else b.cpu().numpy().astype(np.float32))


def cpu_baseline(spec, budget_s=20.0, inputs=None, fp8=False, gate=None, threads=0):
    import oracle
    oracle.build()
    oracle.set_threads(threads)
    x_loc, lg_loc, wgu, wd, l2p, nrep = inputs or oracle_inputs(spec)
    wall1, _ = oracle_sample_step(spec, 1, x_loc, lg_loc, wgu, wd, l2p, nrep, fp8, gate)
    n = int(max(1, min(spec.T, budget_s / max(wall1, 1e-3))))
    wall, cpu = oracle_sample_step(spec, n, x_loc, lg_loc, wgu, wd, l2p, nrep, fp8, gate)
    ffn = "FP8 (e4m3) SwiGLU FFN in fp64" if fp8 else "fp64 SwiGLU FFN"
    return {"value": round(n / wall, 3), "unit": UNIT, "cores": round(cpu / wall, 2),
            "kind": "oracle",
            "sample": f"first {n} of the {spec.T} tokens of {spec.name}, whole layer (gather, "
                      f"top-{spec.k}, dispatch, {ffn}, combine, scatter), "
                      f"{wall:.1f} s wall; cores = CPU time / wall time"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    spec = make_spec(args.config, args.seed, args.experts, args.tokens)
    import oracle
    oracle.build()
    oracle.set_threads(args.cpu_threads)
    inputs = oracle_inputs(spec)
    gate = gate_to_host(*synth.router_gate(spec, "cpu")) if args.router == "gemm" else None
    wall1, _ = oracle_sample_step(spec, 1, *inputs, args.fp8, gate)
    budget = 120.0
    n = int(max(1, min(spec.T, budget / (args.steps + args.warmup) / max(wall1, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_step(spec, n, *inputs, args.fp8, gate)
    walls, cpus = [], []
    for _ in range(args.steps):
        w, c = oracle_sample_step(spec, n, *inputs, args.fp8, gate)
        walls.append(w)
        cpus.append(c)
    tot = sum(walls)
    value = n * args.steps / tot
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": dict(synth.describe(spec), sample_tokens_per_step=n,
                           fp8="e4m3 operands, fp64 arithmetic" if args.fp8 else None),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT,
                             "cores": round(sum(cpus) / tot, 2), "kind": "oracle",
                             "sample": f"first {n} tokens of {spec.name} per step"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main
def aggregate(ms_total: float, tokens: float, e2e_ms: float, world: int, device):
    """Whole-job figures: the slowest rank's times and the tokens of all ranks."""
    t = torch.tensor([ms_total, e2e_ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(n, op=torch.distributed.ReduceOp.SUM)
    return {"ms_max": float(t[0].item()), "e2e_ms_max": float(t[1].item()),
            "tokens": float(n.item())}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    if world > 1:
        backend = "nccl" if args.impl == "native" else "gloo"
        if args.impl == "native":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        r = run_native(args, rank, world, local_rank)
        spec = r["spec"]
        agg = aggregate(r["ms_total"], spec.T * args.steps,
                        r["e2e"]["ms_total"] if r["e2e"] else 0.0, world,
                        torch.device("cuda", local_rank))
        if rank != 0:
            return
        ms_total = agg["ms_max"]
        value = agg["tokens"] / (ms_total / 1e3)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8-e4m3" if args.fp8 else spec.dtype, "data": "synthetic",
            "config": dict(synth.describe(spec), global_rows=r["rows"], l2=L2_NOTE, **r["extra"],
                           ffn_split=("slots with >= %d rows on %d SMs of a second stream"
                                      % ffn_split_of(args) if ffn_split_of(args) else None),
                           boundary=args.boundary, shared_experts=spec.n_shared,
                           router=("gate GEMM fused ahead of top-k, W_r N(0, 1/H) plus the Zipf "
                                   "bias" if args.router == "gemm" else "given logits"),
                           execution=("CUDA graph of the layer step, replayed" if args.exec == "graph"
                                      else "stream launches"),
                           stage_events=f"every {stage_every(args)}th timed step",
                           fp8=("e4m3 codes, UE8M0 scales per 128-token group and 128x128 "
                                "weight block; bf16 layer input/output") if args.fp8 else None,
                           parallelism=f"{world} independent replica(s), one per GPU",
                           stage_ms={k: round(v, 4) for k, v in r["stage_ms"].items()}),
            "roofline": r["roof"],
            "clocks": r["clocks"],
            "gpu_launches": args.steps * r["launches"],
        }
        if r["e2e"]:
            e = r["e2e"]
            e2e_val = float(spec.T * e["steps"] * world) / (agg["e2e_ms_max"] / 1e3)
            line["e2e"] = {"value": round(e2e_val, 1), "unit": UNIT,
                           "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                           "ms_per_step": round(agg["e2e_ms_max"] / e["steps"], 4)}
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(spec, inputs=r["inputs"], fp8=args.fp8,
                                                gate=r["gate"], threads=args.cpu_threads)
        print(json.dumps(line), flush=True)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

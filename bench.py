"""Benchmark of the AWQ int4 MoE expert stage on GB300.

Workload (the line's `value`): the decode sweep on the single-layer decode
shape -- E=512 experts, top-10, hidden 2560, intermediate 160, int4 group-32
with 4-byte metadata -- at M = 1, 2, 4, 8 tokens under two routing regimes,
"hot" (every token picks the same 10 experts) and "rotating" (iid router
logits, so the union grows towards 80 experts). Each layer call is one pass
of the whole hot path: routing metadata, W13 + SwiGLU, W2 + weighted top-k
sum.

A round is one replay, for each case, of a CUDA graph holding a stack of 48
independently seeded layers (18.9 GB of weight banks), so weights stream
cold from HBM (inputs larger than L2; no flush needed). A step is R rounds,
R chosen so that the K timed steps last at least about a second. Metric:
microseconds per layer call and effective HBM GB/s, where the effective
bytes of a call are the packed weights plus metadata of its distinct active
experts (768,000 B each); value = total effective bytes / total time.

The `configs` block of the same line times the other workload
configurations the same way, each on its own 48-layer stack: compact 3-byte
metadata (M = 1, 8), the prefill-sized Zipf(1.1) batches (M = 128, 256, 512;
on the path AWQ_PATH_AUTO takes and on the tensor-core prefill path), NVFP4
weights, and the unsharded intermediate 640 with 3-byte metadata
(M = 1..16).

After the timed regions one sampled layer of every case is compared with the
FP64 CPU oracle (outside the timing); a mismatch ends the run with an error.
Then the same graphs are rebuilt with every layer call replaced by
awq_moe_latency_floor (the call's dependency chain with no arithmetic: ids,
one bulk read of the active experts' banks, a grid barrier, the output rows)
and timed the same way: each case row's `latency_floor_us` and the
roofline's `latency_floor` block say how far the layer kernels sit above
what that chain costs on this GPU.

Flags: --gpus N --steps K --warmup W [--impl reference] [--layers L]
[--cases 8:rotating,...] [--no-configs]. Under torchrun each rank runs an
independent replica (the stage does not shard: no collective), timing is max
over ranks.
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

import synth  # noqa: E402

METRIC = "µs per MoE layer call and effective HBM GB/s (% of peak) at M=1..8, E512 top-10"
WORKLOAD = "decode sweep M=1,2,4,8 x {hot, rotating}, E512 top-10 H2560 I160 int4 g32 4-byte meta"
DEFAULT_CASES = [(1, "hot"), (1, "rotating"), (2, "hot"), (4, "hot"), (8, "hot"),
                 (2, "rotating"), (4, "rotating"), (8, "rotating")]
# The other workload configurations, reported in the line's `configs` block.
CONFIGS = [
    ("compact_3byte", dict(meta_bytes=3, inter=160, cases=[(1, "rotating"), (8, "hot"), (8, "rotating")])),
    ("prefill_zipf_M128", dict(meta_bytes=4, inter=160, cases=[(128, "zipf")])),
    ("prefill_zipf_M128_tc", dict(meta_bytes=4, inter=160, cases=[(128, "zipf")], path="prefill")),
    ("prefill_zipf_M512", dict(meta_bytes=4, inter=160, cases=[(256, "zipf"), (512, "zipf")])),
    ("prefill_zipf_M512_tc", dict(meta_bytes=4, inter=160, cases=[(256, "zipf"), (512, "zipf")], path="prefill")),
    # NVFP4 weights (E2M1 codes, E4M3 scales per 16 K, fp32 globals): decode
    # and prefill-sized batches on the path AWQ_PATH_AUTO takes (the fused
    # kernel up to 16 tokens, hybrid above), decode on the hybrid path, and
    # batches on the tensor-core prefill path
    ("nvfp4_g16_decode", dict(group=16, meta_bytes=1, inter=160,
                              cases=[(1, "rotating"), (2, "hot"), (4, "rotating"), (8, "hot"), (8, "rotating")])),
    ("nvfp4_g16_decode_hybrid", dict(group=16, meta_bytes=1, inter=160, path="hybrid",
                                     cases=[(1, "rotating"), (8, "rotating")])),
    ("nvfp4_g16_zipf", dict(group=16, meta_bytes=1, inter=160, cases=[(128, "zipf"), (256, "zipf"), (512, "zipf")])),
    ("nvfp4_g16_zipf_tc", dict(group=16, meta_bytes=1, inter=160, path="prefill",
                               cases=[(128, "zipf"), (512, "zipf")])),
    ("inter640_3byte", dict(meta_bytes=3, inter=640,
                            cases=[(1, "rotating"), (2, "rotating"), (4, "rotating"), (8, "rotating"),
                                   (16, "rotating")])),
]
BASE_SEED = 7
MIN_TIMED_S = 1.2          # the K timed steps last at least this long


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--layers", type=int, default=48)
    p.add_argument("--cases", default=None,
                   help="comma list of M:regime (default: the eight sweep cases)")
    p.add_argument("--meta-bytes", type=int, default=4, choices=[3, 4])
    p.add_argument("--inter", type=int, default=160, choices=[160, 640])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workload configurations")
    p.add_argument("--no-check", action="store_true",
                   help="skip the post-timing oracle check of sampled layers")
    p.add_argument("--stage-breakdown", action="store_true",
                   help="also time the three-launch path's W13 and W2 kernels alone")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--router", action="store_true",
                   help="route on the device from the router logits (awq_moe_layer_logits) "
                        "instead of passing top-k ids and weights; no e2e leg")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--path", default="auto", choices=["auto", "fused", "sliced", "staged", "prefill", "hybrid"],
                   help="execution path of the layer call (awq_moe_layer_ex); auto is what awq_moe_layer takes")
    p.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S)
    return p.parse_args(argv)


def parse_cases(s):
    if not s:
        return list(DEFAULT_CASES)
    out = []
    for part in s.split(","):
        m, r = part.split(":")
        out.append((int(m), r))
    return out


# ------------------------------------------------------------------ helpers

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (the job's time is the slowest
    replica's); the tensor lives where the process group's backend wants it."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else device
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job rate: every rank (an independent replica) processes
    `units_per_rank` in the slowest rank's `seconds`."""
    return world * units_per_rank / seconds


def case_row(M, regime, active, step_bytes, graph_ms, layers, peak):
    """One case of the sweep: `graph_ms` is the median time of one replay of
    the graph of all `layers` layer calls (with 48 layers, the MoE time of a
    whole decode step), `step_bytes` the weight bytes that replay streams."""
    gbs = step_bytes / (graph_ms * 1e-3) / 1e9
    return {"M": M, "regime": regime, "mean_active_experts": float(np.mean(active)),
            "us_per_call": round(graph_ms * 1e3 / layers, 3), "effective_GBps": round(gbs, 1),
            "pct_of_hbm_peak": round(100 * gbs / peak, 1),
            "layers_step_ms": round(graph_ms, 4)}


def l2_label(layers: int, case_bytes, l2_bytes: int) -> str:
    """How the timed weight stream meets the L2: cold when every case streams
    more weight bytes per step than the L2 holds (a layer's experts are
    evicted before the next step reads them again), else which cases are
    L2-warm (their numbers are not cold-HBM figures)."""
    mb = l2_bytes / 1e6
    small = [i for i, b in enumerate(case_bytes) if b <= l2_bytes]
    if not small:
        return (f"inputs larger than L2: {layers}-layer stack streamed cold, no flush "
                f"(each case streams >= {min(case_bytes) / 1e6:.0f} MB of weights per step; L2 {mb:.0f} MB)")
    return (f"L2-warm: case(s) {small} stream at most {l2_bytes / 1e6:.0f} MB of weights per step "
            f"({layers} layer(s)), so their weights stay in L2; not cold-HBM figures")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []                 # (host monotonic time, csv line)
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def wait_first(self, timeout=5.0):
        """Block until nvidia-smi printed its first sample (it takes a moment
        to start), so that the timed region is sampled from its beginning."""
        t0 = time.monotonic()
        while self.proc is not None and not self.lines and time.monotonic() - t0 < timeout:
            time.sleep(0.01)

    def mark(self, t_start, t_stop):
        self.window = (t_start, t_stop)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.window is not None:
            # samples taken while the timed region ran (one period of slack)
            lo, hi = self.window
            inside = [(t, ln) for t, ln in lines if lo <= t <= hi + 0.025]
            lines = inside if inside else lines
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


KERNEL_FILES = {"fused_layer_kernel": "awq_moe_fused.cu", "sliced_layer_kernel": "awq_moe_sliced.cu"}


def kernel_source_hash(kernel="fused_layer_kernel"):
    """Hash of a persistent kernel's sources (its file and the device headers)
    with comments and blank space removed, so that neither an edit of
    comments nor one of the host code or of other kernels voids a profile of
    unchanged kernel code."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "awq_int4_moe_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name == KERNEL_FILES.get(kernel) or name.endswith(".cuh"):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(name.encode())
            h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, active_experts_per_launch: float):
    """Per-launch DRAM bytes (read + write) of `kernel` from the committed ncu
    capture in profiles/traffic.json, if it was taken on the current kernel
    sources (else None). The capture is of one smaller launch; its bytes per
    active expert are scaled to the mean active experts of a bench launch
    (the traffic grows in proportion to the experts streamed)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if ent and ent.get("source_hash") == kernel_source_hash(kernel):
            return round(ent["dram_bytes_per_active_expert"] * active_experts_per_launch)
    except (OSError, ValueError, KeyError):
        pass
    return None


# ------------------------------------------------------------------ workload

class LayerStack:
    """`layers` independently seeded layers resident on the device, in the
    prepared layout (each layer generated into one reused canonical scratch
    set, then permuted by awq_moe_prepare_weights, as a loader would do once)."""

    def __init__(self, layers, shape, seed, device):
        import torch

        import awq_int4_moe_gb300 as awq
        import synth.device as sd
        E, H, I, G, mb = shape.num_experts, shape.hidden, shape.inter, shape.group, shape.meta_bytes
        self.shape, self.seed, self.layers = shape, seed, layers
        self.banks, self.weights = [], []
        canon = (torch.empty((E, H // 8, 2 * I), dtype=torch.int32, device=device),
                 torch.empty((E, H // G, 2 * I, mb), dtype=torch.uint8, device=device),
                 torch.empty((E, I // 8, H), dtype=torch.int32, device=device),
                 torch.empty((E, I // G, H, mb), dtype=torch.uint8, device=device))
        c_shape = awq.Shape.of(shape)
        self.globals = []
        for layer in range(layers):
            sd.fill_layer(shape, seed, layer, *canon)
            bank = tuple(torch.empty_like(t) for t in canon)
            w = awq.moe_prepare_weights(c_shape, awq.Weights.of(*canon), awq.Weights.of(*bank),
                                        torch.cuda.current_stream())
            if G == 16:     # NVFP4 banks: per-expert global scales of the layer
                g = torch.from_numpy(synth.nvfp4_global(seed, layer, E)).to(device)
                w.global_scale = g.data_ptr()
                self.globals.append(g)
            self.banks.append(bank)
            self.weights.append(w)
        torch.cuda.synchronize()
        del canon

    def bytes(self):
        return sum(sum(t.numel() * t.element_size() for t in b) for b in self.banks)


def case_seed(seed, M, regime):
    return seed + M * 1000 + {"hot": 0, "rotating": 500, "zipf": 700}[regime]


def case_inputs(seed, layers, M, regime, shape, with_logits=False):
    """Per layer: x, top-k ids and weights (the harness's router on the seeded
    logits), and, when asked, the logits themselves."""
    xs, ids, ws, lgs = [], [], [], []
    cs = case_seed(seed, M, regime)
    for layer in range(layers):
        x = synth.hidden_states(cs, layer, M, shape.hidden)
        lg = synth.router_logits(cs, layer, M, shape.num_experts, regime, shape.top_k)
        i, w = synth.router_topk(lg, shape.top_k)
        xs.append(x)
        ids.append(i)
        ws.append(w)
        if with_logits:
            lgs.append(lg)
    return (xs, ids, ws, lgs) if with_logits else (xs, ids, ws)


def distinct(ids):
    return len(set(int(v) for v in np.asarray(ids).ravel()))


def make_case(M, regime, stack, device, router=False):
    """Inputs of one case for every layer of `stack`, on the device: one
    tensor per input kind (per-layer views), so a host step moves each kind in
    one copy; plus the output buffer of every layer."""
    import torch
    shape, L = stack.shape, stack.layers
    xs, ids, wts, lgs = case_inputs(stack.seed, L, M, regime, shape, with_logits=True)
    A = [distinct(i) for i in ids]
    x_all = torch.from_numpy(np.stack([x.view(np.int16) for x in xs])).to(device)
    i_all = torch.from_numpy(np.stack(ids)).to(device)
    w_all = torch.from_numpy(np.stack(wts)).to(device)
    out = torch.empty((L, M, shape.hidden), dtype=torch.int16, device=device)
    return dict(M=M, regime=regime, xs=xs, ids=ids, wts=wts, A=A,
                x_d=list(x_all.unbind(0)), i_d=list(i_all.unbind(0)), w_d=list(w_all.unbind(0)),
                l_d=[torch.from_numpy(lg).to(device) for lg in lgs] if router else None,
                x_all=x_all, i_all=i_all, w_all=w_all, out=out,
                bytes=sum(A) * shape.expert_bytes())


PATHS = {"auto": 0, "fused": 1, "staged": 2, "sliced": 3, "prefill": 4, "hybrid": 5}


def enqueue_layers(case, stack, ws, ws_bytes, status, stream, router=False, path="auto"):
    """Enqueue the layer calls of every layer of the stack, in order, on
    `stream` (one awq_moe_layer, or awq_moe_layer_logits, per layer), all on
    the one workspace -- exactly what a decode step does. `path` other than
    "auto" forces an execution path through awq_moe_layer_ex."""
    import awq_int4_moe_gb300 as awq
    c_shape = awq.Shape.of(stack.shape)
    for layer in range(stack.layers):
        if router:
            # the router's choice is written over the harness's ids/weights
            awq.moe_layer_logits(case["x_d"][layer], case["l_d"][layer], case["M"], c_shape,
                                 stack.weights[layer], case["out"][layer], case["i_d"][layer],
                                 case["w_d"][layer], ws, ws_bytes, status, path=PATHS[path], stream=stream)
        elif path == "auto":
            awq.moe_layer(case["x_d"][layer], case["i_d"][layer], case["w_d"][layer], case["M"], c_shape,
                          stack.weights[layer], case["out"][layer], ws, ws_bytes, status, stream)
        else:
            awq.moe_layer_ex(case["x_d"][layer], case["i_d"][layer], case["w_d"][layer], case["M"], c_shape,
                             stack.weights[layer], case["out"][layer], ws, ws_bytes, status, path=PATHS[path],
                             stream=stream)


def capture_stack_graph(case, stack, ws, ws_bytes, status, stream, router=False, path="auto"):
    """One CUDA graph of all layer calls of the stack for `case` (programmatic
    dependent launch between consecutive calls is kept inside the graph)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue_layers(case, stack, ws, ws_bytes, status, stream, router, path)
    return g


PREFILL_KERNELS = ("w13_tc_kernel", "w2_tc_kernel", "combine_kernel")
HYBRID_MAX_TOKENS = 512          # AWQ_PATH_AUTO: hybrid path for 17..512 tokens (int4 and NVFP4 banks)


def kernel_of(M, top_k, sms, path="auto", inter=160, nvfp4=False):
    """The kernel one layer call of M tokens launches (auto path rules of
    awq_moe_layer_ex; NVFP4 banks take the fused kernel up to 16 tokens and
    the hybrid path above)."""
    if nvfp4 and path == "auto":
        path = "fused" if M <= 16 else "hybrid" if M <= HYBRID_MAX_TOKENS else "prefill"
    sliced_auto = M * top_k <= sms and (M == 2 or (M == 1 and inter == 160))
    if path == "sliced" or (path == "auto" and sliced_auto):
        return "sliced_layer_kernel"
    if path == "fused" or (path == "auto" and M <= 16):
        return "fused_layer_kernel"
    if path == "prefill" or (path == "auto" and M > HYBRID_MAX_TOKENS):
        return "route_kernel + " + " + ".join(PREFILL_KERNELS)
    if path == "hybrid" or path == "auto":
        return "route_kernel + w13_swiglu_kernel + " + " + ".join(PREFILL_KERNELS[1:])
    return "route_kernel + w13_swiglu_kernel + w2_reduce_kernel"


def tc_path_of(kernels):
    """"prefill" or "hybrid" when every launch list is that path's, else None."""
    if all(k.startswith("route_kernel + w13_tc") for k in kernels):
        return "prefill"
    if all(k.startswith("route_kernel + w13_swiglu") and k.endswith("combine_kernel") for k in kernels):
        return "hybrid"
    return None


def oracle_check(case, stack, layer):
    """Compare layer `layer` of `case`'s output buffer with the FP64 oracle at
    |gpu - oracle| <= 4e-3 + 1e-2 |oracle|; returns (ok, max abs error)."""
    import oracle
    shape = stack.shape
    ref, _ = oracle.layer_from_synth(shape, stack.seed, layer, case["xs"][layer], case["ids"][layer],
                                     case["wts"][layer])
    got = case["out"][layer].cpu().numpy().view(np.float16).astype(np.float64)
    err = np.abs(got - ref)
    return bool(np.all(err <= 4e-3 + 1e-2 * np.abs(ref))), float(err.max())


def sampled_check(per_case, stack, tag):
    """One sampled layer per case against the oracle (after the timing)."""
    rows = []
    for i, c in enumerate(per_case):
        layer = (7 * i + 3) % stack.layers
        ok, err = oracle_check(c, stack, layer)
        rows.append({"case": f"M={c['M']} {c['regime']}", "layer": layer, "max_abs_err": err, "ok": ok})
        if not ok:
            raise RuntimeError(f"{tag}: layer {layer} of M={c['M']} {c['regime']} differs from the "
                               f"oracle (max abs err {err:.3e})")
    return rows


# ------------------------------------------------------------------ our arm

def time_rounds(per_case, stream, rounds):
    """Replay every case's graph `rounds` times; per-replay event times."""
    import torch
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(rounds):
            for c in per_case:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                c["graph"].replay()
                e1.record(stream)
                evs.append((c, e0, e1))
    return evs


def latency_floor(per_case, stack, ws, ws_bytes, status, stream, reps):
    """Time, for each decode-sized case (M <= 16), a graph of the stack's
    layer calls replaced by awq_moe_latency_floor calls: the persistent
    kernels' dependency chain (ids, one read of the active experts' banks, a
    grid barrier, the output rows) with no arithmetic, on the same workspace
    and stream. Sets c["floor_ms"] (median replay) and returns the summary
    the roofline carries, or None when no case is decode-sized. Run after the
    sweep's checks: it overwrites the cases' outputs with zeros."""
    import torch

    import awq_int4_moe_gb300 as awq
    c_shape = awq.Shape.of(stack.shape)
    dec = [c for c in per_case if c["M"] <= 16]
    if not dec:
        return None

    def enqueue(c):
        for layer in range(stack.layers):
            awq.moe_latency_floor(c["i_d"][layer], c["M"], c_shape, stack.weights[layer], c["out"][layer],
                                  ws, ws_bytes, status, stream=stream)

    for c in dec:
        with torch.cuda.stream(stream):
            enqueue(c)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue(c)
        c["floor_graph"] = g
    torch.cuda.synchronize()
    for _ in range(3):
        for c in dec:
            c["floor_graph"].replay()
    times = {id(c): [] for c in dec}
    with torch.cuda.stream(stream):
        evs = []
        for _ in range(reps):
            for c in dec:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                c["floor_graph"].replay()
                e1.record(stream)
                evs.append((c, e0, e1))
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the latency-floor graphs")
    for c, e0, e1 in evs:
        times[id(c)].append(e0.elapsed_time(e1))
    for c in dec:
        c["floor_ms"] = statistics.median(times[id(c)])
        del c["floor_graph"]
    floor_ms = sum(c["floor_ms"] for c in dec)
    layer_ms = sum(c["graph_ms"] for c in dec)
    b = sum(c["bytes"] for c in dec)
    return {"kernel": "floor_kernel (awq_moe_latency_floor)",
            "cases": len(dec),
            "avg_launch_us": round(floor_ms * 1e3 / (stack.layers * len(dec)), 3),
            "achieved_GBps": round(b / (floor_ms * 1e-3) / 1e9, 1),
            "layer_time_over_floor": round(layer_ms / floor_ms, 3),
            "what": ("same graph of layer calls with each call replaced by its dependency chain alone: "
                     "ids, one bulk read of the active experts' prepared banks, one grid barrier, "
                     "the output rows")}


def fused_roofline(per_case, ev, L, expert_bytes, peak, peak_kind, case_kernels, profiled=True):
    """Dominant kernels of a step whose every layer call is one launch (the
    kernel of each case in `case_kernels`): the average launch duration is the
    graph time per layer call (launch gaps included); algorithmic bytes are the
    distinct active experts' weights; traffic is the mean over the step's
    launches of each case's kernel's profiled DRAM bytes (null unless every
    kernel has a profile of its current sources)."""
    tot_ms = sum(statistics.median(ev[id(c)]) for c in per_case)
    tot_bytes = sum(c["bytes"] for c in per_case)
    launches = L * len(per_case)
    achieved = tot_bytes / (tot_ms * 1e-3) / 1e9
    # the committed captures are of 4-byte int4 launches at intermediate 160
    # (profiled=False for other banks or widths: no traffic figure)
    per = [profiled_traffic(k, sum(c["A"]) / L) if profiled else None for c, k in zip(per_case, case_kernels)]
    traffic = round(sum(per) / len(per)) if per and all(p is not None for p in per) else None
    return {"bound": "hbm", "kernel": " + ".join(sorted(set(case_kernels))), "achieved": round(achieved, 1),
            "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "avg_launch_us": round(tot_ms * 1e3 / launches, 3),
            "algorithmic_bytes": "per launch: distinct active experts x %d B" % expert_bytes}


def run_ours(args, cases, rank, world, local):
    import torch

    import awq_int4_moe_gb300 as awq

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    shape = synth.ExpertShape(num_experts=512, top_k=10, hidden=2560, inter=args.inter,
                              meta_bytes=args.meta_bytes)
    c_shape = awq.Shape.of(shape)
    L = args.layers
    stack = LayerStack(L, shape, BASE_SEED, device)
    expert_bytes = shape.expert_bytes()
    stream = torch.cuda.Stream(device)
    M_max = max(m for m, _ in cases)
    ws_bytes = awq.moe_workspace_bytes(c_shape, M_max)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)

    per_case = [make_case(M, regime, stack, device, args.router) for M, regime in cases]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for c in per_case:
            enqueue_layers(c, stack, ws, ws_bytes, status, stream, args.router, args.path)   # eager warm-up
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    for c in per_case:
        c["graph"] = capture_stack_graph(c, stack, ws, ws_bytes, status, stream, args.router, args.path)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        for c in per_case:
            c["graph"].replay()
    torch.cuda.synchronize()

    # rounds per step: the K timed steps last at least args.min_timed_s
    t0 = time.perf_counter()
    time_rounds(per_case, stream, 2)
    torch.cuda.synchronize()
    round_s = (time.perf_counter() - t0) / 2
    rounds = max(1, math.ceil(args.min_timed_s / max(1e-9, args.steps * round_s)))

    ev = {id(c): [] for c in per_case}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        clocks.wait_first()
        t_host0 = time.monotonic()
        with torch.cuda.stream(stream):
            start = torch.cuda.Event(enable_timing=True)
            start.record(stream)
        events = time_rounds(per_case, stream, args.steps * rounds)
        with torch.cuda.stream(stream):
            stop = torch.cuda.Event(enable_timing=True)
            stop.record(stream)
        torch.cuda.synchronize()
        clocks.mark(t_host0, time.monotonic())
    if world > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(stop)
    for c, e0, e1 in events:
        ev[id(c)].append(e0.elapsed_time(e1))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the timed region")
    total_ms = max_over_ranks(total_ms, world, device)

    peak, peak_kind = measured_peaks()
    case_rows = [case_row(c["M"], c["regime"], c["A"], c["bytes"], statistics.median(ev[id(c)]), L, peak)
                 for c in per_case]
    round_bytes = sum(c["bytes"] for c in per_case)
    step_ms = total_ms / args.steps
    value = job_throughput(round_bytes * rounds, step_ms * 1e-3, world) / 1e9
    clk = clocks.summary()

    sms = torch.cuda.get_device_properties(device).multi_processor_count
    case_kernels = [kernel_of(c["M"], shape.top_k, sms, args.path, shape.inter) for c in per_case]
    fused = args.path not in ("staged", "prefill", "hybrid") and all(c["M"] <= 16 for c in per_case)
    roof = fused_roofline(per_case, ev, L, expert_bytes, peak, peak_kind, case_kernels) if fused else None
    tc_path = tc_path_of(case_kernels)
    if tc_path and not args.router:
        roof = prefill_roofline(args, per_case, stack, ws, ws_bytes, stream, device, peak, peak_kind, tc_path)
    elif args.stage_breakdown or not fused:
        stage = stage_roofline(args, per_case, stack, c_shape, stream, device, peak, peak_kind)
        if roof is None:
            roof = stage
        else:
            roof["staged_path"] = stage

    checks = None if args.no_check else sampled_check(per_case, stack, "sweep")

    e2e = None
    if not args.no_e2e and not args.router:
        e2e = run_e2e(args, per_case, stack, ws, ws_bytes, status, stream, device, world)

    for c in per_case:
        c["graph_ms"] = statistics.median(ev[id(c)])
    floor = latency_floor(per_case, stack, ws, ws_bytes, status, stream, max(5, min(20, args.steps)))
    for c, row in zip(per_case, case_rows):
        if "floor_ms" in c:
            row["latency_floor_us"] = round(c["floor_ms"] * 1e3 / L, 3)
    if roof is not None and floor is not None:
        roof["latency_floor"] = floor

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s (effective HBM)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 weights x fp16 activations, fp32 accumulate",
        "data": "synthetic (seeded counter-based int4 banks, fp16 N(0,0.5) activations, softmax top-10 routing)",
        "config": {"workload": WORKLOAD, "layers": L, "cases": [f"M={m} {r}" for m, r in cases],
                   "meta_bytes": shape.meta_bytes, "inter": shape.inter,
                   "weights_resident_GB": round(stack.bytes() / 1e9, 2),
                   "l2": l2_label(L, [c["bytes"] for c in per_case],
                                  getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 126 << 20)),
                   "parallelism": "replicas only" if world > 1 else "single GPU",
                   "step": (f"{rounds} round(s); a round is one CUDA-graph replay of the {L}-layer stack "
                            "for each case"),
                   "rounds_per_step": rounds,
                   "timed_s": round(total_ms / 1e3, 3),
                   "routing": ("device router from fp32 logits (awq_moe_layer_logits)" if args.router
                               else "top-k ids and weights given (awq_moe_layer)"),
                   "path": args.path},
        "cases": case_rows,
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "hbm_peak_GBps": peak, "hbm_peak_kind": peak_kind,
        "roofline": roof,
        "clocks": clk,
        "e2e": e2e,
        "oracle_checks": checks,
        "gpu_launches": sum(len(k.split(" + ")) + (1 if args.router and k.startswith("route_kernel") else 0)
                            for k in case_kernels)
                        * L * args.steps * rounds,
    }
    del per_case, ws
    if not args.no_configs and args.cases is None:
        del stack
        torch.cuda.empty_cache()
        result["configs"] = run_configs(args, device, stream, peak, peak_kind)
    return result


def run_configs(args, device, stream, peak, peak_kind):
    """The other workload configurations, each on its own 48-layer stack
    (freed before the next): per case µs per call, effective GB/s, % of the
    HBM peak, and the dominant kernel's roofline."""
    import torch

    import awq_int4_moe_gb300 as awq
    out = {}
    for name, cfg in CONFIGS:
        shape = synth.ExpertShape(num_experts=512, top_k=10, hidden=2560, inter=cfg["inter"],
                                  group=cfg.get("group", 32), meta_bytes=cfg["meta_bytes"])
        c_shape = awq.Shape.of(shape)
        L = args.layers
        stack = LayerStack(L, shape, BASE_SEED + 31, device)
        M_max = max(m for m, _ in cfg["cases"])
        ws_bytes = awq.moe_workspace_bytes(c_shape, M_max)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        per_case = [make_case(M, r, stack, device) for M, r in cfg["cases"]]
        path = cfg.get("path", "auto")
        for c in per_case:
            with torch.cuda.stream(stream):
                enqueue_layers(c, stack, ws, ws_bytes, status, stream, path=path)
            torch.cuda.synchronize()
            c["graph"] = capture_stack_graph(c, stack, ws, ws_bytes, status, stream, path=path)
        torch.cuda.synchronize()
        time_rounds(per_case, stream, 3)
        torch.cuda.synchronize()
        reps = max(5, min(40, args.steps))
        evs = time_rounds(per_case, stream, reps)
        torch.cuda.synchronize()
        times = {id(c): [e0.elapsed_time(e1) for c2, e0, e1 in evs if c2 is c] for c in per_case}
        if int(status.item()) != 0:
            raise RuntimeError(f"{name}: device status {int(status.item())}")
        rows = [case_row(c["M"], c["regime"], c["A"], c["bytes"], statistics.median(times[id(c)]), L, peak)
                for c in per_case]
        tot_b = sum(c["bytes"] for c in per_case)
        tot_ms = sum(statistics.median(times[id(c)]) for c in per_case)
        entry = {"meta_bytes": shape.meta_bytes, "inter": shape.inter, "layers": L, "path": path,
                 "weights_resident_GB": round(stack.bytes() / 1e9, 2),
                 "cases": rows, "effective_GBps": round(tot_b / (tot_ms * 1e-3) / 1e9, 1),
                 "pct_of_hbm_peak": round(100 * tot_b / (tot_ms * 1e-3) / 1e9 / peak, 1)}
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        nv = shape.group == 16
        kernels = [kernel_of(c["M"], shape.top_k, sms, path, shape.inter, nv) for c in per_case]
        if all(k in ("fused_layer_kernel", "sliced_layer_kernel") for k in kernels):
            # the committed captures are of 4-byte int4 banks at intermediate 160
            entry["roofline"] = fused_roofline(per_case, times, L, shape.expert_bytes(), peak, peak_kind, kernels,
                                               profiled=not nv and shape.meta_bytes == 4 and shape.inter == 160)
        elif tc_path_of(kernels):
            entry["roofline"] = prefill_roofline(args, per_case, stack, ws, ws_bytes, stream, device, peak,
                                                 peak_kind, tc_path_of(kernels))
        else:
            entry["roofline"] = stage_roofline(args, per_case, stack, c_shape, stream, device, peak, peak_kind)
        if not args.no_check:
            # the oracle's cost grows with experts x intermediate; two cases per
            # configuration keep the check within seconds
            entry["oracle_checks"] = sampled_check(per_case[:2], stack, name)
        out[name] = entry
        del per_case, ws, stack
        torch.cuda.empty_cache()
    return out


def stage_roofline(args, per_case, stack, c_shape, stream, device, peak, peak_kind):
    """Time the W13 and W2 stages alone (graphs of one launch per layer per
    case, same inputs) to find the dominant kernel and its achieved bandwidth."""
    import torch

    import awq_int4_moe_gb300 as awq
    L, shape, weights = stack.layers, stack.shape, stack.weights
    st = torch.zeros(1, dtype=torch.int32, device=device)
    tot = {"w13": [0.0, 0], "w2": [0.0, 0]}
    alg = {"w13": 0, "w2": 0}
    mb = shape.meta_bytes
    w13_b = 4 * shape.w13_words + mb * shape.w13_records
    w2_b = 4 * shape.w2_words + mb * shape.w2_records
    for c in per_case:
        M, S = c["M"], c["M"] * shape.top_k
        routes = []
        for layer in range(L):
            act = torch.empty(S, dtype=torch.int32, device=device)
            off = torch.empty(S + 1, dtype=torch.int32, device=device)
            srt = torch.empty(S, dtype=torch.int32, device=device)
            na = torch.empty(1, dtype=torch.int32, device=device)
            awq.moe_route(c["i_d"][layer], M, c_shape, act, off, srt, na, st, stream)
            routes.append((act, off, srt, na))
        h = torch.empty((L, S, shape.inter), dtype=torch.int16, device=device)
        out = torch.empty((L, M, shape.hidden), dtype=torch.int16, device=device)
        torch.cuda.synchronize()

        def w13():
            for layer in range(L):
                a, o, s, n = routes[layer]
                awq.moe_w13_swiglu(c["x_d"][layer], M, c_shape, weights[layer], a, o, s, n, h[layer], st, stream)

        def w2():
            for layer in range(L):
                a, o, s, n = routes[layer]
                awq.moe_w2_reduce(h[layer], c["w_d"][layer], M, c_shape, weights[layer], a, o, s, n,
                                  out[layer], st, stream)
        for name, fn, b in (("w13", w13, w13_b), ("w2", w2, w2_b)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            reps = max(3, args.steps // 3)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            tot[name][0] += e0.elapsed_time(e1) / reps
            tot[name][1] += L
            alg[name] += sum(c["A"]) * b
    dom = max(tot, key=lambda k: tot[k][0])
    dur_s = tot[dom][0] * 1e-3 / tot[dom][1]
    achieved = alg[dom] / tot[dom][1] / dur_s / 1e9
    kname = {"w13": "w13_swiglu_kernel", "w2": "w2_reduce_kernel"}[dom]
    return {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": None,
            "avg_launch_us": round(dur_s * 1e6, 3),
            "stage_ms_per_stack": {k: round(v[0] / max(1, v[1] / L), 4) for k, v in tot.items()},
            "algorithmic_bytes": (f"distinct active experts x (W13: {w13_b:,} B; W2: {w2_b:,} B) per launch "
                                  f"({mb}-byte metadata)")}


def prefill_roofline(args, per_case, stack, ws, ws_bytes, stream, device, peak, peak_kind, path="prefill"):
    """Per-launch durations of the prefill path's tensor-core launches inside
    the layer calls: a graph of the stack's calls with the options' trace
    buffer (one per layer call), where each launch records its earliest CTA
    start and latest CTA end (%globaltimer); replayed a few times. The
    dominant launch's achieved bandwidth is its algorithmic bytes over its
    mean duration."""
    import torch

    import awq_int4_moe_gb300 as awq
    L, shape = stack.layers, stack.shape
    c_shape = awq.Shape.of(shape)
    mb = shape.meta_bytes
    w13_b = 4 * shape.w13_words + mb * shape.w13_records
    w2_b = 4 * shape.w2_words + mb * shape.w2_records
    status = torch.zeros(1, dtype=torch.int32, device=device)
    # the hybrid path's W13 is the stage kernel; it traces as launch 0 too
    kernels = (("w13_swiglu_kernel",) if path == "hybrid" else PREFILL_KERNELS[:1]) + PREFILL_KERNELS[1:]
    dur = {k: 0.0 for k in kernels}
    alg = {k: 0.0 for k in kernels}
    n_launch = 0
    for c in per_case:
        M, S = c["M"], c["M"] * shape.top_k
        trace = torch.zeros((L, 8), dtype=torch.int64, device=device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for layer in range(L):
                awq.moe_layer_ex(c["x_d"][layer], c["i_d"][layer], c["w_d"][layer], M, c_shape,
                                 stack.weights[layer], c["out"][layer], ws, ws_bytes, status,
                                 path=PATHS[path], trace=trace[layer], stream=stream)
        reps = max(3, min(10, args.steps // 2))
        for rep in range(reps + 1):
            with torch.cuda.stream(stream):
                trace[:, 0:6:2].fill_(2 ** 63 - 1)
                trace[:, 1:6:2].zero_()
                g.replay()
            torch.cuda.synchronize()
            if rep == 0:
                continue                      # warm-up replay
            t = trace.cpu().numpy().astype(np.float64)
            for k, name in enumerate(kernels):
                dur[name] += float(np.sum(t[:, 2 * k + 1] - t[:, 2 * k])) * 1e-9
        n_launch += L * reps
        for name, b in zip(kernels, (w13_b, w2_b, None)):
            per = sum(c["A"]) * b if b else L * (S * shape.hidden * 4 + M * shape.hidden * 2)
            alg[name] += per * reps
        if int(status.item()) != 0:
            raise RuntimeError(f"prefill trace run: device status {int(status.item())}")
    dom = max(dur, key=dur.get)
    achieved = alg[dom] / dur[dom] / 1e9
    return {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": None, "avg_launch_us": round(dur[dom] / n_launch * 1e6, 3),
            "launch_us": {k: round(v / n_launch * 1e6, 3) for k, v in dur.items()},
            "launch_GBps": {k: round(alg[k] / dur[k] / 1e9, 1) for k in kernels if dur[k] > 0},
            "timing": "per launch from %globaltimer (earliest CTA start to latest CTA end), "
                      "traced graph replays",
            "algorithmic_bytes": (f"W13: distinct active experts x {w13_b:,} B; W2: x {w2_b:,} B; "
                                  f"combine: M k H x 4 B read + M H x 2 B written ({mb}-byte metadata)")}


def run_e2e(args, per_case, stack, ws, ws_bytes, status, stream, device, world):
    """Same sweep through the C ABI's awq_moe_layer, not graph-captured: every
    step copies each case's inputs for all layers from pinned host memory
    (one copy per input kind), makes one C call per layer and reads the
    case's outputs back. The calls go to the library through ctypes with
    their arguments marshalled once (the buffers do not move); the Python
    binding's per-call tensor checks run in the warm-up pass, whose calls
    go through it."""
    import ctypes as C

    import torch

    import awq_int4_moe_gb300 as awq
    lib = awq.lib()
    c_shape = awq.Shape.of(stack.shape)
    st_ptr = C.c_void_p(stream.cuda_stream)
    calls = [[(c["x_d"][layer].data_ptr(), c["i_d"][layer].data_ptr(), c["w_d"][layer].data_ptr(), c["M"],
               C.byref(c_shape), C.byref(stack.weights[layer]), c["out"][layer].data_ptr(), ws.data_ptr(),
               ws_bytes, status.data_ptr(), st_ptr) for layer in range(stack.layers)] for c in per_case]
    host = []
    h2d = d2h = 0
    for c in per_case:
        xs = torch.from_numpy(np.stack([x.view(np.int16) for x in c["xs"]])).pin_memory()
        ids = torch.from_numpy(np.stack(c["ids"])).pin_memory()
        ws_ = torch.from_numpy(np.stack(c["wts"])).pin_memory()
        out_h = torch.empty(tuple(c["out"].shape), dtype=torch.int16).pin_memory()
        host.append((xs, ids, ws_, out_h))
        h2d += sum(t.numel() * t.element_size() for t in (xs, ids, ws_))
        d2h += out_h.numel() * out_h.element_size()

    def step(checked=False):
        for c, (xs, ids, ws_, out_h), cl in zip(per_case, host, calls):
            c["x_all"].copy_(xs, non_blocking=True)
            c["i_all"].copy_(ids, non_blocking=True)
            c["w_all"].copy_(ws_, non_blocking=True)
            if checked:
                enqueue_layers(c, stack, ws, ws_bytes, status, stream)
            else:
                for a in cl:
                    r = lib.awq_moe_layer(*a)
                    if r:
                        raise awq.AwqError(r, "awq_moe_layer")
            out_h.copy_(c["out"], non_blocking=True)

    with torch.cuda.stream(stream):
        step(checked=True)
        for _ in range(max(1, args.warmup)):
            step()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 2)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(steps):
            step()
    stream.synchronize()
    dt = time.perf_counter() - t0
    dt = max_over_ranks(dt, world, device)
    tot_bytes = sum(c["bytes"] for c in per_case)
    return {"value": round(job_throughput(tot_bytes * steps, dt, world) / 1e9, 1), "unit": "GB/s (effective HBM)",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(dt * 1e3 / steps, 3)}


# ------------------------------------------------------------ oracle timing

def _oracle_calls(cases, inter, meta_bytes, layers):
    order = [(M, r, layer) for layer in (0, min(23, layers - 1), layers - 1) for M, r in cases]
    return order


def _oracle_worker(job):
    """One worker of the oracle baseline: layer calls `calls[start::stride]`
    until `seconds` of oracle time are spent. Runs in a spawned process."""
    calls, start, stride, seconds, inter, meta_bytes = job
    import oracle
    shape = synth.ExpertShape(num_experts=512, top_k=10, hidden=2560, inter=inter, meta_bytes=meta_bytes)
    eb = shape.expert_bytes()
    done_bytes, spent, n = 0, 0.0, 0
    t_first = t_last = None
    i = start
    while spent < seconds and n < 10 * len(calls):
        M, regime, layer = calls[i % len(calls)]
        i += stride
        cs = case_seed(BASE_SEED, M, regime)
        x = synth.hidden_states(cs, layer, M, shape.hidden)
        ids, w = synth.routing(cs, layer, M, shape.num_experts, shape.top_k, regime)
        banks = ({}, {}, {}, {})
        for e in sorted(set(int(v) for v in ids.ravel())):
            for d, p in zip(banks, synth.expert_weights(shape, BASE_SEED, layer, e, meta_bytes)):
                d[e] = p
        t0 = time.time()
        oracle.moe_layer(x, ids, w, shape, *banks, meta_bytes)
        t1 = time.time()
        t_first = t0 if t_first is None else t_first
        t_last = t1
        spent += t1 - t0
        done_bytes += distinct(ids) * eb
        n += 1
    return done_bytes, spent, n, t_first, t_last


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(cases, seconds, inter=160, meta_bytes=4, layers=48, cores=None, one_core=True):
    """Time the FP64 CPU oracle, as it stands (single-threaded C), on layer
    calls of the sweep (cases x layers 0, 23, 47): once on one core for about
    `seconds`, then on every host core (one spawned worker process per core,
    independent layer calls) for about the same wall time. The rate over all
    cores is the line's value; the one-core rate is reported beside it."""
    import multiprocessing as mp
    calls = _oracle_calls(cases, inter, meta_bytes, layers)
    one = _oracle_worker((calls, 0, 1, seconds / 2, inter, meta_bytes)) if one_core else None
    n = cores or host_cores()
    if one is None and n <= 1:
        one = _oracle_worker((calls, 0, 1, seconds / 2, inter, meta_bytes))
    if n > 1:
        ctx = mp.get_context("spawn")
        with ctx.Pool(n) as pool:
            res = pool.map(_oracle_worker, [(calls, r, n, seconds / 2, inter, meta_bytes) for r in range(n)])
        tot_b = sum(r[0] for r in res)
        wall = max(r[4] for r in res) - min(r[3] for r in res)
        ncalls = sum(r[2] for r in res)
        value = tot_b / wall / 1e9
    else:
        value, ncalls, wall = one[0] / one[1] / 1e9, one[2], one[1]
    res = {"value": round(value, 4), "unit": "GB/s (effective HBM)", "cores": n, "kind": "oracle",
           "sample": (f"{ncalls} layer calls of the sweep (cases x layers 0/23/47) on {n} worker "
                      f"processes, {wall:.1f} s wall, FP64 C oracle (single-threaded per call)")}
    if one is not None:
        res["sample"] += f"; one-core run: {one[2]} calls in {one[1]:.1f} s"
        res["one_core_value"] = round(one[0] / one[1] / 1e9, 4)
        res["us_per_call_one_core"] = round(one[1] / max(1, one[2]) * 1e6, 1)
    return res


def run_reference(args, cases, rank):
    """--impl reference: the oracle on the host cores, bounded sample per step."""
    if rank != 0:
        return None
    per_step = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    n = host_cores()
    for _ in range(min(1, args.warmup)):
        oracle_sample(cases[:1], per_step / 2, args.inter, args.meta_bytes, args.layers, cores=n,
                      one_core=False)
    t0 = time.perf_counter()
    samples = [oracle_sample(cases, per_step, args.inter, args.meta_bytes, args.layers, cores=n,
                             one_core=(i == 0)) for i in range(args.steps)]
    dt = time.perf_counter() - t0
    value = statistics.mean(s["value"] for s in samples)
    return {"metric": METRIC, "value": value, "unit": "GB/s (effective HBM)", "impl": "reference",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": args.layers,
                       "cases": [f"M={m} {r}" for m, r in cases]},
            "cpu_baseline": {"value": value, "unit": "GB/s (effective HBM)", "cores": n,
                             "kind": "oracle", "sample": samples[0]["sample"],
                             "one_core_value": samples[0].get("one_core_value")},
            "e2e": {"value": value, "unit": "GB/s (effective HBM)", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    cases = parse_cases(args.cases)
    rank, world, local = dist_info()
    if args.impl == "reference":
        res = run_reference(args, cases, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, cases, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_sample(cases, args.cpu_seconds, args.inter, args.meta_bytes,
                                            args.layers)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the MoE decode layer on one GB300 (or N replicas).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload r1_decode_t128] [--seed S]

A step is one pass of the whole hot path over one batch: routing, FP8
quantisation of x, dispatch permutation, the expert FFN (one persistent
kernel for decode batches and BF16 layers; for wide FP8 batches the gate/up
GEMM with its SwiGLU + requantisation epilogue, then the down GEMM), combine.  Inputs are seeded synthetic
tensors of the workload's shape, resident in HBM before timing starts; the
11 GB of expert weights streamed per step are far larger than L2, so no L2
flush is needed between steps.

Prints one JSON line (rank 0).  `value` is tokens/s over all ranks;
`layer_roofline_frac` divides the bytes the layer must move by its definition
by the measured HBM copy bandwidth (`layer_roofline_frac_nominal`: by the
nominal 8 TB/s, which a read-dominated stream cannot exceed); `roofline`
describes the dominant kernel (the one-kernel expert FFN at decode, the
gate/up GEMM for wide batches) by the weight bytes it streams; `e2e` is the
same metric through the layer's public call with pinned host buffers copied
in and out each step; `cpu_baseline` times the CPU oracle on a bounded
sample of the workload.  On the default workload the line also carries
`workloads`: the same measurements (no CPU baseline) of the 1024-token
Zipf-skewed layer behind its balanced permutation and of the 4096-token
layer, timed in the same process one layer at a time.
--impl reference times the CPU oracle itself as the reference arm.
Several GPUs run independent replicas (the layer has no exchange step on one
node here): the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at R1 shape (bs 128/1024); HBM GB/s and % of roofline"
DEFAULT_WORKLOAD = "r1_decode_t128"
EXTRA_WORKLOADS = ("r1_zipf_t1024", "r1_prefill_t4096")
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, about 8 TB/s
L2_BYTES = 126 << 20       # GB300 L2 (about 129 MB)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during timing."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workload
def setup(shape, seed, device):
    import torch
    import moe_expert_layer_07_gb300 as moe
    import synth

    inp = synth.make_inputs(shape, seed=seed, device=device)
    layer = moe.MoELayer(shape, inp)
    log2phys = None
    info = {}
    if shape.balanced_perm:
        # calibration with the product path: count rows per expert on the
        # device over one routed batch, derive the balanced permutation and
        # re-lay the expert weights on a side stream
        reb = moe.ExpertRebalancer(layer, shape.num_sets)
        out = torch.empty((shape.tokens, shape.hidden), device=device)
        layer.forward(inp["x"], out)
        reb.observe()
        before, after = reb.rebalance()
        ms = reb.last_relayout_ms()
        log2phys = reb.log2phys
        info = {"set_imbalance": round(after, 4), "set_imbalance_contiguous": round(before, 4),
                "relayout_ms": round(ms, 3),
                "relayout_gbs": round(reb.relayout_bytes / (ms * 1e-3) / 1e9, 1)}
        # the oracle's view: row-major weights in the same physical order (the
        # layer holds its own tile-packed copy)
        inp = synth.relayout_experts(inp, shape, np.argsort(log2phys))
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return inp, layer, log2phys, info


class Stepper:
    """The hot path as its C-ABI steps on one stream, CUDA events around each."""

    # "route" includes the FP8 quantisation of x (done by the selection kernel)
    NAMES_FUSED = ["route", "permute", "expert_ffn", "combine"]
    # wide FP8 batches: the one-kernel FFN on the groups of at most 32 rows, the
    # two GEMMs on the others (as moe_layer_forward splits them)
    NAMES_WIDE = ["route", "permute", "expert_ffn", "gemm_gate_up_swiglu", "gemm_down", "combine"]
    SMALL_GROUP_ROWS = 32

    def __init__(self, layer, x, out):
        import torch
        import moe_expert_layer_07_gb300 as moe
        self.moe, self.torch = moe, torch
        self.layer, self.x, self.out = layer, x, out
        s = layer.shape
        self.fp8 = s.dtype == "fp8"
        L, ws = layer.layout, layer.ws
        base = ws.data_ptr()
        self.p = {n: base + getattr(L, n) for n in
                  ("status", "logits", "topk_ids", "topk_w", "xq", "xs", "expert_offsets",
                   "src_of_row", "row_of_slot", "perm_scratch", "xp", "xp_scales", "h",
                   "h_scales", "y", "ffn_sched")}
        self.perm_bytes = moe.permute_workspace_size(layer.cfg, s.tokens)
        rows = s.tokens * (s.top_k + s.num_shared)
        self.wide = self.fp8 and rows >= 32 * s.groups   # as moe_layer_forward decides
        self.fused = not self.wide   # as moe_layer_forward decides
        self.NAMES = self.NAMES_FUSED if self.fused else self.NAMES_WIDE
        self.sched_bytes = moe.expert_ffn_sched_bytes(s.groups, rows)
        ws[L.status:L.status + 4].zero_()   # the device status word starts clear
        self.k = {}
        self.events = []
        self.top_events = []

    # stage index of the dominant kernel: the expert FFN, or, in wide batches,
    # whichever of the FFN and the gate/up GEMM takes longer (set_top)
    TOP = 2

    def set_top(self):
        """Picks the longest expert stage from a pass with events between all stages."""
        if self.fused:
            return
        self.events = []
        for _ in range(3):
            self.step(record="all")
        self.torch.cuda.synchronize()
        kms = self.kernel_ms()
        self.TOP = 2 if kms["expert_ffn"] >= kms["gemm_gate_up_swiglu"] else 3
        self.events = []

    def step(self, record=None):
        """One pass of the layer.  record="all": CUDA events between all stages
        (they break the programmatic launch overlap at every boundary);
        record="top": events around the dominant kernel only."""
        moe, p, lay, s = self.moe, self.p, self.layer, self.layer.shape
        cfg, w, wl = lay.cfg, lay._keep, lay.expert_layout
        T, G, H, I = s.tokens, s.groups, s.hidden, s.inter
        rows = T * (s.top_k + s.num_shared)
        ev = []
        n_mark = [0]

        def mark():
            i = n_mark[0]
            n_mark[0] += 1
            if record == "all" or (record == "top" and i in (self.TOP, self.TOP + 1)):
                e = self.torch.cuda.Event(enable_timing=True)
                e.record()
                ev.append(e)

        mark()
        if self.fp8:
            moe.route_quantize(cfg, T, self.x, w["wg"], w.get("e_bias"), w.get("logit_offset"),
                               w.get("log2phys"), p["logits"], p["topk_ids"], p["topk_w"],
                               p["xq"], p["xs"], p["status"])
        else:
            moe.route(cfg, T, self.x, w["wg"], w.get("e_bias"), w.get("logit_offset"),
                      w.get("log2phys"), p["logits"], p["topk_ids"], p["topk_w"], p["status"])
        mark()
        moe.permute(cfg, T, p["topk_ids"], p["xq"] if self.fp8 else self.x,
                    p["xs"] if self.fp8 else None, p["expert_offsets"], p["src_of_row"],
                    p["row_of_slot"], p["xp"], p["xp_scales"] if self.fp8 else None,
                    p["perm_scratch"], self.perm_bytes, p["status"])
        mark()
        if self.fused:   # decode batches: both expert GEMMs in one persistent kernel
            q = self.fp8
            moe.expert_ffn(cfg, G, rows, p["xp"], p["xp_scales"] if q else None,
                           p["expert_offsets"], w["w13"], w.get("w13_s"), w["w2"], w.get("w2_s"),
                           p["h"], p["h_scales"] if q else None, p["y"], p["ffn_sched"],
                           self.sched_bytes, p["status"], w_layout=wl)
            mark()
            moe.combine(cfg, T, p["y"], p["row_of_slot"], p["topk_w"], p["expert_offsets"],
                        self.out, moe.OUT_F32)
            mark()
            self._keep_events(record, ev)
            return
        # wide FP8 batches: the groups of few rows in the one-kernel FFN, then the
        # layer's gate/up GEMM with the SwiGLU epilogue and the down GEMM on the rest
        small = self.SMALL_GROUP_ROWS
        moe.expert_ffn(cfg, G, rows, p["xp"], p["xp_scales"], p["expert_offsets"], w["w13"],
                       w.get("w13_s"), w["w2"], w.get("w2_s"), p["h"], p["h_scales"], p["y"],
                       p["ffn_sched"], self.sched_bytes, p["status"], w_layout=wl,
                       max_group_rows=small)
        mark()
        moe.grouped_gemm_swiglu(cfg, G, I, H, rows, p["xp"], p["xp_scales"],
                                p["expert_offsets"], w["w13"], w.get("w13_s"), p["h"],
                                p["h_scales"], p["status"], w_layout=wl, min_group_rows=small + 1)
        mark()
        moe.grouped_gemm(cfg, G, H, I, rows, p["h"], p["h_scales"] if self.fp8 else None,
                         p["expert_offsets"], w["w2"], w.get("w2_s"), p["y"], moe.OUT_F32,
                         p["status"], w_layout=wl, min_group_rows=small + 1)
        mark()
        moe.combine(cfg, T, p["y"], p["row_of_slot"], p["topk_w"], p["expert_offsets"], self.out,
                    moe.OUT_F32)
        mark()
        self._keep_events(record, ev)

    def _keep_events(self, record, ev):
        if record == "all":
            self.events.append(ev)
        elif record == "top":
            self.top_events.append(ev)

    def top_ms(self):
        """Average ms of the dominant kernel over the steps recorded with "top"."""
        k = max(1, len(self.top_events))
        return sum(a.elapsed_time(b) for a, b in self.top_events) / k

    def kernel_ms(self):
        """Average ms per step of each stage over the recorded steps."""
        acc = {n: 0.0 for n in self.NAMES}
        for ev in self.events:
            for i, n in enumerate(self.NAMES):
                acc[n] += ev[i].elapsed_time(ev[i + 1])
        k = max(1, len(self.events))
        return {n: v / k for n, v in acc.items()}


def path_bytes(shape, offsets):
    """Bytes this path moves, per stage, given the rows per group: the method's
    bytes plus the intermediate it keeps at higher precision (fp32 Y).  Used
    for the per-stage split only."""
    T, H, I, E, S, k = (shape.tokens, shape.hidden, shape.inter, shape.num_experts,
                        shape.num_shared, shape.top_k)
    fp8 = shape.dtype == "fp8"
    eb = 1 if fp8 else 2
    rows = T * (k + S)
    counts = np.diff(offsets)
    active = int((counts > 0).sum())
    w13, w2 = expert_weight_bytes(shape)
    sc_h = 4 * (H // 128) if fp8 else 0
    sc_i = 4 * (I // 128) if fp8 else 0
    b = {}
    b["route"] = 2 * T * H + 2 * E * H + 4 * T * E * 2 + 8 * T * k
    b["quant_x"] = (2 * T * H + T * H + T * sc_h) if fp8 else 0
    b["permute"] = 4 * T * k * 3 + rows * (H * eb + sc_h) * 2
    wide = fp8 and rows >= 32 * (E + S)
    if wide:   # gate/up GEMM with the SwiGLU + requantisation epilogue
        b["gemm_gate_up_swiglu"] = active * w13 + rows * (H * eb + sc_h) + rows * (I * eb + sc_i)
    b["gemm_down"] = active * w2 + rows * (I * eb + sc_i) + rows * H * 4
    if not wide:   # one kernel holds both GEMMs (gate/up with SwiGLU, then down)
        b["expert_ffn"] = active * w13 + rows * (H * eb + sc_h) + rows * (I * eb + sc_i) + \
            b.pop("gemm_down")
    b["combine"] = T * (k + S) * H * 4 + 8 * T * k + T * H * 4
    flops = 2 * T * H * E + 6 * H * I * (T * k + S * T)
    return b, active, flops


def expert_weight_bytes(shape):
    """Weights + block scales of one expert group: (gate/up, down).  R1:
    29,360,128 + 7,168 and 14,680,064 + 3,584 bytes."""
    H, I = shape.hidden, shape.inter
    fp8 = shape.dtype == "fp8"
    eb = 1 if fp8 else 2
    w13 = 2 * I * H * eb + (4 * (2 * I // 128) * (H // 128) if fp8 else 0)
    w2 = H * I * eb + (4 * (H // 128) * (I // 128) if fp8 else 0)
    return w13, w2


def method_bytes(shape, active):
    """Bytes the layer must move by its definition, whatever the kernels keep
    in between: every active group's weights and block scales once, the gate
    weights, x read, its FP8 codes (and row scales) written and read, the
    dispatched rows written and read, h written and read, the expert outputs Y
    as bf16 written and read, and the bf16 output.  This path's wider
    intermediate (fp32 Y) is not counted, so the layer's roofline fraction is
    not flattered by it."""
    T, H, I, E, S, k = (shape.tokens, shape.hidden, shape.inter, shape.num_experts,
                        shape.num_shared, shape.top_k)
    fp8 = shape.dtype == "fp8"
    eb = 1 if fp8 else 2
    rows = T * (k + S)
    sc_h = 4 * (H // 128) if fp8 else 0
    sc_i = 4 * (I // 128) if fp8 else 0
    w13, w2 = expert_weight_bytes(shape)
    b = active * (w13 + w2) + 2 * E * H            # experts + gate
    b += 2 * T * H                                 # x
    if fp8:
        b += 2 * T * (H + sc_h)                    # x codes written and read
    b += 2 * rows * (H * eb + sc_h)                # dispatched rows
    b += 2 * rows * (I * eb + sc_i)                # h
    b += 2 * rows * H * 2                          # Y (bf16)
    b += 2 * T * H                                 # output (bf16)
    return b


# --------------------------------------------------------------- CPU oracle
def oracle_single_thread_rate(shape, inp, log2phys, seed=0, n_tokens=None):
    """Tokens/s of the CPU oracle with its C loops on one thread, on a few
    tokens of the workload (a few seconds of work); the thread count is
    restored afterwards."""
    import oracle
    n = n_tokens or min(shape.tokens, 4 if shape.hidden >= 7168 else 32)
    before = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        rate, dt, _, _ = oracle_sample_rate(shape, inp, log2phys, n, seed=seed, min_seconds=0.0,
                                            max_passes=1)
    finally:
        oracle.set_num_threads(before)
    return rate, n, dt


def oracle_sample_rate(shape, inp, log2phys, n_tokens, seed=0, min_seconds=10.0, max_passes=8):
    """Tokens/s of the CPU oracle on `n_tokens` tokens of the workload,
    repeated until about `min_seconds` of CPU work (at most `max_passes`)."""
    import synth
    import oracle
    from oracle import layer as olayer
    npin = synth.to_numpy(inp, log2phys)
    rng = np.random.default_rng(seed)
    sample = np.sort(rng.choice(shape.tokens, n_tokens, replace=False))
    sub = dict(npin)
    sub["x_bits"] = np.ascontiguousarray(npin["x_bits"][sample])
    sub_shape = shape.with_tokens(n_tokens)
    passes, dt = 0, 0.0
    while passes < max_passes and (passes == 0 or dt < min_seconds):
        t0 = time.perf_counter()
        olayer.layer_forward(sub_shape, sub)
        dt += time.perf_counter() - t0
        passes += 1
    return n_tokens * passes / dt, dt, oracle.num_threads(), passes


# ----------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-tokens", type=int, default=None,
                    help="tokens of the CPU-oracle sample (default: sized to ~10-30 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the 1024- and 4096-token layers measured after the default one")
    args = ap.parse_args()

    import torch
    import torch.distributed as dist
    import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    shape = synth.CONFIGS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return 0
        return reference_arm(args, shape)

    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    import moe_expert_layer_07_gb300 as moe

    line = {"metric": METRIC}
    head = measure(shape, args, world, rank, local, device,
                   cpu=not args.no_cpu_baseline and rank == 0)
    line.update(head)
    if args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        line["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            m = measure(synth.CONFIGS[name], args, world, rank, local, device, cpu=False)
            for k in ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                      "vs_baseline", "data", "cpu_baseline"):
                m.pop(k, None)
            line["workloads"][name] = m
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


_READ_STREAM = {}


def read_stream_gbs(layer, device):
    """This GPU's read-only HBM rate, GB/s: the library's stream-read utility
    over the layer's gate/up weights (several GB, far beyond L2), best of five
    passes; measured once per process.  None when the weights fit in L2."""
    import torch
    import moe_expert_layer_07_gb300 as moe
    if "gbs" in _READ_STREAM:
        return _READ_STREAM["gbs"]
    w = layer._keep["w13"]
    g = moe.stream_read_granule()
    nbytes = (w.numel() * w.element_size()) // g * g
    if nbytes < (1 << 30):
        return None
    st = torch.zeros(1, dtype=torch.int32, device=device)
    for _ in range(3):
        moe.stream_read(w, nbytes, st)
    best = None
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        moe.stream_read(w, nbytes, st)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    if int(st.item()) != 0:
        return None
    _READ_STREAM["gbs"] = nbytes / (best * 1e-3) / 1e9
    return _READ_STREAM["gbs"]


def l2_rotation(shape):
    """How many copies of the layer the timed loops take in turn so that no
    step finds its expert weights in L2: 1 when one layer's weights are more
    than twice L2, else enough copies for two and a half L2s between two uses
    of the same copy."""
    w13, w2 = expert_weight_bytes(shape)
    per_layer = shape.groups * (w13 + w2)
    if per_layer > 2 * L2_BYTES:
        return 1
    return -(-(5 * L2_BYTES // 2) // per_layer) + 1


class Rotation:
    """Steppers over several copies of the layer (same inputs, own weights and
    workspace), stepped in turn."""

    def __init__(self, steppers):
        self.all = steppers
        self.i = 0

    def __getattr__(self, name):
        return getattr(self.all[0], name)

    def step(self, record=None):
        self.all[self.i % len(self.all)].step(record)
        self.i += 1

    def set_top(self):
        for st in self.all:
            st.set_top()

    def top_ms(self):
        ev = [e for st in self.all for e in st.top_events]
        return sum(a.elapsed_time(b) for a, b in ev) / max(1, len(ev))

    def kernel_ms(self):
        n = [len(st.events) for st in self.all]
        acc = {}
        for st, k in zip(self.all, n):
            for name, v in st.kernel_ms().items():
                acc[name] = acc.get(name, 0.0) + v * k
        return {name: v / max(1, sum(n)) for name, v in acc.items()}


def measure(shape, args, world, rank, local, device, cpu):
    """All measurements of one workload (the layer resident only meanwhile)."""
    import torch
    import moe_expert_layer_07_gb300 as moe

    inp, layer, log2phys, perm_info = setup(shape, replica_seed(args.seed, rank), device)
    T, H = shape.tokens, shape.hidden
    x = inp["x"]
    out = torch.empty((T, H), dtype=torch.float32, device=device)
    # weights that fit in L2 are taken from several copies in turn, so that
    # every step streams them from HBM as the larger layers do
    layers = [layer] + [moe.MoELayer(shape, inp, log2phys=log2phys)
                        for _ in range(l2_rotation(shape) - 1)]
    stepper = Rotation([Stepper(lay, x, out) for lay in layers])
    for _ in range(args.warmup * len(layers)):
        stepper.step()
    torch.cuda.synchronize()
    stepper.set_top()
    for lay in layers:
        if lay.status() != 0:
            raise RuntimeError(f"device status {lay.status()} after warm-up ({shape.name})")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(args.steps):
            stepper.step(record="top")   # events around the dominant kernel only
        end.record()
        torch.cuda.synchronize()
        barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, device)
    status = max(lay.status() for lay in layers)
    top_ms = stepper.top_ms()
    # per-stage split, after the timed region (events between all stages)
    for _ in range(min(args.steps, 50)):
        stepper.step(record="all")
    torch.cuda.synchronize()
    kms = stepper.kernel_ms()
    offsets = layer.view("expert_offsets", torch.int32, (shape.groups + 1,)).cpu().numpy()
    bytes_per, active, flops = path_bytes(shape, offsets)
    ms_step = elapsed_ms / args.steps
    value = job_tokens_per_s(T, world, args.steps, elapsed_ms)

    hbm_peak, bf16_peak, peak_src = load_peaks()
    layer_bytes = method_bytes(shape, active)      # the method's bytes per step
    path_total = sum(bytes_per.values())           # + this path's wider intermediates
    # the dominant launch and the active groups it streams: the one-kernel FFN
    # (all groups, or in wide batches those of at most 32 rows) moves every
    # weight and block scale of its groups once; the wide gate/up GEMM (groups
    # of more than 32 rows) their gate/up weights
    counts = np.diff(offsets)
    small = Stepper.SMALL_GROUP_ROWS
    if stepper.fused:
        top_groups, top_label = counts > 0, "expert_ffn (gate/up + SwiGLU + down, one kernel)"
    elif stepper.TOP == 2:
        top_groups = (counts > 0) & (counts <= small)
        top_label = (f"expert_ffn on the groups of at most {small} rows (gate/up + SwiGLU + "
                     "down, one kernel)")
    else:
        top_groups = counts > small
        top_label = (f"swiglu_wide gate/up GEMM on the groups of more than {small} rows "
                     "(SwiGLU + FP8 requantisation epilogue)")
    top_ffn = stepper.fused or stepper.TOP == 2
    top_units = int(top_groups.sum())
    w13_b, w2_b = expert_weight_bytes(shape)
    unit_bytes = w13_b + w2_b if top_ffn else w13_b
    top_bytes = top_units * unit_bytes
    achieved = top_bytes / (top_ms / 1e3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath) and shape.dtype == "fp8" and shape.hidden == 7168:
        with open(tpath) as f:
            tr = json.load(f).get("expert_ffn" if top_ffn else "swiglu_wide")
        rows_per_group = counts[top_groups].sum() / max(1, top_units)
        if tr and (top_ffn or abs(rows_per_group / tr["rows_per_active_group"] - 1.0) <= 0.2):
            # ncu DRAM bytes per active group (small R1 case) x this launch's groups
            traffic = tr["bytes_per_active_group"] * top_units

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(layers, shape, x, device, args.steps, args.warmup, world)
    replay = graph_replay(layer, shape, x, device)
    read_gbs = read_stream_gbs(layer, device)

    cpu_line = None
    if cpu:
        n = args.cpu_tokens or default_cpu_tokens(shape)
        rate, dt, cores, passes = oracle_sample_rate(shape, inp, log2phys, n, seed=args.seed)
        cpu_line = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                    "sample": f"{passes} pass(es) over {n} of {T} tokens of the same workload "
                              f"(routing + expert FFNs + combine in fp64), {dt:.1f} s"}
        rate1, n1, dt1 = oracle_single_thread_rate(shape, inp, log2phys, seed=args.seed)
        cpu_line["single_thread"] = {"value": rate1, "unit": "tokens/s",
                                     "sample": f"{n1} tokens, the oracle's C loops on one "
                                               f"thread, {dt1:.1f} s"}

    result = {
        "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8e4m3" if shape.dtype == "fp8" else "bf16", "data": "synthetic",
        "config": {**workload_config(shape, world), **perm_info},
        "hbm_gbs": layer_bytes / (ms_step / 1e3) / 1e9,
        "layer_roofline_frac": (layer_bytes / (hbm_peak * 1e9)) / (ms_step / 1e3),
        "layer_roofline_frac_nominal": (layer_bytes / (NOMINAL_HBM_GBS * 1e9)) / (ms_step / 1e3),
        "read_stream_gbs": read_gbs,
        "layer_roofline_frac_read_stream": (None if not read_gbs else
                                            (layer_bytes / (read_gbs * 1e9)) / (ms_step / 1e3)),
        "roofline_note": "headline fractions (`layer_roofline_frac`, `roofline.frac`) are of "
                         "the measured copy bandwidth (a read + write figure, which a "
                         "read-dominated weight stream can exceed); the `_read_stream` "
                         "fractions are of this GPU's read-only rate measured in this run "
                         "(`read_stream_gbs`: the library's stream-read utility over the "
                         "layer's weights); the `_nominal` fractions are of the nominal 8 TB/s",
        "layer_bytes": layer_bytes,
        "path_bytes": path_total,
        "path_hbm_gbs": path_total / (ms_step / 1e3) / 1e9,
        "active_experts": active,
        "kernels_ms": {k: round(v, 5) for k, v in kms.items()},
        "kernels_ms_note": "per-stage split from a separate pass with events between all "
                           "stages; the timed region records events around the dominant "
                           "kernel only",
        "roofline": {"bound": "hbm", "kernel": top_label, "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": traffic, "peak_source": f"{peak_src} (hbm_gbs)",
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "peak_nominal": NOMINAL_HBM_GBS,
                     "frac_read_stream": None if not read_gbs else achieved / read_gbs,
                     "peak_read_stream": read_gbs,
                     "bytes_per_unit": unit_bytes, "units": top_units,
                     "work_unit": "active expert group (weights + block scales)",
                     "ms_per_launch": top_ms},
        "tensor_pipe_frac_of_bf16x2": (flops / (ms_step / 1e3)) / (2 * bf16_peak * 1e12),
        "gpu_launches": args.steps * moe.layer_kernel_count(layer.cfg, T),
        "device_status": status,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "graph_replay": replay,
        "cpu_baseline": cpu_line,
    }
    del stepper, layers, layer, inp, x, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return result


def workload_config(shape, world):
    """The `config` object of both arms' JSON lines."""
    return {"workload": shape.name, "tokens": shape.tokens, "hidden": shape.hidden,
            "inter": shape.inter, "experts": shape.num_experts, "shared": shape.num_shared,
            "top_k": shape.top_k, "parallelism": "replicas" if world > 1 else "single",
            "l2": l2_note(shape)}


def l2_note(shape):
    r = l2_rotation(shape)
    if r == 1:
        return "inputs larger than L2 (expert weights streamed each step), no flush"
    return (f"inputs larger than L2: the timed loops take {r} copies of the layer's expert "
            f"weights in turn, so no step finds its weights in L2; no flush")


def replica_seed(seed, rank):
    """Each rank's replica draws its own batch (weak scaling: per-GPU work fixed)."""
    return seed + rank


def max_over_ranks(elapsed_ms, world, device=None):
    """The job's time is the slowest rank's (all_reduce MAX on the default group)."""
    if world <= 1:
        return float(elapsed_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_step, world, steps, elapsed_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_step * world * steps / (elapsed_ms / 1e3)


def default_cpu_tokens(shape):
    # the whole batch up to 256 tokens: a pass of the R1 decode batch is a
    # few seconds of oracle work on a 16-core host
    return min(shape.tokens, 256)


def graph_replay(layer, shape, x_dev, device, replays=50):
    """The layer call captured once as a CUDA graph and replayed: the median of
    `replays` replays, each timed alone with CUDA events on its stream, with a
    256 MB fill (about twice L2) before each one, outside the events, so that
    no replay finds the previous one's data in L2."""
    import torch
    T, H = shape.tokens, shape.hidden
    out = torch.empty((T, H), dtype=torch.float32, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x_dev, out)       # outside the capture: any lazy set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x_dev, out)
    times = []
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(replays + 3):
        flush.fill_(i & 255)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(a.elapsed_time(b))
    med = float(np.median(times))
    del graph, flush, out
    return {"median_ms": med, "value": T / (med / 1e3), "unit": "tokens/s", "replays": replays,
            "l2_flush": "256 MB fill before every replay, outside the timed events",
            "api": "moe_layer_forward captured in a CUDA graph"}


def end_to_end(layers, shape, x_dev, device, steps, warmup, world):
    """Tokens/s through the public layer call with every step's input copied
    from pinned host memory and its output read back.  As in a serving loop,
    step i+1's input copy and step i-1's output copy run on side streams
    while step i computes (device buffers double-buffered); the layer calls
    themselves run in order on one stream, step i on layers[i % len(layers)]."""
    import torch
    T, H = shape.tokens, shape.hidden
    x_host = x_dev.cpu().pin_memory()
    out_host = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x_dev) for _ in range(2)]
    od = [torch.empty((T, H), dtype=torch.float32, device=device) for _ in range(2)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    x_used, x_ready, o_ready, o_read = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in x_used + o_read:
        e.record(torch.cuda.current_stream())
    torch.cuda.synchronize()

    def step(i):
        b = i & 1
        with torch.cuda.stream(s_in):       # input of step i (its buffer's last reader done)
            s_in.wait_event(x_used[b])
            xd[b].copy_(x_host, non_blocking=True)
            x_ready[b].record(s_in)
        with torch.cuda.stream(s_run):      # the layer, in order
            s_run.wait_event(x_ready[b])
            s_run.wait_event(o_read[b])
            layers[i % len(layers)].forward(xd[b], od[b], stream=s_run)
            x_used[b].record(s_run)
            o_ready[b].record(s_run)
        with torch.cuda.stream(s_out):      # result of step i back to the host
            s_out.wait_event(o_ready[b])
            out_host[b].copy_(od[b], non_blocking=True)
            o_read[b].record(s_out)

    for i in range(warmup * len(layers)):
        step(i)
    torch.cuda.synchronize()
    n = max(1, steps // 2)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(n):
        step(i)
    s_in.wait_stream(s_out)                 # the last output is on the host
    t1.record(s_in)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    return {"value": T * world * n / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4,
            "steps": n, "api": "MoELayer.forward -> moe_layer_forward",
            "copies": "every step: x from pinned host memory in, fp32 out back to pinned host "
                      "memory, on side streams overlapping the neighbouring steps"}


def reference_arm(args, shape):
    """The CPU oracle as the reference: tokens/s on bounded samples."""
    import torch
    import synth
    import oracle
    from oracle import layer as olayer

    oracle.build()
    device = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_inputs(shape, seed=args.seed, device=device)
    # no expert permutation: the oracle's layer is the same, bit for bit, with
    # or without one (routing is defined on logical experts), so the reference
    # arm runs the oracle alone on the workload's un-permuted weights
    log2phys = None
    npin = synth.to_numpy(inp, log2phys)
    per_step = max(1, min(shape.tokens, 2 if shape.hidden >= 7168 else shape.tokens // 4))
    rng = np.random.default_rng(args.seed)
    t_total, n_total = 0.0, 0
    for i in range(args.warmup + args.steps):
        sample = np.sort(rng.choice(shape.tokens, per_step, replace=False))
        sub = dict(npin)
        sub["x_bits"] = np.ascontiguousarray(npin["x_bits"][sample])
        t0 = time.perf_counter()
        olayer.layer_forward(shape.with_tokens(per_step), sub)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            t_total += dt
            n_total += per_step
    value = n_total / t_total
    cores = oracle.num_threads()
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "impl": "reference",
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape, 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} tokens per step of the same workload"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())

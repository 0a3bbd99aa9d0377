#!/usr/bin/env python
"""Throughput of the LoRA adapter-product hot path on one GB300 (one JSON line).

Headline workload (the timed step): the wide-MLP LoRA training step, bf16,
16384 tokens, r = 64, scale 0.5, through the C ABI of liblora.so:
  up_proj   K = 4096 -> L = 14336:  lora_forward_h, then lora_backward
  down_proj K = 14336 -> L = 4096:  lora_forward_h, then lora_backward
(the forward adds s (X A) B into Y and saves h = X A; the backward writes dX,
dA and dB from dY and the saved h).  value = 16384 tokens / step time.

Per-configuration parts (each op timed alone with CUDA events, L2 flushed
before every launch, median of the repetitions) cover the other seeded
configurations of the benchmark:
  c1  fp32 256 x 512 x 512, r = 8:          lora_forward, lora_backward_dx_da, lora_backward_db
  c2  bf16 q_proj 8192 x 4096 x 4096, r=16: the same three, and lora_forward_h + lora_backward
  c3  the headline ops, one by one
  c4  prefill T = 4096, in = 4096, QKV [4096, 1024, 1024], 32 slots (R = 64):
      lora_group_by_slot, lora_shrink, lora_expand, lora_apply_linear
  c5  decode T = 256 over 128 slots, in = out = 8192 (R = 64): lora_shrink,
      lora_expand, lora_apply_linear, and lora_gather_shrink over a
      128256-entry axis with 5% of the ids = -1
Each part carries its algorithmic bytes (what must cross HBM once), GB/s and
the fraction of the measured copy bandwidth.

Inputs are resident in HBM before the timed region; the headline step rotates
two input sets (every op's operands are larger than the 129 MB L2, and
consecutive ops read different sets).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
"""
import argparse
import hashlib
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

METRIC = "LoRA fwd+bwd & multi-adapter shrink/expand tokens/s; % of HBM roofline"
UNIT = "tokens/s"
SEED = 0
NSETS = 2
WORKLOAD = ("wide-MLP LoRA training step (c3): M=16384 tokens, r=64, s=0.5, bf16; up_proj 4096->14336 and "
            "down_proj 14336->4096, each lora_forward_h + lora_backward (dX, dA, dB)")
C3_TOKENS = 16384
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--part-reps", type=int, default=30, help="repetitions of each per-configuration part")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parts", action="store_true", help="skip the per-configuration parts")
    ap.add_argument("--parts", default="", help="comma-separated configurations for the parts (c1..c5)")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of CUDA-graph replays")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (timestamped on the host) while the benchmark runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        self.dev = str(device_index)
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.dev, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "25"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:   # timed region shorter than the sampling period: nearest samples after it
            inside = [p for (t, p) in self.samples if t >= t0][:3]
            window = "after-timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(inside[0][1]),
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((num(p[2]) or 0.0) for p in inside)}


# ----------------------------------------------------------------------------- algorithmic bytes
def single_bytes(M, K, L, r, e):
    """What each single-adapter op must move across HBM once (e = element size
    of X, Y, dY, dX; h, dA and dB are fp32)."""
    X, Y, Ab, Bb = M * K * e, M * L * e, K * r * e, r * L * e
    h, dA, dB = M * r * 4, K * r * 4, r * L * 4
    return {
        "lora_forward": X + 2 * Y + Ab + Bb,
        "lora_forward_h": X + 2 * Y + Ab + Bb + h,
        "lora_backward_dx_da": Y + 2 * X + Ab + Bb + dA,      # dY, X, dX
        "lora_backward_db": X + Y + Ab + dB,                   # X, dY
        "lora_backward": Y + 2 * X + Ab + Bb + h + dA + dB,    # dY, X, dX (h saved)
    }


def multi_bytes(w):
    """Algorithmic bytes of the segmented ops: active tokens only, rank-limited
    columns, each used slot's adapter rows once."""
    slots = w["slots"].cpu().tolist()
    ranks = w["ranks"].cpu().tolist()
    S, R, IN = w["S"], w["R"], w["IN"]
    osl = w["out_slices"]
    n, O = len(osl), sum(osl)
    act = [t for t, s in enumerate(slots) if 0 <= s < S and 1 <= ranks[s] <= R]
    used = sorted({slots[t] for t in act})
    na = len(act)
    hcols = sum(n * ranks[slots[t]] for t in act)          # specified h entries
    a_b = sum(n * ranks[s] * IN * 2 for s in used)
    b_b = sum(ranks[s] * O * 2 for s in used)
    out = {
        "lora_group_by_slot": len(slots) * 4 + S * 4 + na * 4,
        "lora_shrink": na * IN * 2 + a_b + hcols * 4,
        "lora_expand": hcols * 4 + 2 * na * O * 2 + b_b,
        "lora_apply_linear": na * IN * 2 + a_b + b_b + 2 * na * O * 2,
    }
    if "ga" in w:
        V = w["V"]
        ids = w["ids"].cpu().tolist()
        out["lora_gather_shrink"] = (sum(ranks[s] * (2 + 4) for t, s in enumerate(slots)
                                         if 0 <= s < S and 1 <= ranks[s] <= R and 0 <= ids[t] < V)
                                     + 12 * len(slots))
    return out


# ----------------------------------------------------------------------------- workloads
def make_single_set(torch, synth, binding, dev, name, seed, prefix, peft=True):
    spec = synth.single_spec(name)
    w = synth.make_single(spec, seed=seed, device=dev, prefix=prefix)
    M, K = w["X"].shape
    r, L = w["B"].shape
    if peft:
        # adapter weights in the PEFT layout: lora_A.weight [r, K], lora_B.weight [L, r]
        w["A"] = w["A"].t().contiguous().t()
        w["B"] = w["B"].t().contiguous().t()
    dt = binding.LORA_BF16 if spec["dtype"] == "bf16" else binding.LORA_F32
    w["Y"] = w["Y0"].clone()
    del w["Y0"]
    w["dX"] = torch.empty_like(w["X"])
    w["dA"] = torch.empty((K, r), dtype=torch.float32, device=dev)
    w["dB"] = torch.empty((r, L), dtype=torch.float32, device=dev)
    w["h"] = torch.empty((M, r), dtype=torch.float32, device=dev)
    w["s"] = spec["s"]
    w["ws"] = {op: binding.workspace(op, dt, M, K, L, r, device=dev)
               for op in (binding.OP_FORWARD, binding.OP_BACKWARD, binding.OP_BACKWARD_DX_DA,
                          binding.OP_BACKWARD_DB)}
    w["dims"] = (M, K, L, r, 2 if spec["dtype"] == "bf16" else 4)
    return w


def single_fns(lora, binding):
    def fwd(w):
        lora.lora_forward(w["X"], w["A"], w["B"], w["Y"], w["s"], ws=w["ws"][binding.OP_FORWARD])

    def fwd_h(w):
        lora.lora_forward_h(w["X"], w["A"], w["B"], w["Y"], w["s"], w["h"], ws=w["ws"][binding.OP_FORWARD])

    def bwd(w):
        lora.lora_backward(w["X"], w["dY"], w["A"], w["B"], w["h"], w["s"], w["dX"], w["dA"], w["dB"],
                           ws=w["ws"][binding.OP_BACKWARD])

    def dxda(w):
        lora.lora_backward_dx_da(w["X"], w["dY"], w["A"], w["B"], w["s"], w["dX"], w["dA"],
                                 ws=w["ws"][binding.OP_BACKWARD_DX_DA])

    def db(w):
        lora.lora_backward_db(w["X"], w["A"], w["dY"], w["s"], w["dB"], ws=w["ws"][binding.OP_BACKWARD_DB])

    return {"lora_forward": fwd, "lora_forward_h": fwd_h, "lora_backward": bwd,
            "lora_backward_dx_da": dxda, "lora_backward_db": db}


def make_multi_set(torch, synth, binding, dev, name, seed):
    spec = synth.multi_spec(name)
    w = synth.make_multi(spec, seed=seed, device=dev)
    n, R, T = len(spec["out_slices"]), spec["R"], spec["T"]
    O = sum(spec["out_slices"])
    w["y"] = w["y0"].clone()
    w["h"] = torch.zeros((T, n * R), dtype=torch.float32, device=dev)
    w["ws"] = {op: binding.workspace(op, binding.LORA_BF16, T, w["IN"], O, R, w["S"], device=dev)
               for op in (binding.OP_GROUP_BY_SLOT, binding.OP_SHRINK, binding.OP_EXPAND, binding.OP_APPLY_LINEAR)}
    w["counts"] = torch.empty(w["S"], dtype=torch.int32, device=dev)
    w["perm"] = torch.empty(max(T, 1), dtype=torch.int32, device=dev)
    w["nact"] = torch.empty(1, dtype=torch.int32, device=dev)
    if "ga" in w:
        w["hg"] = torch.zeros((T, R), dtype=torch.float32, device=dev)
    return w


def multi_fns(lora, binding, sched=False):
    """The segmented ops; with sched=True they reuse the batch's prebuilt schedule
    (m["sched"], from lora_build_schedule) instead of grouping the tokens again."""
    def sc(m):
        return m["sched"] if sched else None

    def group(m):
        lora.lora_group_by_slot(m["slots"], m["ranks"], m["R"], m["counts"], m["perm"], m["nact"],
                                ws=m["ws"][binding.OP_GROUP_BY_SLOT])

    def build(m):
        m["sched"] = lora.lora_build_schedule(m["slots"], m["ranks"], m["R"])

    def shrink(m):
        lora.lora_shrink(m["x"], m["a"], m["slots"], m["ranks"], m["R"], m["h"], num_slices=len(m["out_slices"]),
                         ws=m["ws"][binding.OP_SHRINK], schedule=sc(m))

    def expand(m):
        lora.lora_expand(m["h"], m["b"], m["slots"], m["ranks"], m["scalings"], m["y"], m["out_slices"], m["R"],
                         ws=m["ws"][binding.OP_EXPAND], schedule=sc(m))

    def apply(m):
        lora.lora_apply_linear(m["x"], m["a"], m["b"], m["slots"], m["ranks"], m["scalings"], m["y"],
                               m["out_slices"], m["R"], ws=m["ws"][binding.OP_APPLY_LINEAR], schedule=sc(m))

    def gather(m):
        lora.lora_gather_shrink(m["ids"], m["ga"], m["slots"], m["ranks"], m["R"], m["hg"])

    return {"lora_group_by_slot": group, "lora_build_schedule": build, "lora_shrink": shrink,
            "lora_expand": expand, "lora_apply_linear": apply, "lora_gather_shrink": gather}


def c3_step_ops(sets, lora, binding):
    """The headline step: (name, fn(step index), bytes) for up and down."""
    F = single_fns(lora, binding)
    ops = []
    j = 0
    for proj in ("up", "down"):
        for op in ("lora_forward_h", "lora_backward"):
            by = single_bytes(*sets[0][proj]["dims"])[op]
            ops.append((f"c3_{proj}.{op}", (lambda i, proj=proj, op=op, j=j: F[op](sets[(i + j) % NSETS][proj])), by))
            j += 1
    return ops


def h2d_d2h_tensors(S):
    """(inputs copied in, results copied out) of one set, for the end-to-end leg."""
    ins, outs = [], []
    for proj in ("up", "down"):
        w = S[proj]
        ins += [w["X"], w["Y"], w["dY"]]
        outs += [w["Y"], w["dX"], w["dA"], w["dB"]]
    return ins, outs


# ----------------------------------------------------------------------------- oracle timing
def oracle_c3_sample(O, synth, torch, tokens):
    """A `tokens`-row sample of the headline workload and a function that runs
    its step through the fp64 oracle and returns the seconds it took."""
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    f = lambda t: t.double().cpu().numpy()
    data = {}
    for proj, name in (("up", "single_c3_up"), ("down", "single_c3_down")):
        spec = synth.single_spec(name, M=tokens)
        w = synth.make_single(spec, seed=SEED, device=gen, prefix="cpu_" + proj)
        data[proj] = ({k: f(w[k]) for k in ("X", "A", "B", "Y0", "dY")}, spec["s"])

    def run():
        t0 = time.perf_counter()
        for proj in ("up", "down"):
            d, s = data[proj]
            O.forward(d["X"], d["A"], d["B"], d["Y0"], s)
            O.backward_dx_da(d["X"], d["dY"], d["A"], d["B"], s)
            O.backward_db(d["X"], d["A"], d["dY"], s)
        return time.perf_counter() - t0

    return run


def cpu_baseline(torch, synth, tokens=512, target_s=12.0, max_passes=400):
    """Oracle throughput on the host cores: passes over a fixed sample of the
    headline workload, repeated until about `target_s` seconds of oracle work."""
    from oracle import oracle as O
    O.build()
    cores = O.num_threads()
    run = oracle_c3_sample(O, synth, torch, tokens)
    run()   # first touch of the inputs and the library
    tot, passes = 0.0, 0
    while tot < target_s and passes < max_passes:
        tot += run()
        passes += 1
    return {"value": tokens * passes / tot, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{tokens} of the {C3_TOKENS} tokens through the up and down forward + backward, "
                      f"{passes} passes, {tot:.1f} s of fp64 oracle work"}


# ----------------------------------------------------------------------------- arms
def run_reference(args, rank, world):
    import torch
    from lora_rank_adapter_gb300 import synth
    if rank != 0:
        return
    from oracle import oracle as O
    O.build()
    cores = O.num_threads()
    tokens = 128
    run = oracle_c3_sample(O, synth, torch, tokens)
    for _ in range(args.warmup):
        run()
    times = [run() for _ in range(args.steps)]
    tot = sum(times)
    value = tokens * len(times) / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64)",
            "config": {"workload": WORKLOAD, "global_batch": C3_TOKENS, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{tokens} of the {C3_TOKENS} tokens per step through the up and down "
                                       "forward + backward (fp64 oracle)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reduce_max(value, device):
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank, world, ms_per_step_max):
    """Whole-job tokens/s: every rank processes its own batch; the slowest rank sets the time."""
    return world * tokens_per_rank / (ms_per_step_max / 1e3)


def traffic_from_profiles(op_key):
    """Per-launch DRAM bytes of `op_key` from the committed ncu summary, if the
    kernel source it was taken from is unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    for parts in lines:
        kv = dict(p.split("=", 1) for p in parts if "=" in p)
        if kv.get("op") == op_key:
            src = os.path.join(ROOT, kv.get("source", ""))
            try:
                with open(src, "rb") as f:
                    sha = hashlib.sha256(f.read()).hexdigest()[:16]
            except OSError:
                return None
            if sha == kv.get("source_sha"):
                return int(kv["dram_bytes_per_launch"])
    return None


def time_part(torch, stream, fn, reps, flush):
    """Median device time (ms) of fn() over `reps` launches, L2 flushed before each."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(2):
        flush()
        fn(i)
    for i in range(reps):
        flush()
        evs[i][0].record(stream)
        fn(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def run_parts(torch, lora, binding, synth, dev, stream, c3_sets, args, peak, peak_kind):
    """Per-configuration op times, bytes and roofline fractions."""
    which = set(args.parts.split(",")) if args.parts else {"c1", "c2", "c3", "c4", "c5"}
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.zero_()
    reps = args.part_reps
    SF, MF, MS = single_fns(lora, binding), multi_fns(lora, binding), multi_fns(lora, binding, sched=True)
    out = {}

    def add(cfg, op, fn, nbytes, tokens, bound="hbm"):
        ms = time_part(torch, stream, fn, reps, flush)
        d = {"ms": ms, "bytes": nbytes, "tokens/s": tokens / (ms / 1e3)}
        if bound == "hbm":
            gbs = nbytes / (ms / 1e3) / 1e9
            d.update({"GB/s": gbs, "frac_of_" + peak_kind: gbs / peak})
        else:
            d["bound"] = bound
        out[f"{cfg}.{op}"] = d

    if "c1" in which:
        w = make_single_set(torch, synth, binding, dev, "single_c1", SEED, "part_c1", peft=False)
        by = single_bytes(*w["dims"])
        for op in ("lora_forward", "lora_backward_dx_da", "lora_backward_db"):
            add("c1", op, lambda i, op=op: SF[op](w), by[op], w["dims"][0], bound="launch")
        del w
    if "c2" in which:
        w = make_single_set(torch, synth, binding, dev, "single_c2", SEED, "part_c2")
        by = single_bytes(*w["dims"])
        for op in ("lora_forward", "lora_backward_dx_da", "lora_backward_db", "lora_forward_h", "lora_backward"):
            add("c2", op, lambda i, op=op: SF[op](w), by[op], w["dims"][0])
        del w
    if "c3" in which:
        for proj in ("up", "down"):
            by = single_bytes(*c3_sets[0][proj]["dims"])
            for op in ("lora_forward_h", "lora_backward"):
                add(f"c3_{proj}", op, lambda i, op=op, proj=proj: SF[op](c3_sets[i % NSETS][proj]), by[op],
                    C3_TOKENS)
    for cfg, name in (("c4", "multi_c4"), ("c5", "multi_c5")):
        if cfg not in which:
            continue
        m = make_multi_set(torch, synth, binding, dev, name, SEED)
        by = multi_bytes(m)
        ops = ["lora_group_by_slot", "lora_shrink", "lora_expand", "lora_apply_linear"]
        if "ga" in m:
            ops.append("lora_gather_shrink")
        for op in ops:
            lat = op in ("lora_group_by_slot", "lora_gather_shrink")
            add(cfg, op, lambda i, op=op: MF[op](m), by[op], m["T"], bound="latency" if lat else "hbm")
        # the batch's schedule built once and reused by every op (how a serving
        # engine runs the adapted layers of one batch)
        add(cfg, "lora_build_schedule", lambda i: MF["lora_build_schedule"](m), by["lora_group_by_slot"], m["T"],
            bound="latency")
        MF["lora_build_schedule"](m)
        for op in ("lora_shrink", "lora_expand", "lora_apply_linear"):
            add(cfg, op + ".prebuilt_schedule", lambda i, op=op: MS[op](m), by[op], m["T"])
        del m
    del flush_buf
    torch.cuda.empty_cache()
    return out


def run_gb300(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from lora_rank_adapter_gb300 import _build
    from lora_rank_adapter_gb300 import binding
    from lora_rank_adapter_gb300 import binding as lora
    from lora_rank_adapter_gb300 import synth

    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    sets = [{proj: make_single_set(torch, synth, binding, dev, f"single_c3_{proj}", SEED + k, f"bench{k}_{proj}")
             for proj in ("up", "down")} for k in range(NSETS)]
    ops = c3_step_ops(sets, lora, binding)
    tokens = C3_TOKENS
    torch.cuda.synchronize()

    def step(i, events=None):
        for j, (name, fn, _) in enumerate(ops):
            if events is not None:
                events[j][0].record(stream)
            fn(i)
            if events is not None:
                events[j][1].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0

    # one CUDA graph per input-set rotation: a step's launches (with their
    # programmatic-dependent-launch edges) replay without host overhead
    graphs = None
    if not args.no_graph:
        try:
            graphs = []
            cap_stream = torch.cuda.Stream()
            cap_stream.wait_stream(stream)
            with torch.cuda.stream(cap_stream):
                for j in range(NSETS):
                    step(j)                       # warm the capture stream
                torch.cuda.synchronize()
                for j in range(NSETS):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=cap_stream):
                        step(j)
                    graphs.append(g)
            torch.cuda.synchronize()
            for i in range(max(args.warmup, 3)):
                graphs[i % NSETS].replay()
            torch.cuda.synchronize()
        except Exception as exc:                  # capture unsupported: time eager launches
            sys.stderr.write(f"CUDA graph capture failed ({exc}); timing eager launches\n")
            graphs = None
            torch.cuda.synchronize()

    def run_step(i):
        if graphs is not None:
            graphs[i % NSETS].replay()
        else:
            step(i)

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.35)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    launches0 = lora.lora_kernel_launches()
    t_host0 = time.time()
    e0.record(stream)
    for i in range(K):
        run_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier()
    # graph replays do not pass through the library's launch counter: count one
    # step's launches eagerly and scale
    launches = lora.lora_kernel_launches() - launches0
    if graphs is not None:
        c0 = lora.lora_kernel_launches()
        step(0)
        torch.cuda.synchronize()
        launches = (lora.lora_kernel_launches() - c0) * K
    time.sleep(0.25)
    sampler.stop()
    ms = reduce_max(e0.elapsed_time(e1), dev)
    ms_per_step = ms / K
    value = weak_scaling_value(tokens, world, ms_per_step)

    # per-op device times inside the step (eager launches, events around each op, same rotation)
    KP = max(10, min(K, 50))
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ops]
           for _ in range(KP)]
    for i in range(KP):
        step(i, evs[i])
    torch.cuda.synchronize()

    peak, peak_kind = peaks()
    step_parts = {}
    for j, (name, _, nbytes) in enumerate(ops):
        t_ms = statistics.mean(evs[i][j][0].elapsed_time(evs[i][j][1]) for i in range(KP))
        gbs = nbytes / (t_ms / 1e3) / 1e9
        step_parts[name] = {"ms": t_ms, "bytes": nbytes, "GB/s": gbs, "frac_of_" + peak_kind: gbs / peak,
                            "tokens/s": tokens / (t_ms / 1e3)}
    dom = max(step_parts, key=lambda n: step_parts[n]["ms"])
    roof = {"bound": "hbm", "op": dom, "achieved": step_parts[dom]["GB/s"], "peak": peak, "unit": "GB/s",
            "frac": step_parts[dom]["GB/s"] / peak, "peak_kind": peak_kind,
            "traffic": traffic_from_profiles(dom), "bytes_per_launch": step_parts[dom]["bytes"]}
    step_bytes = sum(p["bytes"] for p in step_parts.values())

    # end to end: pinned host inputs in, results out, every step.  The copies in
    # and out run on streams of their own, so that one step's results go out
    # while the next step's inputs come in (host<->device copies in opposite
    # directions overlap; one direction does not gain from splitting); alternate
    # steps use two device copies of the step's input sets, and a copy's inputs
    # go in only after that copy's previous results have been read out.
    E = min(args.e2e_steps, K)
    e_ms = None
    h2d = sum(t.numel() * t.element_size() for S in sets for t in h2d_d2h_tensors(S)[0])
    d2h = sum(t.numel() * t.element_size() for S in sets for t in h2d_d2h_tensors(S)[1])
    if E > 0:
        sets2 = [{proj: make_single_set(torch, synth, binding, dev, f"single_c3_{proj}", SEED + NSETS + k,
                                        f"bench{NSETS + k}_{proj}") for proj in ("up", "down")} for k in range(NSETS)]
        pairs = [(sets, ops), (sets2, c3_step_ops(sets2, lora, binding))]
        host_in = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in h2d_d2h_tensors(S)[0]]
                   for S in sets]
        host_out = [[[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in h2d_d2h_tensors(S)[1]]
                     for S in sets] for _ in pairs]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in pairs]
        ev_comp = [torch.cuda.Event() for _ in pairs]
        ev_out = [torch.cuda.Event() for _ in pairs]
        out_pending = [False for _ in pairs]

        def e2e_step(i):
            c = i % len(pairs)
            psets, pops = pairs[c]
            if out_pending[c]:
                s_in.wait_event(ev_out[c])
            with torch.cuda.stream(s_in):
                for k, S in enumerate(psets):
                    for dst, src in zip(h2d_d2h_tensors(S)[0], host_in[k]):
                        dst.copy_(src, non_blocking=True)
                ev_in[c].record(s_in)
            stream.wait_event(ev_in[c])
            for _, fn, _ in pops:
                fn(i)
            ev_comp[c].record(stream)
            s_out.wait_event(ev_comp[c])
            with torch.cuda.stream(s_out):
                for k, S in enumerate(psets):
                    for dst, src in zip(host_out[c][k], h2d_d2h_tensors(S)[1]):
                        dst.copy_(src, non_blocking=True)
                ev_out[c].record(s_out)
            out_pending[c] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        s_in.wait_event(f0)
        s_out.wait_event(f0)
        for i in range(E):
            e2e_step(i)
        stream.wait_stream(s_out)
        f1.record(stream)
        torch.cuda.synchronize()
        e_ms = reduce_max(f0.elapsed_time(f1) / E, dev)
        del sets2, pairs
    if E > 0:
        del host_in, host_out
    assert lora.lora_device_error() == 0

    parts = None
    if not args.no_parts:
        parts = run_parts(torch, lora, binding, synth, dev, stream, sets, args, peak, peak_kind)
        assert lora.lora_device_error() == 0

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(torch, synth)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded SplitMix64; inputs resident in HBM)",
                "config": {"workload": WORKLOAD, "model": "Llama-like MLP (4096 <-> 14336) LoRA r=64",
                           "global_batch": C3_TOKENS * world, "parallelism": f"replicas x{world}",
                           "l2": f"{NSETS} rotating input sets; every operand > L2; consecutive ops use "
                                 "different sets",
                           "launch": "eager" if graphs is None else "CUDA graph per step (PDL edges kept)",
                           "step_bytes": step_bytes},
                "step_parts": step_parts, "parts": parts, "roofline": roof, "cpu_baseline": cpu,
                "e2e": None if e_ms is None else {
                    "value": weak_scaling_value(tokens, world, e_ms), "unit": UNIT, "steps": E,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "copies": "pinned host buffers; inputs in and results out on streams of their own, "
                              "alternate steps on two device copies of the inputs"},
                "gpu_launches": int(launches), "clocks": sampler.summary(t_host0, t_host1)}
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

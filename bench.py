#!/usr/bin/env python
"""Decode-attention benchmark on GB300: achieved HBM GB/s and attention calls/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 1|2|3|4|4b|5] [--sub 2,3,4,4b | --no-sub]

A step is one decode-attention call (for workload 5: one whole decode step,
40 sliding + 8 global layer calls) over synthetic inputs already resident in
HBM.  The default workload is workload 5, the Gemma-4-12B decode step at
B=64 with seq_lens log-uniform in [16, 262144], the largest configuration
that fits one GPU; its JSON line also carries one object per target
workload (2, 3, 4a and 4b), each timed with CUDA events the same way.
Throughput counts algorithmic bytes only: the visible K and V rows, q and o.

Inputs larger than L2 are used as they are; smaller ones are rotated over
enough distinct copies that every step reads from HBM, not L2.  Calls are
replayed from a CUDA graph (the decode step of a serving loop); ``e2e`` times
the same calls through the public API with the per-step inputs (q, block
table, seq_lens) copied from pinned host memory and o copied back.

With --gpus N > 1 (under torchrun) every rank runs an independent replica
(the attention of different sequences shares nothing): value is the bytes of
all ranks over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention achieved HBM GB/s (% of GB300 peak) and attention calls/sec"
UNIT = "GB/s"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
# NVIDIA's nominal HBM3e bandwidth of a GB300.  The measured peak above is a
# device-to-device copy, which a pure read stream can exceed; fractions are
# also given against this figure (ncu's DRAM peak on this GPU agrees with it:
# 6.87 TB/s of DRAM traffic reads as 87 % of peak).
NOMINAL_DRAM_GBS = 7900.0
# Workloads timed beside the headline (workload 5): the other targets.
DEFAULT_SUBS = ["2", "3", "4", "4b"]
FALLBACK_BF16_TFLOPS = 1900.0

# Multi-query (prefill) workloads timed beside the decode: new tokens whose
# keys and values are already in the cache attend to it (no such workload is
# given with the decode configurations; these are chosen to span both layer
# types at prompt-chunk sizes).
PREFILL_WORKLOADS = {
    "sliding": dict(seq_lens=[8192] * 4, q_lens=[2048] * 4,
                    name="sliding prefill: B=4 x 2048 new tokens on 8192-token contexts, 16/8 heads, D=256, window 1024"),
    "global": dict(seq_lens=[32768], q_lens=[4096],
                   name="global prefill: B=1 x 4096 new tokens on a 32768-token context, 16/1 heads, D=512"),
}
NUM_SPLITS = 0  # --num-splits: thread blocks per KV head, 0 = automatic

# DRAM bytes per launch of the dominant decode kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture of this benchmark's own
# workload, with the hash of the kernel sources it was taken from; reported
# only while the sources still hash to that value (profiles/ has the
# captures and their commands).
NCU_TRAFFIC = {
    ("global", "2"): (63_961_705, "6886be9625dd5e2a"),
    ("global", "4b"): (2_150_904_388, "6886be9625dd5e2a"),
    ("global", "5"): (4_315_656_713, "6886be9625dd5e2a"),
    ("global_shared", "2"): (32_073_892, "6886be9625dd5e2a"),
    ("global_shared", "4b"): (1_074_527_616, "6886be9625dd5e2a"),
    ("sliding", "3"): (2_184_783_705, "fa5274c6beb31627"),
    # a whole 48-layer step: 40 sliding decodes, 8 global decodes and their combines
    ("step", "5"): (50_372_611_502, "20ccbb5b18bae52d"),
}
KERNEL_SOURCES = {
    "global": ["global.cuh", "common.cuh", "ptx.cuh", "rope.cuh"],
    "global_shared": ["global.cuh", "common.cuh", "ptx.cuh", "rope.cuh"],
    "sliding": ["sliding.cuh", "common.cuh", "ptx.cuh"],
    # a whole decode step: both decode kernels and the combine
    "step": ["sliding.cuh", "global.cuh", "combine.cuh", "common.cuh", "ptx.cuh", "rope.cuh"],
}


def _code_only(text):
    """C++ source without comments, trailing blanks or empty lines (a comment edit keeps the hash)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.split("\n") if ln.strip())


def kernel_source_hash(kind):
    import hashlib
    m = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "paged_decode_attention_gb300", "csrc", f)) as fh:
            m.update(_code_only(fh.read()).encode())
    return m.hexdigest()[:16]


def recorded_traffic(kind, cfg):
    """ncu DRAM bytes per launch for (kernel, workload), or None if absent or stale."""
    entry = NCU_TRAFFIC.get((kind, cfg))
    if entry is None or kernel_source_hash(kind) != entry[1]:
        return None
    return entry[0]


# ---------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by tests/test_bench_host.py)
# ---------------------------------------------------------------------------

def algorithmic_bytes(kind, seq_lens, window, Hq=16, out_bytes=2):
    """Visible K and V rows + q + o of one call (block table and seq_lens not counted)."""
    Hkv, D = (8, 256) if kind == "sliding" else (1, 512)
    vis = sum(min(L, window) if window > 0 else L for L in seq_lens)
    B = len(seq_lens)
    return vis * Hkv * D * 2 * 2 + B * Hq * D * 2 + B * Hq * D * out_bytes


def shared_bytes(seq_lens, window, Hq=16, D=512, out_bytes=2):
    """Values-only global cache: visible V rows + q + o + w_k of one call."""
    vis = sum(min(L, window) if window > 0 else L for L in seq_lens)
    B = len(seq_lens)
    return vis * D * 2 + B * Hq * D * 2 + B * Hq * D * out_bytes + D * 2


def rotation_count(bytes_per_set, floor=1, cap=16):
    """Distinct input sets so that consecutive reuse of a set is separated by > 3x L2."""
    if bytes_per_set <= 0:
        return floor
    return max(floor, min(cap, int(math.ceil(4 * L2_BYTES / bytes_per_set))))


def aggregate(per_rank, steps, warmup, n_gpus, config, dtype="bf16"):
    """Combine per-rank results {bytes, ms, calls, ...} into the JSON line (rank 0)."""
    ms = max(r["ms"] for r in per_rank)
    total_bytes = sum(r["bytes"] for r in per_rank)
    total_calls = sum(r["calls"] for r in per_rank)
    value = total_bytes / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": n_gpus,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms / steps, 6),
        "calls_per_s": round(total_calls / (ms * 1e-3), 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic",
        "config": config,
    }


def prefill_flops(seq_lens, q_lens, window, D, Hq=16):
    """4 D flops (q.k and p.v) per query head per visible key: query i of a
    sequence's last n tokens sits at position L - n + i and sees min(p + 1, window) keys."""
    total = 0
    for L, n in zip(seq_lens, q_lens):
        for i in range(n):
            p = L - n + i
            total += min(p + 1, window) if window > 0 else p + 1
    return 4 * D * Hq * total


def load_bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def time_prefill(stream, dev, reps=20):
    """attn_prefill_* on PREFILL_WORKLOADS: TFLOP/s of the algorithmic flops,
    CUDA events on the launching stream around `reps` back-to-back calls."""
    import torch
    import paged_decode_attention_gb300 as pda
    from workloads import make_prefill_case
    out = {}
    for kind, w in PREFILL_WORKLOADS.items():
        case = make_prefill_case(kind, w["seq_lens"], w["q_lens"], seed=9, device=dev, poison=False, window_only=True)
        c = case.cache
        fn = pda.attn_prefill_sliding if kind == "sliding" else pda.attn_prefill_global
        o = torch.empty_like(case.q)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        kw = dict(window=c.window, max_q=max(w["q_lens"]), status=status, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                fn(case.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, case.cu_q, o, **kw)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn(case.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, case.cu_q, o, **kw)
            e1.record(stream)
        e1.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError("device status %d in the prefill" % int(status.item()))
        ms = e0.elapsed_time(e1) / reps
        flops = prefill_flops(w["seq_lens"], w["q_lens"], c.window, c.D)
        out[kind] = {"workload": w["name"], "ms_per_call": round(ms, 4), "flops_per_call": flops,
                     "value": round(flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                     "launch": "%d back-to-back calls, CUDA events" % reps}
        del case, o
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.windows = {}  # key -> [t0, t1]: the timed regions (None: the main one)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin, key=None):
        w = self.windows.setdefault(key, [None, None])
        w[0 if begin else 1] = time.time()

    def stop(self):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.proc = None

    def summary(self, key=None):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((t, parts))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        t0, t1 = self.windows.get(key, [None, None])
        lo = (t0 or 0) - 0.15
        hi = (t1 or time.time()) + 0.15
        inside = [p for t, p in rows if lo <= t <= hi] or [min(rows, key=lambda r: abs(r[0] - lo))[1]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[2]) for p in inside if num(p[2]) is not None]
        smax = [num(p[3]) for p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def workload_calls(cfg, device, seed_offset=0):
    """The calls (DecodeCase) of one step of workload `cfg`."""
    from workloads import config_case, N_LAYERS
    if cfg == "5":
        calls = [config_case(5, device=device, layer=i, poison=False, seed_offset=seed_offset)
                 for i in range(N_LAYERS)]
        # the layers of one type share one page layout: one block-table tensor per type
        first = {}
        for c in calls:
            f = first.setdefault(c.kind, c)
            if f is not c:
                assert torch_equal(f.block_table, c.block_table), "layers of one type share a page layout"
                c.block_table = f.block_table
        return calls
    if cfg == "4b":
        return [config_case(4, device=device, variant="b", poison=False, seed_offset=seed_offset)]
    return [config_case(int(cfg), device=device, poison=False, seed_offset=seed_offset)]


def torch_equal(a, b):
    import torch
    return bool(torch.equal(a, b))


def workload_name(cfg):
    from workloads import WORKLOADS
    if cfg == "4b":
        return "long-context global decode: B=4 x 262144, 16/1 heads, D=512"
    return WORKLOADS[int(cfg)]


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def prepare_workload(cfg, dev):
    """The calls of one step of workload `cfg` and their per-call buffers, over
    enough rotating input sets that consecutive reuse of a set is separated by
    more than 3x L2 (one set when a step's cache alone exceeds that)."""
    import torch
    import paged_decode_attention_gb300 as pda
    calls0 = workload_calls(cfg, dev)
    step_bytes = sum(algorithmic_bytes(c.kind, c.seq_lens_host, c.window) for c in calls0)
    kv_bytes = sum(c.k_pool.numel() * 2 * 2 for c in calls0)
    n_sets = rotation_count(kv_bytes)
    sets = [calls0] + [workload_calls(cfg, dev, seed_offset=100000 * k) for k in range(1, n_sets)]
    plans = []
    for cs in sets:
        pl = []
        for c in cs:
            kind = pda.KIND_SLIDING if c.kind == "sliding" else pda.KIND_GLOBAL
            ws_bytes = pda.attn_decode_workspace_size(kind, c.B, c.max_seq_len, c.window, NUM_SPLITS)
            ws = pda.new_workspace(ws_bytes, dev)
            o = torch.empty((c.B, c.Hq, c.D), dtype=torch.bfloat16, device=dev)
            pl.append((c, ws, o))
        plans.append(pl)
    return dict(calls0=calls0, plans=plans, n_sets=n_sets, step_bytes=step_bytes, kv_bytes=kv_bytes)


def launch_calls(pl, status, stream, idx=None):
    """The decode calls of one step (or those listed in idx), on `stream`."""
    import paged_decode_attention_gb300 as pda
    for j, (c, ws, o) in enumerate(pl):
        if idx is not None and j not in idx:
            continue
        fn = pda.attn_decode_sliding if c.kind == "sliding" else pda.attn_decode_global
        fn(c.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, o, window=c.window,
           max_seq_len=c.max_seq_len, workspace=ws, status=status, stream=stream,
           num_splits=NUM_SPLITS)


def time_graph(launch_i, n, rounds, stream, use_graph=True):
    """ms per launch_i(i) call: a CUDA graph of launch_i(0..n-1) back to back,
    replayed `rounds` times between CUDA events on `stream` after a warm replay
    (direct calls with use_graph=False)."""
    import torch
    g = None
    if use_graph:
        with torch.cuda.stream(stream):
            for i in range(min(n, 2)):
                launch_i(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                launch_i(i)

    def one_round():
        if g is not None:
            g.replay()
        else:
            for i in range(n):
                launch_i(i)
    with torch.cuda.stream(stream):
        one_round()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(rounds):
            one_round()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (rounds * n)
    del g
    return ms


def hbm_roofline(nbytes, ms, peak, peak_src, kernel, traffic=None):
    """The roofline object of an HBM-bound measurement: algorithmic bytes over
    the event-timed duration, against the measured copy peak and, beside it,
    NVIDIA's nominal DRAM peak (a read stream may exceed the copy figure)."""
    achieved = nbytes / (ms * 1e-3) / 1e9
    out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
           "frac": round(achieved / peak, 4), "traffic": traffic, "algorithmic_bytes": nbytes,
           "peak_source": peak_src, "kernel": kernel,
           "frac_of_dram_peak": round(achieved / NOMINAL_DRAM_GBS, 4),
           "dram_peak": NOMINAL_DRAM_GBS, "dram_peak_source": "nominal HBM3e (NVIDIA)"}
    if achieved > peak:
        out["note"] = ("above the copy-based peak: a pure read stream exceeds a device-to-device copy; "
                       "frac_of_dram_peak is the fraction of the nominal DRAM bandwidth")
    return out


def measure_sub(cfg, dev, stream, status, args, peak, peak_src, sampler=None):
    """One target workload timed on its own: ms per call from a CUDA graph of
    back-to-back calls over the rotating input sets, its HBM roofline, and for
    global layers the values-only cache and (workload 2) the library's
    one-launch step object on the same calls."""
    import torch
    import paged_decode_attention_gb300 as pda
    W = prepare_workload(cfg, dev)
    plans, n_sets, calls0 = W["plans"], W["n_sets"], W["calls0"]
    n = max(8, 2 * n_sets)
    est_ms = W["step_bytes"] / (peak * 1e6)
    rounds = max(3, min(200, int(math.ceil(50.0 / max(est_ms * n, 1e-3)))))
    if sampler:
        sampler.mark(True, key=cfg)
    ms = time_graph(lambda i: launch_calls(plans[i % n_sets], status, stream), n, rounds, stream,
                    use_graph=not args.no_graph)
    if sampler:
        sampler.mark(False, key=cfg)
    kind = calls0[0].kind
    c0 = calls0[0]
    nk = pda.attn_decode_launches(pda.KIND_SLIDING if kind == "sliding" else pda.KIND_GLOBAL, c0.B, c0.max_seq_len,
                                  c0.window, NUM_SPLITS, torch.cuda.get_device_properties(dev).multi_processor_count)
    kernels = ("%s decode + combine (2 launches per call, timed together)" % kind if nk == 2 else
               "%s decode, split sequences merged in the grid (1 launch per call)" % kind)
    out = {"workload": workload_name(cfg), "calls_per_step": len(calls0), "ms_per_call": round(ms, 6),
           "calls_per_s": round(1e3 / ms, 1), "value": round(W["step_bytes"] / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "roofline": hbm_roofline(W["step_bytes"], ms, peak, peak_src, kernels,
                                    recorded_traffic(kind, cfg)),
           "l2": ("inputs %.0f MB > L2; 1 set" % (W["kv_bytes"] / 1e6) if n_sets == 1 else
                  "rotating %d input sets (%.0f MB in all) so every call reads HBM" % (n_sets, n_sets * W["kv_bytes"] / 1e6)),
           "launch": "%d calls back to back in one CUDA graph, %d replays, CUDA events" % (n, rounds)}
    if kind == "global":
        sh = time_global_shared(plans, n_sets, stream, status, dev)
        sh["traffic"] = recorded_traffic("global_shared", cfg)
        sh["frac_of_peak"] = round(sh["value"] / peak, 4)
        sh["frac_of_dram_peak"] = round(sh["value"] / NOMINAL_DRAM_GBS, 4)
        out["values_only_cache"] = sh
    if cfg == "2":
        ws = time_whole_step(plans, n_sets, stream, status, max(50, min(args.steps, 400)))
        ws["frac_of_peak"] = round(ws["value"] / peak, 4)
        ws["graph_replayed_us_per_step"] = round(ms * 1e3, 3)
        out["whole_step_launch"] = ws
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in workload %s" % (int(status.item()), cfg))
    del W, plans, calls0
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_decode_attention_gb300 as pda

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pda.load()
    stream = torch.cuda.Stream(device=dev)

    # --- inputs: one or more rotating sets of the step's calls ---
    W = prepare_workload(args.config, dev)
    calls0, plans, n_sets = W["calls0"], W["plans"], W["n_sets"]
    step_bytes, kv_bytes = W["step_bytes"], W["kv_bytes"]
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch(pl):
        launch_calls(pl, status, stream)

    # the decode kernel, and a combine kernel unless the call merges in the grid
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kernels_per_call = [pda.attn_decode_launches(pda.KIND_SLIDING if c.kind == "sliding" else pda.KIND_GLOBAL,
                                                 c.B, c.max_seq_len, c.window, NUM_SPLITS, sms) for c in calls0]

    # Warm-up with direct calls; then the W warm-up steps and the K timed steps
    # are each captured as one CUDA graph (step i reads input set i % n_sets),
    # so the timed region is the K steps' kernels back to back.
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            launch(plans[i % n_sets])
    stream.synchronize()
    timed_graph = None
    if not args.no_graph:
        warm_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(warm_graph, stream=stream):
            for i in range(max(args.warmup, 3)):
                launch(plans[i % n_sets])
        timed_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(timed_graph, stream=stream):
            for i in range(args.steps):
                launch(plans[i % n_sets])
        with torch.cuda.stream(stream):
            warm_graph.replay()
        stream.synchronize()

    def run_timed_steps():
        if timed_graph is not None:
            timed_graph.replay()
        else:
            for i in range(args.steps):
                launch(plans[i % n_sets])

    # --- timed region ---
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-%s" % props.uuid) if getattr(props, "uuid", None) else str(local_rank)
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark(True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run_timed_steps()
        ev1.record(stream)
    ev1.synchronize()
    if sampler:
        sampler.mark(False)
    torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    st = int(status.item())
    if st != 0:
        raise RuntimeError("device status %d during the benchmark" % st)

    res = {"bytes": step_bytes * args.steps, "ms": ms, "calls": len(calls0) * args.steps}

    # --- dominant kernel: per-launch duration of the heaviest call, timed with
    #     events on its stream around a graph of back-to-back copies of it ---
    heavy = max(range(len(calls0)), key=lambda j: algorithmic_bytes(calls0[j].kind, calls0[j].seq_lens_host,
                                                                    calls0[j].window))
    reps = 2 * n_sets if n_sets > 1 else 8
    rounds = max(8, min(200, args.steps)) if args.no_graph else max(3, min(50, args.steps // reps + 1))
    heavy_ms = time_graph(lambda i: launch_calls(plans[i % n_sets], status, stream, idx=(heavy,)), reps, rounds,
                          stream, use_graph=not args.no_graph)
    hc = calls0[heavy]
    heavy_bytes = algorithmic_bytes(hc.kind, hc.seq_lens_host, hc.window)

    # --- mixed workloads: each layer type's calls of one step, timed apart ---
    per_type = {}
    kinds = sorted(set(c.kind for c in calls0))
    if len(kinds) > 1:
        for kind in kinds:
            idx = tuple(j for j, c in enumerate(calls0) if c.kind == kind)
            kms = time_graph(lambda i, idx=idx: launch_calls(plans[i % n_sets], status, stream, idx=idx), 1, 5,
                             stream, use_graph=not args.no_graph)
            kbytes = sum(algorithmic_bytes(calls0[j].kind, calls0[j].seq_lens_host, calls0[j].window) for j in idx)
            per_type[kind] = {"calls_per_step": len(idx), "ms_per_step": round(kms, 6),
                              "value": round(kbytes / (kms * 1e-3) / 1e9, 2), "unit": UNIT}

    # --- end to end through the public API with host buffers ---
    # a step of one call batches 4 steps per wait; a 48-call step needs no batching
    e2e = run_e2e(args, plans, n_sets, stream, status, dev, batch=max(1, 4 // len(calls0)))

    # --- the step before the decode: norms, RoPE and the cache append ---
    append = time_append(calls0, stream, status, dev)
    # --- multi-query attention over the paged cache (prefill) ---
    prefill = None if args.no_prefill else time_prefill(stream, dev)
    # --- the global calls again over a values-only cache ---
    shared = time_global_shared(plans, n_sets, stream, status, dev)
    if shared is not None:
        shared["traffic"] = recorded_traffic("global_shared", args.config)
    # --- the step as the library's own one-launch object ---
    whole = time_whole_step(plans, n_sets, stream, status, max(3, min(args.steps, 200)))
    whole_append = time_whole_step(plans, n_sets, stream, status, max(3, min(args.steps, 200)), with_append=True)
    if int(status.item()) != 0:
        raise RuntimeError("device status %d after the cache append" % int(status.item()))

    res.update(per_type=per_type, append=append, prefill=prefill, shared=shared, whole_step=whole,
               whole_step_append=whole_append)
    res.update(heavy_ms=heavy_ms, heavy_bytes=heavy_bytes, heavy_kind=hc.kind,
               heavy_kernels=kernels_per_call[heavy], e2e=e2e, n_sets=n_sets,
               launches_per_step=sum(kernels_per_call), kv_bytes=kv_bytes,
               timed_ms_per_step=ms / args.steps)

    # --- the other target workloads, one at a time (rank 0 reports them) ---
    del W, plans, calls0
    torch.cuda.empty_cache()
    subs = {}
    for cfg in args.sub:
        if cfg == args.config:
            continue
        subs[cfg] = measure_sub(cfg, dev, stream, status, args, *load_peaks(), sampler=sampler)
    res["subs"] = subs
    res["clocks"] = None
    if sampler:
        sampler.stop()
        res["clocks"] = sampler.summary()
        for cfg, d in subs.items():
            d["clocks"] = sampler.summary(key=cfg)
    return res


def time_whole_step(plans, n_sets, stream, status, steps, with_append=False):
    """The step's decode calls recorded into one pda.Step per input set and
    launched with one attn_step_launch per step (one CUDA graph of the step's
    calls), `steps` launches back to back between CUDA events.

    with_append: each layer's cache append runs first, as in a real decode
    step: it writes the token at position seq_len - 1 into the layer's pools
    and the decode's q, which the decode then reads."""
    import torch
    import paged_decode_attention_gb300 as pda
    from workloads import append_row_len, key_weight
    objs = []
    gen = torch.Generator(device=stream.device)
    gen.manual_seed(78)
    w = {k: key_weight(D, 79 + D, device=stream.device) for k, D in (("sliding", 256), ("global", 512))}
    keep = []
    for pl in plans:
        st = pda.Step()
        for c, ws, o in pl:
            if with_append:
                qkv = torch.randn((c.B, append_row_len(c.kind)), generator=gen, device=stream.device).to(torch.bfloat16)
                positions = (c.seq_lens - 1).clamp(min=0).to(torch.int32)
                keep.append((qkv, positions))
                add_app = st.add_kv_append_sliding if c.kind == "sliding" else st.add_kv_append_global
                add_app(qkv, w[c.kind], w[c.kind], c.block_table, positions, c.k_pool, c.v_pool, c.q, status=status)
            add = st.add_decode_sliding if c.kind == "sliding" else st.add_decode_global
            add(c.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, o, window=c.window, max_seq_len=c.max_seq_len,
                workspace=ws, status=status, num_splits=NUM_SPLITS)
        objs.append(st.finalize())
    for i in range(max(3, n_sets)):
        objs[i % n_sets].launch(stream)
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            objs[i % n_sets].launch(stream)
        e1.record(stream)
    e1.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the step launch" % int(status.item()))
    ms = e0.elapsed_time(e1) / steps
    calls = [c for c, _, _ in plans[0]]
    nbytes = sum(algorithmic_bytes(c.kind, c.seq_lens_host, c.window) for c in calls)
    out = {"calls_per_step": len(calls), "kernels_per_step": objs[0].num_kernels, "us_per_step": round(ms * 1e3, 3),
           "value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "launch": "one attn_step_launch (one CUDA graph of the step's calls) per step, %d steps back to back"
                     % steps}
    if with_append:
        app = sum(append_bytes(c.kind, c.B) for c in calls)
        out["append_bytes_per_step"] = app
        out["value_with_append_bytes"] = round((nbytes + app) / (ms * 1e-3) / 1e9, 2)
        out["note"] = "value counts the decode bytes only; each layer's append precedes its decode in the graph"
    for st in objs:
        st.close()
    return out


def time_global_shared(plans, n_sets, stream, status, dev, rounds=5):
    """The step's global calls with a values-only cache (attn_decode_global_shared:
    each call's v_pool as the cache, keys rebuilt in the kernel) and, timed the
    same way, with the separate key and value pools.  Each timing is a CUDA
    graph of the calls over every rotating input set, replayed `rounds` times."""
    import torch
    import paged_decode_attention_gb300 as pda
    from workloads import key_weight
    idx = [j for j, c in enumerate(plans[0]) if c[0].kind == "global"]
    if not idx:
        return None
    w_k = key_weight(512, 5, device=dev)
    reps = max(2, n_sets)

    def launch(shared):
        for i in range(reps):
            for j in idx:
                c, ws, o = plans[i % n_sets][j]
                if shared:
                    pda.attn_decode_global_shared(c.q, c.v_pool, w_k, c.block_table, c.seq_lens, o,
                                                  max_seq_len=c.max_seq_len, workspace=ws, status=status,
                                                  stream=stream, num_splits=NUM_SPLITS)
                else:
                    pda.attn_decode_global(c.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, o,
                                           max_seq_len=c.max_seq_len, workspace=ws, status=status, stream=stream,
                                           num_splits=NUM_SPLITS)
    ms = {}
    for shared in (True, False):
        with torch.cuda.stream(stream):
            launch(shared)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch(shared)
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(rounds):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        ms[shared] = e0.elapsed_time(e1) / (rounds * reps)
        del g
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the values-only decode" % int(status.item()))
    calls = [plans[0][j][0] for j in idx]
    nbytes = sum(shared_bytes(c.seq_lens_host, c.window) for c in calls)
    sep_bytes = sum(algorithmic_bytes(c.kind, c.seq_lens_host, c.window) for c in calls)
    return {"calls_per_step": len(idx), "us_per_step": round(ms[True] * 1e3, 3),
            "bytes_per_step": nbytes, "value": round(nbytes / (ms[True] * 1e-3) / 1e9, 2), "unit": "GB/s",
            "separate_cache_us_per_step": round(ms[False] * 1e3, 3),
            "separate_cache_value": round(sep_bytes / (ms[False] * 1e-3) / 1e9, 2),
            "cache_bytes_per_position": {"values_only": 1024, "separate": 2048},
            "launch": "%d steps of the global calls (input sets rotating) in one CUDA graph, %d replays"
                      % (reps, rounds)}


def append_bytes(kind, B):
    """qkv row read, q write and the key and value rows written, per call of B tokens."""
    from workloads import append_row_len
    Hq, Hkv, D = (16, 8, 256) if kind == "sliding" else (16, 1, 512)
    return B * (append_row_len(kind) * 2 + Hq * D * 2 + 2 * Hkv * D * 2) + 2 * D * 2


def time_append(calls0, stream, status, dev, rounds=20):
    """The norm + RoPE + cache-append step for one new token per sequence,
    at position seq_len - 1 of each decode call of the step, per layer type.
    Each call reads its own qkv and writes its own q, rotating over enough
    sets that a set is reused only after more than L2's worth of others."""
    import torch
    import paged_decode_attention_gb300 as pda
    from workloads import append_row_len
    out = {}
    for kind in sorted(set(c.kind for c in calls0)):
        c = next(c for c in calls0 if c.kind == kind)
        D = c.D
        per_call = append_bytes(kind, c.B)
        n = rotation_count(per_call, floor=2, cap=256)
        gen = torch.Generator(device=dev)
        gen.manual_seed(77)
        qkv = [torch.randn((c.B, append_row_len(kind)), generator=gen, device=dev).to(torch.bfloat16)
               for _ in range(n)]
        q_out = [torch.empty((c.B, c.Hq, D), dtype=torch.bfloat16, device=dev) for _ in range(n)]
        w_q = (1.0 + 0.1 * torch.randn(D, generator=gen, device=dev)).to(torch.bfloat16)
        w_k = (1.0 + 0.1 * torch.randn(D, generator=gen, device=dev)).to(torch.bfloat16)
        positions = (c.seq_lens - 1).to(torch.int32)
        fn = pda.attn_kv_append_sliding if kind == "sliding" else pda.attn_kv_append_global

        def launch_all():
            for i in range(n):
                fn(qkv[i], w_q, w_k, c.block_table, positions, c.k_pool, c.v_pool, q_out[i],
                   status=status, stream=stream)
        with torch.cuda.stream(stream):
            launch_all()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch_all()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(rounds):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / (rounds * n)
        out[kind] = {"tokens_per_call": c.B, "us_per_call": round(ms * 1e3, 3),
                     "bytes_per_call": per_call, "value": round(per_call / (ms * 1e-3) / 1e9, 2),
                     "unit": "GB/s", "sets": n,
                     "launch": "%d calls back to back in one CUDA graph, %d replays" % (n, rounds)}
    return out


def _packed_inputs(parts, dev):
    """One pinned host buffer and one device buffer holding the tensors `parts`
    back to back (256-byte aligned), with device views of each part."""
    import torch

    def a256(n):
        return (n + 255) // 256 * 256
    sizes = [t.numel() * t.element_size() for t in parts]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += a256(n)
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    devbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, off, n in zip(parts, offs, sizes):
        host[off:off + n].copy_(t.detach().cpu().contiguous().view(torch.uint8).reshape(-1))
        views.append(devbuf[off:off + n].view(t.dtype).view(t.shape))
    return host, devbuf, views


def run_e2e(args, plans, n_sets, stream, status, dev, batch=4):
    """End to end through the public binding.  Every step: an H2D copy from
    pinned memory of each block table the step's calls use (once per table:
    the layers of one type share one) and, for every call, of its packed q
    and seq_lens; the call (a PreparedDecode of the binding); and a D2H copy
    of o into pinned memory.  The KV cache stays resident.  Steps are pipelined as a serving
    loop runs them, `batch` steps at a time: a batch's input copies run on
    their own stream while the compute stream works on the previous batch,
    its output copies on a third stream once its calls are done, and 2*batch
    buffer slots alternate between batches, with events ordering every reuse.
    The compute stream waits once per batch, so the calls inside a batch stay
    chained by programmatic launch.  The K steps are captured as one CUDA
    graph (eager with --no-graph)."""
    import torch
    import paged_decode_attention_gb300 as pda
    slots = 2 * batch
    staged = {}  # (input set, slot) -> [(host, device, prepared call, o, pinned o), ...]

    def stage(i):
        key = (i % n_sets, i % slots)
        if key not in staged:
            calls = []
            tables = {}  # id of a case's block table -> its device view in this slot
            for c, ws, o in plans[key[0]]:
                if id(c.block_table) not in tables:
                    hbuf, dbuf, (btv,) = _packed_inputs([c.block_table], dev)
                    tables[id(c.block_table)] = btv
                    calls.append((hbuf, dbuf, None, None, None))
                btv = tables[id(c.block_table)]
                hbuf, dbuf, (qv, slv) = _packed_inputs([c.q, c.seq_lens], dev)
                o_dev = torch.empty_like(o)
                prep = pda.PreparedDecode(pda.KIND_SLIDING if c.kind == "sliding" else pda.KIND_GLOBAL,
                                          qv, c.k_pool, c.v_pool, btv, slv, o_dev, window=c.window,
                                          max_seq_len=c.max_seq_len, num_splits=NUM_SPLITS, workspace=ws,
                                          status=status)
                calls.append((hbuf, dbuf, prep, o_dev, torch.empty(o.shape, dtype=o.dtype).pin_memory()))
            staged[key] = calls
        return staged[key]

    steps = max(3, min(args.steps, 200))
    for i in range(max(steps, 3)):
        stage(i)
    first = staged[(0, 0)]
    h2d = sum(hbuf.numel() for hbuf, _, _, _, _ in first)
    d2h = sum(oh.numel() * oh.element_size() for _, _, _, _, oh in first if oh is not None)
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # a batch's inputs copied
    ev_comp = [torch.cuda.Event() for _ in range(2)]  # its calls done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # its outputs read back

    def run_steps(n):
        fork = torch.cuda.Event()
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        nb = 0
        for i0 in range(0, n, batch):
            par = nb % 2
            idx = range(i0, min(n, i0 + batch))
            if nb >= 2:
                s_in.wait_event(ev_comp[par])  # batch nb-2 no longer reads these slots
            with torch.cuda.stream(s_in):
                for i in idx:
                    for hbuf, dbuf, _, _, _ in stage(i):
                        dbuf.copy_(hbuf, non_blocking=True)
            ev_in[par].record(s_in)
            stream.wait_event(ev_in[par])
            if nb >= 2:
                stream.wait_event(ev_out[par])  # batch nb-2's outputs have been read back
            for i in idx:
                for _, _, prep, _, _ in stage(i):
                    if prep is not None:
                        prep.run(stream)
            ev_comp[par].record(stream)
            s_out.wait_event(ev_comp[par])
            with torch.cuda.stream(s_out):
                for i in idx:
                    for _, _, _, o_dev, oh in stage(i):
                        if oh is not None:
                            oh.copy_(o_dev, non_blocking=True)
            ev_out[par].record(s_out)
            nb += 1
        for par in range(min(nb, 2)):  # join
            stream.wait_event(ev_out[par])

    with torch.cuda.stream(stream):
        run_steps(min(steps, 2 * batch))
    torch.cuda.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            run_steps(steps)
        graph.replay()  # warm
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            run_steps(steps)
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    step_bytes = sum(algorithmic_bytes(c.kind, c.seq_lens_host, c.window) for c, _, _ in plans[0])
    return {"value": round(step_bytes * steps / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 6),
            "pipelined": ("every step copies its inputs in and its output back; %d steps per batch, one "
                          "input copy stream, one output copy stream, the compute stream waits once per batch"
                          % batch)}


def oracle_sample(cfg, budget_s=2.0, threads=None):
    """A bounded sample of workload `cfg` for the fp64 oracle: (callable, bytes, description)."""
    import numpy as np
    import oracle
    from workloads import bits, config_seq_lens, make_case
    lens = config_seq_lens(5 if cfg == "5" else (4 if cfg == "4b" else int(cfg)), "b" if cfg == "4b" else None)
    kind = "sliding" if cfg in ("1", "3") else "global"
    if cfg == "5":
        kind = "global"
    window = 1024 if kind == "sliding" else 0
    # the first sequences of the workload, as many as fit a per-position budget
    per_pos_s = 2.0e-7 if kind == "global" else 4.0e-7   # rough fp64 cost per position (16 heads)
    take, acc = [], 0.0
    for L in lens:
        n = min(L, window) if window > 0 else L
        if take and acc + n * per_pos_s > budget_s:
            break
        if n * per_pos_s > budget_s and not take:
            L = max(1, int(budget_s / per_pos_s))
            n = L
        take.append(L)
        acc += n * per_pos_s
    case = make_case(kind, take, seed=5150, device="cpu", window=window,
                     window_only=(kind == "sliding"), poison=False)
    if threads is None:
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    args = (bits(case.q), bits(case.k_pool), bits(case.v_pool), case.block_table.numpy(),
            case.seq_lens.numpy(), case.window)

    def run():
        oracle.decode_paged(*args, threads=threads)

    nbytes = algorithmic_bytes(kind, take, window)
    desc = "%s decode, %d sequence(s) of the workload's seq_lens (%s), all 16 heads" % (
        kind, len(take), ",".join(str(x) for x in take[:6]) + ("..." if len(take) > 6 else ""))
    return run, nbytes, desc, threads


def cpu_baseline(cfg, budget_s=2.0, reps=3):
    """The oracle on all the host cores the process may use, and on one core
    (over a sample scaled down by the core count)."""
    def timed(run):
        run()
        t = []
        for _ in range(reps):
            t0 = time.perf_counter()
            run()
            t.append(time.perf_counter() - t0)
        return min(t)
    run, nbytes, desc, threads = oracle_sample(cfg, budget_s)
    sec = timed(run)
    run1, nbytes1, desc1, _ = oracle_sample(cfg, budget_s / max(threads, 1), threads=1)
    sec1 = timed(run1)
    return {"value": round(nbytes / sec / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc, "seconds_per_sample": round(sec, 4),
            "one_core": {"value": round(nbytes1 / sec1 / 1e9, 4), "unit": UNIT, "sample": desc1}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    run, nbytes, desc, threads = oracle_sample(args.config, budget_s=0.5)
    for _ in range(max(args.warmup, 0)):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    sec = time.perf_counter() - t0
    value = round(nbytes * args.steps / sec / 1e9, 4)
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(args.config), "sample": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------

_PG = None


def init_dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local_rank


def setup_pg(world, backend):
    global _PG
    if world > 1 and _PG is None:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        _PG = dist


def barrier(world):
    if world > 1 and _PG is not None:
        _PG.barrier()


def gather_results(res, world):
    if world == 1:
        return [res]
    out = [None] * world
    _PG.all_gather_object(out, res)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="5", choices=["1", "2", "3", "4", "4b", "5"])
    ap.add_argument("--sub", default=None,
                    help="comma-separated workloads timed beside the headline (default with --config 5: "
                         "2,3,4,4b; otherwise none)")
    ap.add_argument("--no-sub", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-graph", action="store_true", help="launch every call directly (no CUDA graph)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill timing")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="thread blocks per KV head (0 = the library's automatic plan)")
    args = ap.parse_args(argv)
    global NUM_SPLITS
    NUM_SPLITS = args.num_splits
    if args.warmup < 3:
        args.warmup = 3
    if args.no_sub:
        args.sub = []
    elif args.sub is None:
        args.sub = list(DEFAULT_SUBS) if args.config == "5" else []
    else:
        args.sub = [s for s in args.sub.split(",") if s]
        bad = [s for s in args.sub if s not in ("1", "2", "3", "4", "4b", "5")]
        if bad:
            ap.error("unknown workload(s) in --sub: %s" % ",".join(bad))
    rank, world, local_rank = init_dist()

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    setup_pg(world, "nccl")
    res = run_ours(args, rank, world, local_rank)
    allres = gather_results(res, world)
    if rank != 0:
        return 0
    print(json.dumps(make_line(args, allres)), flush=True)
    return 0


def sub_key(cfg):
    """JSON key of a workload: 4a and 4b are the two variants of workload 4."""
    return "4a" if cfg == "4" else cfg


def make_line(args, allres):
    """The JSON line of our arm from every rank's results (rank 0)."""
    peak, peak_src = load_peaks()
    r0 = allres[0]
    config = {"workload": workload_name(args.config), "config_id": sub_key(args.config),
              "l2": ("inputs %.0f MB > L2; %d set(s)" % (r0["kv_bytes"] / 1e6, r0["n_sets"])
                     if r0["n_sets"] == 1 else
                     "rotating %d input sets (%.0f MB in all) so every step reads HBM"
                     % (r0["n_sets"], r0["n_sets"] * r0["kv_bytes"] / 1e6)),
              "launch": ("the K timed steps replayed as one CUDA graph" if not args.no_graph
                         else "direct calls")}
    line = aggregate(allres, args.steps, args.warmup, args.gpus, config)
    # The roofline of the whole step: its algorithmic bytes over its event-timed
    # duration on the launching stream (for a one-call workload, that call).
    n_calls = r0["calls"] // args.steps
    step_kernel = ("the whole decode step: %d decode calls (%s), each a decode kernel and, where split "
                   "sequences are not merged in the grid, a combine (%d launches), timed together" % (
                       n_calls, ", ".join("%d %s" % (v["calls_per_step"], k) for k, v in sorted(r0["per_type"].items()))
                       if r0.get("per_type") else r0["heavy_kind"], r0["launches_per_step"]))
    line["roofline"] = hbm_roofline(r0["bytes"] / args.steps, r0["timed_ms_per_step"], peak, peak_src, step_kernel,
                                    recorded_traffic("step", args.config) if n_calls > 1 else
                                    recorded_traffic(r0["heavy_kind"], args.config))
    # the heaviest call of the step on its own (the dominant kernel)
    line["dominant_kernel"] = hbm_roofline(
        r0["heavy_bytes"], r0["heavy_ms"], peak, peak_src,
        "%s decode (%d launch%s per call, timed together)"
        % (r0["heavy_kind"], r0["heavy_kernels"], "es" if r0["heavy_kernels"] > 1 else ""),
        recorded_traffic(r0["heavy_kind"], args.config))
    line["dominant_kernel"]["ms_per_call"] = round(r0["heavy_ms"], 6)
    line["hbm_frac_of_peak"] = round(line["value"] / peak, 4)
    line["hbm_frac_of_dram_peak"] = round(line["value"] / NOMINAL_DRAM_GBS, 4)
    if r0.get("per_type"):
        line["per_layer_type"] = {k: dict(v, frac_of_peak=round(v["value"] / peak, 4),
                                          frac_of_dram_peak=round(v["value"] / NOMINAL_DRAM_GBS, 4))
                                  for k, v in r0["per_type"].items()}
    line["gpu_launches"] = r0["launches_per_step"] * args.steps
    if r0.get("subs"):
        line["workloads"] = {sub_key(k): v for k, v in r0["subs"].items()}
    if r0.get("prefill"):
        tpeak, tsrc = load_bf16_peak()
        line["prefill"] = {k: dict(v, roofline={"bound": "tensor", "achieved": v["value"], "peak": tpeak,
                                                "unit": "TFLOP/s", "frac": round(v["value"] / tpeak, 4),
                                                "peak_source": tsrc})
                           for k, v in r0["prefill"].items()}
    if r0.get("append"):
        line["append"] = {k: dict(v, frac_of_peak=round(v["value"] / peak, 4)) for k, v in r0["append"].items()}
    if r0.get("whole_step"):
        line["whole_step_launch"] = dict(r0["whole_step"], frac_of_peak=round(r0["whole_step"]["value"] / peak, 4),
                                         graph_replayed_us_per_step=round(r0["timed_ms_per_step"] * 1e3, 3))
    if r0.get("whole_step_append"):
        line["whole_step_launch_with_append"] = dict(r0["whole_step_append"],
                                                     frac_of_peak=round(r0["whole_step_append"]["value"] / peak, 4))
    if r0.get("shared"):
        line["global_values_only_cache"] = dict(r0["shared"], frac_of_peak=round(r0["shared"]["value"] / peak, 4))
    line["e2e"] = r0["e2e"]
    line["clocks"] = r0["clocks"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config)
    return line


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python3
"""BitLinear W1.58A8 forward benchmark (B300, sm_103a).

Headline workload, one step: decode at M = 1 over a ~2B-class ternary model's
projections -- 30 layers x {QKV 2560->3840, O 2560->2560, up 2560->6912,
down 6912->2560} with distinct weights (388 MB packed, three times the 126 MB
L2, so every step streams the weights from HBM; no L2 flush is needed) and a
bf16 N(0, 1) input per projection (the down projection's relu(z)^2-shaped).
A step is the 120 single-token forwards (activation quantisation + packed-
ternary contraction + rescale) as one bitlinear_forward_chain launch: the
inputs are independent, so the chain streams the weights of all 120 calls
without waiting between them.  Captured once in a CUDA graph and replayed.
Metric: GB/s of algorithmic bytes (packed weights + bf16 activations + fp32
outputs + gamma).

"extras" adds the same weights run as dependent calls (each call waits for
the one before: per-call launches, the chain with a grid barrier before every
call, the chain passing each output on as the next input), as independent
per-call launches, with grouped scales, batched decode M in {8,16,32,64},
prefill M = 2048 (tensor-core path; dense-equivalent 2*M*N*K ops/s) and the
100B-class shapes (80 layers, 9.4 GB resident).

--impl reference times the CPU oracle instead (the repository's plain C
restatement of the method) on a bounded sample of the same workload.

--profile CASE runs one case of these workloads a few times, untimed, and
exits: the command the kernel profiles under profiles/ are captured with.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BitLinear GB/s (decode, % HBM peak) and int8 TOPS (prefill, % INT8 peak)"
WORKLOAD = "decode_2b"

# DRAM bytes (read + write) of one chain launch of the headline step, from
# one ncu capture of the kernel source whose sha256 starts with `src`;
# reported as null once that source has changed.
CHAIN_TRAFFIC = {"bytes_per_launch": 389954304, "src": "31941f8aee9f025a",
                 "file": "w1_a8_bitlinear_02_b300/csrc/bl_chain.cuh"}


def measured_traffic():
    import hashlib
    path = os.path.join(ROOT, CHAIN_TRAFFIC["file"])
    try:
        h = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    ok = CHAIN_TRAFFIC["src"] and h.startswith(CHAIN_TRAFFIC["src"])
    return CHAIN_TRAFFIC["bytes_per_launch"] if ok else None


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons during the timed region.

    Uses the nvidia-smi query loop (the GPU picked by UUID, since nvidia-smi
    numbers every GPU of the machine), or NVML when nvidia-smi is missing."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index, self.period_ms = index, period_ms
        self.rows: list[list[str]] = []
        self.error = None
        self._proc = None
        self._t = None

    def _uuid(self):
        import torch
        try:
            u = str(torch.cuda.get_device_properties(self.index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def __enter__(self):
        import shutil
        import subprocess
        exe = shutil.which("nvidia-smi")
        if exe is None:
            self.error = "nvidia-smi not found"
            return self
        sel = self._uuid() or str(self.index)
        cmd = [exe, "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(self.period_ms)]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                          text=True)
        except Exception as e:
            self.error = repr(e)
            return self
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)  # let the first sample land before the timed region
        return self

    def _read(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def __exit__(self, *a):
        time.sleep(0.1)
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=5)

    def summary(self) -> dict:
        mhz, mx, reasons = [], None, set()
        for r in self.rows:
            try:
                mhz.append(float(r[0]))
                mx = float(r[1])
            except ValueError:
                continue
            for name, v in zip(self.NAMES, r[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz),
                **({"error": self.error} if self.error else {})}


# ------------------------------------------------------------------ helpers
def algorithmic_bytes(M: int, N: int, K: int, x_bytes: int = 2) -> int:
    """Bytes a BitLinear forward must move: packed weights, x, y and gamma."""
    row = ((K + 63) // 64) * 16
    return N * row + M * K * x_bytes + M * N * 4 + 4


def prepare(bl, wl, mats, M: int, device, x_dtype):
    """Pack each matrix's weights (seeded, drawn on the GPU) and draw x."""
    import torch
    out = []
    for mt in mats:
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, device)
        packed, gamma = bl.bitlinear_pack_weights(W)
        del W
        x = wl.activations(M, mt.K, mt.x_kind if M == 1 else "outliers1pct",
                           mt.seed + 500, device, x_dtype)
        y = torch.empty((M, mt.N), dtype=torch.float32, device=device)
        ws_n = bl.workspace_bytes(M, mt.N, mt.K)
        ws = torch.empty(ws_n, dtype=torch.uint8, device=device) if ws_n else None
        out.append(dict(mt=mt, packed=packed, gamma=gamma, x=x, y=y, ws=ws, M=M))
    torch.cuda.synchronize()
    return out


def to_slabs(items, torch):
    """Move every call's x (and y) into one contiguous device buffer, so an
    end-to-end step copies all inputs in with one transfer and all outputs out
    with one.  Each call keeps a view; offsets stay 16-byte aligned."""
    for key in ("x", "y"):
        ts = [it[key] for it in items]
        slab = torch.empty(sum(t.numel() for t in ts), dtype=ts[0].dtype, device=ts[0].device)
        off = 0
        for it, t in zip(items, ts):
            v = slab[off:off + t.numel()].view(t.shape)
            v.copy_(t)
            it[key] = v
            off += t.numel()
            assert (v.data_ptr() % 16) == 0
        items[0]["_" + key + "_slab"] = slab
    return items[0]["_x_slab"], items[0]["_y_slab"]


def sweep_calls(bl, items):
    for it in items:
        mt = it["mt"]
        bl.bitlinear_forward(it["packed"], it["gamma"], mt.N, mt.K, it["x"], y=it["y"],
                             workspace=it["ws"])


def capture(bl, items, stream):
    import torch
    # the inputs, outputs and workspaces were made on the current stream
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        sweep_calls(bl, items)  # warm (first launches set kernel attributes)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            sweep_calls(bl, items)
    return g


def time_graph(g, stream, steps: int, warmup: int, dist_mod, device) -> float:
    """Seconds for `steps` replays, CUDA events on `stream`, barrier-bracketed."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        stream.synchronize()
        dist_mod.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    dist_mod.barrier()
    return e0.elapsed_time(e1) / 1e3


def launches_per_call(bl, M: int, N: int, K: int) -> int:
    return 1 if bl.workspace_bytes(M, N, K) == 0 else 2


# ------------------------------------------------------------------ CPU oracle timing
ORACLE_WARM_S = 1.5  # thread pool up, caches warm, other CPU work settled


def oracle_warm(items_host, seconds: float = ORACLE_WARM_S) -> float:
    """Run the oracle's forward over the items for `seconds`; return the mean
    seconds per call seen (used to size a bounded sample)."""
    import oracle
    oracle.set_threads(os.cpu_count() or 1)
    t0 = time.perf_counter()
    calls = 0
    while True:
        for (packed, g, N, K, x) in items_host:
            oracle.forward_packed(packed, g, N, K, x)
            calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return el / calls


def oracle_timing(items_host, budget_s: float):
    """Time the CPU oracle's forward on host copies of (packed, gamma, x) for
    about `budget_s` seconds after the same warm-up as the reference arm.
    Returns (seconds, algorithmic bytes, calls, threads)."""
    import oracle
    oracle_warm(items_host)
    t0 = time.perf_counter()
    nbytes, calls = 0, 0
    while True:
        for (packed, g, N, K, x) in items_host:
            oracle.forward_packed(packed, g, N, K, x)
            nbytes += algorithmic_bytes(x.shape[0], N, K)
            calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el, nbytes, calls, oracle.get_threads()


def oracle_table(wl, torch) -> list:
    """The CPU oracle on bounded samples of every workload configuration, at
    one thread and at all host threads (the cpu_baseline leg, --cpu-table):
    weights packed and activations drawn on the host by the oracle and the
    seeded generators; per entry the seconds per unit and the rate."""
    import oracle

    def rate(fn, min_s=0.5):
        fn()
        t0 = time.perf_counter()
        n = 0
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                return el / n

    def packed_host(mt):
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, "cpu").numpy()
        p, g = oracle.pack_weights(W)
        del W
        return p, float(g)

    rows = []
    all_threads = os.cpu_count() or 1
    plans = []
    t = wl.matrices("tiny")[0]
    tp = packed_host(t)
    tx = wl.activations(4, t.K, t.x_kind, t.seed + 500, "cpu", torch.float32).numpy()
    plans.append(("1 tiny", "one forward, M=4, 256x512", [(tp, t.N, t.K, tx)], "GB/s"))
    mats = wl.matrices(WORKLOAD, layers=1)
    packs = [packed_host(mt) for mt in mats]
    x1 = [wl.activations(1, mt.K, mt.x_kind, mt.seed + 500, "cpu", torch.bfloat16).float().numpy() for mt in mats]
    plans.append(("2 decode M=1", "layer 0's four projections (QKV, O, up, down), M=1",
                  [(p, mt.N, mt.K, x) for p, mt, x in zip(packs, mats, x1)], "GB/s"))
    for M in (8, 16, 32, 64):
        xm = [wl.activations(M, mt.K, "outliers1pct", mt.seed + 500, "cpu", torch.bfloat16).float().numpy()
              for mt in mats]
        plans.append((f"3 decode M={M}", f"layer 0's four projections, M={M}",
                      [(p, mt.N, mt.K, x) for p, mt, x in zip(packs, mats, xm)], "GB/s"))
    T = 16
    for name, mt, kind in (("up", mats[2], "normal"), ("down", mats[3], "relu2")):
        p = packs[2] if name == "up" else packs[3]
        xt = wl.activations(T, mt.K, kind, mt.seed + 900, "cpu", torch.bfloat16).float().numpy()
        plans.append((f"4 prefill {name}", f"{T} of the 2048 tokens (tokens are independent) on "
                      f"{mt.N}x{mt.K}", [(p, mt.N, mt.K, xt)], "TOPS"))
    big = wl.matrices("decode_100b", layers=1)
    bpk = [packed_host(mt) for mt in big]
    for M in (1, 8):
        xb = [wl.activations(M, mt.K, "normal", mt.seed + 500, "cpu", torch.bfloat16).float().numpy() for mt in big]
        plans.append((f"5 100B M={M}", f"layer 0's two matrices (28672x8192, 8192x28672), M={M}",
                      [(p, mt.N, mt.K, x) for p, mt, x in zip(bpk, big, xb)], "GB/s"))
    for cfg, sample, calls, unit in plans:
        ent = {"config": cfg, "sample": sample, "unit": unit}
        for th in (1, all_threads):
            oracle.set_threads(th)
            sec = rate(lambda: [oracle.forward_packed(p[0], p[1], N, K, x) for (p, N, K, x) in calls])
            if unit == "GB/s":
                v = sum(algorithmic_bytes(x.shape[0], N, K) for (_, N, K, x) in calls) / sec / 1e9
            else:
                v = sum(2.0 * x.shape[0] * N * K for (_, N, K, x) in calls) / sec / 1e12
            ent[f"threads_{th}"] = {"s_per_sample": sec, unit: v}
        rows.append(ent)
        print(json.dumps(ent), file=sys.stderr, flush=True)
    oracle.set_threads(all_threads)
    return rows


def host_items(items, limit: int):
    out = []
    for it in items[:limit]:
        mt = it["mt"]
        out.append((it["packed"].cpu().numpy(), float(it["gamma"].item()), mt.N, mt.K,
                    it["x"].float().cpu().numpy()))
    return out


# ------------------------------------------------------------------ profiling cases
PROFILE_CASES = {
    # name: (M, N, K, activation kind, weight std, calls)
    "decode_2b_qkv": (1, 3840, 2560, "normal", 0.02, 6),
    "decode_100b_up": (1, 28672, 8192, "normal", 0.01, 6),
    "decode_100b_down": (1, 8192, 28672, "normal", 0.01, 6),
    "batch_m16_qkv": (16, 3840, 2560, "outliers1pct", 0.02, 6),
    "batch_m64_up": (64, 6912, 2560, "outliers1pct", 0.02, 6),
    "batch_m8_100b_up": (8, 28672, 8192, "normal", 0.01, 6),
    "prefill_up": (2048, 6912, 2560, "normal", 0.02, 6),
    "prefill_down": (2048, 2560, 6912, "relu2", 0.02, 6),
}


# decode-chain cases: (workload, layers, tokens, launches)
PROFILE_CHAINS = {
    "chain_2b": ("decode_2b", 30, 1, 4),       # the headline step
    "chain_2b_10": ("decode_2b", 10, 1, 4),    # 130 MB of weights (above L2), for full captures
    "chain_2b_m8": ("decode_2b", 10, 8, 4),
    "chain_100b_8": ("decode_100b", 8, 1, 4),  # 8 layers, 470 MB
}


def run_profile_chain(name: str):
    """A few untimed chain launches of one case on cuda:0 (for ncu captures)."""
    import torch
    import w1_a8_bitlinear_02_b300 as bl
    from w1_a8_bitlinear_02_b300 import workloads as wl
    wname, layers, M, n = PROFILE_CHAINS[name]
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    items = prepare(bl, wl, wl.matrices(wname, layers=layers), M, dev, torch.bfloat16)
    calls = chain_calls(items)
    ws = bl.chain_workspace(calls, dev)
    for _ in range(n):
        bl.bitlinear_forward_chain(calls, ws)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    print(json.dumps({"profile_chain": name, "calls": len(calls), "launches": n}), flush=True)


def run_profile_case(name: str):
    """A few untimed forward calls of one case on cuda:0 (for ncu captures)."""
    import torch
    import w1_a8_bitlinear_02_b300 as bl
    from w1_a8_bitlinear_02_b300 import workloads as wl
    if name in PROFILE_CHAINS:
        run_profile_chain(name)
        return
    M, N, K, kind, std, calls = PROFILE_CASES[name]
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    W = wl.weight(N, K, std, wl.weight_seed("decode_2b", 0, 0) + N, dev)
    packed, gamma = bl.bitlinear_pack_weights(W)
    del W
    x = wl.activations(M, K, kind, 4500 + K, dev, torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    wsn = bl.workspace_bytes(M, N, K)
    ws = torch.empty(wsn, dtype=torch.uint8, device=dev) if wsn else None
    for _ in range(calls):
        bl.bitlinear_forward(packed, gamma, N, K, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    print(json.dumps({"profile_case": name, "M": M, "N": N, "K": K, "calls": calls}), flush=True)


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank: int):
    """The CPU oracle on a bounded sample of the headline workload: layer 0's
    four projections at M = 1 (inputs drawn and packed on the host by the
    oracle itself).  A step is R forward calls cycling through the four
    projections, R sized from the warm-up so that the K timed steps take about
    REF_TIMED_S seconds; value = algorithmic bytes / time."""
    if rank != 0:
        return
    import oracle
    import torch
    from w1_a8_bitlinear_02_b300 import workloads as wl
    mats = wl.matrices(WORKLOAD, layers=1)  # one layer's four projections
    items = []
    for mt in mats:
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, "cpu").numpy()
        packed, g = oracle.pack_weights(W)
        x = wl.activations(1, mt.K, mt.x_kind, mt.seed + 500, "cpu", torch.bfloat16)
        items.append((packed, float(g), mt.N, mt.K, x.float().numpy()))
    t_call = oracle_warm(items)
    for i in range(args.warmup):
        p, g, N, K, x = items[i % len(items)]
        oracle.forward_packed(p, g, N, K, x)
    R = int(min(1000, max(len(items), -(-REF_TIMED_S // (args.steps * t_call)))))
    t0 = time.perf_counter()
    nbytes, c = 0, 0
    for _ in range(args.steps):
        for _ in range(R):
            p, g, N, K, x = items[c % len(items)]
            oracle.forward_packed(p, g, N, K, x)
            nbytes += algorithmic_bytes(1, N, K)
            c += 1
    el = time.perf_counter() - t0
    gbs = nbytes / el / 1e9
    cores = oracle.get_threads()
    sample = (f"{R} oracle forwards per step at M=1, cycling through layer 0's four projections "
              f"(QKV, O, up, down) of the ~2B decode workload; {args.steps * R} calls, "
              f"{el:.1f} s timed after {ORACLE_WARM_S} s of warm-up calls")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": "decode_2b M=1 (CPU oracle, bounded sample)", "sample": sample},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


REF_TIMED_S = 6.0


# ------------------------------------------------------------------ our arm
def chain_calls(items, mode="independent"):
    """Chain descriptors for the items: independent inputs (each call its own
    x), "barrier" (the same, each call waiting for every earlier one) or
    "dataflow" (each call's input is the previous call's output, cut to K;
    the down projection squares its ReLU)."""
    calls, prev = [], None
    for it in items:
        mt = it["mt"]
        c = dict(packed=it["packed"], gamma=it["gamma"], x=it["x"], y=it["y"], N=mt.N, K=mt.K,
                 wait_prev=1 if mode == "barrier" else 0)
        if mode == "dataflow" and prev is not None and prev.shape[1] >= mt.K:
            c["x"] = prev[:, :mt.K]
            c["act"] = 1 if mt.name == "down" else 0
        calls.append(c)
        prev = it["y"]
    return calls


def capture_chain(bl, calls, ws, stream):
    import torch
    # the workspace was zero-filled (and the inputs made) on the current stream
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        bl.bitlinear_forward_chain(calls, ws)  # warm (kernel attributes)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            bl.bitlinear_forward_chain(calls, ws)
    return g


def capture_chains(bl, parts, wss, stream):
    """One CUDA graph of several chain launches (one per part, each with its
    own workspace), in order."""
    import torch
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for calls, ws in zip(parts, wss):
            bl.bitlinear_forward_chain(calls, ws)  # warm (kernel attributes)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for calls, ws in zip(parts, wss):
                bl.bitlinear_forward_chain(calls, ws)
    return g


def chain_launches(calls) -> int:
    """Launches of one chain call: the set-up kernel (the call table into the
    workspace and the inputs no earlier call writes quantised into their
    records) and the chain itself."""
    return 2


def run_ours(args, rank: int, world: int, local: int):
    import torch

    import w1_a8_bitlinear_02_b300 as bl
    from w1_a8_bitlinear_02_b300 import dist as D
    from w1_a8_bitlinear_02_b300 import workloads as wl

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peaks = load_peaks()
    bl.set_launch_overlap(not args.no_overlap)
    stream = torch.cuda.Stream(device)

    mats = wl.matrices(WORKLOAD, layers=args.layers)
    items = prepare(bl, wl, mats, 1, device, torch.bfloat16)
    x_slab, y_slab = to_slabs(items, torch)
    step_bytes = sum(algorithmic_bytes(1, it["mt"].N, it["mt"].K) for it in items)
    packed_bytes = sum(it["packed"].numel() for it in items)
    calls = chain_calls(items)
    ws = bl.chain_workspace(calls, device)
    g = capture_chain(bl, calls, ws, stream)
    launches_step = chain_launches(calls)

    with ClockSampler(local) as clk:
        secs = time_graph(g, stream, args.steps, args.warmup, D, device)
    secs_max, bytes_all = D.aggregate(secs, step_bytes * args.steps, device)
    gbs = bytes_all / secs_max / 1e9
    ms_step = secs_max / args.steps * 1e3
    assert bl.device_error() == 0, "a kernel reported a device-side failure"

    # the dominant kernel: the chain, one launch per step; its duration is
    # taken as the whole step's (the two small set-up launches included), so
    # the achieved rate is a lower bound of the chain kernel's own
    per_launch_s = secs / args.steps
    achieved = step_bytes / per_launch_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic(),
                "traffic_unit": "bytes per launch (dram read + write, ncu)",
                "algorithmic_bytes_per_launch": step_bytes,
                "kernel": "bl::chain::chain_kernel",
                "duration": "step time (CUDA events on the launching stream) per chain launch, the "
                            "step's set-up launch (call table, input quantisation) included",
                "peak_source": f"{peaks['source']} (copy bandwidth)"}

    # end to end: every step copies its x in from pinned host memory and its
    # y out to pinned host memory (one slab each way).  Two buffer sets and
    # three streams pipeline the steps: step i's copies overlap the chain
    # launches of steps i - 1 and i + 1 (events keep a buffer from being
    # overwritten before its step has finished with it)
    items_b = [dict(it) for it in items]
    for it in items_b:
        it["x"] = it["x"].clone()
        it["y"] = torch.empty_like(it["y"])
    x_slab_b, y_slab_b = to_slabs(items_b, torch)
    calls_b = chain_calls(items_b)
    ws_b = bl.chain_workspace(calls_b, device)
    g_b = capture_chain(bl, calls_b, ws_b, stream)
    graphs = (g, g_b)
    x_slabs, y_slabs = (x_slab, x_slab_b), (y_slab, y_slab_b)
    x_hosts = tuple(xs.cpu().pin_memory() for xs in x_slabs)
    y_hosts = tuple(torch.empty_like(ys, device="cpu").pin_memory() for ys in y_slabs)
    h2d = x_hosts[0].numel() * x_hosts[0].element_size()
    d2h = y_hosts[0].numel() * y_hosts[0].element_size()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        if used[b]:
            s_in.wait_event(ev["comp"][b])    # the chain that read x_slabs[b] is done
            stream.wait_event(ev["out"][b])   # y_slabs[b] has been copied out
        with torch.cuda.stream(s_in):
            x_slabs[b].copy_(x_hosts[b], non_blocking=True)
        ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        graphs[b].replay()
        ev["comp"][b].record(stream)
        s_out.wait_event(ev["comp"][b])
        with torch.cuda.stream(s_out):
            y_hosts[b].copy_(y_slabs[b], non_blocking=True)
        ev["out"][b].record(s_out)
        used[b] = True

    with torch.cuda.stream(stream):
        e2e_steps = max(2, min(args.steps, 1000))
        for i in range(max(4, min(args.warmup, 20))):
            e2e_step(i)
        torch.cuda.synchronize()
        D.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        stream.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i)
        s_out.wait_stream(stream)
        s_out.wait_stream(s_in)
        e1.record(s_out)
        torch.cuda.synchronize()
    e2e_s, e2e_bytes = D.aggregate(e0.elapsed_time(e1) / 1e3, step_bytes * e2e_steps, device)
    e2e = {"value": e2e_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h,
           "how": "per step: one pinned-host -> device copy of the step's x slab (every call's x), "
                  "the chain launch, one device -> pinned-host copy of the step's y slab; two "
                  "buffer sets and separate copy streams overlap a step's copies with the chain "
                  "launches of its neighbours (events order each buffer's reuse); timed from "
                  "the first copy in to the last copy out"}
    del g_b, ws_b
    del g

    extras = {}
    if not args.no_extras:
        extras = run_extras(bl, wl, torch, device, stream, peaks, items, args)

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hi = host_items(items, 4)
        el, nb, ncalls, cores = oracle_timing(hi, args.cpu_seconds)
        cpu_baseline = {"value": nb / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                        "sample": f"{ncalls} calls of the oracle's forward on layer 0's four "
                                  "projections at M=1 (host copies of the same packed weights "
                                  f"and activations), {el:.1f} s after {ORACLE_WARM_S} s of warm-up"}
        if args.cpu_table:
            cpu_baseline["table"] = oracle_table(wl, torch)

    if rank == 0:
        line = {
            "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8", "data": "synthetic",
            "config": {"workload": f"decode_2b: M=1 over {args.layers} layers x {{qkv 3840x2560, "
                                   "o 2560x2560, up 6912x2560, down 2560x6912}, an independent "
                                   "x bf16 per projection, fused act-quant",
                       "M": 1, "layers": args.layers, "matrices": len(items),
                       "packed_weight_bytes_per_step": packed_bytes,
                       "algorithmic_bytes_per_step": step_bytes,
                       "l2": (f"inputs larger than L2 (packed weights {packed_bytes / 1e6:.0f} MB vs "
                              "126 MB L2); no flush") if packed_bytes > 126e6 else
                             f"packed weights {packed_bytes / 1e6:.0f} MB fit in L2 (reduced run)",
                       "launch": "CUDA graph of one bitlinear_forward_chain of the 120 calls "
                                 "(independent inputs: no call waits for another)",
                       "parallelism": f"{world} independent replica(s), weak scaling"},
            "roofline": roofline,
            "cpu_baseline": cpu_baseline,
            "e2e": e2e,
            "gpu_launches": launches_step * args.steps,
            "clocks": clk.summary(),
            "frac_of_hbm_peak": gbs / peaks["hbm_gbs"],
            "extras": extras,
        }
        print(json.dumps(line), flush=True)


def run_extras(bl, wl, torch, device, stream, peaks, items2b, args):
    out = {}
    reps = max(3, min(args.steps, 50))

    def timed(fn, n):
        for _ in range(3):
            fn()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    def line(nb, s, how, **kw):
        return {"GB/s": nb / s / 1e9, "frac_hbm": nb / s / 1e9 / peaks["hbm_gbs"], "ms_per_sweep": s * 1e3,
                "us_per_call": s * 1e6 / len(items2b), "how": how, **kw}

    nb = sum(algorithmic_bytes(1, it["mt"].N, it["mt"].K) for it in items2b)
    with torch.cuda.stream(stream):
        # dependent calls, per-call launches (launch overlap mode 1: a kernel
        # may prefetch its weights, then waits for the previous one)
        bl.set_launch_overlap(0 if args.no_overlap else 1)
        g = capture(bl, items2b, stream)
        out["decode_2b_per_call_dependent"] = line(nb, timed(g.replay, max(3, min(args.steps, 200))),
                                                   "120 bitlinear_forward launches, each waiting for the "
                                                   "previous (launch overlap mode 1)")
        del g
        # independent per-call launches (mode 2: the GEMV does not wait)
        bl.set_launch_overlap(2)
        g = capture(bl, items2b, stream)
        out["decode_2b_per_call_independent"] = line(nb, timed(g.replay, max(3, min(args.steps, 200))),
                                                     "120 bitlinear_forward launches, launch overlap mode 2")
        bl.set_launch_overlap(0 if args.no_overlap else 1)
        del g
        # the chain with every call waiting for all earlier ones (grid barrier)
        for mode, how in (("barrier", "bitlinear_forward_chain, every call waiting for all earlier calls "
                                      "at a grid barrier (independent inputs)"),
                          ("dataflow", "bitlinear_forward_chain, each call's input the previous call's "
                                       "output (fp32, read from its tagged output words as it lands); "
                                       "without normalisation between layers the values shrink layer "
                                       "by layer, the work per call is the same")):
            calls = chain_calls(items2b, mode)
            ws = bl.chain_workspace(calls, device)
            g = capture_chain(bl, calls, ws, stream)
            s = timed(g.replay, max(3, min(args.steps, 200)))
            out[f"decode_2b_chain_{mode}"] = line(nb, s, how)
            del g, ws

        # grouped scales: one weight scale per 128 output rows, dependent
        # per-call launches (the grouped forward has no chain form)
        G = 128
        gits = []
        for it in items2b:
            mt = it["mt"]
            W = wl.weight(mt.N, mt.K, mt.std, mt.seed, device)
            pk, gv = bl.bitlinear_pack_weights_grouped(W, G)
            del W
            gits.append(dict(mt=mt, packed=pk, gamma=gv, x=it["x"], y=it["y"], ws=it["ws"]))
        torch.cuda.synchronize()

        def grouped_sweep():
            for it in gits:
                mt = it["mt"]
                bl.bitlinear_forward_grouped(it["packed"], it["gamma"], G, mt.N, mt.K, it["x"], y=it["y"],
                                             workspace=it["ws"])
        gg = torch.cuda.CUDAGraph()
        grouped_sweep()
        stream.synchronize()
        with torch.cuda.graph(gg, stream=stream):
            grouped_sweep()
        s = timed(gg.replay, max(3, min(args.steps, 200)))
        nbg = nb + sum(4 * (it["mt"].N // G - 1) for it in items2b)  # the scale vectors
        out["decode_2b_grouped128"] = line(nbg, s, "bitlinear_forward_grouped, one weight scale per 128 "
                                                   "output rows, 120 dependent per-call launches")
        del gg, gits

        # batched decode on the same weights: dependent per-call launches,
        # and (8 and 16 tokens) the chain of independent calls -- 16 tokens as
        # two 8-token calls per projection, each streaming the weights
        mats = [it["mt"] for it in items2b]
        bd = {}
        for M in (8, 16, 32, 64):
            its = []
            for it in items2b:
                mt = it["mt"]
                x = wl.activations(M, mt.K, "outliers1pct", mt.seed + 600 + M, device, torch.bfloat16)
                y = torch.empty((M, mt.N), dtype=torch.float32, device=device)
                wsn = bl.workspace_bytes(M, mt.N, mt.K)
                ws = torch.empty(wsn, dtype=torch.uint8, device=device) if wsn else None
                its.append(dict(mt=mt, packed=it["packed"], gamma=it["gamma"], x=x, y=y, ws=ws))
            nbm = sum(algorithmic_bytes(M, m.N, m.K) for m in mats)
            ops = sum(2 * M * m.N * m.K for m in mats)
            g = capture(bl, its, stream)
            s = timed(g.replay, reps)
            bd[f"M={M}"] = {"GB/s": nbm / s / 1e9, "frac_hbm": nbm / s / 1e9 / peaks["hbm_gbs"],
                            "TOPS_dense_equiv": ops / s / 1e12, "ms_per_sweep": s * 1e3,
                            "how": "120 dependent bitlinear_forward launches (launch overlap mode 1)"}
            del g
            # the chain: calls of up to 16 tokens (the token rows of x in
            # slices of 16; each slice streams the weights again), at most
            # 240 calls a launch
            calls = []
            for it in its:
                mt = it["mt"]
                for h in range(0, M, 16):
                    calls.append(dict(packed=it["packed"], gamma=it["gamma"], x=it["x"][h:h + 16],
                                      y=it["y"][h:h + 16], N=mt.N, K=mt.K))
            parts = [calls[i:i + 240] for i in range(0, len(calls), 240)]
            wss = [bl.chain_workspace(pc, device) for pc in parts]
            gch = capture_chains(bl, parts, wss, stream)
            s = timed(gch.replay, reps)
            per = min(M, 16)
            bd[f"M={M} chain"] = {"GB/s": nbm / s / 1e9, "frac_hbm": nbm / s / 1e9 / peaks["hbm_gbs"],
                                  "TOPS_dense_equiv": ops / s / 1e12, "ms_per_sweep": s * 1e3,
                                  "how": (f"{len(parts)} bitlinear_forward_chain launch(es) of {len(calls)} calls "
                                          f"of {per} tokens (independent inputs)" +
                                          ("" if M <= 16 else f"; the weights stream {M // 16} times, the bytes "
                                                              "count them once"))}
            del gch, wss, calls, parts
            del its
        out["decode_2b_batch"] = bd

        # prefill M = 2048 on the tensor-core path (forward = activation
        # quantisation kernel + GEMM kernel).  The GEMM's own time is
        # estimated as the forward's minus that of bitlinear_quant_act on the
        # same x (the same one-pass quantisation, int8 instead of bf16 codes).
        pf = {}
        for name, N, K, kind in (("up", 6912, 2560, "normal"), ("down", 2560, 6912, "relu2")):
            W = wl.weight(N, K, 0.02, wl.weight_seed("prefill_2b", 0, 0) + N, device)
            packed, gamma = bl.bitlinear_pack_weights(W)
            del W
            x = wl.activations(2048, K, kind, 4500 + K, device, torch.bfloat16)
            y = torch.empty((2048, N), dtype=torch.float32, device=device)
            ws = torch.empty(bl.workspace_bytes(2048, N, K), dtype=torch.uint8, device=device)
            xq = torch.empty((2048, K), dtype=torch.int8, device=device)
            sc = torch.empty((2048,), dtype=torch.float32, device=device)
            s = timed(lambda: bl.bitlinear_forward(packed, gamma, N, K, x, y=y, workspace=ws), reps)
            # the same forward in plain stream order (no launch overlap): the
            # quantisation kernel, then the GEMM kernel
            mode = bl.get_launch_overlap()
            bl.set_launch_overlap(0)
            try:
                s_serial = timed(lambda: bl.bitlinear_forward(packed, gamma, N, K, x, y=y, workspace=ws), reps)
            finally:
                bl.set_launch_overlap(mode)
            sq = timed(lambda: bl.bitlinear_quant_act(x, xq=xq, scale=sc), reps)
            ops = 2 * 2048 * N * K
            tops = ops / s / 1e12
            tops_g = ops / max(s_serial - sq, 1e-9) / 1e12
            pf[name] = {"N": N, "K": K, "M": 2048, "ms": s * 1e3, "TOPS_dense_equiv": tops,
                        "frac_bf16_peak": tops / peaks["bf16_tflops"],
                        "ms_serial": s_serial * 1e3, "quant_ms": sq * 1e3, "gemm_ms_est": (s_serial - sq) * 1e3,
                        "gemm_roofline": {"bound": "tensor", "achieved": tops_g,
                                          "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                          "frac": tops_g / peaks["bf16_tflops"],
                                          "duration": "an estimate: the forward in plain stream order (no "
                                                      "launch overlap) minus bitlinear_quant_act's time (the "
                                                      "same one-pass quantisation writing int8 instead of "
                                                      "bf16 codes); CUDA events, same stream"},
                        "note": "sm_103a has no integer MMA; int8 x ternary runs exactly as "
                                "bf16 x bf16 -> fp32 on tcgen05 (kind::f16); peak = measured "
                                "dense bf16 (burst)"}
            del packed, gamma, x, y, ws, xq, sc
        out["prefill_2b"] = pf

        # the tiny configuration: one forward, M = 4, 256 x 512, fp32 x
        t = wl.matrices("tiny")[0]
        Wt = wl.weight(t.N, t.K, t.std, t.seed, device)
        tp, tg = bl.bitlinear_pack_weights(Wt)
        tx = wl.activations(4, t.K, t.x_kind, t.seed + 500, device, torch.float32)
        ty = torch.empty((4, t.N), dtype=torch.float32, device=device)
        gt = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            bl.bitlinear_forward(tp, tg, t.N, t.K, tx, y=ty)
            stream.synchronize()
            with torch.cuda.graph(gt, stream=stream):
                for _ in range(100):
                    bl.bitlinear_forward(tp, tg, t.N, t.K, tx, y=ty)
            st = timed(gt.replay, max(3, min(args.steps, 50))) / 100
        out["tiny"] = {"us_per_call": st * 1e6, "GB/s": algorithmic_bytes(4, t.N, t.K) / st / 1e9,
                       "how": "100 dependent bitlinear_forward calls (M=4, 256x512, fp32 x) in one graph"}
        del gt, Wt, tp, tg, tx, ty

        # 100B-class decode: 80 layers x {28672x8192, 8192x28672}, 9.4 GB
        # resident: M = 1 as one chain (independent inputs), as dependent and
        # as independent per-call launches; M = 8 dependent per-call launches
        if not args.no_100b:
            mats = wl.matrices("decode_100b")
            its = prepare(bl, wl, mats, 1, device, torch.bfloat16)
            nb1 = sum(algorithmic_bytes(1, it["mt"].N, it["mt"].K) for it in its)
            res = {}
            calls = chain_calls(its)
            ws = bl.chain_workspace(calls, device)
            gch = capture_chain(bl, calls, ws, stream)
            s = timed(gch.replay, max(3, min(args.steps, 20)))
            res["M=1 chain"] = {"GB/s": nb1 / s / 1e9, "frac_hbm": nb1 / s / 1e9 / peaks["hbm_gbs"],
                                "ms_per_sweep": s * 1e3, "us_per_call": s * 1e6 / len(its),
                                "how": "one bitlinear_forward_chain of the 160 calls (independent inputs)"}
            del gch, ws
            x8 = [wl.activations(8, it["mt"].K, "normal", it["mt"].seed + 508, device, torch.bfloat16) for it in its]
            y8 = [torch.empty((8, it["mt"].N), dtype=torch.float32, device=device) for it in its]
            calls = [dict(packed=it["packed"], gamma=it["gamma"], x=x, y=y, N=it["mt"].N, K=it["mt"].K)
                     for it, x, y in zip(its, x8, y8)]
            ws = bl.chain_workspace(calls, device)
            gch = capture_chain(bl, calls, ws, stream)
            s = timed(gch.replay, max(3, min(args.steps, 20)))
            nb8 = sum(algorithmic_bytes(8, it["mt"].N, it["mt"].K) for it in its)
            res["M=8 chain"] = {"GB/s": nb8 / s / 1e9, "frac_hbm": nb8 / s / 1e9 / peaks["hbm_gbs"],
                                "ms_per_sweep": s * 1e3, "us_per_call": s * 1e6 / len(its),
                                "how": "one bitlinear_forward_chain of the 160 calls of 8 tokens (independent inputs)"}
            del gch, ws, calls, x8, y8
            for M, mode in ((1, 1), (1, 2), (8, 1)):
                if M == 8:
                    for it in its:
                        mt = it["mt"]
                        it["x"] = wl.activations(8, mt.K, "normal", mt.seed + 508, device, torch.bfloat16)
                        it["y"] = torch.empty((8, mt.N), dtype=torch.float32, device=device)
                        wsn = bl.workspace_bytes(8, mt.N, mt.K)
                        it["ws"] = torch.empty(wsn, dtype=torch.uint8, device=device) if wsn else None
                bl.set_launch_overlap(mode)
                g = capture(bl, its, stream)
                s = timed(g.replay, max(3, min(args.steps, 20)))
                bl.set_launch_overlap(0 if args.no_overlap else 1)
                nbm = sum(algorithmic_bytes(M, it["mt"].N, it["mt"].K) for it in its)
                res[f"M={M} per-call " + ("dependent" if mode == 1 else "independent")] = {
                    "GB/s": nbm / s / 1e9, "frac_hbm": nbm / s / 1e9 / peaks["hbm_gbs"],
                    "ms_per_sweep": s * 1e3, "us_per_call": s * 1e6 / len(its),
                    "resident_packed_GB": sum(it["packed"].numel() for it in its) / 1e9,
                    "how": ("per-call launches, launch overlap mode 1" if mode == 1 else
                            "per-call launches, launch overlap mode 2")}
                del g
            del its
            out["decode_100b"] = res
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=30)
    ap.add_argument("--no-overlap", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-100b", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-table", action="store_true",
                    help="also time the CPU oracle on every configuration at 1 and all threads")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES) + sorted(PROFILE_CHAINS),
                    help="run one case a few times untimed (for ncu) and exit")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from w1_a8_bitlinear_02_b300 import dist as D
    rank, world, local = D.init()
    try:
        if args.impl == "reference":
            run_reference(args, rank)
        else:
            run_ours(args, rank, world, local)
    finally:
        D.finalize()


if __name__ == "__main__":
    main()

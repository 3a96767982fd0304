#!/usr/bin/env python
"""Benchmark: MoE decode layer latency and achieved HBM bandwidth on GB300.

One step = one decode-layer call (moe_layer: gate/up pass + down pass) on one
batch of B tokens of the Qwen3-style layer (E=128 experts, top-8, d=2048,
I=768, MXFP8 weights), seeded synthetic inputs already resident in HBM.
`value` = algorithmic bytes of all steps of all ranks / max-over-ranks time,
in TB/s, where a step's bytes are
    U*3*I*d*33/32 (+ shared) + 2Bd (x) + 8Bk (ids, w) + 4B(k+S)I (h) + 2Bd (y)
with U the exact number of distinct experts of that step's routing.

The timed region (K steps in CUDA graphs between CUDA events, barrier and
synchronize on both sides) is repeated and the median region is reported.

Also reported: the same-run copy-kernel peak, each pass alone with the
dominant kernel's roofline and the whole layer's fraction, the end-to-end
number through moe_layer_host (host buffers, copies inside the timed
region), align at prefill scale for two routings, the router, the MXFP8
activation round trip, the MXFP4 passes, the expert-centric grouped layer
against the decode layer from B=32 to 4096, the sweep of every decode
config (Qwen3 B=1..32, the routing-locality configs, DeepSeek-V3 with its
shared expert), the SM clocks sampled during the timed region and the CPU
oracle on a bounded sample.  `--impl reference` times the CPU oracle itself
on this workload; `--profile` runs a few plain calls of one path for ncu.

N > 1 (torchrun): every rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE decode layer µs and achieved HBM TB/s (% of copy peak) at B=1–32"
PAGE_TBPS_B32 = 3.95          # warp decode page, B=32, measured on B200 (context)
L2_BYTES = 129 * 1024 * 1024  # GB300 L2 (also queried at run time)
PROFILES = os.path.join(ROOT, "profiles")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--batch", type=int, default=32)
    p.add_argument("--routing", default="softmax_uniform")
    p.add_argument("--config", default="qwen3", choices=["qwen3", "deepseek", "tiny"])
    p.add_argument("--no-sweep", action="store_true", help="skip the B / routing / config sweep")
    p.add_argument("--min-seconds", type=float, default=0.5,
                   help="repeat the K-step timed region until this much timed work (median reported)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--ref-seconds", type=float, default=90.0)
    p.add_argument("--profile", choices=["layer", "fp4", "grouped"], default=None,
                   help="profiler run: --warmup + --steps plain calls of one path on the workload (one weight "
                        "copy, no timing, no other sections), then exit")
    return p.parse_args(argv)


# ------------------------------------------------------------ multi-rank ---

class Ranks:
    """Rank bookkeeping; torch.distributed only when WORLD_SIZE > 1."""

    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend or "nccl")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def reduce(self, value: float, op: str) -> float:
        if not self.pg:
            return value
        import torch
        dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
        if self.pg.get_backend() == "gloo":
            dev = "cpu"
        t = torch.tensor([value], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(bytes_per_rank: float, seconds_per_rank: float, ranks: Ranks):
    """Whole-job rate: all ranks' bytes over the slowest rank's time."""
    total = ranks.reduce(bytes_per_rank, "sum")
    slowest = ranks.reduce(seconds_per_rank, "max")
    return total, slowest, (total / slowest if slowest > 0 else 0.0)


# ------------------------------------------------------------- accounting ---

def layer_bytes(cfg, ids, B: int) -> dict:
    """Algorithmic bytes of one layer call on a routing `ids` [B, k]."""
    import torch
    U = int(torch.unique(ids).numel())
    S = 1 if cfg.shared else 0
    expert = cfg.I * cfg.d * 33 // 32            # one [I, d] MXFP8 matrix incl. scales
    gate_up = (U + S) * 2 * expert + 2 * B * cfg.d + 4 * B * cfg.k + 2 * B * (cfg.k + S) * cfg.I
    down = (U + S) * expert + 2 * B * (cfg.k + S) * cfg.I + 8 * B * cfg.k + 2 * B * cfg.d
    layer = (U + S) * 3 * expert + 2 * B * cfg.d + 8 * B * cfg.k + 4 * B * (cfg.k + S) * cfg.I + 2 * B * cfg.d
    return {"U": U, "gate_up": gate_up, "down": down, "layer": layer}


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_decode_gb300", "csrc")
    for name in ("common.cuh", "decode_common.cuh", "gate_up.cu", "down.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(PROFILES, f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_tr.group(1))


# ----------------------------------------------------------------- clocks ---

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.err = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.target = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.target = str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        except Exception as e:  # no nvidia-smi: report, do not fail the bench
            self.err = str(e)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


# ---------------------------------------------------------- GPU helpers ---

def graph_replayer(fn_steps, n_steps: int, stream):
    """Capture n_steps calls fn_steps(i) into one CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                fn_steps(i)
    return g


def time_steps(fn_steps, K: int, W: int, stream, ranks: Ranks, chunk: int = 250, sampler=None,
               min_seconds: float = 0.0, min_repeats: int = 1, max_repeats: int = 1):
    """W untimed warm-up steps, then the timed region: exactly K steps (CUDA
    graphs of `chunk` steps) between CUDA events on `stream`, with a barrier
    and a device synchronize on both sides.  The region is repeated at least
    `min_repeats` times and until `min_seconds` of timed work, at most
    `max_repeats` times; returns (median seconds of one K-step region, clock
    record, all region times)."""
    import torch
    chunk = max(1, min(chunk, K))
    with torch.cuda.stream(stream):     # first calls outside capture (one-time setup)
        fn_steps(0)
        fn_steps(1)
    stream.synchronize()
    g_main = graph_replayer(fn_steps, chunk, stream)
    rem = K % chunk
    g_rem = graph_replayer(fn_steps, rem, stream) if rem else None
    wq, wr = divmod(W, chunk)
    g_wr = graph_replayer(fn_steps, wr, stream) if wr else None
    with torch.cuda.stream(stream):
        for _ in range(wq):
            g_main.replay()
        if g_wr:
            g_wr.replay()
    stream.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.15)
    times = []
    while True:
        ranks.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(K // chunk):
                g_main.replay()
            if g_rem:
                g_rem.replay()
            t1.record(stream)
        t1.synchronize()
        torch.cuda.synchronize()
        ranks.barrier()
        times.append(t0.elapsed_time(t1) / 1e3)
        if len(times) >= max_repeats or (len(times) >= min_repeats and sum(times) >= min_seconds):
            break
    clocks = sampler.stop() if sampler else None
    return statistics.median(times), clocks, times


def measure_copy_peak(dev, nbytes=1 << 30, reps=10) -> float:
    import torch
    import mixture_experts_decode_gb300 as moe
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev).fill_(7)
    b = torch.empty_like(a)
    for _ in range(3):
        moe.copy(b, a)
    best = math.inf
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        moe.copy(b, a)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    del a, b
    torch.cuda.empty_cache()
    return 2 * nbytes / best / 1e9


def make_replicas(cfg, dev, R, start=0):
    """Weight replicas start .. R-1 of a layer config on the device."""
    import mixture_experts_decode_gb300 as moe
    from mixture_experts_decode_gb300 import inputs
    out = []
    for r in range(start, R):
        W = inputs.layer_weights(cfg, dev, replica=r)
        mx = lambda a, b: moe.MX(W[a], W[b])
        sh = None
        if W["shared"] is not None:
            s = W["shared"]
            sh = (moe.MX(s[0], s[1]), moe.MX(s[2], s[3]), moe.MX(s[4], s[5]))
        out.append((mx("w_gate", "s_gate"), mx("w_up", "s_up"), mx("w_down", "s_down"), sh))
    return out


class Workload:
    """Device-resident weights (R replicas) and NB batches of one layer config."""

    def __init__(self, cfg, B, routing, dev, n_batches=64, min_bytes=None, replicas=None):
        import torch
        import mixture_experts_decode_gb300 as moe
        from mixture_experts_decode_gb300 import inputs
        self.cfg, self.B, self.dev, self.routing = cfg, B, dev, routing
        self.batches = [inputs.layer_batch(cfg, B, routing=routing, step=i) for i in range(n_batches)]
        self.bytes = [layer_bytes(cfg, ids, B) for _, ids, _ in self.batches]
        mean_layer = statistics.mean(b["layer"] for b in self.bytes)
        l2 = min_bytes or 4 * L2_BYTES
        # replicas so that consecutive steps stream more than 4x L2 of weights
        R = max(1, math.ceil(l2 / mean_layer))
        full = (cfg.E + (1 if cfg.shared else 0)) * 3 * cfg.I * cfg.d * 33 // 32
        R = min(R, max(1, int(0.5 * torch.cuda.mem_get_info(dev)[0] // full)))
        if replicas is not None and len(replicas) >= R:
            self.replicas = replicas[:R]
        else:
            have = list(replicas or [])
            self.replicas = have + make_replicas(cfg, dev, R, start=len(have))
        self.R = len(self.replicas)
        self.x = [x.to(dev) for x, _, _ in self.batches]
        self.ids = [i.to(dev) for _, i, _ in self.batches]
        self.w = [w.to(dev) for _, _, w in self.batches]
        S = 1 if cfg.shared else 0
        self.ws = torch.empty(moe.layer_workspace_bytes(B, cfg.k, cfg.I, bool(S)), dtype=torch.uint8, device=dev)
        self.y = torch.empty((B, cfg.d), dtype=torch.bfloat16, device=dev)
        self.h = [torch.zeros((B, cfg.k + S, cfg.I), dtype=torch.bfloat16, device=dev)
                  for _ in range(n_batches)]

    def step(self, i):
        import mixture_experts_decode_gb300 as moe
        g, u, d, sh = self.replicas[i % self.R]
        j = i % len(self.batches)
        moe.layer(self.x[j], self.ids[j], self.w[j], g, u, d, shared=sh, workspace=self.ws, y=self.y)

    def gate_up(self, i):
        import mixture_experts_decode_gb300 as moe
        g, u, _, sh = self.replicas[i % self.R]
        j = i % len(self.batches)
        moe.gate_up(self.x[j], self.ids[j], g, u, shared_gate=sh[0] if sh else None,
                    shared_up=sh[1] if sh else None, h=self.h[j])

    def down(self, i):
        import mixture_experts_decode_gb300 as moe
        _, _, d, sh = self.replicas[i % self.R]
        j = i % len(self.batches)
        moe.down(self.h[j], self.ids[j], self.w[j], d, shared_down=sh[2] if sh else None, y=self.y)

    def mean_bytes(self, K, key="layer"):
        return sum(self.bytes[i % len(self.bytes)][key] for i in range(K)) / K


def cpu_oracle_sample(wl: "Workload", seconds: float):
    """Time the CPU oracle on the first tokens of batch 0 (~`seconds` of CPU),
    single-threaded and pinned to one host core."""
    import numpy as np
    import torch
    import oracle
    cfg = wl.cfg
    x, ids, w = wl.batches[0]
    g, u, d, sh = wl.replicas[0]
    host_cores = sorted(os.sched_getaffinity(0))

    def run(tokens):
        sub = ids[:tokens]
        uniq = sorted(set(sub.reshape(-1).tolist()))
        remap = np.full(max(uniq) + 1, -1, np.int64)
        remap[uniq] = np.arange(len(uniq))
        idx = torch.tensor(uniq, dtype=torch.long, device=wl.dev)
        host = [t.index_select(0, idx).cpu().numpy() for t in (g.w, g.s, u.w, u.s, d.w, d.s)]
        shared = None
        if sh is not None:
            shared = tuple(t.cpu().numpy() for m in sh for t in (m.w, m.s))
        xb = x[:tokens].contiguous().view(torch.int16).numpy().astype(np.uint16)
        t0 = time.perf_counter()
        oracle.moe_layer(xb, remap[sub.numpy()].astype(np.int32), w[:tokens].numpy(), *host, shared=shared)
        return time.perf_counter() - t0

    try:
        os.sched_setaffinity(0, {host_cores[-1]})
        t1 = run(1)
        n = int(max(1, min(wl.B, seconds / max(t1, 1e-6))))
        dt = run(n) if n > 1 else t1
    finally:
        os.sched_setaffinity(0, set(host_cores))
    nbytes = layer_bytes(cfg, ids[:n], n)["layer"]
    return {"value": nbytes / dt / 1e12, "unit": "TB/s", "cores": 1, "kind": "oracle",
            "host_cores": len(host_cores), "host_cpu_count": os.cpu_count(),
            "sample": f"oracle (single-threaded C, FP64, pinned to one host core) on the first {n} of {wl.B} "
                      f"tokens of one batch: {dt:.2f} s; value = that sub-batch's algorithmic layer bytes / time"}


def measure_layer(wl, stream, ranks, K, W, hbm_peak, copy_gbs, kernels=True):
    """Layer, and optionally each pass alone, on one workload: µs and TB/s."""
    secs, _, _ = time_steps(wl.step, K, W, stream, ranks, chunk=min(K, 250), min_seconds=0.1, min_repeats=3, max_repeats=10)
    nb = wl.mean_bytes(K)
    us = secs / K * 1e6
    out = {"B": wl.B, "routing": wl.routing, "replicas": wl.R,
           "unique_experts_mean": statistics.mean(b["U"] for b in wl.bytes),
           "algorithmic_bytes_mean": nb, "us": us, "tbps": nb / (us * 1e-6) / 1e12,
           "frac_of_measured_peak": nb / (us * 1e-6) / 1e9 / hbm_peak,
           "frac_of_copy_peak": nb / (us * 1e-6) / 1e9 / copy_gbs}
    if kernels:
        wl.gate_up(0)
        for name, fn in (("gate_up", wl.gate_up), ("down", wl.down)):
            ks, _, _ = time_steps(fn, K, W, stream, ranks, chunk=min(K, 250), min_seconds=0.1, min_repeats=3, max_repeats=10)
            kus = ks / K * 1e6
            kb = wl.mean_bytes(K, name)
            out[name] = {"us": kus, "gbs": kb / (kus * 1e-6) / 1e9,
                         "frac_of_measured_peak": kb / (kus * 1e-6) / 1e9 / hbm_peak}
    return out


def measure_grouped(wl, stream, ranks, K):
    """µs per moe_layer_grouped call on a workload's batches and weights
    (shared expert included); None if the call is refused."""
    import torch
    import mixture_experts_decode_gb300 as moe
    cfg = wl.cfg
    try:
        ws = torch.empty(moe.layer_grouped_workspace_bytes(wl.B, cfg.k, cfg.E, cfg.d, cfg.I, cfg.shared),
                         dtype=torch.uint8, device=wl.dev)

        def step(i):
            g, u, d, sh = wl.replicas[i % wl.R]
            j = i % len(wl.batches)
            moe.layer_grouped(wl.x[j], wl.ids[j], wl.w[j], g, u, d, shared=sh, workspace=ws, y=wl.y)

        secs, _, _ = time_steps(step, K, 3, stream, ranks, chunk=K, min_seconds=0.05, min_repeats=3, max_repeats=10)
        del ws
        return secs / K * 1e6
    except Exception:  # reported as missing, never fatal to the bench line
        return None


def sweep(dev, stream, ranks, hbm_peak, copy_gbs, qwen_replicas):
    """Every decode config of the workload list: the Qwen3-style B sweep, the
    routing-locality sweep at B=32 (with the contiguous - scattered gap) and
    the DeepSeek-V3-style B sweep with its shared expert (at B = 32 and 64
    also the expert-centric layer, `grouped_us`)."""
    import torch
    from mixture_experts_decode_gb300 import inputs
    out = {"qwen3": [], "locality_b32": {}, "deepseek_v3": []}
    reps = list(qwen_replicas)
    for B in (1, 2, 4, 8, 16, 32):
        wl = Workload(inputs.QWEN3, B, "softmax_uniform", dev, n_batches=16, replicas=reps)
        reps = wl.replicas if len(wl.replicas) > len(reps) else reps
        out["qwen3"].append(measure_layer(wl, stream, ranks, 400, 20, hbm_peak, copy_gbs))
        if B == 32:
            out["locality_b32"]["softmax_uniform"] = out["qwen3"][-1]
        del wl
    for routing in ("contiguous", "zipf"):
        wl = Workload(inputs.QWEN3, 32, routing, dev, n_batches=16, replicas=reps)
        out["locality_b32"][routing] = measure_layer(wl, stream, ranks, 400, 20, hbm_peak, copy_gbs)
        del wl
    loc = out["locality_b32"]
    loc["gap_tbps_contiguous_minus_uniform"] = loc["contiguous"]["tbps"] - loc["softmax_uniform"]["tbps"]
    loc["gap_tbps_contiguous_minus_zipf"] = loc["contiguous"]["tbps"] - loc["zipf"]["tbps"]
    del reps
    torch.cuda.empty_cache()
    ds = []
    for B in (1, 8, 32, 64):
        wl = Workload(inputs.DEEPSEEK_V3, B, "sigmoid_scaled", dev, n_batches=8, replicas=ds)
        ds = wl.replicas if len(wl.replicas) > len(ds) else ds
        row = measure_layer(wl, stream, ranks, 40, 5, hbm_peak, copy_gbs)
        if B >= 32:  # the expert-centric layer (with its shared-expert pass) on the same batches
            row["grouped_us"] = measure_grouped(wl, stream, ranks, 20)
        out["deepseek_v3"].append(row)
        del wl
    del ds
    torch.cuda.empty_cache()
    return out


def run_align(dev, stream, ranks, routing="softmax_normal", K=200):
    import torch
    import mixture_experts_decode_gb300 as moe
    from mixture_experts_decode_gb300 import inputs
    T, k, E, bs = 16384, 8, 256, 64
    ids = inputs.align_ids(T, k, E, routing).to(dev)
    ns, nb, wsb = moe.align_sizes(T, k, E, bs)
    s = torch.empty(ns, dtype=torch.int32, device=dev)
    e = torch.empty(nb, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    secs, _, _ = time_steps(lambda i: moe.align_block_size(ids, E, bs, s, e, n, ws), K, 20, stream, ranks,
                            chunk=100, min_seconds=0.1, min_repeats=3, max_repeats=10)
    nbytes = 4 * (T * k + ns + nb + 1)
    return {"workload": f"align T=16384 k=8 E=256 block_size=64 {routing}", "us": secs / K * 1e6,
            "gbs": nbytes / (secs / K) / 1e9, "algorithmic_bytes": nbytes}


def run_router(dev, stream, ranks, cfg, B, K=200):
    """The routing step for this workload's routing at this batch (one launch)."""
    import torch
    import mixture_experts_decode_gb300 as moe
    from mixture_experts_decode_gb300 import inputs
    score, scale = ("sigmoid", 2.5) if cfg.routing == "sigmoid_scaled" else ("softmax", 1.0)
    kind = cfg.routing if cfg.routing in ("softmax_uniform", "softmax_normal", "sigmoid_scaled") else "softmax_normal"
    lg = inputs.router_logits(kind, B, cfg.E, "bench-router", B).to(dev)
    ids = torch.empty((B, cfg.k), dtype=torch.int32, device=dev)
    w = torch.empty((B, cfg.k), dtype=torch.float32, device=dev)
    secs, _, _ = time_steps(lambda i: moe.router_topk(lg, cfg.k, score, scale, ids, w), K, 20, stream, ranks,
                            chunk=100)
    return {"workload": f"router {score} top-{cfg.k} of E={cfg.E}, B={B}" + (f" x{scale}" if score == "sigmoid" else ""),
            "us": secs / K * 1e6}


def run_requant(dev, stream, ranks, copy_gbs, rows=16384, K=4096, reps=50):
    """The MXFP8 activation round trip (moe_mx_requant) on a BF16 [rows, K]
    tensor larger than L2: read 2 B + write 2 B per value."""
    import torch
    import mixture_experts_decode_gb300 as moe
    from mixture_experts_decode_gb300 import inputs
    x = inputs.randn((rows, K), dev, "bench-requant").to(torch.bfloat16)
    out = torch.empty_like(x)
    secs, _, _ = time_steps(lambda i: moe.mx_requant(x, out), reps, 5, stream, ranks, chunk=25)
    nbytes = 4 * rows * K
    gbs = nbytes / (secs / reps) / 1e9
    return {"workload": f"BF16 [{rows}, {K}] -> MXFP8 -> BF16", "us": secs / reps * 1e6, "gbs": gbs,
            "algorithmic_bytes": nbytes, "frac_of_copy_peak": gbs / copy_gbs}


def run_fp4(dev, stream, ranks, cfg, B, routing, copy_gbs, K=100, n_batches=16):
    """The MXFP4-weight passes (moe_gate_up_fp4 + moe_down_fp4) on this
    workload with MXFP4 weights.  Algorithmic bytes count each distinct
    expert's codes once (I*d/2 per matrix) plus its scales (I*d/32) and the
    activations; this path streams a shared expert's rows once per token
    that routes to it, so its achieved GB/s is a floor, not a traffic
    figure.  A failure here leaves an "error" field instead of a number."""
    try:
        import torch
        import mixture_experts_decode_gb300 as moe
        from mixture_experts_decode_gb300 import inputs
        W = inputs.layer_weights(cfg, dev, fp4=True)
        mx = lambda a, b: moe.MX(W[a], W[b])
        G, Uw, D = mx("w_gate", "s_gate"), mx("w_up", "s_up"), mx("w_down", "s_down")
        sh = None
        if W.get("shared") is not None:
            s = W["shared"]
            sh = (moe.MX(s[0], s[1]), moe.MX(s[2], s[3]), moe.MX(s[4], s[5]))
        S = 1 if sh else 0
        bt = []
        nbytes = []
        expert = cfg.I * cfg.d // 2 + cfg.I * cfg.d // 32
        for i in range(n_batches):
            x, ids, w = inputs.layer_batch(cfg, B, routing=routing, step=i)
            U = int(torch.unique(ids).numel())
            nbytes.append((U + S) * 3 * expert + 4 * B * cfg.d + 8 * B * cfg.k + 4 * B * (cfg.k + S) * cfg.I)
            bt.append((x.to(dev), ids.to(dev), w.to(dev)))
        h = torch.empty((B, cfg.k + S, cfg.I), dtype=torch.bfloat16, device=dev)
        y = torch.empty((B, cfg.d), dtype=torch.bfloat16, device=dev)

        def step(i):
            x, ids, w = bt[i % n_batches]
            moe.gate_up(x, ids, G, Uw, shared_gate=sh[0] if sh else None, shared_up=sh[1] if sh else None,
                        h=h, fp4=True)
            moe.down(h, ids, w, D, shared_down=sh[2] if sh else None, y=y, fp4=True)

        secs, _, _ = time_steps(step, K, 5, stream, ranks, chunk=50)
        mean_bytes = sum(nbytes[i % n_batches] for i in range(K)) / K
        us = secs / K * 1e6
        gbs = mean_bytes / (secs / K) / 1e9
        del W, bt
        torch.cuda.empty_cache()
        return {"workload": f"{cfg.name} B={B} routing={routing}, MXFP4 weights (E2M1, E8M0 per 32)",
                "kernels": "the row-tile gate/up and down kernels with MXFP4 tiles (one warp per output "
                           "value at B=1)",
                "us": us, "gbs": gbs, "algorithmic_bytes_mean": mean_bytes,
                "frac_of_copy_peak": gbs / copy_gbs}
    except Exception as exc:  # reported, never fatal to the bench line
        return {"error": repr(exc)[:300]}


def run_grouped(dev, stream, ranks, hbm_peak, tensor_peak, reps, batches=(32, 64, 128, 256, 1024, 4096)):
    """The expert-centric layer (moe_layer_grouped) against the decode layer
    on the Qwen3-style workload, per B: µs of each (the decode layer up to its
    B <= 256 limit), the grouped layer with MXFP8 activations too, and the
    grouped layer's achieved HBM GB/s (algorithmic bytes: each distinct
    expert's weights once, x, ids, w and y) and tensor TFLOP/s (2 * B * k * 3
    * d * I).  One weight copy per replica, cycled; a failure leaves an
    "error" field."""
    try:
        import torch
        import mixture_experts_decode_gb300 as moe
        from mixture_experts_decode_gb300 import inputs
        cfg = inputs.QWEN3
        rows = []
        for B in batches:
            n_b = 4
            bt = [inputs.layer_batch(cfg, B, step=i) for i in range(n_b)]
            by = [layer_bytes(cfg, ids, B) for _, ids, _ in bt]
            dv = [(x.to(dev), i.to(dev), w.to(dev)) for x, i, w in bt]
            ws = torch.empty(moe.layer_grouped_workspace_bytes(B, cfg.k, cfg.E, cfg.d, cfg.I),
                             dtype=torch.uint8, device=dev)
            y = torch.empty((B, cfg.d), dtype=torch.bfloat16, device=dev)

            def grouped(i, act=False):
                g, u, d, _ = reps[i % len(reps)]
                x, ids, w = dv[i % n_b]
                moe.layer_grouped(x, ids, w, g, u, d, act_mx=act, workspace=ws, y=y)

            K = 40 if B <= 1024 else 10
            gs, _, _ = time_steps(grouped, K, 3, stream, ranks, chunk=K, min_seconds=0.05, min_repeats=3,
                                  max_repeats=10)
            gms, _, _ = time_steps(lambda i: grouped(i, True), K, 3, stream, ranks, chunk=K, min_seconds=0.05,
                                   min_repeats=3, max_repeats=10)
            alg = statistics.mean(b["U"] for b in by) * 3 * cfg.I * cfg.d * 33 // 32 + 4 * B * cfg.d + 8 * B * cfg.k
            flops = 2.0 * B * cfg.k * 3 * cfg.d * cfg.I
            row = {"B": B, "grouped_us": gs / K * 1e6, "grouped_act_mx_us": gms / K * 1e6,
                   "unique_experts_mean": statistics.mean(b["U"] for b in by),
                   "grouped_gbs": alg / (gs / K) / 1e9, "grouped_frac_of_hbm_peak": alg / (gs / K) / 1e9 / hbm_peak,
                   "grouped_tflops": flops / (gs / K) / 1e12,
                   "grouped_frac_of_tensor_peak": flops / (gs / K) / 1e12 / tensor_peak}
            if B <= 256:
                wsd = torch.empty(moe.layer_workspace_bytes(B, cfg.k, cfg.I, False), dtype=torch.uint8, device=dev)

                def decode(i):
                    g, u, d, _ = reps[i % len(reps)]
                    x, ids, w = dv[i % n_b]
                    moe.layer(x, ids, w, g, u, d, workspace=wsd, y=y)

                ds, _, _ = time_steps(decode, K, 3, stream, ranks, chunk=K, min_seconds=0.05, min_repeats=3,
                                      max_repeats=10)
                row["decode_us"] = ds / K * 1e6
                row["faster"] = "grouped" if gs < ds else "decode"
            rows.append(row)
            del ws, dv
        torch.cuda.empty_cache()
        return {"workload": f"{cfg.name} routing={cfg.routing}, moe_layer_grouped vs moe_layer",
                "kernels": "align + grouped_mma_kernel<2> (gate/up) + grouped_mma_kernel<1> (down) + combine; "
                           "tcgen05.mma kind::f16, BF16 operands dequantised from MXFP8 in shared memory",
                "tensor_peak_tflops": tensor_peak, "rows": rows}
    except Exception as exc:  # reported, never fatal to the bench line
        return {"error": repr(exc)[:300]}


# -------------------------------------------------------------------- arms ---

def run_e2e(wl, stream, ranks, K, W):
    """The same layer through moe_layer_host (pinned host x / topk_ids /
    topk_w in, y out; the copies inside the timed region, every step).  Two
    streams with their own workspace and host y take alternate steps, so one
    step's copies overlap the other's kernels, as a serving loop would run."""
    import torch
    import mixture_experts_decode_gb300 as moe
    cfg, B, dev = wl.cfg, wl.B, wl.dev
    S = 1 if cfg.shared else 0
    xh = [x.pin_memory() for x, _, _ in wl.batches]
    ih = [i.pin_memory() for _, i, _ in wl.batches]
    wh = [w.pin_memory() for _, _, w in wl.batches]
    streams = [stream, torch.cuda.Stream(dev)]
    yh = [torch.empty((B, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in streams]
    nws = moe.layer_host_workspace_bytes(B, cfg.d, cfg.k, cfg.I, bool(S))
    hws = [torch.empty(nws, dtype=torch.uint8, device=dev) for _ in streams]

    def e2e_step(i):
        g, u, d, sh = wl.replicas[i % wl.R]
        j = i % len(wl.batches)
        q = i % 2
        with torch.cuda.stream(streams[q]):
            moe.layer_host(xh[j], ih[j], wh[j], g, u, d, shared=sh, workspace=hws[q], y_host=yh[q], device=dev)

    for i in range(max(3, W)):
        e2e_step(i)
    torch.cuda.synchronize()
    ranks.barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    streams[1].wait_event(s0)
    for i in range(K):
        e2e_step(i)
    done = torch.cuda.Event()
    done.record(streams[1])
    stream.wait_event(done)
    s1.record(stream)
    s1.synchronize()
    torch.cuda.synchronize()
    ranks.barrier()
    secs = s0.elapsed_time(s1) / 1e3
    _, slow, rate = aggregate(wl.mean_bytes(K) * K, secs, ranks)
    return {"value": rate / 1e12, "unit": "TB/s", "us_per_step": slow / K * 1e6,
            "h2d_bytes_per_step": B * cfg.d * 2 + B * cfg.k * 8, "d2h_bytes_per_step": B * cfg.d * 2,
            "api": "moe_layer_host (pinned host x/topk_ids/topk_w -> y), two streams taking alternate steps"}


def run_ours(args):
    import torch
    import __graft_entry__
    from mixture_experts_decode_gb300 import inputs

    ranks = Ranks()
    torch.cuda.set_device(ranks.local)
    dev = torch.device("cuda", ranks.local)
    __graft_entry__.build()
    global L2_BYTES
    L2_BYTES = torch.cuda.get_device_properties(dev).L2_cache_size or L2_BYTES
    cfg = {"qwen3": inputs.QWEN3, "deepseek": inputs.DEEPSEEK_V3, "tiny": inputs.TINY}[args.config]
    B, K, W = args.batch, args.steps, args.warmup
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "MEASURED_PEAKS.json hbm_gbs (burst copy), of measured"
    if not hbm_peak:
        hbm_peak, peak_src = 6800.0, "fallback 6.8 TB/s, of fallback"
    copy_gbs = measure_copy_peak(dev)

    wl = Workload(cfg, B, args.routing, dev)
    stream = torch.cuda.Stream(dev)
    sampler = ClockSampler(ranks.local)
    secs, clocks, region_times = time_steps(wl.step, K, W, stream, ranks, sampler=sampler,
                                            min_seconds=args.min_seconds, min_repeats=5, max_repeats=1000)
    nbytes = wl.mean_bytes(K) * K
    total_bytes, slowest, rate = aggregate(nbytes, secs, ranks)
    value = rate / 1e12
    us_per_step = slowest / K * 1e6

    # each pass alone on the same inputs, timed on the stream it launches on
    kk = max(50, min(K, 1000))
    wl.gate_up(0)
    gu_secs, _, _ = time_steps(wl.gate_up, kk, 10, stream, ranks, min_seconds=0.1, min_repeats=3, max_repeats=20)
    dn_secs, _, _ = time_steps(wl.down, kk, 10, stream, ranks, min_seconds=0.1, min_repeats=3, max_repeats=20)
    gu_us, dn_us = gu_secs / kk * 1e6, dn_secs / kk * 1e6
    gu_gbs = wl.mean_bytes(kk, "gate_up") / (gu_us * 1e-6) / 1e9
    dn_gbs = wl.mean_bytes(kk, "down") / (dn_us * 1e-6) / 1e9
    workload_tag = f"{args.config}_b{B}"
    dom = "gate_up" if gu_us >= dn_us else "down"
    dom_gbs = gu_gbs if dom == "gate_up" else dn_gbs
    layer_gbs = value * 1e3
    roofline = {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": dom_gbs / hbm_peak, "traffic": profiled_traffic(dom, workload_tag),
                "peak_source": peak_src, "algorithmic_bytes_per_launch": wl.mean_bytes(kk, dom),
                "layer": {"achieved": layer_gbs, "frac": layer_gbs / hbm_peak,
                          "note": "the whole layer (both passes) against the same peak"}}

    Ke = min(K, 2000)
    e2e = run_e2e(wl, stream, ranks, Ke, W)
    align = run_align(dev, stream, ranks)
    align_zipf = run_align(dev, stream, ranks, routing="zipf")
    router = run_router(dev, stream, ranks, cfg, B)
    requant = run_requant(dev, stream, ranks, copy_gbs)
    fp4 = run_fp4(dev, stream, ranks, cfg, B, args.routing, copy_gbs)

    cpu = None
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(wl, args.cpu_seconds)
    qwen_reps = wl.replicas if cfg is inputs.QWEN3 else []
    wl_bytes = wl.bytes
    del wl
    torch.cuda.empty_cache()
    tensor_peak = peaks.get("bf16_tflops") or 1900.0
    grouped = None if args.no_sweep else run_grouped(dev, stream, ranks, hbm_peak, tensor_peak,
                                                     qwen_reps[:2] or make_replicas(inputs.QWEN3, dev, 2))
    sw = None if args.no_sweep else sweep(dev, stream, ranks, hbm_peak, copy_gbs, qwen_reps)

    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": ranks.world, "steps": K, "warmup": W,
        "ms_per_step": us_per_step / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGE_TBPS_B32 if (args.config == "qwen3" and B == 32) else None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{cfg.name} B={B} routing={args.routing}", "E": cfg.E, "k": cfg.k,
                   "d": cfg.d, "I": cfg.I, "B": B, "shared_expert": cfg.shared,
                   "weights": "MXFP8 (E4M3, E8M0 per 32 along K); BF16 activations; FP32 accumulation",
                   "l2": f"inputs larger than L2: {nbytes / K / 1e6:.0f} MB streamed per step, "
                         f"weight replicas x 64 batches cycled (L2 {L2_BYTES / 2**20:.0f} MiB)",
                   "parallelism": f"replicas x{ranks.world}"},
        "timing": {"repeats": len(region_times), "statistic": "median over repeats of the K-step region",
                   "region_ms_min": min(region_times) * 1e3, "region_ms_max": max(region_times) * 1e3},
        "layer_us": us_per_step, "unique_experts_mean": statistics.mean(b["U"] for b in wl_bytes),
        "copy_peak_gbs": copy_gbs, "pct_of_copy_peak": 100 * value * 1e3 / copy_gbs,
        "pct_of_measured_peak": 100 * value * 1e3 / hbm_peak, "pct_of_8tbs_nominal": 100 * value / 8.0,
        "kernels": {"gate_up_us": gu_us, "gate_up_gbs": gu_gbs, "down_us": dn_us, "down_gbs": dn_gbs},
        "roofline": roofline, "e2e": e2e, "gpu_launches": 2 * K * len(region_times), "clocks": clocks,
        "align": align, "align_zipf": align_zipf, "router": router, "mx_requant": requant, "fp4_layer": fp4,
        "cpu_baseline": cpu, "grouped": grouped, "sweep": sw,
    }
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)
    ranks.close()


def run_reference(args):
    """The CPU oracle as it stands, on this workload's shapes (rank 0 only)."""
    ranks_rank = int(os.environ.get("RANK", "0"))
    if ranks_rank != 0:
        return
    import numpy as np
    import torch
    import oracle
    from mixture_experts_decode_gb300 import inputs
    cfg = {"qwen3": inputs.QWEN3, "deepseek": inputs.DEEPSEEK_V3, "tiny": inputs.TINY}[args.config]
    B, K, W = args.batch, args.steps, args.warmup
    x, ids, w = inputs.layer_batch(cfg, B, routing=args.routing)
    # a step = the oracle layer on one token restricted to its first routed
    # expert and the first `m` intermediate neurons (a slice of the same
    # matrices); m sized so that warm-up + K steps take about ref-seconds
    e0 = int(ids[0, 0])
    Wt = inputs.expert_weights(cfg, [e0], "cpu")

    def sliced(m):
        arrs = [Wt["w_gate"][:, :m], Wt["s_gate"][:, :m], Wt["w_up"][:, :m], Wt["s_up"][:, :m],
                Wt["w_down"][:, :, :m], Wt["s_down"][:, :, :m // 32]]
        return [np.ascontiguousarray(a.numpy()) for a in arrs]

    xb = x[:1].contiguous().view(torch.int16).numpy().astype(np.uint16)
    one = np.zeros((1, 1), np.int32)
    w1 = np.ones((1, 1), np.float32)

    def step(arrs):
        oracle.moe_layer(xb, one, w1, *arrs)

    host_cores = sorted(os.sched_getaffinity(0))
    os.sched_setaffinity(0, {host_cores[-1]})   # single-threaded oracle, one pinned core
    probe = sliced(32)
    t = time.perf_counter()
    step(probe)
    t_unit = max(time.perf_counter() - t, 1e-6)
    units = int(max(1, min(cfg.I // 32, args.ref_seconds / (K + W) / t_unit)))
    arrs = sliced(32 * units)
    for _ in range(W):
        step(arrs)
    t0 = time.perf_counter()
    for _ in range(K):
        step(arrs)
    dt = time.perf_counter() - t0
    m = 32 * units
    step_bytes = 3 * m * cfg.d * 33 // 32 + 2 * cfg.d + 8 + 4 * m + 2 * cfg.d
    value = step_bytes * K / dt / 1e12
    sample = (f"per step: oracle layer on 1 token x 1 routed expert x {m} of {cfg.I} intermediate "
              f"neurons of the {cfg.name} layer ({step_bytes} algorithmic bytes)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": dt / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{cfg.name} B={B} routing={args.routing}", "E": cfg.E, "k": cfg.k,
                       "d": cfg.d, "I": cfg.I, "B": B},
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": 1, "kind": "oracle", "sample": sample,
                             "host_cores": len(host_cores), "host_cpu_count": os.cpu_count()},
            "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """A short run of one path for a profiler (ncu) to capture: the decode
    layer (gate/up + down), the same with MXFP4 weights (the two passes), or
    the grouped layer; W + K calls on batches of the chosen workload."""
    import torch
    import __graft_entry__
    import mixture_experts_decode_gb300 as moe
    from mixture_experts_decode_gb300 import inputs
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    cfg = {"qwen3": inputs.QWEN3, "deepseek": inputs.DEEPSEEK_V3, "tiny": inputs.TINY}[args.config]
    B = args.batch
    W = inputs.layer_weights(cfg, dev, fp4=args.profile == "fp4")
    mx = lambda a, b: moe.MX(W[a], W[b])
    G, U, D = mx("w_gate", "s_gate"), mx("w_up", "s_up"), mx("w_down", "s_down")
    sh = None
    if W.get("shared") is not None:
        s = W["shared"]
        sh = (moe.MX(s[0], s[1]), moe.MX(s[2], s[3]), moe.MX(s[4], s[5]))
    S = 1 if sh else 0
    batches = [tuple(t.to(dev) for t in inputs.layer_batch(cfg, B, routing=args.routing, step=i)) for i in range(4)]
    y = torch.empty((B, cfg.d), dtype=torch.bfloat16, device=dev)
    h = torch.empty((B, cfg.k + S, cfg.I), dtype=torch.bfloat16, device=dev)
    for i in range(args.warmup + args.steps):
        x, ids, w = batches[i % len(batches)]
        if args.profile == "layer":
            moe.layer(x, ids, w, G, U, D, shared=sh, y=y)
        elif args.profile == "fp4":
            moe.gate_up(x, ids, G, U, shared_gate=sh[0] if sh else None, shared_up=sh[1] if sh else None,
                        h=h, fp4=True)
            moe.down(h, ids, w, D, shared_down=sh[2] if sh else None, y=y, fp4=True)
        else:
            moe.layer_grouped(x, ids, w, G, U, D, y=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "workload": f"{cfg.name} B={B} routing={args.routing}",
                      "calls": args.warmup + args.steps, "device_error": moe.device_error(dev)}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the ternary-g128 product on one GB300 (or N replicas).

Headline (one "step"): a decode sweep at M = 1 over a 64-layer synthetic
backbone, each layer's three MLP projections (gate and up 5120 -> 17408,
down 17408 -> 5120), every projection with its own weights (4.55 GB of packed
codes and scales, far above the 129 MB L2, so every step streams from HBM).
The sweep is captured once in a CUDA graph and replayed; value = weight bytes
(codes + scales) streamed per second.

Also reported (separate timed loops, same process): the small-batch / verify
shapes (M in {1,2,4,5,8,16}), the rotation and the rotation-fused product at
K = 4096, N = 12288, and the pp512 prefill over the 64-layer backbone
(gate, up, qkv-like 5120 -> 6144, down) on the tensor cores.

`--impl reference` times the CPU oracle on the same workload and metric.
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); rank 0 prints the one JSON line.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ternary GEMV M=1 weight GB/s (% HBM peak); pp512 GEMM TFLOP/s (% bf16 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "_source": "fallback"}
DECODE_LAYERS = 64
GEMV_SRC = os.path.join(ROOT, "bit_gemv_gemm_gb300", "csrc", "tern_gemv.cu")
GEMM_SRC = os.path.join(ROOT, "bit_gemv_gemm_gb300", "csrc", "tern_gemm.cu")


def weight_bytes(N: int, K: int) -> int:
    return N * K // 4 + N * K // 64


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["_source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def src_hash(path: str) -> str:
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def load_traffic(kernel: str, src: str):
    """Per-launch DRAM bytes of `kernel` from a committed ncu summary, or None if
    the kernel source changed since the counters were taken."""
    d = traffic_entry(kernel, src)
    return d.get("dram_bytes_per_launch") if d else None


def traffic_entry(kernel: str, src: str):
    """The committed ncu summary entry of `kernel` (the captured launch, its DRAM
    bytes and its algorithmic bytes), or None if the source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_sha256_16") != src_hash(src):
        return None
    return d


def traffic_note(kernel: str, src: str) -> dict:
    """What the roofline's `traffic` figure was taken on: the captured launch and
    that launch's own algorithmic bytes (to compare the DRAM bytes against)."""
    d = traffic_entry(kernel, src)
    if not d:
        return {"traffic_launch": None, "traffic_launch_alg_bytes": None}
    return {"traffic_launch": d.get("workload"), "traffic_launch_alg_bytes": d.get("alg_bytes_per_launch")}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.file.seek(0)
        sms, mx, pw, reasons = [], [], [], set()
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(mx), "power_w_max": max(pw),
                "samples": len(sms), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# multi-rank plumbing (replicas; the only collectives time the ranks)
# ---------------------------------------------------------------------------

def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------

def graph_of(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, steps: int, warmup: int) -> float:
    """Average ms per replay, CUDA events on the launching stream."""
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(steps):
        g.replay()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class DecodeSweep:
    """64 layers x (gate, up, down) at M tokens; each projection its own weights."""

    def __init__(self, tern, layers: int, seed: int = 2):
        import torch
        import synth
        self.tern = tern
        self.layers = []
        self.shapes = [("gate", 5120, 17408), ("up", 5120, 17408), ("down", 17408, 5120)]
        for l in range(layers):
            projs = []
            for name, K, N in self.shapes:
                t = synth.device_trits(seed, f"L{l}.{name}.t", (N, K))
                codes = tern.pack(t)
                del t
                s = synth.device_scales(seed, f"L{l}.{name}.s", (N, K // 128))
                projs.append((name, K, N, codes, s))
            self.layers.append(projs)
        torch.cuda.synchronize()

    def weight_bytes(self) -> int:
        return sum(weight_bytes(N, K) for projs in self.layers for (_, K, N, _, _) in projs)

    def buffers(self, M: int, seed: int = 2, pair: bool = True):
        """x, y and one shared workspace for M tokens.  With `pair`, gate and up
        read one activation (as in the model); otherwise every projection has
        its own."""
        import torch
        import synth
        xs, ys = [], []
        for l, projs in enumerate(self.layers):
            for (name, K, N, _, _) in projs:
                if not (pair and name == "up"):
                    xs.append(synth.device_activations(seed, f"L{l}.{name}.x{M}", (M, K)))
                ys.append(torch.empty((M, N), dtype=torch.float32, device="cuda"))
        need = [self.tern.gemv_workspace_bytes(M, N, K) for (_, K, N) in self.shapes]
        need.append(int(self.tern.lib().tern_gemv_pair_workspace_bytes(M, 17408, 17408, 5120)))
        return xs, ys, self.tern.workspace(max(need))

    def run(self, xs, ys, ws, pair: bool = True):
        """One decode step: with `pair`, gate and up in one tern_gemv_pair call
        on their shared activation, then down; otherwise three tern_gemv calls."""
        if pair:
            for l, (g, u, d) in enumerate(self.layers):
                self.tern.gemv_pair(xs[2 * l], g[3], g[4], u[3], u[4], y_a=ys[3 * l], y_b=ys[3 * l + 1], ws=ws)
                self.tern.gemv(xs[2 * l + 1], d[3], d[4], y=ys[3 * l + 2], ws=ws)
            return
        i = 0
        for projs in self.layers:
            for (_, K, N, codes, s) in projs:
                self.tern.gemv(xs[i], codes, s, y=ys[i], ws=ws)
                i += 1

    def launches(self, pair: bool = True) -> int:
        return (2 if pair else 3) * len(self.layers)

    def alg_bytes(self, M: int, pair: bool = True) -> int:
        """Codes, scales, x (read once per call) and y of one step."""
        b = 0
        for projs in self.layers:
            for (name, K, N, _, _) in projs:
                b += weight_bytes(N, K) + 4 * M * N + (0 if (pair and name == "up") else 2 * M * K)
        return b


def bench_decode(tern, sweep: DecodeSweep, steps: int, warmup: int, ws_count: int, dev_index: int,
                 pair: bool = True):
    import torch
    M = 1
    xs, ys, ws = sweep.buffers(M, pair=pair)
    g = graph_of(lambda: sweep.run(xs, ys, ws, pair))
    time_graph(g, 2, warmup)                       # warm
    with ClockSampler(dev_index) as clk:
        barrier(ws_count)
        torch.cuda.synchronize()
        ms = time_graph(g, steps, 0)
        torch.cuda.synchronize()
        barrier(ws_count)
    ms = max_over_ranks(ms, ws_count)
    launches = sweep.launches(pair)                    # one kernel per tern_gemv / tern_gemv_pair call

    # end to end through the same API: H2D of every projection's x, the sweep,
    # D2H of every y; pinned host buffers, copies inside the timed region.
    # Two buffer sets: step i + 1's input copy and step i - 1's output copy run
    # on a copy stream beside step i's sweep, and every step still copies its
    # own inputs in and its own results out.
    xh = [x.cpu().pin_memory() for x in xs]
    xhost = torch.cat([x.flatten() for x in xh]).pin_memory()
    st = torch.cuda.current_stream()
    cp = torch.cuda.Stream()
    sets = []
    for _ in range(2):
        xin = torch.empty(xhost.numel(), dtype=xhost.dtype, device="cuda")
        yout = torch.empty(sum(y.numel() for y in ys), dtype=torch.float32, device="cuda")
        views, off = [], 0
        for x in xs:
            views.append(xin[off:off + x.numel()].view(x.shape))
            off += x.numel()
        yviews, off = [], 0
        for y in ys:
            yviews.append(yout[off:off + y.numel()].view(y.shape))
            off += y.numel()
        g2 = graph_of(lambda v=views, yv=yviews: sweep.run(v, yv, ws, pair))
        yhost = torch.empty(yout.numel(), dtype=torch.float32).pin_memory()
        sets.append({"xin": xin, "yout": yout, "g": g2, "yhost": yhost,
                     "h2d": torch.cuda.Event(), "comp": torch.cuda.Event()})

    def e2e_run(n):
        """n pipelined steps; returns ms from the first input copy to the last output copy."""
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cp.wait_stream(st)
        with torch.cuda.stream(cp):
            a.record(cp)
            sets[0]["xin"].copy_(xhost, non_blocking=True)
            sets[0]["h2d"].record(cp)
        for i in range(n):
            cur, nxt = sets[i % 2], sets[(i + 1) % 2]
            if i + 1 < n:
                with torch.cuda.stream(cp):
                    if i >= 1:
                        cp.wait_event(nxt["comp"])       # step i - 1's sweep has read its x
                    nxt["xin"].copy_(xhost, non_blocking=True)
                    nxt["h2d"].record(cp)
            st.wait_event(cur["h2d"])
            cur["g"].replay()
            cur["comp"].record(st)
            with torch.cuda.stream(cp):
                cp.wait_event(cur["comp"])
                cur["yhost"].copy_(cur["yout"], non_blocking=True)
        with torch.cuda.stream(cp):
            b.record(cp)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    e2e_run(3)
    e_steps = max(10, steps // 4)
    barrier(ws_count)
    e2e_ms = max_over_ranks(e2e_run(e_steps) / e_steps, ws_count)

    # the same, one step after another on one stream (no overlap), for comparison
    s0 = sets[0]

    def serial_step():
        s0["xin"].copy_(xhost, non_blocking=True)
        s0["g"].replay()
        s0["yhost"].copy_(s0["yout"], non_blocking=True)

    for _ in range(3):
        serial_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_count)
    a.record(st)
    for _ in range(e_steps):
        serial_step()
    b.record(st)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(a.elapsed_time(b) / e_steps, ws_count)
    yhost = s0["yhost"]
    del xh
    return {
        "ms": ms, "clocks": clk.summary(), "launches_per_step": launches,
        "weight_bytes": sweep.weight_bytes(), "alg_bytes": sweep.alg_bytes(M, pair),
        "e2e_ms": e2e_ms, "e2e_serial_ms": serial_ms, "h2d": xhost.numel() * 2, "d2h": yhost.numel() * 4,
    }


def bench_verify(tern, sweep: DecodeSweep, qkv, steps: int, warmup: int):
    """M in {1,2,4,5,8,16} at K=5120, N=17408 (gate weights of all layers) and
    N=6144 (qkv-like weights of all layers)."""
    import torch
    import synth
    out = []
    layers = len(sweep.layers)
    gate = [(p[0][3], p[0][4]) for p in sweep.layers]
    for N, mats in ((17408, gate), (6144, qkv)):
        for M in synth.VERIFY_M:
            K = 5120
            xs = [synth.device_activations(3, f"V{l}.x{M}.{N}", (M, K)) for l in range(layers)]
            ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(layers)]
            ws = tern.workspace(tern.gemv_workspace_bytes(M, N, K))

            def run():
                for l in range(layers):
                    tern.gemv(xs[l], mats[l][0], mats[l][1], y=ys[l], ws=ws)

            g = graph_of(run)
            ms = time_graph(g, max(3, steps // 4), warmup)
            per = ms / layers * 1e-3
            wb = weight_bytes(N, K)
            out.append({"M": M, "K": K, "N": N, "us": per * 1e6, "weight_GBps": wb / per / 1e9,
                        "TFLOPs": 2.0 * M * N * K / per / 1e12})
    return out


def bench_fused_gate_up(tern, sweep: DecodeSweep, steps: int, warmup: int, hbm: float):
    """The decode sweep with each layer's gate and up weights stored as one
    5120 -> 34816 matrix (one call for both, as an engine that keeps a fused
    gate_up projection would run it) and the same down calls: how much of the
    per-call fixed cost two matrices in one launch recover."""
    import torch
    import synth
    layers = len(sweep.layers)
    gu = []
    for l in range(layers):
        t = synth.device_trits(9, f"GU{l}.t", (2 * 17408, 5120))
        gu.append((tern.pack(t), synth.device_scales(9, f"GU{l}.s", (2 * 17408, 40))))
        del t
    x5 = [synth.device_activations(9, f"GU{l}.x", (1, 5120)) for l in range(layers)]
    x17 = [synth.device_activations(9, f"GD{l}.x", (1, 17408)) for l in range(layers)]
    ygu = torch.empty((1, 2 * 17408), dtype=torch.float32, device="cuda")
    yd = torch.empty((1, 5120), dtype=torch.float32, device="cuda")
    ws = tern.workspace(max(tern.gemv_workspace_bytes(1, 2 * 17408, 5120), tern.gemv_workspace_bytes(1, 5120, 17408)))

    def run():
        for l in range(layers):
            tern.gemv(x5[l], gu[l][0], gu[l][1], y=ygu, ws=ws)
            d = sweep.layers[l][2]
            tern.gemv(x17[l], d[3], d[4], y=yd, ws=ws)

    g = graph_of(run)
    ms = time_graph(g, max(3, steps // 4), warmup)
    wb = layers * (weight_bytes(2 * 17408, 5120) + weight_bytes(5120, 17408))
    gbps = wb / (ms * 1e-3) / 1e9
    return {"layers": layers, "launches": 2 * layers, "ms_per_step": ms, "weight_GBps": gbps, "hbm_frac": gbps / hbm}


def bench_verify_step(tern, sweep: DecodeSweep, qkv, steps: int, warmup: int):
    """One speculative-verify step as a CUDA graph: k + 1 = 5 tokens through
    every layer's qkv (5120 -> 6144), gate and up (5120 -> 17408, one pair call
    on their shared activation) and down (17408 -> 5120) products, 64 layers,
    192 launches.  The drafter and the work between the products (attention,
    activations) are not part of it: each call reads a fixed activation."""
    import torch
    import synth
    M = synth.VERIFY_STEP_M
    layers = len(sweep.layers)
    x5 = synth.device_activations(6, "VS.x5120", (M, 5120))
    x17 = synth.device_activations(6, "VS.x17408", (M, 17408))
    ys = {N: torch.empty((M, N), dtype=torch.float32, device="cuda") for N in (6144, 17408, 5120)}
    ws = tern.workspace(max(tern.gemv_workspace_bytes(M, N, K) for (K, N) in ((5120, 6144), (5120, 17408),
                                                                              (17408, 5120))))

    yu = torch.empty((M, 17408), dtype=torch.float32, device="cuda")
    ws = tern.workspace(max(ws.numel(), int(tern.lib().tern_gemv_pair_workspace_bytes(M, 17408, 17408, 5120))))

    def run():
        for l in range(layers):
            tern.gemv(x5, qkv[l][0], qkv[l][1], y=ys[6144], ws=ws)
            g_, u_, d_ = sweep.layers[l]
            tern.gemv_pair(x5, g_[3], g_[4], u_[3], u_[4], y_a=ys[17408], y_b=yu, ws=ws)
            tern.gemv(x17, d_[3], d_[4], y=ys[5120], ws=ws)

    g = graph_of(run)
    ms = time_graph(g, max(3, steps // 10), warmup)
    wb = layers * (weight_bytes(6144, 5120) + 2 * weight_bytes(17408, 5120) + weight_bytes(5120, 17408))
    return {"M": M, "layers": layers, "launches": 3 * layers, "us_per_step": ms * 1e3,
            "weight_GBps": wb / (ms * 1e-3) / 1e9, "tokens_per_s": M / (ms * 1e-3)}


def bench_f3(tern, steps: int, warmup: int, hbm: float, copies: int = 16):
    """Native base-3 packing (five trits per byte): the decode product (M = 1,
    and M = 5) per decode shape, `copies` distinct matrices (more bytes than
    L2) back to back in one graph, beside the 2-bit product on the same shape."""
    import torch
    import synth
    out = []
    for (K, N) in synth.DECODE_SHAPES:
        mats = []
        for c in range(copies):
            t = synth.device_trits(9, f"F{c}.{K}.t", (N, K))
            mats.append((tern.f3_pack(t), synth.device_scales(9, f"F{c}.{K}.s", (N, K // 128))))
            del t
        wb = N * 26 * (K // 128) + N * (K // 128) * 2
        for M in (1, 5):
            xs = [synth.device_activations(9, f"F{c}.{K}.x{M}", (M, K)) for c in range(copies)]
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")

            def run(xs=xs, y=y):
                for c in range(copies):
                    tern.f3_gemv(xs[c], mats[c][0], mats[c][1], y=y)

            g = graph_of(run)
            ms = time_graph(g, max(3, steps // 4), warmup)
            per = ms / copies * 1e-3
            out.append({"M": M, "K": K, "N": N, "us": per * 1e6, "weight_bytes": wb,
                        "weight_GBps": wb / per / 1e9, "hbm_frac": wb / per / 1e9 / hbm,
                        "bits_per_weight": 8.0 * wb / (N * K)})
        del mats
    return out


def bench_binary(tern, steps: int, warmup: int, hbm: float, copies: int = 16):
    """The 1-bit sibling format.  Decode (M = 1): per decode shape, `copies`
    distinct matrices (more bytes than L2) called back to back in one graph.
    Prefill (M = 512): per layer shape, 4 distinct matrices in one graph."""
    import torch
    import synth
    out = {"decode": [], "pp512": []}
    for (K, N) in synth.DECODE_SHAPES:
        mats = []
        for c in range(copies):
            t = synth.device_binary(7, f"B{c}.{K}.t", (N, K))
            mats.append((tern.bin_pack(t), synth.device_scales(7, f"B{c}.{K}.s", (N, K // 128))))
            del t
        xs = [synth.device_activations(7, f"B{c}.{K}.x", (1, K)) for c in range(copies)]
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        ws = tern.workspace(tern.gemv_workspace_bytes(1, N, K))

        def run():
            for c in range(copies):
                tern.bin_gemv(xs[c], mats[c][0], mats[c][1], y=y, ws=ws)

        g = graph_of(run)
        ms = time_graph(g, max(3, steps // 4), warmup)
        per = ms / copies * 1e-3
        wb = N * K // 8 + N * K // 64
        out["decode"].append({"M": 1, "K": K, "N": N, "us": per * 1e6, "weight_bytes": wb,
                              "weight_GBps": wb / per / 1e9, "hbm_frac": wb / per / 1e9 / hbm})
        del mats
    M = synth.PREFILL_M
    for (name, K, N) in synth.PREFILL_LAYER:
        mats = []
        for c in range(4):
            t = synth.device_binary(8, f"BP{c}.{name}.t", (N, K))
            mats.append((tern.bin_pack(t), synth.device_scales(8, f"BP{c}.{name}.s", (N, K // 128))))
            del t
        x = synth.device_activations(8, f"BP.{name}.x", (M, K))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws = tern.workspace(tern.gemm_workspace_bytes(M, N, K))

        def run(mats=mats, x=x, y=y, ws=ws):
            for c in range(4):
                tern.bin_gemm(x, mats[c][0], mats[c][1], y=y, ws=ws)

        g = graph_of(run)
        ms = time_graph(g, max(2, steps // 20), max(1, warmup // 2))
        per = ms / 4 * 1e-3
        out["pp512"].append({"name": name, "K": K, "N": N, "us": per * 1e6, "TFLOPs": 2.0 * M * N * K / per / 1e12})
        del mats
    return out


def bench_affine(tern, steps: int, warmup: int, hbm: float, copies: int = 16):
    """An affine pack (w = s q + b per group of 128, 2.25 bits per weight with
    the biases).  Decode (M = 1): per decode shape, `copies` distinct matrices
    (more bytes than L2) called back to back in one graph.  Prefill (M = 512):
    per layer shape, 4 distinct matrices in one graph."""
    import torch
    import synth
    out = {"decode": [], "pp512": []}

    def mat(seed, key, N, K):
        s = synth.device_scales(seed, f"{key}.s", (N, K // 128))
        return (synth.device_code_words(seed, f"{key}.c", (N, K // 16)), s, synth.device_biases(seed, f"{key}.b", s))

    for (K, N) in synth.DECODE_SHAPES:
        mats = [mat(9, f"A{c}.{K}", N, K) for c in range(copies)]
        xs = [synth.device_activations(9, f"A{c}.{K}.x", (1, K)) for c in range(copies)]
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        ws = tern.workspace(tern.gemv_workspace_bytes(1, N, K))

        def run():
            for c in range(copies):
                tern.affine_gemv(xs[c], *mats[c], y=y, ws=ws)

        g = graph_of(run)
        ms = time_graph(g, max(3, steps // 4), warmup)
        per = ms / copies * 1e-3
        wb = N * K // 4 + 2 * (N * K // 64)
        out["decode"].append({"M": 1, "K": K, "N": N, "us": per * 1e6, "weight_bytes": wb,
                              "weight_GBps": wb / per / 1e9, "hbm_frac": wb / per / 1e9 / hbm})
        del mats
    M = synth.PREFILL_M
    for (name, K, N) in synth.PREFILL_LAYER:
        mats = [mat(10, f"AP{c}.{name}", N, K) for c in range(4)]
        x = synth.device_activations(10, f"AP.{name}.x", (M, K))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws = tern.workspace(tern.gemm_workspace_bytes(M, N, K))

        def run(mats=mats, x=x, y=y, ws=ws):
            for c in range(4):
                tern.affine_gemm(x, *mats[c], y=y, ws=ws)

        g = graph_of(run)
        ms = time_graph(g, max(2, steps // 20), max(1, warmup // 2))
        per = ms / 4 * 1e-3
        out["pp512"].append({"name": name, "K": K, "N": N, "us": per * 1e6, "TFLOPs": 2.0 * M * N * K / per / 1e12})
        del mats
    return out


def bench_rotated(tern, steps: int, warmup: int, peaks: dict, copies: int = 40):
    import torch
    import synth
    K, N = synth.ROTATED["K"], synth.ROTATED["N"]
    mats = []
    for c in range(copies):
        t = synth.device_trits(4, f"R{c}.t", (N, K))
        mats.append((tern.pack(t), synth.device_scales(4, f"R{c}.s", (N, K // 128))))
        del t
    signs = synth.device_signs(4, "R.signs", K)
    out = []
    for M in synth.ROTATED["M"]:
        xs = [synth.device_activations(4, f"R{c}.x{M}", (M, K)) for c in range(copies)]
        xr = [torch.empty_like(x) for x in xs]
        ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(copies)]
        ws = tern.workspace(tern.gemv_workspace_bytes(M, N, K))

        def fused():
            for c in range(copies):
                tern.fwht_gemm(xs[c], signs, mats[c][0], mats[c][1], y=ys[c], ws=ws)

        def separate():
            for c in range(copies):
                tern.fwht(xs[c], signs, y=xr[c])
                tern.gemv(xr[c], mats[c][0], mats[c][1], y=ys[c], ws=ws)

        def rot_only():
            for c in range(copies):
                tern.fwht(xs[c], signs, y=xr[c])

        def product_only():
            for c in range(copies):
                tern.gemv(xr[c], mats[c][0], mats[c][1], y=ys[c], ws=ws)

        res = {"M": M, "K": K, "N": N}
        for name, fn in (("fused", fused), ("separate", separate), ("fwht_only", rot_only),
                         ("product_only", product_only)):
            g = graph_of(fn)
            ms = time_graph(g, max(3, steps // 4), warmup)
            res[f"{name}_us"] = ms / copies * 1e3
        wb = weight_bytes(N, K)
        res["fused_weight_GBps"] = wb / (res["fused_us"] * 1e-6) / 1e9
        res["fwht_GBps"] = 4.0 * M * K / (res["fwht_only_us"] * 1e-6) / 1e9
        res["fused_minus_product_us"] = res["fused_us"] - res["product_only_us"]
        res["fused_hbm_frac"] = res["fused_weight_GBps"] / peaks["hbm_gbs"]
        out.append(res)
    del mats
    # the rotation alone where it is bandwidth-bound: many tokens, inputs and
    # outputs larger than L2 (4 copies of 4096 x 4096 bf16 in and out)
    Mb, nb = 4096, 4
    xb = [synth.device_activations(5, f"RB{c}", (Mb, K)) for c in range(nb)]
    yb = [torch.empty_like(x) for x in xb]

    def big():
        for c in range(nb):
            tern.fwht(xb[c], signs, y=yb[c])

    g = graph_of(big)
    ms = time_graph(g, max(3, steps // 4), warmup)
    us = ms / nb * 1e3
    gbps = 4.0 * Mb * K / (us * 1e-6) / 1e9
    bw = {"M": Mb, "K": K, "us": us, "GBps": gbps,
          "roofline": {"bound": "hbm", "kernel": "fwht_kernel", "achieved": gbps, "peak": peaks["hbm_gbs"],
                       "unit": "GB/s", "frac": gbps / peaks["hbm_gbs"], "peak_source": f"{peaks['_source']} hbm_gbs",
                       "bytes": "bf16 in + bf16 out, 4 K bytes per token"}}
    del xb, yb
    return {"small_batch": out, "bandwidth": bw}


def bench_prefill(tern, sweep: DecodeSweep, qkv, steps: int, warmup: int, peaks: dict, dev_index: int):
    """pp512: 64 layers x (gate, up, qkv, down) at M=512, bf16 in, bf16 out."""
    import torch
    import synth
    M = synth.PREFILL_M
    layers = len(sweep.layers)
    x5 = synth.device_activations(5, "P.x5120", (M, 5120))
    x17 = synth.device_activations(5, "P.x17408", (M, 17408))
    outs = {N: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for N in (17408, 6144, 5120)}
    ws = tern.workspace(max(tern.gemm_workspace_bytes(M, N, K) for (_, K, N) in synth.PREFILL_LAYER))
    try:
        tern.gemm(x5, sweep.layers[0][0][3], sweep.layers[0][0][4], y=outs[17408], ws=ws)
        torch.cuda.synchronize()
    except tern.TernError as e:
        return {"unavailable": f"tern_gemm: {e}"}
    mats = {"gate": [(p[0][3], p[0][4]) for p in sweep.layers],
            "up": [(p[1][3], p[1][4]) for p in sweep.layers],
            "qkv": qkv,
            "down": [(p[2][3], p[2][4]) for p in sweep.layers]}
    per_gemm = {}
    for (name, K, N) in synth.PREFILL_LAYER:
        x = x5 if K == 5120 else x17

        def run(name=name, x=x, N=N):
            for l in range(layers):
                tern.gemm(x, mats[name][l][0], mats[name][l][1], y=outs[N], ws=ws)

        g = graph_of(run)
        ms = time_graph(g, max(2, steps // 20), max(1, warmup // 2))
        per = ms / layers * 1e-3
        per_gemm[name] = {"K": K, "N": N, "us": per * 1e6, "TFLOPs": 2.0 * M * N * K / per / 1e12}

    def full():
        for l in range(layers):
            for (name, K, N) in synth.PREFILL_LAYER:
                tern.gemm(x5 if K == 5120 else x17, mats[name][l][0], mats[name][l][1], y=outs[N], ws=ws)

    g = graph_of(full)
    with ClockSampler(dev_index) as clk:
        ms = time_graph(g, max(2, steps // 20), max(1, warmup // 2))
    flops = layers * sum(2.0 * M * N * K for (_, K, N) in synth.PREFILL_LAYER)
    tf = flops / (ms * 1e-3) / 1e12
    # a pass of ~16 ms timed over a few replays is a burst, not a seconds-long
    # loop under the power cap: the burst peak is the denominator (the
    # sustained one is kept beside it)
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak)
    for v in per_gemm.values():
        v["frac"] = v["TFLOPs"] / peak
    dom = max(per_gemm.items(), key=lambda kv: kv[1]["us"])
    return {
        "M": M, "layers": layers, "ms_per_pass": ms, "TFLOPs": tf, "tokens_per_s": M / (ms * 1e-3),
        "per_gemm": per_gemm, "clocks": clk.summary(),
        "roofline": {"bound": "tensor", "kernel": "tern_gemm (tcgen05)", "achieved": tf, "peak": peak,
                     "unit": "TFLOP/s", "frac": tf / peak, "frac_of_sustained": tf / peak_sus,
                     "peak_source": f"{peaks['_source']} bf16_tflops (burst; pass of {ms:.1f} ms)",
                     "traffic": load_traffic("gemm_kernel", GEMM_SRC), **traffic_note("gemm_kernel", GEMM_SRC)},
        "dominant": dom[0],
    }


def cpu_baseline(budget_s: float = 12.0) -> dict:
    """The oracle, as it stands, on a bounded sample of the decode workload:
    repeated full M=1 products of one gate-shaped (5120 -> 17408) matrix on all
    host cores, then row slices of it on one core."""
    import oracle
    import synth
    oracle.build()
    K, N = 5120, 17408
    p = synth.problem(2, 1, N, K, tag="cpu")
    codes, _ = oracle.pack(p.t)
    oracle.matmul(p.x[:, :], codes[:64], p.s[:64])              # warm the library
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.matmul(p.x, codes, p.s)
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s or calls >= 200:
            break
    gbps = calls * weight_bytes(N, K) / el / 1e9
    cores = oracle.max_threads()
    rows, calls1, t0 = 2048, 0, time.perf_counter()
    while True:
        oracle.matmul(p.x, codes[:rows], p.s[:rows], nthreads=1)
        calls1 += 1
        el1 = time.perf_counter() - t0
        if el1 >= budget_s / 3 or calls1 >= 200:
            break
    gbps1 = calls1 * weight_bytes(rows, K) / el1 / 1e9
    oracle.matmul(p.x, codes[:64], p.s[:64], nthreads=cores)    # the thread count persists: restore it
    return {"value": gbps, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{calls} full M=1 products of one 5120->17408 matrix (23.7 MB packed) in {el:.1f} s "
                      f"with the C oracle (fp64, OpenMP over outputs)", "cpu": cpu_model(),
            "single_thread": {"value": gbps1, "unit": "GB/s", "cores": 1,
                              "sample": f"{calls1} products of {rows} rows of that matrix in {el1:.1f} s, one thread"}}


def cpu_model() -> str:
    """The host CPU's model name, for the record (x86: /proc/cpuinfo; Arm: lscpu)."""
    import platform
    try:
        for line in open("/proc/cpuinfo"):
            k, _, v = line.partition(":")
            if k.strip() == "model name" and v.strip():
                return v.strip()
    except OSError:
        pass
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine() or "unknown"


def cpu_baseline_pp512(budget_s: float = 5.0) -> dict:
    """The oracle, as it stands, on a bounded sample of the pp512 workload: all
    512 tokens against a growing number of rows of one gate-shaped (5120 ->
    17408) matrix, on all host cores and on one; the rates are extrapolated to
    the whole 64-layer pass."""
    import oracle
    import synth
    oracle.build()
    M, K, rows = synth.PREFILL_M, 5120, 64
    p = synth.problem(5, M, rows, K, tag="cpu_pp")
    codes, _ = oracle.pack(p.t)
    oracle.matmul(p.x[:4], codes[:4], p.s[:4])                      # warm the library
    total = sum(2.0 * M * N * K for (_, K, N) in synth.PREFILL_LAYER) * synth.PREFILL_LAYERS

    def rate(nthreads, r, budget):
        calls, t0 = 0, time.perf_counter()
        while True:
            oracle.matmul(p.x, codes[:r], p.s[:r], nthreads=nthreads)
            calls += 1
            el = time.perf_counter() - t0
            if el >= budget or calls >= 50:
                return calls, el, calls * 2.0 * M * r * K / el / 1e12

    cores = oracle.max_threads()
    calls, el, tflops = rate(cores, rows, budget_s)
    calls1, el1, tflops1 = rate(1, 8, budget_s / 3)
    oracle.matmul(p.x[:4], codes[:4], p.s[:4], nthreads=cores)      # the thread count persists: restore it
    return {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{calls} products of 512 tokens x {rows} rows x K={K} (a slice of the gate matrix) in "
                      f"{el:.1f} s with the C oracle (fp64, OpenMP over outputs)",
            "extrapolated_pass_s": total / (tflops * 1e12),
            "single_thread": {"value": tflops1, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"{calls1} products of 512 tokens x 8 rows x K={K} in {el1:.1f} s, one thread",
                              "extrapolated_pass_s": total / (tflops1 * 1e12)}}


def safe_cpu_baseline_pp512(budget_s: float) -> dict:
    """cpu_baseline_pp512, or the reason it could not run (it is an extra row:
    it never takes the benchmark line down)."""
    try:
        return cpu_baseline_pp512(budget_s)
    except Exception as e:                     # noqa: BLE001 - reported, not hidden
        return {"unavailable": f"{type(e).__name__}: {e}"}


def run_reference(args) -> None:
    """The reference arm: the CPU oracle on the decode workload's metric."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    import synth
    oracle.build()
    K, N = 5120, 17408
    p = synth.problem(2, 1, N, K, tag="cpu")
    codes, _ = oracle.pack(p.t)
    # size each step's sample so the whole run stays within about a minute
    t0 = time.perf_counter()
    oracle.matmul(p.x, codes[:1024], p.s[:1024])
    rate = 1024 / max(time.perf_counter() - t0, 1e-6)                 # rows per second
    total_steps = args.steps + args.warmup
    rows = int(max(64, min(N, rate * 60.0 / max(total_steps, 1))))
    for _ in range(args.warmup):
        oracle.matmul(p.x, codes[:rows], p.s[:rows])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(p.x, codes[:rows], p.s[:rows])
    el = time.perf_counter() - t0
    gbps = args.steps * weight_bytes(rows, K) / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbps, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode GEMV M=1, 5120->17408 rows sample (CPU oracle)", "M": 1, "K": K,
                   "N_sampled": rows},
        "cpu_baseline": {"value": gbps, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"{rows} rows x K={K} per step, {args.steps} steps", "cpu": cpu_model()},
        "e2e": {"value": gbps, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "rows": {"pp512": {"cpu_baseline": safe_cpu_baseline_pp512(3.0)}},
    }
    print(json.dumps(line), flush=True)


# Single cases for profiler captures: each runs its launch 3 times unprofiled
# (warm-up) and then 2 more, with synthetic inputs of the bench's shapes.
PROFILE_CASES = ("fwht_bw", "fused_m1", "fused_m16", "separate_m16", "gemm_down", "gemm_qkv", "gemv_m1", "gemv_m8",
                 "gemv_m16", "f3_m1")


def run_profile_case(name: str) -> None:
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import bit_gemv_gemm_gb300 as tern
    import synth
    K4, N4 = synth.ROTATED["K"], synth.ROTATED["N"]
    if name == "fwht_bw":
        # the rotation where it is bandwidth-bound: 4096 tokens x K = 4096
        x = synth.device_activations(5, "PB.x", (4096, K4))
        sg = synth.device_signs(5, "PB.s", K4)
        y = torch.empty_like(x)
        fn = lambda: tern.fwht(x, sg, y=y)
    elif name in ("fused_m1", "fused_m16", "separate_m16"):
        M = 1 if name == "fused_m1" else 16
        c = tern.pack(synth.device_trits(6, "PF.t", (N4, K4)))
        sc = synth.device_scales(6, "PF.sc", (N4, K4 // 128))
        x = synth.device_activations(6, f"PF.x{M}", (M, K4))
        sg = synth.device_signs(6, "PF.s", K4)
        y = torch.empty((M, N4), dtype=torch.float32, device="cuda")
        ws = tern.workspace(tern.gemv_workspace_bytes(M, N4, K4))
        if name == "separate_m16":
            xr = torch.empty_like(x)
            fn = lambda: (tern.fwht(x, sg, y=xr), tern.gemv(xr, c, sc, y=y, ws=ws))
        else:
            fn = lambda: tern.fwht_gemm(x, sg, c, sc, y=y, ws=ws)
    elif name in ("gemm_down", "gemm_qkv"):
        K, N = (17408, 5120) if name == "gemm_down" else (5120, 6144)
        M = 512
        c = tern.pack(synth.device_trits(7, "PG.t", (N, K)))
        sc = synth.device_scales(7, "PG.sc", (N, K // 128))
        x = synth.device_activations(7, "PG.x", (M, K))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ws = tern.workspace(tern.gemm_workspace_bytes(M, N, K))
        fn = lambda: tern.gemm(x, c, sc, y=y, ws=ws)
    elif name == "f3_m1":
        K, N = 5120, 17408
        c = tern.f3_pack(synth.device_trits(8, "P3.t", (N, K)))
        sc = synth.device_scales(8, "P3.sc", (N, K // 128))
        x = synth.device_activations(8, "P3.x", (1, K))
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        fn = lambda: tern.f3_gemv(x, c, sc, y=y)
    else:
        M = int(name.split("_m")[1])
        K, N = 5120, 17408
        c = tern.pack(synth.device_trits(8, "PV.t", (N, K)))
        sc = synth.device_scales(8, "PV.sc", (N, K // 128))
        x = synth.device_activations(8, f"PV.x{M}", (M, K))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        ws = tern.workspace(tern.gemv_workspace_bytes(M, N, K))
        fn = lambda: tern.gemv(x, c, sc, y=y, ws=ws)
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    err = tern.device_error()
    if err:
        raise SystemExit(f"device error {err:#x}")
    print(f"profile case {name}: 5 launches done", flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=DECODE_LAYERS)
    ap.add_argument("--skip", default="", help="comma list of parts to skip: fused,verify,rotated,binary,f3,affine,prefill,cpu")
    ap.add_argument("--profile", default="", choices=["", *PROFILE_CASES],
                    help="run one hot-path case a few times for a profiler capture and exit (no JSON line)")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    ws_count, rank, local = dist_setup()
    import __graft_entry__
    __graft_entry__.build()
    import bit_gemv_gemm_gb300 as tern
    import synth
    peaks = load_peaks()
    skip = set(filter(None, args.skip.split(",")))
    dev_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local

    sweep = DecodeSweep(tern, args.layers)
    qkv = []
    for l in range(args.layers):
        t = synth.device_trits(2, f"L{l}.qkv.t", (6144, 5120))
        qkv.append((tern.pack(t), synth.device_scales(2, f"L{l}.qkv.s", (6144, 40))))
        del t
    torch.cuda.synchronize()

    dec = bench_decode(tern, sweep, args.steps, args.warmup, ws_count, dev_index)
    value = ws_count * dec["weight_bytes"] / (dec["ms"] * 1e-3) / 1e9
    achieved = dec["alg_bytes"] / (dec["ms"] * 1e-3) / 1e9
    hbm = peaks["hbm_gbs"]
    rows = {}
    if "fused" not in skip:
        sep = bench_decode(tern, sweep, args.steps, args.warmup, 1, dev_index, pair=False)
        sgb = sep["weight_bytes"] / (sep["ms"] * 1e-3) / 1e9
        rows["separate_calls"] = {"launches": sep["launches_per_step"], "ms_per_step": sep["ms"],
                                  "weight_GBps": sgb, "hbm_frac": sgb / hbm}
        rows["fused_gate_up"] = bench_fused_gate_up(tern, sweep, args.steps, args.warmup, hbm)
    if "verify" not in skip:
        rows["verify"] = bench_verify(tern, sweep, qkv, args.steps, args.warmup)
        rows["verify_step"] = bench_verify_step(tern, sweep, qkv, args.steps, args.warmup)
    if "rotated" not in skip:
        rows["rotated"] = bench_rotated(tern, args.steps, args.warmup, peaks)
    if "binary" not in skip:
        rows["binary"] = bench_binary(tern, args.steps, args.warmup, hbm)
    if "f3" not in skip:
        rows["f3"] = bench_f3(tern, args.steps, args.warmup, hbm)
    if "affine" not in skip:
        rows["affine"] = bench_affine(tern, args.steps, args.warmup, hbm)
    if "prefill" not in skip:
        rows["pp512"] = bench_prefill(tern, sweep, qkv, args.steps, args.warmup, peaks, dev_index)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": ws_count,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dec["ms"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"decode GEMV M=1 sweep, {args.layers} layers x (gate 5120->17408 and "
                               f"up 5120->17408 reading one activation in one tern_gemv_pair call, "
                               f"down 17408->5120), distinct weights",
                   "M": 1, "layers": args.layers, "weight_bytes_per_step": dec["weight_bytes"],
                   "l2": "inputs larger than L2 (4.55 GB of weights per step vs 129 MB L2)",
                   "parallelism": f"replicas x{ws_count}", "cuda_graph": True},
        "hbm_frac": value / ws_count / hbm,
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel (one launch per tern_gemv_pair or tern_gemv call)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": f"{peaks['_source']} hbm_gbs",
                     "traffic": load_traffic("gemv_kernel", GEMV_SRC), **traffic_note("gemv_kernel", GEMV_SRC)},
        "clocks": dec["clocks"],
        "e2e": {"value": ws_count * dec["weight_bytes"] / (dec["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": dec["h2d"], "d2h_bytes_per_step": dec["d2h"],
                "copies": "copy stream beside the sweep, two buffer sets",
                "serial_value": ws_count * dec["weight_bytes"] / (dec["e2e_serial_ms"] * 1e-3) / 1e9},
        "gpu_launches": dec["launches_per_step"] * args.steps,
        "rows": rows,
    }
    if rank == 0 and "cpu" not in skip:
        line["cpu_baseline"] = cpu_baseline()
        if isinstance(rows.get("pp512"), dict) and "TFLOPs" in rows["pp512"]:
            rows["pp512"]["cpu_baseline"] = safe_cpu_baseline_pp512(5.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_count > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

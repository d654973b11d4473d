#!/usr/bin/env python3
"""Benchmark of the gated delta-rule library on GB300.

Headline: the batched GDN decode step (B=64, Hk=16, Hv=32, Dk=Dv=128, fp32 state of 134 MB), in
state GB/s (state bytes read + written per step / time per step).  The same JSON line also carries
the other operations measured in the same run: the Comba decode step (B=256, H=32, K=V=128), the
varlen chunked prefill (T=15360 over lengths 4096+2048+1024+8192, Hk=16, Hv=32, K=V=128, C=64) in
tokens/s, and the fused decode window (N=32, h_k=16, h_v=48, ntok=8) in verify and commit mode.

Timing: W untimed warm-up steps, then exactly K timed steps bracketed by a barrier and a device
synchronise, CUDA events on the stream the kernels run on, max over ranks.  Every step reads state
last touched more than an L2's worth of traffic earlier (two interleaved decode chains, rotated
window states, inputs larger than L2).  Under torchrun each rank runs its own replica of the
workload (weak scaling; the operations have no exchange step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gdn,reference}]

--impl reference times the CPU oracle (the plain C implementation the tests trust) on the same
workload, a bounded sample of it per step, on this host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gdn_inputs as gi  # noqa: E402

METRIC = "decode state GB/s (% HBM peak); prefill tokens/s (% roofline), 1xGB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 2 ** 20


# ------------------------------------------------------------------------------------------------
# Algorithmic work of each operation (bytes that must cross HBM at least once; flops of the
# contractions).  The Comba formula is the one of the KBench spec (flops_src).
# ------------------------------------------------------------------------------------------------
def decode_state_bytes(B, Hk, Hv, Dk, Dv):
    return 2 * B * Hv * Dv * Dk * 4


def decode_bytes(B, Hk, Hv, Dk, Dv):
    tokens = 2 * B * Hk * Dk * 2 + B * Hv * Dv * 2 + B * Hv * 4 + B * Hv * 2
    return decode_state_bytes(B, Hk, Hv, Dk, Dv) + tokens + B * Hv * Dv * 2  # + y (bf16)


def comba_bytes(B, H, K, V):
    return 2 * B * H * K * V * 4 + B * H * (6 * K + 4 * V + 6)


def comba_forward_bytes(B, T, H, K, V):
    """State read and written once; per token q, k, p, v, beta (bf16), g (f32) read and o (bf16)
    written."""
    return 2 * B * H * K * V * 4 + B * T * H * (3 * K * 2 + V * 2 + 2 + 4 + V * 2)


def prefill_bytes(seqlens, Hk, Hv, K, V):
    T, n = sum(seqlens), len(seqlens)
    return (2 * T * Hk * K * 2 + T * Hv * V * 2 + 2 * T * Hv * 2 + T * Hv * V * 2
            + 2 * n * Hv * V * K * 4 + n * 8 + (n + 1) * 8 + 2 * Hv * 4)


def comba_prefill_bytes(seqlens, H, K, V):
    """q, k, p, v, beta (bf16) and g (f32) read once, out (bf16) written once, the sequences'
    pool slots gathered and scattered."""
    T, n = sum(seqlens), len(seqlens)
    return (3 * T * H * K * 2 + T * H * V * 2 + T * H * (2 + 4) + T * H * V * 2
            + 2 * n * H * K * V * 4 + n * 8 + (n + 1) * 8)


def prefill_flops(seqlens, Hv, K, V, C):
    chunks = sum((s + C - 1) // C for s in seqlens)
    T = sum(seqlens)
    return T * Hv * 2 * (3 * C * K + 2 * C * V + 3 * K * V) + chunks * Hv * C ** 3 // 3


def window_bytes(N, h_k, h_v, D, ntok, commit: bool):
    C = (2 * h_k + h_v) * D
    state = N * D * h_v * D * 4
    act = (N * ntok * C + N * C * 3 + 2 * N * ntok * h_v + 2 * N * ntok * h_v * D) * 4
    weights = (C * 4 + 2 * h_v + D) * 4
    return state + act + weights + ((state + N * C * 3 * 4) if commit else 0)


# ------------------------------------------------------------------------------------------------
# Environment helpers
# ------------------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def profiled_traffic(kernel: str, source):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None when the kernel
    source has changed since the counters were taken.  `source` is one file or a tuple of files
    (the kernel and the launch code that picks its shape), hashed concatenated in that order."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        h = hashlib.sha256()
        for src in ((source,) if isinstance(source, str) else source):
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()[:16]
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == kernel and parts[1] == sha:
                    return int(parts[2])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed regions run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        rows = []
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), max=float(f[2]), util=float(f[4]),
                                 reasons=[n for n, v in zip(
                                     ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                      "sw_power_cap"), f[5:9]) if v.lower() == "active"]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if r["util"] > 0] or rows
        reasons = sorted({x for r in loaded for x in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(loaded)}


# ------------------------------------------------------------------------------------------------
# Distributed plumbing (replicas; one process per GPU)
# ------------------------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if _cuda_ok() else "gloo"
            if backend == "nccl":
                import torch
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = torch.device("cuda", self.local_rank) if _cuda_ok() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# ------------------------------------------------------------------------------------------------
# GPU measurements
# ------------------------------------------------------------------------------------------------
E2E_GRAPH = 8  # decode steps per captured graph of the end-to-end loop


def _timed(torch, dist, steps, fn, finish=None):
    """Run fn(i) for i in range(steps) between barriers and synchronises; return seconds (max over
    ranks) measured with CUDA events on the current stream.  finish() (if given) runs before the
    end event, to join work that fn put on other streams into the current one."""
    dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        fn(i)
    if finish is not None:
        finish()
    end.record()
    torch.cuda.synchronize()
    dist.barrier()
    return dist.max(start.elapsed_time(end) / 1e3)


def _timed_calls(torch, dist, steps, fn, restore):
    """Like _timed, but restore(i) runs before call i outside the timed region: each call is
    bracketed by its own CUDA events on the current stream (restore's work is enqueued before the
    start event, so the stream reaches the start event only once it is done), and the sum of the
    calls' times is returned (max over ranks)."""
    dist.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        restore(i)
        evs[i][0].record()
        fn(i)
        evs[i][1].record()
    torch.cuda.synchronize()
    dist.barrier()
    return dist.max(sum(a.elapsed_time(b) for a, b in evs) / 1e3)


def bench_decode(torch, gdn, dist, steps, warmup, seed):
    c = gi.GDN_DECODE_BATCHED
    B, Hk, Hv, Dk, Dv = c["B"], c["Hk"], c["Hv"], c["Dk"], c["Dv"]
    dev = torch.device("cuda")
    g = gi.rng(seed)
    b16, f32 = torch.bfloat16, torch.float32

    def tok():
        t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
        return tuple(torch.from_numpy(t[n]).to(dt).to(dev) for n, dt in
                     (("q", b16), ("k", b16), ("v", b16), ("g", f32), ("beta", b16)))

    # two independent chains (A: s0 <-> s1, B: s2 <-> s3), interleaved, so that every step reads a
    # state last written two steps (> 2 x 134 MB of traffic) earlier
    states = [torch.zeros((B, Hv, Dv, Dk), dtype=f32, device=dev) for _ in range(4)]
    y = torch.empty((B, Hv, Dv), dtype=b16, device=dev)
    for w in range(c["warmup"]):          # 16 warm-up steps of the recurrence, fresh draws
        gdn.gdn_decode_step(states[w % 2], *tok(), state_out=states[1 - w % 2], y=y)
    states[0].copy_(states[c["warmup"] % 2])
    states[2].copy_(states[0])
    t = tok()                             # the measured draw, reused by every timed step

    def step(i):
        chain, parity = (i % 2) * 2, (i // 2) % 2
        src, dst = states[chain + parity], states[chain + 1 - parity]
        gdn.gdn_decode_step(src, *t, state_out=dst, y=y)

    for i in range(warmup):
        step(i)
    secs = _timed(torch, dist, steps, step)

    # end to end through the public API: per step, the token inputs come from pinned host memory
    # (packed in one buffer, one copy) and y goes back to pinned host memory; the state stays
    # resident in HBM (a serving cache).  The two chains are two independent request batches served
    # alternately: a chain's copies run on copy streams and overlap the other chain's kernel, and a
    # chain's next inputs are sent only after its previous result has arrived on the host side.
    parts = [x.contiguous().view(torch.uint8).reshape(-1) for x in t]
    offs, total = [], 0
    for p_ in parts:
        offs.append(total)
        total += (p_.numel() + 255) // 256 * 256
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for p_, o_ in zip(parts, offs):
        host_in[o_:o_ + p_.numel()].copy_(p_.cpu())
    dev_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [[dev_in[ch][o_:o_ + p_.numel()].view(x.dtype).view(x.shape)
              for p_, o_, x in zip(parts, offs, t)] for ch in range(2)]
    ys = [torch.empty_like(y) for _ in range(2)]
    host_y = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in, ev_k, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i, base):
        """Step i of a sequence of steps starting at step base, on the current stream."""
        comp = torch.cuda.current_stream()
        ch, parity = i % 2, (i // 2) % 2
        if i == base:  # the copy streams follow the current stream from here on
            s_in.wait_stream(comp)
            s_out.wait_stream(comp)
        if i - base >= 2:
            s_in.wait_event(ev_out[ch])  # this chain's previous result is on the host
            s_in.wait_event(ev_k[ch])    # and its previous kernel no longer reads dev_in[ch]
        with torch.cuda.stream(s_in):
            dev_in[ch].copy_(host_in, non_blocking=True)
        ev_in[ch].record(s_in)
        comp.wait_event(ev_in[ch])
        gdn.gdn_decode_step(states[2 * ch + parity], *views[ch], state_out=states[2 * ch + 1 - parity],
                            y=ys[ch])
        ev_k[ch].record(comp)
        s_out.wait_event(ev_k[ch])
        with torch.cuda.stream(s_out):
            host_y[ch].copy_(ys[ch], non_blocking=True)
        ev_out[ch].record(s_out)

    def e2e_finish():
        comp = torch.cuda.current_stream()
        comp.wait_event(ev_out[0])
        comp.wait_event(ev_out[1])

    for i in range(warmup):
        e2e_step(i, 0)
    e2e_finish()
    # a serving loop replays its decode steps from a CUDA graph: E2E_GRAPH steps (both chains, both
    # state parities) are captured once -- the same API calls, copies and stream dependencies -- and
    # replayed; steps past the last whole graph run eagerly.  Exactly `steps` steps are timed.
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph):
            for i in range(E2E_GRAPH):
                e2e_step(i, 0)
            e2e_finish()
        graph.replay()
        torch.cuda.synchronize()
        reps, rem = divmod(steps, E2E_GRAPH)
    except RuntimeError as e:  # no graph: every step eagerly (noted in the JSON line)
        print(f"e2e graph capture failed, eager steps: {e}", file=sys.stderr)
        torch.cuda.synchronize()
        graph, reps, rem = None, 0, steps

    def e2e_call(j):
        if j < reps:
            graph.replay()
        else:
            for i in range(reps * E2E_GRAPH, steps):
                e2e_step(i, reps * E2E_GRAPH)
            e2e_finish()

    e2e_secs = _timed(torch, dist, reps + (1 if rem else 0), e2e_call)
    # the same steps issued eagerly, one API call (and its copies and events) at a time from Python
    e2e_eager_secs = _timed(torch, dist, steps, lambda i: e2e_step(i, 0), finish=e2e_finish)
    h2d = sum(p_.numel() for p_ in parts)
    d2h = host_y[0].numel() * host_y[0].element_size()
    return dict(secs=secs, e2e_secs=e2e_secs, e2e_eager_secs=e2e_eager_secs, h2d=h2d, d2h=d2h,
                e2e_graph=graph is not None,
                state_bytes=decode_state_bytes(B, Hk, Hv, Dk, Dv),
                alg_bytes=decode_bytes(B, Hk, Hv, Dk, Dv), shape=(B, Hk, Hv, Dk, Dv))


def bench_decode_multi(torch, gdn, dist, steps, warmup, seed, T=8):
    """T consecutive decode tokens per call on the batched decode shapes (state on chip across
    the tokens): the speculative-window-sized multi-token path."""
    c = gi.GDN_DECODE_BATCHED
    B, Hk, Hv, Dk, Dv = c["B"], c["Hk"], c["Hv"], c["Dk"], c["Dv"]
    dev = torch.device("cuda")
    g = gi.rng(seed + 5)
    b16, f32 = torch.bfloat16, torch.float32
    toks = [gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv) for _ in range(T)]
    st = {n: torch.from_numpy(np.stack([t[n] for t in toks], axis=1)).to(dt).to(dev)
          for n, dt in (("q", b16), ("k", b16), ("v", b16), ("g", f32), ("beta", b16))}
    states = [(torch.randn((B, Hv, Dv, Dk), device=dev) * 0.1) for _ in range(4)]
    y = torch.empty((B, T, Hv, Dv), dtype=b16, device=dev)

    def step(i):
        chain, parity = (i % 2) * 2, (i // 2) % 2
        gdn.gdn_decode_multi(states[chain + parity], st["q"], st["k"], st["v"], st["g"], st["beta"],
                             state_out=states[chain + 1 - parity], y=y)

    for i in range(warmup):
        step(i)
    secs = _timed(torch, dist, steps, step)
    tok_bytes = T * (2 * B * Hk * Dk * 2 + B * Hv * Dv * 2 + B * Hv * 6 + B * Hv * Dv * 2)
    return dict(secs=secs, T=T, B=B, alg_bytes=decode_state_bytes(B, Hk, Hv, Dk, Dv) + tok_bytes)


def bench_decode_pooled(torch, gdn, dist, steps, warmup, seed, pool=128):
    """The batched decode step on a pooled state: 64 batch rows scattered over a 128-slot pool."""
    c = gi.GDN_DECODE_BATCHED
    B, Hk, Hv, Dk, Dv = c["B"], c["Hk"], c["Hv"], c["Dk"], c["Dv"]
    dev = torch.device("cuda")
    g = gi.rng(seed + 6)
    b16, f32 = torch.bfloat16, torch.float32
    t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
    d = [torch.from_numpy(t[n]).to(dt).to(dev) for n, dt in
         (("q", b16), ("k", b16), ("v", b16), ("g", f32), ("beta", b16))]
    pools = [torch.randn((pool, Hv, Dv, Dk), device=dev) * 0.1 for _ in range(2)]
    idx = torch.from_numpy(g.choice(pool, size=B, replace=False).astype(np.int64)).to(dev)
    y = torch.empty((B, Hv, Dv), dtype=b16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(i):
        gdn.gdn_decode_step_pooled(pools[i % 2], idx, *d, y=y, dev_status=status)

    for i in range(warmup):
        step(i)
    secs = _timed(torch, dist, steps, step)
    return dict(secs=secs, alg_bytes=decode_bytes(B, Hk, Hv, Dk, Dv))


# The Comba spec's measure shapes (B, H, K, V).
COMBA_SWEEP = [(896, 16, 128, 128), (448, 32, 128, 128), (1792, 8, 128, 128), (1280, 16, 64, 128),
               (640, 24, 128, 128)]


def bench_comba_sweep(torch, gdn, dist, steps, warmup, seed):
    dev = torch.device("cuda")
    b16, f32 = torch.bfloat16, torch.float32
    out = []
    for (B, H, K, V) in COMBA_SWEEP:
        g = gi.rng(seed + B + K)
        t = gi.comba_decode_token(g, B, H, K, V)
        d = [torch.from_numpy(t[n]).to(dt).to(dev) for n, dt in
             (("q", b16), ("k", b16), ("v", b16), ("p", b16), ("beta", b16), ("g_log", f32))]
        states = [torch.randn((B, H, K, V), device=dev) * 0.1 for _ in range(2)]
        o = torch.empty((B, H, V), dtype=b16, device=dev)

        def step(i):
            gdn.comba_decode_step(states[i % 2], *d, state_new=states[1 - i % 2], o=o)

        for i in range(warmup):
            step(i)
        secs = _timed(torch, dist, steps, step)
        out.append(dict(shape=[B, H, K, V], secs=secs, alg_bytes=comba_bytes(B, H, K, V)))
        del states
    return out


def bench_comba(torch, gdn, dist, steps, warmup, seed):
    c = gi.COMBA_DECODE
    B, H, K, V = c["B"], c["H"], c["K"], c["V"]
    dev = torch.device("cuda")
    g = gi.rng(seed + 1)
    b16, f32 = torch.bfloat16, torch.float32

    def tok():
        t = gi.comba_decode_token(g, B, H, K, V)
        return tuple(torch.from_numpy(t[n]).to(dt).to(dev) for n, dt in
                     (("q", b16), ("k", b16), ("v", b16), ("p", b16), ("beta", b16),
                      ("g_log", f32)))

    states = [torch.zeros((B, H, K, V), dtype=f32, device=dev) for _ in range(4)]
    o = torch.empty((B, H, V), dtype=b16, device=dev)
    for w in range(c["warmup"]):
        gdn.comba_decode_step(states[w % 2], *tok(), state_new=states[1 - w % 2], o=o)
    states[0].copy_(states[c["warmup"] % 2])
    states[2].copy_(states[0])
    t = tok()

    def step(i):
        chain, parity = (i % 2) * 2, (i // 2) % 2
        gdn.comba_decode_step(states[chain + parity], *t, state_new=states[chain + 1 - parity], o=o)

    for i in range(warmup):
        step(i)
    secs = _timed(torch, dist, steps, step)
    return dict(secs=secs, alg_bytes=comba_bytes(B, H, K, V), shape=(B, H, K, V))


def bench_comba_forward(torch, gdn, dist, steps, warmup, seed):
    c = gi.COMBA_FORWARD
    B, T, H, K, V = c["B"], c["T"], c["H"], c["K"], c["V"]
    x = gi.comba_forward_inputs(gi.rng(seed + 5), B, T, H, K, V)
    dev = torch.device("cuda")
    b16, f32 = torch.bfloat16, torch.float32
    d = {n: torch.from_numpy(x[n]).to(dt).to(dev) for n, dt in
         (("q", b16), ("k", b16), ("v", b16), ("p", b16), ("beta", b16), ("g_log", f32), ("state", f32))}
    o = torch.empty((B, T, H, V), dtype=b16, device=dev)

    def step(i):  # the 537 MB state is larger than L2; it is carried from call to call
        gdn.comba_forward(d["state"], d["q"], d["k"], d["v"], d["p"], d["beta"], d["g_log"], o=o)

    for i in range(warmup):
        step(i)
    secs = _timed(torch, dist, steps, step)
    return dict(secs=secs, alg_bytes=comba_forward_bytes(B, T, H, K, V), B=B, T=T, H=H)


def bench_prefill(torch, gdn, dist, steps, warmup, seed, dtype="bf16"):
    c = gi.GDN_PREFILL
    Hk, Hv, K, V, C = c["Hk"], c["Hv"], c["K"], c["V"], c["chunk"]
    x = gi.gdn_prefill_inputs(gi.rng(seed + 2), c["seqlens"], Hk, Hv, K, V, c["pool"], dtype=dtype)
    dev = torch.device("cuda")
    b16 = torch.float16 if dtype == "f16" else torch.bfloat16  # the token arrays' type
    f32 = torch.float32
    d = {n: torch.from_numpy(x[n]).to(dt).to(dev) for n, dt in
         (("q", b16), ("k", b16), ("v", b16), ("a", b16), ("b", b16), ("A_log", f32),
          ("dt_bias", f32), ("state_pool", f32), ("cache_indices", torch.int64),
          ("cu_seqlens", torch.int64))}
    T = x["T"]
    out = torch.empty((T, Hv, V), dtype=b16, device=dev)
    ws = torch.empty(max(1, gdn.gdn_prefill_workspace_size(len(c["seqlens"]), T, Hk, Hv, K, V, C)),
                     dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    pristine = d["state_pool"].clone()

    def step(i):
        gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                d["state_pool"], d["cache_indices"], d["cu_seqlens"], C, out=out,
                                workspace=ws, dev_status=status)

    def restore(i):  # every call starts from the same pool (the call updates it in place)
        d["state_pool"].copy_(pristine)

    for i in range(warmup):
        restore(i)
        step(i)
    secs = _timed_calls(torch, dist, steps, step, restore)
    return dict(secs=secs, T=T, alg_bytes=prefill_bytes(c["seqlens"], Hk, Hv, K, V),
                flops=prefill_flops(c["seqlens"], Hv, K, V, C))


def bench_window(torch, gdn, dist, steps, warmup, seed, commit):
    c = gi.GDN_WINDOW
    N, h_k, h_v, D, ntok = c["N"], c["h_k"], c["h_v"], c["D"], c["ntok"]
    x = gi.gdn_window_inputs(gi.rng(seed + 3), N, h_k, h_v, D, ntok)
    dev = torch.device("cuda")
    f32 = torch.float32
    d = {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(f32).to(dev) for n in x}
    # rotate three state copies (3 x 100 MB) and three history pairs so that no read hits L2
    states = [d["state"].clone() for _ in range(3)]
    hists = [d["hist"].clone() for _ in range(3)]
    hist_out = [torch.empty_like(d["hist"]) for _ in range(3)]
    y = torch.empty((N, ntok, h_v, D), dtype=f32, device=dev)
    code = 1 if commit else 0

    def step(i):
        j = i % 3
        gdn.gdn_window_fused(states[j], hists[j], hist_out[j], d["qkv"], d["alpha"], d["beta"],
                             d["z"], d["conv_w"], d["dt"], d["ssm_a"], d["gamma"], h_k, code, y=y)

    for i in range(warmup):
        step(i)
    secs = _timed(torch, dist, steps, step)
    return dict(secs=secs, alg_bytes=window_bytes(N, h_k, h_v, D, ntok, commit))


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (the baseline; also the reference arm)
# ------------------------------------------------------------------------------------------------
class OracleSample:
    """The oracle on a bounded sample of one operation's workload, timed on this host's cores.

    The workload is cut into independent units (a batch row, a sequence, a (sequence, head) pair:
    whatever the oracle takes in one call); ``unit(i)`` runs unit ``i`` and ``work`` is what one unit
    contributes to the operation's metric (bytes or tokens).  ``run`` keeps ``threads`` units in
    flight until ``seconds`` have passed (the oracle's C code runs outside the GIL); ``run_one``
    times units on one thread.  The oracle is run as it stands, untuned."""

    def __init__(self, name, unit, n_units, work, unit_desc, scale_to_metric, metric_unit):
        self.name, self.unit, self.n_units, self.work = name, unit, n_units, work
        self.unit_desc, self.scale, self.metric_unit = unit_desc, scale_to_metric, metric_unit
        self.next = 0

    def run(self, seconds: float, threads: int):
        """Returns (value in the metric's unit, units run, seconds)."""
        done = 0
        t0 = time.perf_counter()
        with ThreadPoolExecutor(max_workers=threads) as ex:
            while time.perf_counter() - t0 < seconds:
                list(ex.map(self.unit, [(self.next + i) % self.n_units for i in range(threads)]))
                self.next += threads
                done += threads
        secs = time.perf_counter() - t0
        return done * self.work * self.scale / secs, done, secs

    def run_one(self, seconds: float):
        done = 0
        t0 = time.perf_counter()
        while done == 0 or time.perf_counter() - t0 < seconds:
            self.unit(self.next % self.n_units)
            self.next += 1
            done += 1
        secs = time.perf_counter() - t0
        return done * self.work * self.scale / secs, done, secs

    def baseline(self, seconds: float, threads: int) -> dict:
        """The cpu_baseline object of this operation: all threads, then one thread."""
        value, n, secs = self.run(seconds, threads)
        v1, n1, secs1 = self.run_one(max(1.0, seconds / 4))
        return {"value": value, "unit": self.metric_unit, "cores": threads, "kind": "oracle",
                "sample": f"{n} units ({self.unit_desc}), fp64 oracle, {threads} threads over units, "
                          f"{secs:.2f} s",
                "one_thread": {"value": v1, "unit": self.metric_unit,
                               "sample": f"{n1} units on 1 thread, {secs1:.2f} s"}}


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def oracle_samples() -> dict:
    """One OracleSample per measured operation, on reduced copies of the operations' workloads
    (the same shapes per unit, the same distributions)."""
    import oracle
    oracle.build()
    out = {}

    # GDN decode step: unit = one batch row (Hv heads of Dv x Dk)
    c = gi.GDN_DECODE_BATCHED
    B, Hk, Hv, Dk, Dv = c["B"], c["Hk"], c["Hv"], c["Dk"], c["Dv"]
    g = gi.rng(0)
    t = {n: _f64(x) for n, x in gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv).items()}
    S = _f64(g.standard_normal((B, Hv, Dv, Dk)) * 0.1)
    rows = [dict(S=np.ascontiguousarray(S[b:b + 1]),
                 **{n: np.ascontiguousarray(x[b:b + 1]) for n, x in t.items()}) for b in range(B)]

    def dec_row(b):
        r = rows[b]
        oracle.gdn_decode(r["S"], r["q"], r["k"], r["v"], r["g"], r["beta"], Dk ** -0.5)

    desc = f"batch rows of {Hv} heads of {Dv}x{Dk}"
    out["decode"] = OracleSample("decode", dec_row, B, decode_state_bytes(1, Hk, Hv, Dk, Dv), desc,
                                 1e-9, "GB/s")
    out["decode_pooled"] = OracleSample("decode_pooled", dec_row, B,
                                        decode_bytes(B, Hk, Hv, Dk, Dv) / B, desc, 1e-9, "GB/s")

    # multi-token decode: unit = one batch row stepped through T = 8 tokens
    T8 = 8
    toks = [{n: _f64(x) for n, x in gi.gdn_decode_token(g, 8, Hk, Hv, Dk, Dv).items()}
            for _ in range(T8)]

    def multi_row(b):
        St = rows[b]["S"]
        r = b % 8
        for tk in toks:
            St, _ = oracle.gdn_decode(St, tk["q"][r:r + 1], tk["k"][r:r + 1], tk["v"][r:r + 1],
                                      tk["g"][r:r + 1], tk["beta"][r:r + 1], Dk ** -0.5)

    out["decode_multi"] = OracleSample("decode_multi", multi_row, B, T8,
                                       f"batch rows of {Hv} heads stepped through {T8} tokens", 1.0,
                                       "token-steps/s")

    # Comba decode step: unit = one batch row (H heads of K x V)
    cc = gi.COMBA_DECODE
    H, K, V = cc["H"], cc["K"], cc["V"]
    ct = {n: _f64(x) for n, x in gi.comba_decode_token(g, 8, H, K, V).items()}
    CS = _f64(g.standard_normal((8, H, K, V)) * 0.1)

    def comba_row(b):
        sl = slice(b, b + 1)
        oracle.comba_decode(CS[sl], ct["q"][sl], ct["k"][sl], ct["v"][sl], ct["p"][sl],
                            ct["beta"][sl], ct["g_log"][sl], K ** -0.5)

    out["comba_decode"] = OracleSample("comba_decode", comba_row, 8, comba_bytes(1, H, K, V),
                                       f"batch rows of {H} heads of {K}x{V}", 1e-9, "GB/s")

    # Comba forward: unit = one batch row, T tokens, H heads
    cf = gi.COMBA_FORWARD
    fx = {n: _f64(x) for n, x in gi.comba_forward_inputs(g, 8, cf["T"], H, K, V).items()}

    def cfwd_row(b):
        sl = slice(b, b + 1)
        oracle.comba_forward(fx["state"][sl], fx["q"][sl], fx["k"][sl], fx["v"][sl], fx["p"][sl],
                             fx["beta"][sl], fx["g_log"][sl], K ** -0.5)

    out["comba_forward"] = OracleSample("comba_forward", cfwd_row, 8, H * cf["T"],
                                        f"batch rows of {H} heads x {cf['T']} tokens", 1.0,
                                        "head-token steps/s")

    # chunked prefill: unit = (one 512-token sequence, one value head); tokens/s = token-heads / Hv
    pc = gi.GDN_PREFILL
    L = 512
    px = gi.gdn_prefill_inputs(gi.rng(2), (L,), pc["Hk"], pc["Hv"], pc["K"], pc["V"], pc["pool"])
    pq, pk, pv, pa, pb = (_f64(px[n]) for n in ("q", "k", "v", "a", "b"))
    slot = int(px["cache_indices"][0])
    pS = [_f64(px["state_pool"][slot, h]) for h in range(pc["Hv"])]

    def prefill_unit(h):
        oracle.gdn_prefill_unit(pq, pk, pv, pa, pb, float(px["A_log"][h]), float(px["dt_bias"][h]),
                                pS[h], h, pc["K"] ** -0.5)

    out["prefill_chunked"] = OracleSample(
        "prefill_chunked", prefill_unit, pc["Hv"], L,
        f"(sequence of {L} tokens, value head) pairs of the prefill's shapes", 1.0 / pc["Hv"],
        "tokens/s")

    # Comba chunked prefill: unit = (one 512-token sequence, one head), the oracle's Comba
    # recurrence over the sequence
    cx = gi.comba_prefill_inputs(gi.rng(5), (L,), pc["Hv"], K, V, pc["pool"])
    cslot = int(cx["cache_indices"][0])
    cheads = [dict(q=_f64(cx["q"][None, :, h:h + 1]), k=_f64(cx["k"][None, :, h:h + 1]),
                   v=_f64(cx["v"][None, :, h:h + 1]), p=_f64(cx["p"][None, :, h:h + 1]),
                   beta=_f64(cx["beta"][None, :, h:h + 1]), g=_f64(cx["g_log"][None, :, h:h + 1]),
                   S=_f64(cx["state_pool"][cslot, h][None, None])) for h in range(pc["Hv"])]

    def comba_prefill_unit(h):
        u = cheads[h]
        oracle.comba_forward(u["S"], u["q"], u["k"], u["v"], u["p"], u["beta"], u["g"], K ** -0.5)

    out["comba_prefill_chunked"] = OracleSample(
        "comba_prefill_chunked", comba_prefill_unit, pc["Hv"], L,
        f"(sequence of {L} tokens, head) pairs of the Comba prefill's shapes", 1.0 / pc["Hv"],
        "tokens/s")

    # fused window: unit = one sequence (all value heads, ntok tokens)
    wc = gi.GDN_WINDOW
    wx = {n: _f64(x) for n, x in gi.gdn_window_inputs(gi.rng(3), 4, wc["h_k"], wc["h_v"], wc["D"],
                                                         wc["ntok"]).items()}
    for commit in (False, True):
        def win_seq(n, code=1 if commit else 0):
            sl = slice(n, n + 1)
            oracle.gdn_window(wx["state"][sl], wx["hist"][sl], wx["qkv"][sl], wx["alpha"][sl],
                              wx["beta"][sl], wx["z"][sl], wx["conv_w"], wx["dt"], wx["ssm_a"],
                              wx["gamma"], wc["h_k"], code)

        name = "window_commit" if commit else "window_verify"
        out[name] = OracleSample(
            name, win_seq, 4, window_bytes(1, wc["h_k"], wc["h_v"], wc["D"], wc["ntok"], commit),
            f"sequences of {wc['h_v']} value heads x {wc['ntok']} tokens", 1e-9, "GB/s")
    out["prefill_chunked_f16"] = out["prefill_chunked"]  # the oracle widens either input type
    return out


def bench_comba_prefill(torch, gdn, dist, steps, warmup, seed):
    """The Comba chunked prefill on the GDN prefill's token layout: lengths 4096+2048+1024+8192,
    H=32 heads (each with its own q, k, p), K=V=128, chunk 64, a 16-slot pool."""
    c = gi.GDN_PREFILL
    H, K, V, C = c["Hv"], c["K"], c["V"], c["chunk"]
    x = gi.comba_prefill_inputs(gi.rng(seed + 5), c["seqlens"], H, K, V, c["pool"])
    dev = torch.device("cuda")
    bf, f32 = torch.bfloat16, torch.float32
    d = {n: torch.from_numpy(x[n]).to(dt).to(dev) for n, dt in
         (("q", bf), ("k", bf), ("v", bf), ("p", bf), ("beta", bf), ("g_log", f32), ("state_pool", f32),
          ("cache_indices", torch.int64), ("cu_seqlens", torch.int64))}
    T = x["T"]
    out = torch.empty((T, H, V), dtype=bf, device=dev)
    ws = torch.empty(max(1, gdn.gdn_prefill_workspace_size(len(c["seqlens"]), T, H, H, K, V, C)),
                     dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    pristine = d["state_pool"].clone()

    def step(i):
        gdn.comba_prefill_chunked(d["q"], d["k"], d["v"], d["p"], d["beta"], d["g_log"], d["state_pool"],
                                  d["cache_indices"], d["cu_seqlens"], C, out=out, workspace=ws, dev_status=status)

    def restore(i):  # every call starts from the same pool (the call updates it in place)
        d["state_pool"].copy_(pristine)

    for i in range(warmup):
        restore(i)
        step(i)
    secs = _timed_calls(torch, dist, steps, step, restore)
    return dict(secs=secs, T=T, alg_bytes=comba_prefill_bytes(c["seqlens"], H, K, V),
                flops=prefill_flops(c["seqlens"], H, K, V, C))


# ------------------------------------------------------------------------------------------------
def main_single_op(args, torch, gdn, dist, seed):
    """One operation alone, args.steps timed calls after args.warmup: a small, repeatable command to
    run under a profiler."""
    fns = {
        "decode": lambda: bench_decode(torch, gdn, dist, args.steps, args.warmup, seed),
        "comba": lambda: bench_comba(torch, gdn, dist, args.steps, args.warmup, seed),
        "comba_forward": lambda: bench_comba_forward(torch, gdn, dist, args.steps, args.warmup, seed),
        "prefill": lambda: bench_prefill(torch, gdn, dist, args.steps, args.warmup, seed),
        "prefill_f16": lambda: bench_prefill(torch, gdn, dist, args.steps, args.warmup, seed, "f16"),
        "comba_prefill": lambda: bench_comba_prefill(torch, gdn, dist, args.steps, args.warmup, seed),
        "window_verify": lambda: bench_window(torch, gdn, dist, args.steps, args.warmup, seed, False),
        "window_commit": lambda: bench_window(torch, gdn, dist, args.steps, args.warmup, seed, True),
        "decode_multi": lambda: bench_decode_multi(torch, gdn, dist, args.steps, args.warmup, seed),
        "decode_pooled": lambda: bench_decode_pooled(torch, gdn, dist, args.steps, args.warmup, seed),
    }
    r = fns[args.op]()
    if dist.rank == 0:
        print(json.dumps({"op": args.op, "steps": args.steps, "warmup": args.warmup,
                          "us_per_call": r["secs"] / args.steps * 1e6}))
    dist.close()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gdn", "reference"), default="gdn")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work of the oracle baseline (rank 0, N=1)")
    ap.add_argument("--op", choices=("decode", "comba", "comba_forward", "prefill", "prefill_f16", "comba_prefill",
                                     "window_verify", "window_commit",
                                     "decode_multi", "decode_pooled"),
                    help="time only this operation on its workload and print its time per call "
                         "(for profiling; not the benchmark line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        return main_reference(args)

    import torch
    import gated_deltanet_delta_gb300 as gdn
    from gated_deltanet_delta_gb300 import build as gbuild

    dist = Dist()
    gbuild.build()
    gdn.load()
    torch.cuda.set_device(dist.local_rank)
    hbm_peak, tf_peak, peak_src = load_peaks()
    seed = dist.rank

    if args.op:
        return main_single_op(args, torch, gdn, dist, seed)

    sampler = ClockSampler(dist.local_rank)
    with sampler:
        dec = bench_decode(torch, gdn, dist, args.steps, args.warmup, seed)
        extra = {}
        for name, fn in (("comba", lambda: bench_comba(torch, gdn, dist, args.steps, args.warmup,
                                                         seed)),
                         ("prefill", lambda: bench_prefill(torch, gdn, dist,
                                                           max(3, args.steps // 10),
                                                           args.warmup, seed)),
                         ("prefill_f16", lambda: bench_prefill(torch, gdn, dist,
                                                               max(3, args.steps // 10),
                                                               args.warmup, seed, "f16")),
                         ("comba_prefill", lambda: bench_comba_prefill(torch, gdn, dist,
                                                                       max(3, args.steps // 10),
                                                                       args.warmup, seed)),
                         ("window_verify", lambda: bench_window(torch, gdn, dist, args.steps,
                                                                args.warmup, seed, False)),
                         ("window_commit", lambda: bench_window(torch, gdn, dist, args.steps,
                                                                args.warmup, seed, True)),
                         ("decode_multi", lambda: bench_decode_multi(torch, gdn, dist, args.steps,
                                                                     args.warmup, seed)),
                         ("decode_pooled", lambda: bench_decode_pooled(torch, gdn, dist, args.steps,
                                                                       args.warmup, seed)),
                         ("comba_forward", lambda: bench_comba_forward(torch, gdn, dist,
                                                                       max(3, args.steps // 5),
                                                                       args.warmup, seed)),
                         ("comba_sweep", lambda: bench_comba_sweep(torch, gdn, dist,
                                                                   max(3, args.steps // 5),
                                                                   args.warmup, seed))):
            try:
                extra[name] = fn()
            except gdn.GdnError as e:
                extra[name] = {"unavailable": str(e)}
    clocks = sampler.summary()

    N, K = dist.world, args.steps
    ms = dec["secs"] / K * 1e3
    value = N * dec["state_bytes"] * K / dec["secs"] / 1e9
    e2e_value = N * dec["state_bytes"] * K / dec["e2e_secs"] / 1e9
    per_launch = dec["secs"] / K
    achieved = dec["alg_bytes"] / per_launch / 1e9
    peak_note = "of measured" if peak_src == "measured" else "of fallback"

    ops = {}
    if "secs" in extra.get("comba", {}):
        cb = extra["comba"]
        t1 = cb["secs"] / K
        gbs = cb["alg_bytes"] / t1 / 1e9
        ops["comba_decode"] = {
            "workload": gi.COMBA_DECODE["name"], "value": N * gbs, "unit": "GB/s",
            "us_per_step": t1 * 1e6,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "note": peak_note,
                         "traffic": profiled_traffic("comba_decode_kernel",
                                                     "gated_deltanet_delta_gb300/csrc/comba.cuh")}}
    elif "comba" in extra:
        ops["comba_decode"] = extra["comba"]
    for key, op_name, dt_note in (("prefill", "prefill_chunked", ""),
                                  ("prefill_f16", "prefill_chunked_f16", ", fp16 token arrays"),
                                  ("comba_prefill", "comba_prefill_chunked",
                                   ", Comba recurrence, H=32 (own q, k, p per head)")):
        pf = extra.get(key, {})
        if "secs" not in pf:
            if key in extra:
                ops[op_name] = pf
            continue
        steps_pf = max(3, args.steps // 10)
        t1 = pf["secs"] / steps_pf
        t_hbm = pf["alg_bytes"] / (hbm_peak * 1e9)
        t_tc = pf["flops"] / (tf_peak * 1e12)
        roof = max(t_hbm, t_tc)
        ops[op_name] = {
            "workload": gi.GDN_PREFILL["name"] + dt_note, "value": N * pf["T"] / t1, "unit": "tokens/s",
            "us_per_call": t1 * 1e6,
            "roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                         "achieved": (pf["alg_bytes"] / t1 / 1e9) if t_hbm >= t_tc
                         else (pf["flops"] / t1 / 1e12),
                         "peak": hbm_peak if t_hbm >= t_tc else tf_peak,
                         "unit": "GB/s" if t_hbm >= t_tc else "TFLOP/s",
                         "frac": roof / t1, "note": peak_note,
                         "roofline_us": roof * 1e6, "hbm_us": t_hbm * 1e6, "tensor_us": t_tc * 1e6,
                         "traffic": profiled_traffic({"prefill": "gdn_prefill_call",
                                                      "prefill_f16": "gdn_prefill_f16_call",
                                                      "comba_prefill": "comba_prefill_call"}.get(key, ""),
                                                     "gated_deltanet_delta_gb300/csrc/prefill.cuh")}}
    for key in ("window_verify", "window_commit"):
        w = extra.get(key, {})
        if "secs" in w:
            t1 = w["secs"] / K
            gbs = w["alg_bytes"] / t1 / 1e9
            ops[key] = {"workload": gi.GDN_WINDOW["name"], "value": N * gbs, "unit": "GB/s",
                        "us_per_call": t1 * 1e6,
                        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                                     "unit": "GB/s", "frac": gbs / hbm_peak, "note": peak_note,
                                     "traffic": profiled_traffic(
                                         "gdn_window_kernel" if key == "window_verify"
                                         else "gdn_window_kernel_commit",
                                         ("gated_deltanet_delta_gb300/csrc/window.cuh",
                                          "gated_deltanet_delta_gb300/csrc/window.cu"))}}
        elif key in extra:
            ops[key] = w

    dm = extra.get("decode_multi", {})
    if "secs" in dm:
        t1 = dm["secs"] / K
        gbs = dm["alg_bytes"] / t1 / 1e9
        ops["decode_multi"] = {
            "workload": f"gdn decode, {dm['T']} tokens per call, B64 Hk16 Hv32 D128",
            "value": N * dm["B"] * dm["T"] / t1, "unit": "token-steps/s", "us_per_call": t1 * 1e6,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "note": peak_note,
                         "traffic": profiled_traffic("gdn_decode_multi_kernel",
                                                     ("gated_deltanet_delta_gb300/csrc/decode.cuh",
                                                      "gated_deltanet_delta_gb300/csrc/decode.cu"))}}
    dp = extra.get("decode_pooled", {})
    if "secs" in dp:
        t1 = dp["secs"] / K
        gbs = dp["alg_bytes"] / t1 / 1e9
        ops["decode_pooled"] = {
            "workload": "gdn decode on a 128-slot pool, B64 Hk16 Hv32 D128", "value": N * gbs,
            "unit": "GB/s", "us_per_step": t1 * 1e6,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "note": peak_note,
                         "traffic": profiled_traffic("gdn_decode_kernel_pooled",
                                                     ("gated_deltanet_delta_gb300/csrc/decode.cuh",
                                                      "gated_deltanet_delta_gb300/csrc/decode.cu"))}}
    cf = extra.get("comba_forward", {})
    if "secs" in cf:
        t1 = cf["secs"] / max(3, K // 5)
        gbs = cf["alg_bytes"] / t1 / 1e9
        ops["comba_forward"] = {
            "workload": gi.COMBA_FORWARD["name"], "value": N * cf["B"] * cf["H"] * cf["T"] / t1,
            "unit": "head-token steps/s", "us_per_call": t1 * 1e6,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "note": peak_note,
                         "traffic": profiled_traffic("comba_forward_kernel",
                                                     "gated_deltanet_delta_gb300/csrc/comba_forward.cuh")}}
    elif "comba_forward" in extra:
        ops["comba_forward"] = cf
    if isinstance(extra.get("comba_sweep"), list):
        ksw = max(3, args.steps // 5)
        rows = []
        for r in extra["comba_sweep"]:
            t1 = r["secs"] / ksw
            gbs = r["alg_bytes"] / t1 / 1e9
            rows.append({"shape_BHKV": r["shape"], "GB/s": gbs, "frac": gbs / hbm_peak,
                         "us_per_step": t1 * 1e6})
        ops["comba_sweep"] = {"workload": "Comba spec measure shapes", "rows": rows,
                              "note": peak_note}

    cpu = None
    if dist.rank == 0 and N == 1:
        # the oracle beside every GPU number: the headline on args.cpu_seconds of CPU work, every
        # other operation on a quarter of that (plus a one-thread run each)
        threads = os.cpu_count() or 1
        samples = oracle_samples()
        cpu = samples["decode"].baseline(args.cpu_seconds, threads)
        for op_name, entry in ops.items():
            if op_name in samples and isinstance(entry, dict) and "value" in entry:
                entry["cpu_baseline"] = samples[op_name].baseline(args.cpu_seconds / 4, threads)

    B, Hk, Hv, Dk, Dv = dec["shape"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": N, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": gi.GDN_DECODE_BATCHED["name"], "B": B, "Hk": Hk, "Hv": Hv,
                   "Dk": Dk, "Dv": Dv, "state_bytes_per_step": dec["state_bytes"],
                   "l2": "inputs larger than L2: two interleaved chains over four 134 MB states",
                   "parallelism": f"replicas x{N}"},
        "hbm_frac": value / N / hbm_peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "note": peak_note,
                     "traffic": profiled_traffic("gdn_decode_kernel",
                                                 ("gated_deltanet_delta_gb300/csrc/decode.cuh",
                                                  "gated_deltanet_delta_gb300/csrc/decode.cu"))},
        "e2e": {"value": e2e_value, "unit": "GB/s", "graph": dec["e2e_graph"], "h2d_bytes_per_step": dec["h2d"],
                "d2h_bytes_per_step": dec["d2h"],
                "eager_value": N * dec["state_bytes"] * K / dec["e2e_eager_secs"] / 1e9,
                "note": "value: the steps' API calls, host copies and stream dependencies captured "
                        "once in a CUDA graph and replayed (a device-side pipelined copy + kernel "
                        "figure; the per-call host work runs only at capture); eager_value: every "
                        "step issued from Python through the C ABI"},
        "gpu_launches": K,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "ops": ops,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def main_reference(args):
    """The reference arm: the CPU oracle, timed on this host's cores, each step a bounded sample
    of the batched decode workload.  Under torchrun only rank 0 works and prints."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    per_step = max(0.05, min(1.0, 60.0 / max(1, args.steps + args.warmup)))
    sample = oracle_samples()["decode"]
    for _ in range(args.warmup):
        sample.run(per_step, threads)
    vals, secs, units = [], 0.0, 0
    for _ in range(args.steps):
        v, n, s = sample.run(per_step, threads)
        vals.append(v)
        secs += s
        units += n
    value = statistics.median(vals)
    desc = (f"{units} {sample.unit_desc} over {args.steps} steps of {per_step:.2f} s, fp64 oracle, "
            f"{threads} threads over units")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": gi.GDN_DECODE_BATCHED["name"]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

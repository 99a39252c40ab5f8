"""Benchmark of the routed, quantized expert-FFN MoE layer on GB300.

Workload (default): the 35B-A3B-shaped int4 decode layer -- 40 layers,
hidden 2048, 256 experts, top-8, expert intermediate 512, int4 g64 weights
(1,671,168 B per expert), a slot cache of 2,560 experts (25% of the 10,240
(layer, expert) pairs) warmed from a seeded Zipf(1.1) routing history, and the
full pool (17.1 GB) in pinned host memory as the source of truth.

One step = T tokens through all 40 MoE layers; each layer runs the whole hot
path: route (logits, softmax, top-k) -> resolve (slot or -1, q* split) ->
fetch (misses pool -> cache) -> experts (gate/up, SwiGLU, down, combine).  The
40-layer step is captured once in a CUDA graph and replayed; inputs for every
step are resident in HBM before timing starts.

Printed: one JSON line (rank 0).  --impl reference times the CPU oracle on
the same workload instead.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode expert-weight HBM GB/s; prefill grouped-GEMM TFLOP/s"
# DRAM bytes (read + write) of one experts call (gate/up + down kernels) from
# an ncu capture of the same kernels on this workload's shape, L2 kept
# between the kernels (`bench.py --case decode --tokens T` under
# `ncu --cache-control none`, summarised under profiles/)
TRAFFIC_PER_CALL = {1: 13_372_928, 8: 104_289_536}
# DRAM bytes per ft_moe_decode_layer launch (ncu); empty until captured for the current kernel
LAYER_TRAFFIC_PER_CALL = {}
# the same for one flash-shaped NVFP4 decode experts call at T = 1
# (`bench.py --case decode-flash --tokens 1`)
FLASH_TRAFFIC_PER_CALL = 27_660_544
UNIT = "MoE-layer tokens/s"


# --------------------------------------------------------------- plumbing --
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(rank_units: float, rank_seconds: float, world: int, reduce_fn=None):
    """Whole-job throughput: units summed over ranks / the slowest rank's time."""
    if world == 1 or reduce_fn is None:
        return rank_units / rank_seconds, rank_seconds, rank_units
    units, secs = reduce_fn(rank_units, rank_seconds)
    return units / secs, secs, units


def torch_reduce_fn(device):
    import torch
    import torch.distributed as dist

    def fn(units, secs):
        u = torch.tensor([units], dtype=torch.float64, device=device)
        s = torch.tensor([secs], dtype=torch.float64, device=device)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        dist.all_reduce(s, op=dist.ReduceOp.MAX)
        return float(u.item()), float(s.item())

    return fn


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------- the workload --
def step_inputs(cfg, T: int, n_steps: int):
    """Pinned host inputs [n_steps, L, T, H] bf16 bits: step i's tokens depend
    only on i (x ~ N(0,1), feature 0 = 1.0, the router's bias feature)."""
    import torch

    import synth

    xs = np.stack([synth.normal_bf16(synth.stream_key(cfg.seed, "bench-x", T, i), (cfg.L, T, cfg.H))
                   for i in range(n_steps)])
    xs[..., 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
    return torch.from_numpy(xs.view(np.int16)).pin_memory()


class DecodeWorkload:
    """Device state of the decode benchmark for one config (built untimed)."""

    def __init__(self, cfg, T: int, phi: int, n_steps: int, device, log=print):
        import torch

        import quantized_expert_ffn_router_gb300 as ft
        import synth

        self.ft, self.cfg, self.T, self.phi = ft, cfg, T, phi
        self.dev = device
        L, E, k, H, I, g = cfg.L, cfg.E, cfg.k, cfg.H, cfg.I, cfg.g
        self.block, self.offs = ft.block_bytes(cfg.fmt, H, I, g)
        stride = self.block
        t0 = time.time()
        n_fid = L * E
        if cfg.slots >= n_fid:
            self._init_resident(cfg, T, n_steps, device, log)
            return
        # pool: the source of truth, pinned host memory, indexed by flat id
        self.pool = torch.empty((n_fid, stride), dtype=torch.uint8, pin_memory=True)
        chunk = 128
        tmp = torch.empty((chunk, stride), dtype=torch.uint8, device=device)
        for f0 in range(0, n_fid, chunk):
            n = min(chunk, n_fid - f0)
            synth.bank_blocks_torch(cfg.seed, range(f0, f0 + n), cfg.fmt, H, I, g, tmp[:n], ref_K=cfg.ref_K)
            self.pool[f0:f0 + n].copy_(tmp[:n])
        torch.cuda.synchronize()
        log(f"pool {n_fid} x {stride} B generated in {time.time() - t0:.1f}s")
        ts = synth.tensor_scales(cfg.fmt, H, I, n_fid)
        self.tscale = None if ts is None else torch.from_numpy(ts).to(device)
        self.S = cfg.slots
        self.cache = torch.zeros((self.S, stride), dtype=torch.uint8, device=device)
        self.pool_b = ft.make_bank(cfg.fmt, H, I, g, self.pool, self.tscale)
        self.cache_b = ft.make_bank(cfg.fmt, H, I, g, self.cache, self.tscale)
        # router weights with the Zipf bias feature (column 0)
        self.W = torch.stack([torch.from_numpy(synth.router_weights(cfg.seed, l, E, H, cfg.router_std,
                                                                    zipf_bias=cfg.zipf))
                              for l in range(L)]).to(device)
        # cache state: replay the seeded Zipf history through the GPU resolve
        self.state = ft.DeviceCacheState(L, E, self.S, device=device)
        t0 = time.time()
        hist = synth.zipf_history(cfg.seed, L, E, k, cfg.history_steps)
        hd = torch.from_numpy(hist).to(device)
        sl = torch.empty((1, k), dtype=torch.int32, device=device)
        nf = torch.zeros(1, dtype=torch.int32, device=device)
        ff = torch.empty(k, dtype=torch.int32, device=device)
        fs = torch.empty(k, dtype=torch.int32, device=device)
        for s in range(cfg.history_steps):
            for l in range(L):
                ft.resolve_slots(self.state, l, hd[s, l:l + 1], 65536, sl, nf, ff, fs)
        # fill the cache with its owners' blocks (one fetch over all slots)
        owner = self.state.slot_owner[: self.S]
        idx = torch.nonzero(owner >= 0).flatten().to(torch.int32)
        nfill = torch.tensor([idx.numel()], dtype=torch.int32, device=device)
        ft.fetch(self.pool_b, self.cache_b, nfill, owner[idx.long()].contiguous(), idx.contiguous())
        torch.cuda.synchronize()
        log(f"cache warmed ({int(idx.numel())} slots) from {cfg.history_steps} history steps in "
            f"{time.time() - t0:.1f}s")
        # per-step inputs: x ~ N(0,1) bf16 with feature 0 = 1.0 (the bias feature)
        self.x_host = step_inputs(cfg, T, n_steps)
        self.x_all = self.x_host.to(device)
        self.x_stage = torch.empty((L, T, H), dtype=torch.int16, device=device)
        self.out = torch.empty((L, T, H), dtype=torch.int16, device=device)
        # per-layer buffers
        self.ids = torch.empty((L, T, k), dtype=torch.int32, device=device)
        self.w = torch.empty((L, T, k), dtype=torch.float32, device=device)
        self.slot = torch.empty((L, T, k), dtype=torch.int32, device=device)
        self.nf = torch.zeros((L, 1), dtype=torch.int32, device=device)
        self.ml = T * k
        self.ff = torch.empty((L, self.ml), dtype=torch.int32, device=device)
        self.fs = torch.empty((L, self.ml), dtype=torch.int32, device=device)
        self.rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=device)
        self.ews = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, H, I, E), dtype=torch.uint8,
                               device=device)
        self.lws = torch.zeros(ft.decode_layer_workspace(T, k, H, I, E), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.fused = False

    def _init_resident(self, cfg, T, n_steps, device, log):
        """A cache holding every (layer, expert) block (flash: 24,576 x
        2,764,800 B = 67.9 GB of HBM): slot f holds flat id f, so the cache
        bank doubles as the pool (nothing is ever fetched) and the state is
        the identity map; no pinned pool, no history."""
        import torch

        import synth

        ft = self.ft
        L, E, k, H, I, g = cfg.L, cfg.E, cfg.k, cfg.H, cfg.I, cfg.g
        n_fid = L * E
        t0 = time.time()
        self.S = n_fid
        self.pool = None
        self.cache = torch.empty((n_fid, self.block), dtype=torch.uint8, device=device)
        for f0 in range(0, n_fid, 256):
            n = min(256, n_fid - f0)
            synth.bank_blocks_torch(cfg.seed, range(f0, f0 + n), cfg.fmt, H, I, g, self.cache[f0:f0 + n],
                                    ref_K=cfg.ref_K)
        torch.cuda.synchronize()
        ts = synth.tensor_scales(cfg.fmt, H, I, n_fid)
        self.tscale = None if ts is None else torch.from_numpy(ts).to(device)
        self.cache_b = ft.make_bank(cfg.fmt, H, I, g, self.cache, self.tscale)
        self.pool_b = self.cache_b
        self.W = torch.stack([torch.from_numpy(synth.router_weights(cfg.seed, l, E, H, cfg.router_std,
                                                                    zipf_bias=cfg.zipf))
                              for l in range(L)]).to(device)
        self.state = ft.DeviceCacheState(L, E, self.S, device=device)
        ident = torch.arange(n_fid, dtype=torch.int32, device=device)
        self.state.slot_owner[:n_fid].copy_(ident)
        self.state.map.copy_(ident)
        self.state.usage[:n_fid].zero_()
        self.state.recency.zero_()
        self.state.step.fill_(1)
        log(f"resident cache {n_fid} x {self.block} B ({n_fid * self.block / 1e9:.1f} GB) generated in "
            f"{time.time() - t0:.1f}s")
        self.x_host = step_inputs(cfg, T, n_steps)
        self.x_all = self.x_host.to(device)
        self.x_stage = torch.empty((L, T, H), dtype=torch.int16, device=device)
        self.out = torch.empty((L, T, H), dtype=torch.int16, device=device)
        self.ids = torch.empty((L, T, k), dtype=torch.int32, device=device)
        self.w = torch.empty((L, T, k), dtype=torch.float32, device=device)
        self.slot = torch.empty((L, T, k), dtype=torch.int32, device=device)
        self.nf = torch.zeros((L, 1), dtype=torch.int32, device=device)
        self.ml = T * k
        self.ff = torch.empty((L, self.ml), dtype=torch.int32, device=device)
        self.fs = torch.empty((L, self.ml), dtype=torch.int32, device=device)
        self.rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=device)
        self.ews = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, H, I, E), dtype=torch.uint8,
                               device=device)
        self.lws = torch.zeros(ft.decode_layer_workspace(T, k, H, I, E), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.fused = False

    # one pass of the hot path over all layers (enqueue only).  Fused: one
    # ft_moe_decode_layer kernel per layer.  Separate: route, resolve, fetch,
    # experts (two kernels) per layer.  `ev` holds per-layer events: 2 around
    # the layer kernel (fused) or the experts call (separate) of every
    # EXP_EVERY-th layer (an event node between kernels costs microseconds and
    # breaks the programmatic launch chain, so the timed graph samples), or
    # one around every op of every layer (per_op, the breakdown graph)
    EXP_EVERY = 8

    # the separate calls' router and resolve as one C call (ft_moe_route_resolve:
    # the top-k inside the resolve kernel); False: ft_moe_route + ft_moe_resolve_slots
    combined = True

    @property
    def OPS(self):
        if self.fused:
            return ["layer"]
        return ["route_resolve", "fetch", "experts"] if self.combined else ["route", "resolve", "fetch", "experts"]

    @property
    def KERNELS_PER_LAYER(self):
        return 1 if self.fused else 5

    def step(self, ev=None, per_op=False):
        ft, cfg, T = self.ft, self.cfg, self.T

        def mark(l, i, edge=None):
            # i: op boundary (per-op graph); edge: 0 / 1 = start / end of the
            # sampled kernel (timed graph)
            if ev is None:
                return
            if per_op:
                ev[l][i].record()
            elif edge is not None and l % self.EXP_EVERY == 0:
                ev[l // self.EXP_EVERY][edge].record()

        for l in range(cfg.L):
            if self.fused:
                mark(l, 0, edge=0)
                ft.decode_layer(self.x_stage[l], self.W[l], cfg.k, self.state, l, self.phi, self.cache_b,
                                self.pool_b, self.ids[l], self.w[l], self.slot[l], self.nf[l], self.ff[l],
                                self.fs[l], self.out[l], self.lws, dev_status=self.status)
                mark(l, 1, edge=1)
                continue
            mark(l, 0)
            if self.combined:
                ft.route_resolve(self.x_stage[l], self.W[l], cfg.k, self.ids[l], self.w[l], self.rws, self.state, l,
                                 self.phi, self.slot[l], self.nf[l], self.ff[l], self.fs[l], dev_status=self.status)
            else:
                ft.route(self.x_stage[l], self.W[l], cfg.k, self.ids[l], self.w[l], self.rws)
                mark(l, 1)
                ft.resolve_slots(self.state, l, self.ids[l], self.phi, self.slot[l], self.nf[l], self.ff[l],
                                 self.fs[l], self.status)
            n0 = 1 if self.combined else 2
            mark(l, n0)
            ft.fetch(self.pool_b, self.cache_b, self.nf[l], self.ff[l], self.fs[l], self.status)
            mark(l, n0 + 1, edge=0)
            ft.experts_fwd(self.cache_b, self.pool_b, l, cfg.E, self.x_stage[l], T, cfg.k, self.slot[l],
                           self.ids[l], self.w[l], self.out[l], self.ews, dev_status=self.status)
            mark(l, n0 + 2, edge=1)

    def use_fused(self, want: bool) -> bool:
        """Run the step as one fused kernel per layer when asked and the
        library accepts the shape (one eager layer call decides); else the
        separate calls."""
        self.fused = False
        if not want:
            return False
        import torch

        x0 = self.x_stage[0].clone()
        try:
            self.fused = True
            self.x_stage.copy_(self.x_all[0])
            self.step()
            torch.cuda.synchronize()
        except self.ft.FtError:
            self.fused = False
        self.x_stage[0].copy_(x0)
        return self.fused

    def capture(self):
        """Three graphs of one step: `graph` (timed) with no event inside (an
        event node between kernels breaks the programmatic launch chain),
        `graph_ev` with events around the layer kernel (fused) or the experts
        call (separate) of every EXP_EVERY-th layer (launch durations, replayed
        after the timed region), `graph_ops` with events around every op
        (breakdown).  Each recapture replaces the graphs and their events
        together."""
        import torch

        def events(n, rows):
            return [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(n)]
                    for _ in range(rows)]

        self.graph = self.graph_ev = self.graph_ops = None  # before their events go
        self.ev_exp = events(2, (self.cfg.L + self.EXP_EVERY - 1) // self.EXP_EVERY)
        self.ev_ops = events(len(self.OPS) + 1, self.cfg.L)
        self.x_stage.copy_(self.x_all[0])
        self.step()  # eager warm-up (attributes, lazy init) before capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        self.graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_ev):
            self.step(self.ev_exp)
        self.graph_ops = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_ops):
            self.step(self.ev_ops, per_op=True)
        torch.cuda.synchronize()

    def settle(self, steps: int, seed: int = 1):
        """Replay the step on `steps` fresh random token batches (generated on
        the device, untimed) so the slot cache reaches its steady state under
        the router's own routing before anything is timed: the seeded Zipf
        history that warmed it has the router's popularity but not its
        per-token draws, and the hit rate keeps improving for a few hundred
        steps after it."""
        import torch

        g = torch.Generator(device=self.dev)
        g.manual_seed(seed)
        xv = self.x_stage.view(torch.bfloat16)
        for _ in range(steps):
            xv.normal_(generator=g)
            xv[..., 0] = 1.0  # the router's bias feature
            self.graph.replay()
        torch.cuda.synchronize()

    def fresh_inputs(self, seed: int):
        """Refill the device copy of the per-step inputs with new tokens
        (N(0,1) bf16, feature 0 = 1.0), so that a further timed run meets
        tokens the cache has not adapted to."""
        import torch

        g = torch.Generator(device=self.dev)
        g.manual_seed(seed)
        xv = self.x_all.view(torch.bfloat16)
        xv.normal_(generator=g)
        xv[..., 0] = 1.0

    def fetch_rate(self, first: int, reps: int = 20):
        """Mean fetched experts and host-path pairs per step over `reps` replays
        on the inputs first.. (outside the timed region)."""
        import torch

        nf = hp = 0
        for i in range(reps):
            self.x_stage.copy_(self.x_all[(first + i) % self.x_all.shape[0]])
            self.graph.replay()
            nf += int(self.nf.sum().item())
            hp += int((self.slot < 0).sum().item())
        return nf / reps, hp / reps

    def experts_us(self, first: int = 0, reps: int = 5):
        """Device time (us) of one layer kernel (fused) or one experts call
        (separate: gate/up + down): the median over `reps` replays of the
        sampling graph (on inputs first..) of the mean over its sampled
        layers."""
        import torch

        runs = []
        for i in range(reps):
            self.x_stage.copy_(self.x_all[(first + i) % self.x_all.shape[0]])
            self.graph_ev.replay()
            torch.cuda.synchronize()
            runs.append(sum(e[0].elapsed_time(e[1]) for e in self.ev_exp) * 1e3 / len(self.ev_exp))
        return statistics.median(runs)

    def op_times(self, first: int, reps: int = 5):
        """Per-op device time (us per step, summed over layers): the median of
        a few replays of the per-op graph on fresh inputs (steps first, ...),
        outside the timed region."""
        import torch

        names = self.OPS
        runs = []
        for i in range(reps):
            self.x_stage.copy_(self.x_all[(first + i) % self.x_all.shape[0]])
            self.graph_ops.replay()
            torch.cuda.synchronize()
            tot = {n: 0.0 for n in names}
            for ev in self.ev_ops:
                for j, n in enumerate(names):
                    tot[n] += ev[j].elapsed_time(ev[j + 1]) * 1e3
            runs.append(tot)
        return {n: statistics.median(r[n] for r in runs) for n in names}

    def distinct_expert_bytes(self):
        """Algorithmic expert bytes of the last step: distinct experts per layer
        (cache and pool reads alike) x block bytes."""
        ids = self.ids.cpu().numpy()
        return sum(len(set(ids[l].ravel().tolist())) for l in range(self.cfg.L)) * self.block

    def fetch_bytes(self):
        return int(self.nf.sum().item()) * self.block

    def misses(self):
        sl = self.slot.cpu().numpy()
        return int(self.nf.sum().item()), int((sl < 0).sum())


def time_device(wl, steps: int, warmup: int, reduce_fn, world: int, clocks=None, first: int = 0):
    """Device time of `steps` replays of the captured step on inputs
    first+warmup.. (after `warmup` untimed replays on inputs first..)."""
    import torch

    s = torch.cuda.current_stream()
    n_in = wl.x_all.shape[0]
    for i in range(warmup):
        wl.x_stage.copy_(wl.x_all[(first + i) % n_in])
        wl.graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.cudart().cudaProfilerStart()  # a profiler started with --profile-from-start off sees only this
    e0.record(s)
    for i in range(steps):
        wl.x_stage.copy_(wl.x_all[(first + warmup + i) % n_in])
        wl.graph.replay()
    e1.record(s)
    torch.cuda.synchronize()
    torch.cuda.cudart().cudaProfilerStop()
    if clocks:
        clocks.stop()
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    return e0.elapsed_time(e1) / 1e3


def time_e2e(wl, steps: int, warmup: int):
    """Host buffers in, host buffers out: pinned H2D of the step's inputs,
    graph replay, D2H of the step's outputs, all inside the timed region.
    Uses the inputs after those of the device-timed run (fresh tokens, so
    the cache sees as many misses as there)."""
    import torch

    out_host = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()
    s = torch.cuda.current_stream()
    first = warmup + steps
    n_in = wl.x_host.shape[0]
    for i in range(warmup):
        wl.x_stage.copy_(wl.x_host[i % n_in], non_blocking=True)
        wl.graph.replay()
        out_host.copy_(wl.out, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(steps):
        wl.x_stage.copy_(wl.x_host[(first + i) % n_in], non_blocking=True)
        wl.graph.replay()
        out_host.copy_(wl.out, non_blocking=True)
    e1.record(s)
    torch.cuda.synchronize()
    h2d = wl.x_stage.numel() * wl.x_stage.element_size()
    d2h = wl.out.numel() * wl.out.element_size()
    return e0.elapsed_time(e1) / 1e3, h2d, d2h


# --------------------------------------------------------------- the oracle --
class OracleLayer:
    """The CPU oracle on the same decode workload: route, resolve, fetch (a
    copy) and the fp64 experts for one layer call."""

    def __init__(self, cfg, T: int, phi: int, layers=(0, 1)):
        import oracle
        import synth

        self.o, self.cfg, self.T, self.phi = oracle, cfg, T, phi
        L, E, k, H, I, g = cfg.L, cfg.E, cfg.k, cfg.H, cfg.I, cfg.g
        self.layers = list(layers)
        _, self.stride = synth.block_layout(cfg.fmt, H, I, g)
        # pool slice for the sampled layers, as the oracle reads it (flat ids)
        import torch

        self.blocks = {}
        for l in self.layers:
            blk = torch.empty((E, self.stride), dtype=torch.uint8)
            synth.bank_blocks_torch(cfg.seed, range(l * E, (l + 1) * E), cfg.fmt, H, I, g, blk, ref_K=cfg.ref_K)
            for e in range(E):
                self.blocks[l * E + e] = blk[e].numpy()
        self.W = {l: synth.router_weights(cfg.seed, l, E, H, cfg.router_std, zipf_bias=cfg.zipf)
                  for l in self.layers}
        self.st = oracle.CacheState(L, E, cfg.slots)
        hist = synth.zipf_history(cfg.seed, L, E, k, cfg.history_steps)
        for s in range(cfg.history_steps):
            for l in range(L):
                oracle.resolve(self.st, l, hist[s, l:l + 1], 65536, k)
        xs = synth.normal_bf16(synth.stream_key(cfg.seed, "bench-x", T), (64, L, T, H))
        xs[..., 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
        self.xs = xs
        self.ts = synth.tensor_scales(cfg.fmt, H, I, L * E)

    def layer_call(self, i: int):
        cfg, o = self.cfg, self.o
        l = self.layers[i % len(self.layers)]
        x = self.xs[i % self.xs.shape[0], l]
        ids, w = o.route(x, self.W[l], cfg.k)
        sl, nf, ff, fs = o.resolve(self.st, l, ids, self.phi)
        out = np.zeros((self.T, cfg.H))
        xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        for t in range(self.T):
            for j in range(cfg.k):
                f = l * cfg.E + int(ids[t, j])
                y = o.expert(self.blocks[f], cfg.fmt, cfg.H, cfg.I, cfg.g, xv[t],
                             None if self.ts is None else self.ts[f])
                out[t] += float(np.float32(w[t, j])) * y
        return out


def oracle_rate(cfg, T, phi, budget_s: float = 15.0, min_calls: int = 2, max_calls: int = 10 ** 6):
    ol = OracleLayer(cfg, T, phi)
    t0 = time.perf_counter()
    n = 0
    while n < min_calls or (time.perf_counter() - t0 < budget_s and n < max_calls):
        ol.layer_call(n)
        n += 1
    dt = time.perf_counter() - t0
    return T * n / dt, n, dt


def run_reference(args, cfg, T):
    """The CPU oracle as the reference arm: each step one layer call for T tokens."""
    import oracle

    oracle.build()
    ol = OracleLayer(cfg, T, args.phi)
    for i in range(args.warmup):
        ol.layer_call(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        ol.layer_call(args.warmup + i)
    dt = time.perf_counter() - t0
    value = T * args.steps / dt
    sample = f"{args.steps} single-layer calls of {T} token(s) on layers {ol.layers} (of {cfg.L})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name} decode (35B-A3B-shaped int4 g64, 40x256 experts, top-8, "
                               f"H2048, I512), T={T}, phi={args.phi}",
                   "parallelism": "replicas" if args.gpus > 1 else "single"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------- host link and q* cap -----
def host_link_bench(wl, log=print, reps: int = 3):
    """The host link's copy rate (one 1 GiB cudaMemcpyAsync from the pinned
    pool to the device, best of `reps`) and the fetch kernel's rate moving 64
    cached experts from the pool into the slots that already hold them (the
    same bytes, so the cache stays consistent)."""
    import torch

    if wl.pool is None:
        return None
    ft = wl.ft
    nb = min(wl.pool.shape[0], (1 << 30) // wl.pool.shape[1])
    src = wl.pool[:nb]
    dst = torch.empty(src.shape, dtype=torch.uint8, device=wl.dev)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        best = t if best is None else min(best, t)
    copy_gbs = src.numel() / best / 1e9
    del dst
    owner = wl.state.slot_owner[: wl.S]
    slots = torch.nonzero(owner >= 0).flatten()[:64].to(torch.int32)
    n = int(slots.numel())
    fetch_gbs = None
    if n:
        fids = owner[slots.long()].contiguous()
        nf = torch.tensor([n], dtype=torch.int32, device=wl.dev)
        ft.fetch(wl.pool_b, wl.cache_b, nf, fids, slots.contiguous())  # warm-up
        torch.cuda.synchronize()
        bestf = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ft.fetch(wl.pool_b, wl.cache_b, nf, fids, slots.contiguous())
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1e3
            bestf = t if bestf is None else min(bestf, t)
        fetch_gbs = n * wl.block / bestf / 1e9
    res = {"h2d_copy_GBs": copy_gbs, "h2d_copy_bytes": int(src.numel()),
           "fetch_kernel_GBs": fetch_gbs, "fetch_experts": n,
           "fetch_frac_of_copy": (fetch_gbs / copy_gbs) if fetch_gbs else None,
           "how": "one pinned-host -> device cudaMemcpyAsync of 1 GiB of the pool (best of 3); ft_moe_fetch of "
                  "64 cached experts onto their own slots (best of 3), CUDA events"}
    log(f"host link: copy {copy_gbs:.1f} GB/s, fetch kernel {fetch_gbs} GB/s")
    return res


def phi_bench(wl, phi: int, args, units, reduce_fn, world, log=print):
    """The same decode step with the q* split capping the fetches at
    frac_q16 = phi: the capped misses stay on the host path (the experts read
    them in place from the pinned pool).  Timed like the headline line after
    the cache settles under the new split."""
    import torch

    old = wl.phi
    wl.phi = phi
    wl.use_fused(args.layer_kernel == "fused")
    wl.fresh_inputs(2000 + phi)
    wl.capture()
    wl.settle(max(64, args.settle // 4), seed=2)
    secs = time_device(wl, args.steps, args.warmup, reduce_fn, world, None)
    value, secs_max, _ = aggregate(units, secs, world, reduce_fn)
    nfetch, host_pairs = wl.fetch_rate(first=args.warmup + 2 * args.steps + 5)
    st = wl.ft.get_status(wl.status)
    wl.phi = old
    if st != 0:
        raise RuntimeError(f"device status {st} during the phi={phi} benchmark")
    log(f"phi={phi}: {value:.1f} {UNIT}, {secs_max / args.steps * 1e3:.3f} ms/step, {nfetch:.2f} fetched and "
        f"{host_pairs:.2f} host-path pairs per step")
    torch.cuda.synchronize()
    return {"frac_q16": phi, "value": value, "unit": UNIT, "ms_per_step": secs_max / args.steps * 1e3,
            "fused": wl.fused, "fetched_experts_per_step": nfetch, "host_path_pairs_per_step": host_pairs,
            "launch_us": wl.experts_us()}


# ------------------------------------------------------- flash decode -----
def host_mem_available() -> int:
    """MemAvailable of this host in bytes (0 when unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def flash_bench(steps: int, warmup: int, device, log=print, cache_frac: float = 1.0):
    """The NVFP4 decode step of the flash config (48 layers x 512 experts,
    top-10, H 2560, I 640, 2,764,800 B per expert block), one token per step,
    captured in one CUDA graph; the same timing as the headline decode line.
    cache_frac 1: every expert resident in HBM (67.9 GB), nothing is ever
    fetched; below 1: a slot cache of that fraction of the 24,576 (layer,
    expert) pairs in HBM and the whole pool in pinned host memory, the cache
    settled under the step's own routing before timing."""
    import dataclasses

    import torch

    import synth

    cfg = synth.get_config("flash")
    if cache_frac < 1.0:
        cfg = dataclasses.replace(cfg, slots=int(round(cache_frac * cfg.L * cfg.E)))
    n_steps = warmup + steps + 5 + 20
    wl = DecodeWorkload(cfg, 1, 65536, n_steps, device, log)
    fused = wl.use_fused(True)
    wl.capture()
    wl.settle(8 if cache_frac >= 1.0 else 128)
    secs = time_device(wl, steps, warmup, None, 1)
    nfetch, host_pairs = wl.fetch_rate(first=warmup + steps + 5)
    exp_us = wl.experts_us()
    ebytes = wl.distinct_expert_bytes()
    st = wl.ft.get_status(wl.status)
    if st != 0:
        raise RuntimeError(f"device status {st} during the flash decode benchmark")
    per_call = ebytes / cfg.L + (cfg.E * cfg.H * 4 if fused else 0)
    where = ("every expert resident (67.9 GB)" if cache_frac >= 1.0 else
             f"cache {cfg.slots} slots ({cache_frac:.0%} of 24,576) in HBM, pool in pinned host memory")
    res = {"workload": "flash-shaped NVFP4 decode: 48 layers x 512 experts, top-10, H2560, I640 "
                       f"(2,764,800 B/expert), {where}, T=1",
           "value": cfg.L * steps / secs, "unit": UNIT, "ms_per_step": secs / steps * 1e3,
           "fetched_experts_per_step": nfetch, "host_path_pairs_per_step": host_pairs,
           "model_tokens_per_s": steps / secs, "fused": fused,
           "launch_us": exp_us, "bytes_per_launch": per_call,
           "kernel": "ft_moe_decode_layer (expert + router bytes)" if fused else
                     "ft_moe_experts_fwd decode (expert bytes)",
           "experts_traffic_per_call": None if fused else FLASH_TRAFFIC_PER_CALL,
           "experts_GBs": per_call / (exp_us * 1e-6) / 1e9 if exp_us else None}
    log(f"flash T=1 cache {cache_frac:.0%}: {res['value']:.1f} {UNIT}, {res['ms_per_step']:.3f} ms/step, "
        f"{'layer kernel' if fused else 'experts'} {exp_us:.1f} us/call, {nfetch:.1f} fetched/step")
    del wl
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ prefill -----
def prefill_bench(T: int, steps: int, warmup: int, device, log=print, state=None):
    """One prefill MoE layer of the prefill config (NVFP4, H 4096, I 2048,
    256 experts, top-6): route -> permute (f16 gather) -> grouped SwiGLU
    experts on tcgen05 -> combine, for T prompt tokens, the whole layer's
    experts resident in the cache bank.  Returns the layer time, the grouped
    GEMM (experts call) time and its TFLOP/s; all inputs resident in HBM."""
    import torch

    import quantized_expert_ffn_router_gb300 as ft
    import synth

    cfg = synth.get_config("prefill")
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    if state is None:
        _, stride = synth.block_layout(cfg.fmt, H, I, cfg.g)
        bank = torch.empty((E, stride), dtype=torch.uint8, device=device)
        for e0 in range(0, E, 32):
            synth.bank_blocks_torch(cfg.seed, range(e0, min(E, e0 + 32)), cfg.fmt, H, I, cfg.g, bank[e0:e0 + 32])
        ts = torch.from_numpy(synth.tensor_scales(cfg.fmt, H, I, E)).to(device)
        W = torch.from_numpy(synth.router_weights(cfg.seed, 0, E, H, cfg.router_std)).to(device)
        state = dict(bank=bank, ts=ts, W=W, cb=ft.make_bank(cfg.fmt, H, I, cfg.g, bank, ts),
                     slot=torch.arange(E, dtype=torch.int32, device=device))
    n = T * k
    x = torch.from_numpy(synth.normal_bf16(synth.stream_key(cfg.seed, "prefill-bench-x", T), (T, H))
                         .view(np.int16)).to(device)
    ids = torch.empty((T, k), dtype=torch.int32, device=device)
    w = torch.empty((T, k), dtype=torch.float32, device=device)
    rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=device)
    perm = torch.empty(n, dtype=torch.int32, device=device)
    inv = torch.empty((T, k), dtype=torch.int32, device=device)
    off = torch.empty(E + 1, dtype=torch.int32, device=device)
    xp = torch.empty((n, H), dtype=torch.int16, device=device)
    xs = torch.empty(n, dtype=torch.float32, device=device)
    pws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=device)
    yp = torch.empty((n, H), dtype=torch.int16, device=device)
    ews = torch.empty(ft.experts_workspace(ft.FT_PREFILL, T, k, H, I, E), dtype=torch.uint8, device=device)
    out = torch.empty((T, H), dtype=torch.int16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]

    def layer(timed):
        # events between the ops (timed) break their programmatic overlap: the
        # layer time comes from the loop without them
        if timed:
            ev[0].record()
        ft.route(x, state["W"], k, ids, w, rws)
        if timed:
            ev[1].record()
        ft.permute(ids, E, x, perm, inv, off, xp, pws, dev_status=status, xp_scale=xs)
        if timed:
            ev[2].record()
        ft.experts_fwd(state["cb"], None, 0, E, xp, T, k, state["slot"], None, None, yp, ews,
                       mode=ft.FT_PREFILL, offsets=off, dev_status=status, x_scale=xs)
        if timed:
            ev[3].record()
        ft.combine(yp, inv, w, out)
        if timed:
            ev[4].record()

    for _ in range(warmup):
        layer(False)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        layer(False)
    e1.record()
    torch.cuda.synchronize()
    layer_ms = e0.elapsed_time(e1) / steps
    # each op's interval, one step at a time
    per_op = {"route": [], "permute": [], "grouped_gemm": [], "combine": []}
    for _ in range(steps):
        layer(True)
        torch.cuda.synchronize()
        for i, name in enumerate(per_op):
            per_op[name].append(ev[i].elapsed_time(ev[i + 1]))
    if ft.get_status(status) != 0:
        raise RuntimeError(f"device status {ft.get_status(status)} in prefill")
    flops = 6.0 * H * I * T * k
    gm = statistics.median(per_op["grouped_gemm"])
    res = {"T": T, "layer_ms": layer_ms, "layer_tokens_per_s": T / (layer_ms * 1e-3),
           "grouped_gemm_ms": gm, "grouped_gemm_tflops": flops / (gm * 1e-3) / 1e12,
           "weight_bytes": int(state["bank"].numel()), "flops": flops,
           "per_op_ms": {name: statistics.median(v) for name, v in per_op.items()},
           "per_op_timing": "events around each op, one step at a time (median); the layer time has no events inside"}
    po = res["per_op_ms"]
    log(f"prefill T={T}: layer {layer_ms:.3f} ms, grouped GEMM {gm:.3f} ms = {res['grouped_gemm_tflops']:.0f} TFLOP/s; "
        f"route {po['route']:.3f}, permute {po['permute']:.3f}, combine {po['combine']:.3f} ms")
    return res, state


def prefill_pipeline_bench(T: int, n_layers: int, device, log=print, reps: int = 4):
    """Prefill of n_layers consecutive layers of the prefill config with the
    experts streamed from pinned host memory through the whole-layer double
    buffer (pipeline.PrefillLayers: each layer copied by the copy engine into
    one half of the cache's first 2E slots while the previous layer computes).
    Returns the time per layer, the time of one layer's copy alone, and the
    host-link rate they imply."""
    import torch

    import quantized_expert_ffn_router_gb300 as ft
    import synth
    from quantized_expert_ffn_router_gb300.pipeline import PrefillLayers

    cfg = synth.get_config("prefill")
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    _, stride = synth.block_layout(cfg.fmt, H, I, cfg.g)
    t0 = time.time()
    pool = torch.empty((n_layers * E, stride), dtype=torch.uint8).pin_memory()
    tmp = torch.empty((32, stride), dtype=torch.uint8, device=device)
    for f0 in range(0, n_layers * E, 32):
        synth.bank_blocks_torch(cfg.seed, range(f0, f0 + 32), cfg.fmt, H, I, cfg.g, tmp)
        pool[f0:f0 + 32].copy_(tmp)
    del tmp
    torch.cuda.synchronize()
    log(f"prefill pool: {n_layers} layers x {E} experts ({pool.numel() / 1e9:.1f} GB pinned) in {time.time() - t0:.1f}s")
    ts = torch.from_numpy(synth.tensor_scales(cfg.fmt, H, I, n_layers * E)).to(device)
    cache = torch.empty((2 * E, stride), dtype=torch.uint8, device=device)
    pb = ft.make_bank(cfg.fmt, H, I, cfg.g, pool, ts)
    cb = ft.make_bank(cfg.fmt, H, I, cfg.g, cache, ts)
    state = ft.DeviceCacheState(n_layers, E, 2 * E, device=device)
    xs = [torch.from_numpy(synth.normal_bf16(synth.stream_key(cfg.seed, "prefill-pipe-x", T, l), (T, H))
                           .view(np.int16)).to(device) for l in range(n_layers)]
    Ws = [torch.from_numpy(synth.router_weights(cfg.seed, l, E, H, cfg.router_std)).to(device)
          for l in range(n_layers)]
    outs = [torch.empty((T, H), dtype=torch.int16, device=device) for _ in range(n_layers)]
    pl = PrefillLayers(state, cb, pb, E, k, T, device=device)
    layers = list(range(n_layers))
    pl(layers, xs, Ws, outs)  # warm-up (kernel attributes, tensor maps)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_layer = []
    for _ in range(reps):
        e0.record()
        pl(layers, xs, Ws, outs)
        e1.record()
        torch.cuda.synchronize()
        per_layer.append(e0.elapsed_time(e1) / n_layers)
    copy_ms = []
    for l in range(n_layers):
        e0.record()
        ft.fetch_layer(pb, cb, l, E, 0)
        e1.record()
        torch.cuda.synchronize()
        copy_ms.append(e0.elapsed_time(e1))
    if ft.get_status(pl.status) != 0:
        raise RuntimeError(f"device status {ft.get_status(pl.status)} in the prefill pipeline")
    layer_bytes = E * stride
    res = {"T": T, "layers": n_layers, "ms_per_layer": min(per_layer),
           "tokens_per_s_per_layer": T / (min(per_layer) * 1e-3),
           "layer_copy_ms": statistics.median(copy_ms), "layer_bytes": layer_bytes,
           "host_link_GBs": layer_bytes / (statistics.median(copy_ms) * 1e-3) / 1e9}
    log(f"prefill pipeline T={T}: {res['ms_per_layer']:.2f} ms/layer, one layer's copy {res['layer_copy_ms']:.2f} ms "
        f"({res['host_link_GBs']:.0f} GB/s)")
    return res


# ----------------------------------------------------- small cases for ncu --
def kernel_case(name: str, T: int):
    """A small standalone workload for kernel profiling: a few calls of one
    kernel family on a bank that fits in a few GB (no pool, no history).
      decode:  ft_moe_experts_fwd decode on the d35b or flash shape, fresh
               random experts each call (nothing reused in L2);
      decode-step: the whole decode layer on two d35b-shaped layers over a
               128-slot cache, as separate calls and as the fused kernel;
      prefill-layer: route, permute, grouped experts and combine of one
               prefill layer (256 experts resident, --tokens, default 2048);
      prefill: permute + ft_moe_experts_fwd prefill, NVFP4 H 4096 I 2048,
               16 experts, top-6, 512 tokens (or --tokens >= 16)."""
    import torch

    import quantized_expert_ffn_router_gb300 as ft
    import synth
    from quantized_expert_ffn_router_gb300 import build as ftbuild

    ftbuild.build()
    ft.load()
    dev = "cuda"
    rng = np.random.default_rng(0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if name in ("decode", "decode-flash"):
        cfg = synth.get_config("d35b" if name == "decode" else "flash")
        E, k = cfg.E, cfg.k
        _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
        bank = torch.empty((2 * E, stride), dtype=torch.uint8, device=dev)
        synth.bank_blocks_torch(0, range(2 * E), cfg.fmt, cfg.H, cfg.I, cfg.g, bank, ref_K=cfg.ref_K)
        ts = synth.tensor_scales(cfg.fmt, cfg.H, cfg.I, cfg.L * E)
        cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, bank, None if ts is None else torch.from_numpy(ts).to(dev))
        w = torch.full((T, k), 0.1, device=dev)
        x = torch.from_numpy(synth.normal_bf16(1, (T, cfg.H)).view(np.int16)).to(dev)
        out = torch.empty((T, cfg.H), device=dev)
        ws = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, cfg.H, cfg.I, E), dtype=torch.uint8, device=dev)
        # evict the bank generation's dirty lines so DRAM counters see only the calls
        scratch = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        scratch.zero_()
        scratch.sum()
        torch.cuda.synchronize()
        for c in range(3):
            ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
            slots = torch.from_numpy(ids + (c % 2) * E).to(dev)
            ft.experts_fwd(cb, None, 0, E, x, T, k, slots, torch.from_numpy(ids).to(dev), w, out, ws,
                           dev_status=status)
    elif name == "decode-step":
        # two d35b-shaped layers (256 experts, top-8, H 2048, I 512, int4 g64)
        # over a 128-slot cache, half filled: 4 steps of the separate calls
        # (route, resolve, fetch, experts) then 4 of the fused layer kernel,
        # on fresh tokens (misses, fetches and host-path pairs included)
        cfg = synth.get_config("d35b")
        L, E, k, H, I, g, S = 2, cfg.E, cfg.k, cfg.H, cfg.I, cfg.g, 128
        _, stride = synth.block_layout(cfg.fmt, H, I, g)
        pool = torch.empty((L * E, stride), dtype=torch.uint8).pin_memory()
        tmp = torch.empty((64, stride), dtype=torch.uint8, device=dev)
        for f0 in range(0, L * E, 64):
            synth.bank_blocks_torch(cfg.seed, range(f0, f0 + 64), cfg.fmt, H, I, g, tmp, ref_K=cfg.ref_K)
            pool[f0:f0 + 64].copy_(tmp)
        cache = torch.empty((S, stride), dtype=torch.uint8, device=dev)
        st = ft.DeviceCacheState(L, E, S, device=dev)
        fids = torch.from_numpy(rng.choice(L * E, S // 2, replace=False).astype(np.int32)).to(dev)
        slots = torch.arange(S // 2, dtype=torch.int32, device=dev)
        st.slot_owner[: S // 2].copy_(fids)
        st.map[fids.long()] = slots
        st.usage[: S // 2].copy_(torch.arange(S // 2, dtype=torch.int64, device=dev))
        st.step.fill_(S)
        pb, cb = ft.make_bank(cfg.fmt, H, I, g, pool), ft.make_bank(cfg.fmt, H, I, g, cache)
        ft.fetch(pb, cb, torch.tensor([S // 2], dtype=torch.int32, device=dev), fids, slots)
        Ws = [torch.from_numpy(synth.router_weights(cfg.seed, l, E, H, cfg.router_std, zipf_bias=cfg.zipf)).to(dev)
              for l in range(L)]
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        sl = torch.empty((T, k), dtype=torch.int32, device=dev)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        ff = torch.empty(T * k, dtype=torch.int32, device=dev)
        fs = torch.empty(T * k, dtype=torch.int32, device=dev)
        out = torch.empty((T, H), dtype=torch.int16, device=dev)
        rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=dev)
        ews = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, H, I, E), dtype=torch.uint8, device=dev)
        lws = torch.zeros(ft.decode_layer_workspace(T, k, H, I, E), dtype=torch.uint8, device=dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(5)
        x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        for fused in (False, True):
            for step in range(4):
                for l in range(L):
                    x.normal_(generator=gen)
                    x[:, 0] = 1.0
                    xi = x.view(torch.int16)
                    if fused:
                        ft.decode_layer(xi, Ws[l], k, st, l, 65536, cb, pb, ids, w, sl, nf, ff, fs, out, lws,
                                        dev_status=status)
                    else:
                        ft.route(xi, Ws[l], k, ids, w, rws)
                        ft.resolve_slots(st, l, ids, 65536, sl, nf, ff, fs, status)
                        ft.fetch(pb, cb, nf, ff, fs, status)
                        ft.experts_fwd(cb, pb, l, E, xi, T, k, sl, ids, w, out, ews, dev_status=status)
    elif name == "prefill":
        # --tokens 128: ~48 rows per expert (the 2048-token layer's regime);
        # 512 (the default): ~192 rows per expert (the 8192-token layer's)
        H, I, E, k = 4096, 2048, 16, 6
        Tp = T if T >= 16 else 512
        _, stride = synth.block_layout(synth.gen.FMT_NVFP4, H, I, 16)
        bank = torch.empty((E, stride), dtype=torch.uint8, device=dev)
        synth.bank_blocks_torch(0, range(E), synth.gen.FMT_NVFP4, H, I, 16, bank)
        ts = torch.from_numpy(synth.tensor_scales(synth.gen.FMT_NVFP4, H, I, E)).to(dev)
        cb = ft.make_bank(synth.gen.FMT_NVFP4, H, I, 16, bank, ts)
        ids = torch.from_numpy(np.stack([rng.choice(E, k, replace=False) for _ in range(Tp)]).astype(np.int32)).to(dev)
        x = torch.from_numpy(synth.normal_bf16(1, (Tp, H)).view(np.int16)).to(dev)
        n = Tp * k
        perm = torch.empty(n, dtype=torch.int32, device=dev)
        inv = torch.empty((Tp, k), dtype=torch.int32, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        xp = torch.empty((n, H), dtype=torch.int16, device=dev)
        xs = torch.empty(n, device=dev)
        pws = torch.empty(ft.permute_workspace(Tp, k, E), dtype=torch.uint8, device=dev)
        yp = torch.empty((n, H), dtype=torch.int16, device=dev)
        ews = torch.empty(ft.experts_workspace(ft.FT_PREFILL, Tp, k, H, I, E), dtype=torch.uint8, device=dev)
        slot = torch.arange(E, dtype=torch.int32, device=dev)
        ft.permute(ids, E, x, perm, inv, off, xp, pws, dev_status=status, xp_scale=xs)
        for _ in range(2):
            ft.experts_fwd(cb, None, 0, E, xp, Tp, k, slot, None, None, yp, ews, mode=ft.FT_PREFILL,
                           offsets=off, dev_status=status, x_scale=xs)
    elif name == "prefill-layer":
        # one whole prefill layer at the benchmark's shape (NVFP4, H 4096,
        # I 2048, 256 experts resident, top-6) for --tokens (default 2048)
        # tokens: route (tiled logits + top-k), permute, grouped experts,
        # combine; twice
        cfg = synth.get_config("prefill")
        H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
        Tp = T if T >= 16 else 2048
        _, stride = synth.block_layout(cfg.fmt, H, I, cfg.g)
        bank = torch.empty((E, stride), dtype=torch.uint8, device=dev)
        synth.bank_blocks_torch(cfg.seed, range(E), cfg.fmt, H, I, cfg.g, bank)
        ts = torch.from_numpy(synth.tensor_scales(cfg.fmt, H, I, E)).to(dev)
        cb = ft.make_bank(cfg.fmt, H, I, cfg.g, bank, ts)
        W = torch.from_numpy(synth.router_weights(cfg.seed, 0, E, H, cfg.router_std)).to(dev)
        x = torch.from_numpy(synth.normal_bf16(synth.stream_key(cfg.seed, "prefill-x", Tp), (Tp, H)).view(np.int16)).to(dev)
        n = Tp * k
        ids = torch.empty((Tp, k), dtype=torch.int32, device=dev)
        w = torch.empty((Tp, k), dtype=torch.float32, device=dev)
        rws = torch.zeros(ft.route_workspace(Tp, E, H), dtype=torch.uint8, device=dev)
        perm = torch.empty(n, dtype=torch.int32, device=dev)
        inv = torch.empty((Tp, k), dtype=torch.int32, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        xp = torch.empty((n, H), dtype=torch.int16, device=dev)
        xs = torch.empty(n, device=dev)
        pws = torch.empty(ft.permute_workspace(Tp, k, E), dtype=torch.uint8, device=dev)
        yp = torch.empty((n, H), dtype=torch.int16, device=dev)
        out = torch.empty((Tp, H), dtype=torch.int16, device=dev)
        ews = torch.empty(ft.experts_workspace(ft.FT_PREFILL, Tp, k, H, I, E), dtype=torch.uint8, device=dev)
        slot = torch.arange(E, dtype=torch.int32, device=dev)
        for _ in range(2):
            ft.route(x, W, k, ids, w, rws)
            ft.permute(ids, E, x, perm, inv, off, xp, pws, dev_status=status, xp_scale=xs)
            ft.experts_fwd(cb, None, 0, E, xp, Tp, k, slot, None, None, yp, ews, mode=ft.FT_PREFILL,
                           offsets=off, dev_status=status, x_scale=xs)
            ft.combine(yp, inv, w, out)
    else:
        raise SystemExit(f"unknown case {name}")
    torch.cuda.synchronize()
    if ft.get_status(status) != 0:
        raise RuntimeError(f"device status {ft.get_status(status)}")
    print("ok", flush=True)


# ---------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--tokens", type=int, default=1, help="decode batch (1 or 8)")
    ap.add_argument("--phi", type=int, default=65536, help="frac_q16 of the q* split")
    ap.add_argument("--settle", type=int, default=512,
                    help="untimed steps on fresh tokens before timing, so the cache reaches steady state")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-batch", type=int, default=8, help="also time this batch (0: off)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill layer measurement")
    ap.add_argument("--no-flash", action="store_true", help="skip the NVFP4 (flash) decode measurement")
    ap.add_argument("--prefill-layers", type=int, default=3,
                    help="layers streamed from host memory through the prefill double buffer (0: skip)")
    ap.add_argument("--route-resolve", choices=["combined", "separate"], default="combined",
                    help="the separate-calls step's router and resolve: ft_moe_route_resolve, or the two calls")
    ap.add_argument("--layer-kernel", choices=["fused", "separate"], default="separate",
                    help="decode step as the separate route / resolve / fetch / experts calls (measured faster) or "
                         "as one ft_moe_decode_layer kernel per layer (when the shape fits); the other form is "
                         "timed too and reported in detail")
    ap.add_argument("--case", choices=["decode", "decode-flash", "decode-step", "prefill", "prefill-layer"],
                    help="run a small kernel case for a profiler instead of the benchmark")
    args = ap.parse_args()
    if args.case:
        kernel_case(args.case, args.tokens)
        return
    if args.warmup < 3:
        args.warmup = 3

    import synth

    cfg = synth.get_config("d35b")
    world, rank, local = dist_info()
    log = (lambda *a: print(*a, file=sys.stderr, flush=True)) if rank == 0 else (lambda *a: None)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, cfg, args.tokens)
        return

    import torch

    import quantized_expert_ffn_router_gb300 as ft

    from quantized_expert_ffn_router_gb300 import build as ftbuild

    ftbuild.build()
    ft.load()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    reduce_fn = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
        reduce_fn = torch_reduce_fn(device)

    # device-timed steps, e2e steps, per-op breakdown, fetch statistics
    n_steps = args.warmup + 2 * args.steps + 5 + 20
    results = {}
    batches = [args.tokens] + ([args.extra_batch] if args.extra_batch and args.extra_batch != args.tokens else [])
    wl = None
    for bi, T in enumerate(batches):
        if wl is None:
            wl = DecodeWorkload(cfg, T, args.phi, n_steps, device, log)
        else:
            wl = reshape_workload(wl, T, n_steps)
        wl.combined = args.route_resolve == "combined"
        fused = wl.use_fused(args.layer_kernel == "fused")
        wl.capture()
        wl.settle(args.settle)
        clocks = ClockSampler(local) if bi == 0 else None
        secs = time_device(wl, args.steps, args.warmup, reduce_fn, world, clocks)
        units = T * cfg.L * args.steps
        value, secs_max, units_all = aggregate(units, secs, world, reduce_fn)
        exp_us = wl.experts_us()
        ebytes = wl.distinct_expert_bytes()
        kt = None
        nfetch, host_pairs = wl.fetch_rate(first=args.warmup + 2 * args.steps + 5)
        e2e_secs, h2d, d2h = time_e2e(wl, args.steps, args.warmup)
        kt = wl.op_times(first=args.warmup + 2 * args.steps)
        e2e_val, _, _ = aggregate(units, e2e_secs, world, reduce_fn)
        results[T] = dict(value=value, secs=secs_max, kt=kt, exp_us=exp_us, ebytes=ebytes, nfetch=nfetch,
                          host_pairs=host_pairs, e2e=e2e_val, h2d=h2d, d2h=d2h,
                          clocks=clocks.summary() if clocks else None, fused=fused, combined=wl.combined,
                          kernels_per_layer=wl.KERNELS_PER_LAYER)
        st = ft.get_status(wl.status)
        if st != 0:
            raise RuntimeError(f"device status {st} during the benchmark")
        log(f"T={T}: {value:.1f} {UNIT}, {secs_max / args.steps * 1e3:.3f} ms/step, "
            f"{'fused' if fused else 'separate'}, kernels {kt}")
        # the same step in the other form (one fused kernel per layer, or the
        # separate calls), timed the same way after the headline runs
        if wl.use_fused(not fused) != fused:
            wl.fresh_inputs(1000 + T)
            wl.capture()
            wl.settle(max(32, args.settle // 8), seed=3)
            secs_o = time_device(wl, args.steps, args.warmup, reduce_fn, world, None)
            v_o, s_o, _ = aggregate(units, secs_o, world, reduce_fn)
            results[T]["other_form"] = {"form": "fused" if wl.fused else "separate", "value": v_o,
                                        "ms_per_step": s_o / args.steps * 1e3,
                                        "us_per_layer": s_o / args.steps / cfg.L * 1e6,
                                        "launch_us_sampled": wl.experts_us(),
                                        "fetched_experts_per_step": wl.fetch_rate(first=args.warmup + 2 * args.steps
                                                                                  + 5)[0]}
            log(f"T={T} {'fused' if wl.fused else 'separate'} form: {v_o:.1f} {UNIT}, "
                f"{s_o / args.steps * 1e3:.3f} ms/step")
            st = ft.get_status(wl.status)
            if st != 0:
                raise RuntimeError(f"device status {st} during the benchmark")
            wl.use_fused(fused)
            wl.capture()
        if bi == 0:
            results[T]["host_link"] = host_link_bench(wl, log)
            if args.phi != 26214:
                results[T]["phi_26214"] = phi_bench(wl, 26214, args, units, reduce_fn, world, log)

    prefill = None
    if not args.no_prefill:
        del wl
        torch.cuda.empty_cache()
        pst = None
        prefill = {}
        for Tp in synth.get_config("prefill").tokens:
            res, pst = prefill_bench(Tp, max(3, min(args.steps, 20)), args.warmup, device, log, pst)
            prefill[str(Tp)] = res
        del pst
        torch.cuda.empty_cache()
        if args.prefill_layers > 0:
            prefill["streamed"] = prefill_pipeline_bench(synth.get_config("prefill").tokens[0], args.prefill_layers,
                                                         device, log)
    flash = None
    if not args.no_flash:
        if args.no_prefill:
            del wl
        torch.cuda.empty_cache()
        flash = flash_bench(max(3, min(args.steps, 100)), args.warmup, device, log)
        need = 24576 * 2764800 * 1.5
        if host_mem_available() >= need:
            torch.cuda.empty_cache()
            flash["cache_25pct"] = flash_bench(max(3, min(args.steps, 50)), args.warmup, device, log,
                                               cache_frac=0.25)
        else:
            flash["cache_25pct"] = {"skipped": f"host memory available {host_mem_available() / 1e9:.0f} GB "
                                               f"< {need / 1e9:.0f} GB for the pinned 67.9 GB pool"}
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    r = results[args.tokens]
    kt = r["kt"] or {}
    dom = max(kt, key=kt.get) if kt else "experts"
    exp_us = r["exp_us"]
    if r["fused"]:
        # one kernel per layer and nothing else in the step: the timed
        # region's CUDA events over steps x L launches give its duration
        exp_us = r["secs"] / args.steps / cfg.L * 1e6
    roof = None
    router_bytes = cfg.E * cfg.H * 4
    if exp_us:
        # algorithmic bytes of one launch (each distinct expert's block once,
        # plus the router rows when the router runs in the same kernel) / its
        # event-timed duration
        per_call = r["ebytes"] / cfg.L + (router_bytes if r["fused"] else 0)
        achieved = per_call / (exp_us * 1e-6) / 1e9
        kname = ("ft_moe_decode_layer (route, resolve, fetch, experts, combine: one kernel per layer)" if r["fused"]
                 else "ft_moe_experts_fwd decode (gate/up + down kernels)")
        roof = {"bound": "hbm", "kernel": kname,
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": (LAYER_TRAFFIC_PER_CALL if r["fused"] else TRAFFIC_PER_CALL).get(args.tokens),
                "peak_kind": peak_kind, "frac_of_8tbs_nominal": achieved / 8000.0,
                "algorithmic_bytes_per_launch": per_call,
                "launch_us": exp_us,
                "launch_us_sampled": r["exp_us"],
                "timing": ("CUDA events around the timed region on the launching stream / (steps x 40 launches): the "
                           "step is one ft_moe_decode_layer kernel per layer and nothing else; launch_us_sampled: "
                           "events around every 8th layer's kernel in a copy of the graph replayed after the timed "
                           "region (each event node also breaks the launch chain)") if r["fused"] else
                          (f"events around the experts calls of every {DecodeWorkload.EXP_EVERY}th layer in a copy of "
                           "the step's graph replayed after the timed region"),
                "step_us_per_layer": r["secs"] / args.steps / cfg.L * 1e6,
                "dominant_op_by_time": dom}
    cpu = None
    if not args.no_cpu_baseline:
        rate, n, dt = oracle_rate(cfg, args.tokens, args.phi)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n} single-layer calls of {args.tokens} token(s) (route, resolve, fp64 experts) "
                         f"on 2 of 40 layers, {dt:.1f} s, single-threaded C++"}
    launches_per_step = cfg.L * r["kernels_per_layer"]
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["secs"] / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4-w/bf16-x/f32-acc", "data": "synthetic",
        "config": {"workload": f"35B-A3B-shaped decode: 40 layers x 256 experts, top-8, H2048, I512, "
                               f"int4 g64 (1,671,168 B/expert), cache 2560 slots (25%) from a Zipf(1.1) "
                               f"history, pool in pinned host memory, T={args.tokens} tokens/step, "
                               f"frac_q16={args.phi}",
                   "tokens_per_step": args.tokens, "layers": cfg.L,
                   "l2": "inputs larger than L2: each step streams "
                         f"{r['ebytes'] / 1e6:.0f} MB of expert bytes (L2 129 MB)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "clocks": r["clocks"],
        "e2e": {"value": r["e2e"], "unit": UNIT, "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "cpu_baseline": cpu,
        "detail": {
            "model_tokens_per_s": r["value"] / cfg.L,
            "per_op_us_per_step": kt,
            "expert_bytes_per_step": r["ebytes"],
            "step": ("per layer: ft_moe_decode_layer (one kernel: route, resolve with the q* split, fetch, "
                     "experts, combine)" if r["fused"] else
                     ("per layer: ft_moe_route_resolve (router logits grid, then one resolve CTA that takes the "
                      "top-k first), ft_moe_fetch, ft_moe_experts_fwd (two kernels)" if r.get("combined", True) else
                      "per layer: ft_moe_route, ft_moe_resolve_slots, ft_moe_fetch, ft_moe_experts_fwd (two kernels)")),
            "other_form": r.get("other_form"),
            "phi_26214": r.get("phi_26214"),
            "host_link": r.get("host_link"),
            "settle_steps": args.settle,
            "fetched_experts_per_step": r["nfetch"],
            "host_path_pairs_per_step": r["host_pairs"],
            "fetch_stats": "mean of 20 steps after the timed region",
            "prefill": None if prefill is None else {
                "workload": "one prefill MoE layer: NVFP4, H 4096, I 2048, 256 experts, top-6, all experts "
                            "resident; route -> permute -> grouped SwiGLU on tcgen05 -> combine",
                "tensor_peak_tflops": peaks["bf16_tflops"],
                "tensor_peak_kind": f"{peak_kind} bf16 dense (f16 runs at the bf16 rate)",
                "by_tokens": {t: dict(v, tensor_frac=v["grouped_gemm_tflops"] / peaks["bf16_tflops"])
                              for t, v in prefill.items() if t != "streamed"},
                "streamed_from_host": prefill.get("streamed")},
            "flash_nvfp4_decode": None if flash is None else dict(
                flash, experts_frac_of_hbm=(flash["experts_GBs"] / peaks["hbm_gbs"]
                                            if flash["experts_GBs"] else None)),
            "other_batches": {str(T): {"value": v["value"], "ms_per_step": v["secs"] / args.steps * 1e3,
                                       "per_op_us_per_step": v["kt"], "expert_bytes_per_step": v["ebytes"],
                                       "fused": v["fused"], "launch_us": v["exp_us"],
                                       "other_form": v.get("other_form"),
                                       "e2e": v["e2e"]}
                              for T, v in results.items() if T != args.tokens},
        },
    }
    print(json.dumps(line), flush=True)


def reshape_workload(wl, T, n_steps):
    """Reuse pool, cache, router and warmed state for another batch size."""
    import torch

    import synth

    cfg, dev, ft = wl.cfg, wl.dev, wl.ft
    L, E, k, H = cfg.L, cfg.E, cfg.k, cfg.H
    wl.T = T
    wl.x_host = step_inputs(cfg, T, n_steps)
    wl.x_all = wl.x_host.to(dev)
    wl.x_stage = torch.empty((L, T, H), dtype=torch.int16, device=dev)
    wl.out = torch.empty((L, T, H), dtype=torch.int16, device=dev)
    wl.ids = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    wl.w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    wl.slot = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    wl.ml = T * k
    wl.ff = torch.empty((L, wl.ml), dtype=torch.int32, device=dev)
    wl.fs = torch.empty((L, wl.ml), dtype=torch.int32, device=dev)
    wl.rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=dev)
    wl.ews = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, H, cfg.I, E), dtype=torch.uint8, device=dev)
    wl.lws = torch.zeros(ft.decode_layer_workspace(T, k, H, cfg.I, E), dtype=torch.uint8, device=dev)
    return wl


if __name__ == "__main__":
    main()

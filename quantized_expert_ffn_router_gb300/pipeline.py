"""Decode layer pipelines and the calibration of the q* split, over the C ABI.

Stream orchestration only: every step is a call into libft_moe.so.

* DecodeLayer runs one decode layer call:
    serial      route -> resolve -> fetch -> experts (cache and host path in
                one call, combine fused)
    overlapped  route -> resolve -> fork:
                  host stream  experts FT_DECODE_HOST (the -1 pairs, read in
                               place from the pinned pool)
                  main stream  fetch -> experts FT_DECODE on the cache
                -> join -> merge_partials
  The overlapped form follows the pages' decode step ("FreeToken 딥다이브",
  design pattern 3: the host work is submitted first, the copy of the
  missing experts runs meanwhile, then the GPU experts, and the two partial
  sums are added; "FreeToken: 让消费级电脑跑起 284B MoE", sec. 6: the merge is
  exact).  Both forms capture into one CUDA graph (the fork and join are
  events).

* frac_q16_from_bandwidths and calibrate_frac_q16: the split fraction
  phi = B_P / B_H in Q16 (deep-dive pattern 2; paper post sec. 6, q* = m *
  B_P / B_H), where B_P is the bandwidth of copying expert blocks from the
  pool into the cache and B_H that of computing experts in place on the pool.
  The deep-dive notes that the profile prefers the two measured while both
  run at once (they share host memory), and calibrate_frac_q16 does so.

* SpeculativeDecode runs a decode step over consecutive layers with the
  speculative next-layer copies of the NVMe-streaming post ("Where the time
  actually goes"): layer l+1's router on layer l's input predicts its
  experts, ft_moe_prefetch plans their copies and ft_moe_fetch starts them on
  a second stream while layer l computes.

* PrefillLayers runs prefill over consecutive layers through the whole-layer
  double buffer: layer l's experts in cache slots (l%2)*E .., copied from the
  pool by the copy engine (ft_moe_fetch_layer, then ft_moe_cache_install) on
  a second stream while the previous layer computes on the main stream
  (route -> permute -> grouped experts -> combine); the last two layers stay
  in the cache and seed decode ("FreeToken 딥다이브", design pattern 1;
  "FreeToken: 让消费级电脑跑起 284B MoE", sec. 5).  With fewer than 2E slots the
  buffer is single: each layer is copied after the previous one's experts.

* resize_cache rebuilds the slot cache at a new size: every new buffer is
  allocated first, then ft_moe_cache_rebuild validates and copies; a failed
  allocation or a refused rebuild leaves the running cache untouched
  ("FreeToken 딥다이브", design pattern 7: validate before destroy;
  "FreeToken: 让消费级电脑跑起 284B MoE", sec. 7).
"""

from __future__ import annotations

import ctypes

from . import (FT_DECODE, FT_DECODE_HOST, FT_PREFILL, DeviceCacheState, FtBank, cache_install, combine, experts_fwd,
               experts_workspace, fetch, fetch_layer, make_bank, merge_partials, permute, permute_workspace, prefetch,
               resolve_slots, route, route_resolve, route_workspace)
from . import cache_rebuild as _cache_rebuild


def frac_q16_from_bandwidths(b_p: float, b_h: float) -> int:
    """phi = B_P / B_H as a Q16 integer in [1, 65536].  B_P >= B_H means every
    miss is worth fetching (65536); phi is never 0, which the split reads as
    "no cap"."""
    if not (b_p > 0 and b_h > 0):
        raise ValueError("bandwidths must be positive")
    return int(min(65536, max(1, round(65536.0 * b_p / b_h))))


class DecodeLayer:
    """Buffers and streams for decode layer calls of T tokens (allocated once,
    so that calls can be captured in a CUDA graph)."""

    def __init__(self, state: DeviceCacheState, cache: FtBank, pool: FtBank | None, E: int, k: int, T: int,
                 device="cuda"):
        import torch

        self.state, self.cache, self.pool, self.E, self.k, self.T = state, cache, pool, E, k, T
        H, I = cache.H, cache.I
        n = T * k
        ml = max(min(n, state.S), 1)
        i32 = dict(dtype=torch.int32, device=device)
        self.ids = torch.empty((T, k), **i32)
        self.w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.slot_ids = torch.empty((T, k), **i32)
        self.num_fetch = torch.zeros(1, **i32)
        self.fetch_fid = torch.empty(ml, **i32)
        self.fetch_slot = torch.empty(ml, **i32)
        self.route_ws = torch.zeros(route_workspace(T, E, H), dtype=torch.uint8, device=device)
        wsb = experts_workspace(FT_DECODE, T, k, H, I, E)
        self.ws = torch.zeros(wsb, dtype=torch.uint8, device=device)
        self.ws_host = torch.zeros(wsb, dtype=torch.uint8, device=device)
        self.part_cache = torch.empty((T, H), dtype=torch.float32, device=device)
        self.part_host = torch.empty((T, H), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, **i32)
        self.host_stream = torch.cuda.Stream(device=device)
        self.ev_fork = torch.cuda.Event()
        self.ev_join = torch.cuda.Event()

    def __call__(self, layer: int, x, w_router, frac_q16: int, out, overlapped: bool = True):
        """x [T,H] bf16, w_router [E,H] fp32 -> out [T,H] (fp32 or bf16), on the
        current stream (plus the host stream when overlapped)."""
        import torch

        main = torch.cuda.current_stream()
        # route + resolve in one call (the top-k inside the resolve kernel where the shape allows)
        route_resolve(x, w_router, self.k, self.ids, self.w, self.route_ws, self.state, layer, frac_q16,
                      self.slot_ids, self.num_fetch, self.fetch_fid, self.fetch_slot, dev_status=self.status,
                      stream=main)
        if not overlapped or self.pool is None:
            if self.pool is not None:
                fetch(self.pool, self.cache, self.num_fetch, self.fetch_fid, self.fetch_slot, self.status,
                      stream=main)
            experts_fwd(self.cache, self.pool, layer, self.E, x, self.T, self.k, self.slot_ids, self.ids, self.w,
                        out, self.ws, dev_status=self.status, stream=main)
            return out
        self.ev_fork.record(main)
        self.host_stream.wait_event(self.ev_fork)
        experts_fwd(self.cache, self.pool, layer, self.E, x, self.T, self.k, self.slot_ids, self.ids, self.w,
                    self.part_host, self.ws_host, mode=FT_DECODE_HOST, dev_status=self.status,
                    stream=self.host_stream)
        self.ev_join.record(self.host_stream)
        fetch(self.pool, self.cache, self.num_fetch, self.fetch_fid, self.fetch_slot, self.status, stream=main)
        experts_fwd(self.cache, None, layer, self.E, x, self.T, self.k, self.slot_ids, self.ids, self.w,
                    self.part_cache, self.ws, dev_status=self.status, stream=main)
        main.wait_event(self.ev_join)
        merge_partials(self.part_cache, self.part_host, out, stream=main)
        return out


class SpeculativeDecode:
    """One decode step over consecutive layers with speculative next-layer
    copies (NVMe-streaming post, "Where the time actually goes": layer l+1's
    router run on layer l's MoE input picks most of layer l+1's experts, so
    their copies can start a layer early).

    Per layer l, on the current (main) stream: route -> resolve -> fetch ->
    experts (the serial DecodeLayer call, the pool as host path).  After
    layer l's resolve, a second stream runs layer l+1's router on layer l's
    input, plans the prefetch of the predicted misses (ft_moe_prefetch) and
    copies them (ft_moe_fetch) while layer l's fetch and experts run.  Layer
    l+1's resolve waits for the plan (the state), its fetch for the copy (the
    slots).  The prefetch never evicts a slot that layer l uses (usage >=
    step-1 after layer l's resolve), so the two streams touch disjoint slots.
    Outputs equal the non-speculative step's bit for bit: only which bytes
    come from a cache slot or from the pool changes.  Buffers are allocated
    once, so a step captures into one CUDA graph."""

    def __init__(self, state: DeviceCacheState, cache: FtBank, pool: FtBank, E: int, k: int, T: int,
                 max_prefetch: int | None = None, device="cuda"):
        import torch

        if pool is None:
            raise ValueError("speculative decode copies from a pool")
        self.layer = DecodeLayer(state, cache, pool, E, k, T, device)
        self.max_prefetch = T * k if max_prefetch is None else int(max_prefetch)
        n = T * k
        ml = max(min(n, state.S), 1)
        i32 = dict(dtype=torch.int32, device=device)
        self.pred_ids = torch.empty((T, k), **i32)
        self.pred_w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.pred_ws = torch.zeros(route_workspace(T, E, cache.H), dtype=torch.uint8, device=device)
        self.pf_num = torch.zeros(1, **i32)
        self.pf_fid = torch.empty(ml, **i32)
        self.pf_slot = torch.empty(ml, **i32)
        self.spec_stream = torch.cuda.Stream(device=device)
        self.ev_resolved = torch.cuda.Event()
        self.ev_plan = [torch.cuda.Event() for _ in range(2)]
        self.ev_copy = [torch.cuda.Event() for _ in range(2)]

    def __call__(self, xs, w_routers, frac_q16: int, outs, speculate: bool = True, layers=None):
        """xs[i] [T,H] bf16 MoE input and w_routers[i] [E,H] fp32 router of
        layer layers[i] (default i) -> outs[i].  Enqueues on the current stream
        (and the speculation stream)."""
        import torch

        d = self.layer
        main = torch.cuda.current_stream()
        P = self.spec_stream
        n = len(xs)
        layers = list(range(n)) if layers is None else list(layers)
        for i in range(n):
            l = layers[i]
            route(xs[i], w_routers[i], d.k, d.ids, d.w, d.route_ws, stream=main)
            if speculate and i > 0:
                main.wait_event(self.ev_plan[i % 2])  # the prefetch's state update is in
            resolve_slots(d.state, l, d.ids, frac_q16, d.slot_ids, d.num_fetch, d.fetch_fid, d.fetch_slot,
                          d.status, stream=main)
            if speculate and i + 1 < n:
                b = (i + 1) % 2
                self.ev_resolved.record(main)
                P.wait_event(self.ev_resolved)
                route(xs[i], w_routers[i + 1], d.k, self.pred_ids, self.pred_w, self.pred_ws, stream=P)
                prefetch(d.state, layers[i + 1], self.pred_ids, self.max_prefetch, self.pf_num, self.pf_fid,
                         self.pf_slot, d.status, stream=P)
                self.ev_plan[b].record(P)
                fetch(d.pool, d.cache, self.pf_num, self.pf_fid, self.pf_slot, d.status, stream=P)
                self.ev_copy[b].record(P)
            if speculate and i > 0:
                main.wait_event(self.ev_copy[i % 2])  # the prefetched blocks are in their slots
            fetch(d.pool, d.cache, d.num_fetch, d.fetch_fid, d.fetch_slot, d.status, stream=main)
            experts_fwd(d.cache, d.pool, l, d.E, xs[i], d.T, d.k, d.slot_ids, d.ids, d.w, outs[i], d.ws,
                        dev_status=d.status, stream=main)
        if speculate:
            main.wait_stream(P)
        return outs


def calibrate_frac_q16(pool: FtBank, cache: FtBank, E: int, k: int, n_fetch: int, reps: int = 10,
                       device="cuda") -> dict:
    """Measure B_P (ft_moe_fetch of n_fetch blocks pool -> cache slots) and
    B_H (FT_DECODE_HOST experts over k pool experts of one token), each alone
    and both at once on two streams, and derive frac_q16 from the pair
    measured at once.  Repetition i draws n_fetch + k distinct experts of
    layer i mod (pool blocks / E), so that repetitions read different blocks.
    Needs E >= n_fetch + k and n_fetch cache slots."""
    import torch

    from . import block_bytes

    nbytes = block_bytes(cache.fmt, cache.H, cache.I, cache.group)[0]
    n_layers = int(pool.n_blocks) // E
    if n_layers < 1 or E < n_fetch + k or int(cache.n_blocks) < n_fetch:
        raise ValueError("calibrate: pool or cache too small for the requested sizes")
    gen = torch.Generator().manual_seed(0)
    i32 = dict(dtype=torch.int32, device=device)
    draws = []
    for i in range(reps):
        layer = i % n_layers
        perm = torch.randperm(E, generator=gen)
        draws.append((layer, (perm[:n_fetch] + layer * E).to(**i32), perm[n_fetch:n_fetch + k].view(1, k).to(**i32)))
    fs = torch.arange(n_fetch, **i32)
    nf = torch.tensor([n_fetch], **i32)
    slots = torch.full((1, k), -1, **i32)
    w = torch.full((1, k), 1.0 / k, dtype=torch.float32, device=device)
    x = torch.randn((1, cache.H), generator=gen).to(torch.bfloat16).view(torch.int16).to(device)
    out = torch.empty((1, cache.H), dtype=torch.float32, device=device)
    ws = torch.zeros(experts_workspace(FT_DECODE, 1, k, cache.H, cache.I, E), dtype=torch.uint8, device=device)
    status = torch.zeros(1, **i32)
    s_p, s_h = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

    def run_fetch(i, st):
        fetch(pool, cache, nf, draws[i][1], fs, status, stream=st)

    def run_host(i, st):
        experts_fwd(cache, pool, draws[i][0], E, x, 1, k, slots, draws[i][2], w, out, ws, mode=FT_DECODE_HOST,
                    dev_status=status, stream=st)

    def timed(st, fn, i):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn(i, st)
        e1.record(st)
        return e0, e1

    torch.cuda.synchronize()
    run_fetch(0, s_p)  # warm-up: loads the kernels
    run_host(0, s_h)
    torch.cuda.synchronize()
    us = {"alone_fetch": [], "alone_host": [], "both_fetch": [], "both_host": []}
    for i in range(reps):
        j = (i + reps // 2) % reps
        ev = {"alone_fetch": timed(s_p, run_fetch, i)}
        torch.cuda.synchronize()
        ev["alone_host"] = timed(s_h, run_host, j)
        torch.cuda.synchronize()
        ev["both_fetch"] = timed(s_p, run_fetch, j)
        ev["both_host"] = timed(s_h, run_host, i)
        torch.cuda.synchronize()
        for key, (e0, e1) in ev.items():
            us[key].append(e0.elapsed_time(e1) * 1e3)
    med = {key: sorted(v)[len(v) // 2] for key, v in us.items()}
    gbs = lambda n, t_us: n / (t_us * 1e-6) / 1e9
    res = {
        "B_P_alone_GBs": gbs(n_fetch * nbytes, med["alone_fetch"]),
        "B_H_alone_GBs": gbs(k * nbytes, med["alone_host"]),
        "B_P_GBs": gbs(n_fetch * nbytes, med["both_fetch"]),
        "B_H_GBs": gbs(k * nbytes, med["both_host"]),
        "n_fetch": n_fetch, "k": k, "block_bytes": nbytes, "reps": reps,
    }
    res["frac_q16"] = frac_q16_from_bandwidths(res["B_P_GBs"], res["B_H_GBs"])
    res["frac_q16_alone"] = frac_q16_from_bandwidths(res["B_P_alone_GBs"], res["B_H_alone_GBs"])
    res["status"] = int(status.item())
    return res


class PrefillLayers:
    """Buffers, streams and events for prefill of T tokens through a run of
    layers, each layer's experts loaded whole into the cache's first slots.

    The cache must hold at least E slots (state.S and cache.n_blocks); with
    2E or more the buffer is double (the next layer's copy overlaps this
    layer's experts), otherwise single.  Routing, permutation, the grouped
    experts and the combine are the library's calls; the cache state records
    every installed layer, so afterwards the last layer (two layers, double
    buffered) are resident for decode."""

    def __init__(self, state: DeviceCacheState, cache: FtBank, pool: FtBank, E: int, k: int, T: int,
                 device="cuda"):
        import torch

        slots = min(state.S, int(cache.n_blocks))
        if slots < E:
            raise ValueError(f"prefill needs a whole layer in the cache: {slots} slots < E = {E}")
        self.state, self.cache, self.pool, self.E, self.k, self.T = state, cache, pool, E, k, T
        self.n_buf = 2 if slots >= 2 * E else 1
        H, I = cache.H, cache.I
        n = T * k
        i32 = dict(dtype=torch.int32, device=device)
        self.slot_of = [torch.arange(b * E, (b + 1) * E, **i32) for b in range(self.n_buf)]
        self.ids = torch.empty((T, k), **i32)
        self.w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.route_ws = torch.zeros(route_workspace(T, E, H), dtype=torch.uint8, device=device)
        self.perm = torch.empty(n, **i32)
        self.inv = torch.empty((T, k), **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.xp = torch.empty((n, H), dtype=torch.int16, device=device)
        self.xp_scale = torch.empty(n, dtype=torch.float32, device=device)
        self.perm_ws = torch.empty(permute_workspace(T, k, E), dtype=torch.uint8, device=device)
        self.yp = torch.empty((n, H), dtype=torch.int16, device=device)
        self.ws = torch.empty(experts_workspace(FT_PREFILL, T, k, H, I, E), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, **i32)
        self.copy_stream = torch.cuda.Stream(device=device)
        self.ev_loaded = [torch.cuda.Event() for _ in range(self.n_buf)]
        self.ev_free = [torch.cuda.Event() for _ in range(self.n_buf)]

    def __call__(self, layers, xs, ws_router, outs):
        """layers: flat-id layer indices in order; xs[i] [T,H] bf16 input of
        layers[i]; ws_router[i] [E,H] fp32 its router; outs[i] [T,H] bf16 its
        MoE output.  Enqueues on the current stream (and the copy stream)."""
        import torch

        main = torch.cuda.current_stream()
        E, k, T, nb = self.E, self.k, self.T, self.n_buf

        def load(i):
            b = i % nb
            if i == 0:
                self.copy_stream.wait_stream(main)  # the state and slots as earlier work on the stream left them
            if i >= nb:
                self.copy_stream.wait_event(self.ev_free[b])  # buffer b's previous layer has run its experts
            fetch_layer(self.pool, self.cache, layers[i], E, b * E, stream=self.copy_stream)
            cache_install(self.state, layers[i], b * E, stream=self.copy_stream)
            self.ev_loaded[b].record(self.copy_stream)

        load(0)
        for i, layer in enumerate(layers):
            b = i % nb
            if nb == 2 and i + 1 < len(layers):
                load(i + 1)  # copied while this layer computes
            main.wait_event(self.ev_loaded[b])
            route(xs[i], ws_router[i], k, self.ids, self.w, self.route_ws, stream=main)
            permute(self.ids, E, xs[i], self.perm, self.inv, self.offsets, self.xp, self.perm_ws,
                    dev_status=self.status, stream=main, xp_scale=self.xp_scale)
            experts_fwd(self.cache, None, layer, E, self.xp, T, k, self.slot_of[b], None, None, self.yp, self.ws,
                        mode=FT_PREFILL, offsets=self.offsets, dev_status=self.status, stream=main,
                        x_scale=self.xp_scale)
            self.ev_free[b].record(main)
            combine(self.yp, self.inv, self.w, outs[i], stream=main)
            if nb == 1 and i + 1 < len(layers):
                load(i + 1)  # single buffer: after this layer's experts
        main.wait_stream(self.copy_stream)
        return outs


def resize_cache(state: DeviceCacheState, cache, fmt: int, H: int, I: int, group: int, new_S: int,
                 budget_bytes: int, tensor_scale=None, alloc=None, rebuild=None, dev_status=None, stream=None):
    """Rebuild the slot cache (state + its bank tensor `cache` [S, stride]) at
    new_S slots.  Returns (new_state, new_cache, new_bank); the caller switches
    to them and frees the old ones once the stream has passed the rebuild.

    Everything the new cache needs is allocated before the library is
    called, through alloc(shape, dtype, fill) (default: torch.full on the old
    cache's device), and the rebuild itself validates before it writes.  So
    an allocation that fails (out of memory) raises before any device work,
    and a rebuild the library refuses (FtError FT_ERR_REJECTED: over budget,
    wrong shape) raises after nothing was changed: either way the old state
    and bank keep serving."""
    import torch

    if new_S < 0:
        raise ValueError("new_S < 0")
    device = cache.device
    if alloc is None:
        def alloc(shape, dtype, fill):
            return torch.full(shape, fill, dtype=dtype, device=device)
    stride = int(cache.stride(0)) * cache.element_size()
    new_state = DeviceCacheState(state.L, state.E, new_S, device=device, alloc=alloc)
    new_cache = alloc((max(new_S, 1), stride), torch.uint8, 0)
    old_bank = make_bank(fmt, H, I, group, cache, tensor_scale)
    new_bank = make_bank(fmt, H, I, group, new_cache, tensor_scale)
    (rebuild or _cache_rebuild)(state, old_bank, new_state, new_bank, budget_bytes, dev_status=dev_status,
                                stream=stream)
    return new_state, new_cache, new_bank

"""GPU: the fused decode layer (ft_moe_decode_layer, one kernel per layer
call) against the separate calls (route, resolve, fetch, experts) and the
oracle, over several steps and layers on an evolving slot cache.

Integers (top-k ids, slot ids, fetch lists, the whole cache state, the cache
bytes) must equal the separate calls' bit for bit; outputs must be within
the tolerance of the oracle, and at the 35B shape with one token (where both
paths run the same arithmetic in the same order) equal to the separate
calls' bit for bit.  Also: replay from a CUDA graph, a shape it refuses, and
a bounded wait that runs out."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import assert_close, oracle_pairs_output
from test_gpu_decode_layers import _Layer, _cache_from_state, _dev_state, _pool, _seeded_host_state, _t

pytestmark = pytest.mark.gpu
DEV = "cuda"


class _Fused:
    """One fused layer call's buffers (the same outputs as _Layer's)."""

    def __init__(self, ft, T, k, E, H, I, ml):
        self.ft = ft
        self.ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        self.w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        self.sl = torch.empty((T, k), dtype=torch.int32, device=DEV)
        self.nf = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.ff = torch.empty(ml, dtype=torch.int32, device=DEV)
        self.fs = torch.empty(ml, dtype=torch.int32, device=DEV)
        self.ws = torch.zeros(ft.decode_layer_workspace(T, k, H, I, E), dtype=torch.uint8, device=DEV)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def __call__(self, st, cache_b, pool_b, layer, E, k, phi, x, W, out):
        self.ft.decode_layer(x, W, k, st, layer, phi, cache_b, pool_b, self.ids, self.w, self.sl, self.nf, self.ff,
                             self.fs, out, self.ws, dev_status=self.status)


def _states_equal(a, b):
    for x, y in [(a.map, b.map), (a.slot_owner, b.slot_owner), (a.usage, b.usage), (a.recency, b.recency),
                 (a.step, b.step)]:
        if not torch.equal(x, y):
            return False
    return True


CASES = [("tiny", 8, 6, 26214, 1), ("d35b", 1, 48, 65536, 2), ("d35b", 1, 48, 26214, 2), ("d35b", 1, 0, 65536, 2),
         ("d35b", 1, 48, 0, 2), ("flash", 1, 64, 65536, 1)]


@pytest.mark.parametrize("name,T,S,phi,L", CASES)
def test_fused_layer_matches_separate_calls_and_oracle(cuda_lib, name, T, S, phi, L):
    ft = cuda_lib
    cfg = synth.get_config(name)
    E, k, H, I = cfg.E, cfg.k, cfg.H, cfg.I
    pool, stride = _pool(cfg, L)
    ts_np = synth.tensor_scales(cfg.fmt, H, I, cfg.L * E)
    ts = None if ts_np is None else _t(ts_np)
    host = _seeded_host_state(L, E, S, seed=7, filled=0.5)
    states = [_dev_state(ft, host), _dev_state(ft, host)]
    caches = [_cache_from_state(host, pool, stride) for _ in range(2)]
    pb = ft.make_bank(cfg.fmt, H, I, cfg.g, pool, ts)
    cbs = [ft.make_bank(cfg.fmt, H, I, cfg.g, c, ts) for c in caches]
    Ws = [_t(synth.router_weights(cfg.seed, l, E, H, cfg.router_std, zipf_bias=cfg.zipf)) for l in range(L)]
    ml = min(T * k, max(S, 1))
    fused, sep = _Fused(ft, T, k, E, H, I, T * k), _Layer(ft, T, k, E, H, I, T * k)
    steps = 5
    xs = synth.normal_bf16(synth.stream_key(cfg.seed, "fused-layer", name, T), (steps, L, T, H))
    if cfg.zipf is not None:
        xs[..., 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
    x_all = _t(xs)
    same_order = name == "d35b" and T == 1
    fetched = host_pairs = 0
    for s in range(steps):
        for l in range(L):
            out_f = torch.full((T, H), float("nan"), device=DEV)
            out_s = torch.full((T, H), float("nan"), device=DEV)
            fused(states[0], cbs[0], pb, l, E, k, phi, x_all[s, l], Ws[l], out_f)
            sep(states[1], cbs[1], pb, l, E, k, phi, x_all[s, l], Ws[l], out_s)
            torch.cuda.synchronize()
            what = f"{name} T={T} S={S} phi={phi} step {s} layer {l}"
            assert torch.equal(fused.ids, sep.ids), what
            assert torch.equal(fused.sl, sep.sl), what
            assert torch.equal(fused.nf, sep.nf), what
            n = int(fused.nf.item())
            assert torch.equal(fused.ff[:ml], sep.ff[:ml]) and torch.equal(fused.fs[:ml], sep.fs[:ml]), what
            assert _states_equal(states[0], states[1]), what
            np.testing.assert_allclose(fused.w.cpu().numpy(), sep.w.cpu().numpy(), rtol=1e-5, atol=1e-8)
            fetched += n
            host_pairs += int((fused.sl < 0).sum().item())
            if same_order:
                assert torch.equal(fused.w, sep.w), what
                assert torch.equal(out_f, out_s), what
            else:
                assert_close(out_f.cpu().numpy(), out_s.cpu().numpy(), what, rel_l2=1e-4, max_abs=1e-4,
                             ref_max=None)
            # the oracle, fed the ids and weights this call chose (pairs from the cache or the pool)
            ids, w = fused.ids.cpu().numpy(), fused.w.cpu().numpy()
            blocks = {l * E + int(e): pool[l * E + int(e)].numpy() for e in set(ids.ravel().tolist())}
            ref = oracle_pairs_output(blocks, cfg, ts_np, xs[s, l], ids, w, l)
            assert_close(out_f.cpu().numpy(), ref, what)
    assert torch.equal(caches[0], caches[1])
    assert ft.get_status(fused.status) == 0 and ft.get_status(sep.status) == 0
    if S > 0 and phi in (0, 65536):
        assert fetched > 0  # the fetch hand-off ran
    if S == 0 or phi == 26214:
        assert host_pairs > 0  # pairs read the pool in place


def test_fused_layer_graph_replay_is_bit_identical(cuda_lib):
    """Two layers of fused calls captured in one CUDA graph and replayed give
    the eager calls' outputs, caches and states bit for bit."""
    ft = cuda_lib
    cfg = synth.get_config("d35b")
    L, T, S, phi = 2, 1, 48, 26214
    E, k, H, I = cfg.E, cfg.k, cfg.H, cfg.I
    pool, stride = _pool(cfg, L)
    host = _seeded_host_state(L, E, S, seed=11, filled=0.5)
    states = [_dev_state(ft, host), _dev_state(ft, host)]
    caches = [_cache_from_state(host, pool, stride) for _ in range(2)]
    pb = ft.make_bank(cfg.fmt, H, I, cfg.g, pool)
    cbs = [ft.make_bank(cfg.fmt, H, I, cfg.g, c) for c in caches]
    Ws = [_t(synth.router_weights(cfg.seed, l, E, H, cfg.router_std, zipf_bias=cfg.zipf)) for l in range(L)]
    runs = [[_Fused(ft, T, k, E, H, I, T * k) for _ in range(L)] for _ in range(2)]
    xs = synth.normal_bf16(synth.stream_key(cfg.seed, "fused-graph"), (4, L, T, H))
    xs[..., 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
    x_all = _t(xs)
    x_stage = torch.empty((L, T, H), dtype=torch.int16, device=DEV)
    outs = [torch.empty((L, T, H), dtype=torch.float32, device=DEV) for _ in range(2)]
    x_stage.copy_(x_all[0])
    for l in range(L):  # one eager call each first (attributes, lookups) before the capture
        runs[0][l](states[0], cbs[0], pb, l, E, k, phi, x_stage[l], Ws[l], outs[0][l])
        runs[1][l](states[1], cbs[1], pb, l, E, k, phi, x_stage[l], Ws[l], outs[1][l])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for l in range(L):
                runs[0][l](states[0], cbs[0], pb, l, E, k, phi, x_stage[l], Ws[l], outs[0][l])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for s in range(1, 4):
        x_stage.copy_(x_all[s])
        g.replay()
        for l in range(L):
            runs[1][l](states[1], cbs[1], pb, l, E, k, phi, x_stage[l], Ws[l], outs[1][l])
        torch.cuda.synchronize()
        assert torch.equal(outs[0], outs[1]), s
        assert _states_equal(states[0], states[1]), s
        assert torch.equal(caches[0], caches[1]), s
        for l in range(L):
            assert torch.equal(runs[0][l].ids, runs[1][l].ids) and torch.equal(runs[0][l].sl, runs[1][l].sl)


def test_fused_layer_refuses_a_plan_that_does_not_fit(cuda_lib):
    """Eight tokens at the 35B shape need more shared memory than one SM has:
    the call is refused on the host and nothing is launched."""
    ft = cuda_lib
    cfg = synth.get_config("d35b")
    T, E, k, H, I = 8, cfg.E, cfg.k, cfg.H, cfg.I
    pool, stride = _pool(cfg, 1)
    st = ft.DeviceCacheState(1, E, 16, device=DEV)
    cache = torch.zeros((16, stride), dtype=torch.uint8, device=DEV)
    pb, cb = ft.make_bank(cfg.fmt, H, I, cfg.g, pool), ft.make_bank(cfg.fmt, H, I, cfg.g, cache)
    f = _Fused(ft, T, k, E, H, I, T * k)
    x = torch.zeros((T, H), dtype=torch.int16, device=DEV)
    W = torch.zeros((E, H), dtype=torch.float32, device=DEV)
    out = torch.zeros((T, H), dtype=torch.float32, device=DEV)
    with pytest.raises(ft.FtError) as ei:
        f(st, cb, pb, 0, E, k, 65536, x, W, out)
    assert ei.value.status == ft.FT_ERR_INVALID
    torch.cuda.synchronize()
    assert int(st.step.item()) == 0  # nothing ran


def test_fused_layer_bounded_wait_runs_out(cuda_lib):
    """With the wait limit at 1 ns, a hand-off wait that does not find its
    data at the first look gives up (the workers look for the leader's plan
    microseconds before it can exist): the kernel returns with FT_ERR_TIMEOUT
    in the status word, the next call on that status does nothing, and after
    the caller clears the workspace and the status and restores the limit the
    layer runs normally again on the same context."""
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    L, T, S, phi = 1, 8, 6, 26214
    E, k, H, I = cfg.E, cfg.k, cfg.H, cfg.I
    pool, stride = _pool(cfg, L)
    host = _seeded_host_state(L, E, S, seed=3, filled=0.5)
    st = _dev_state(ft, host)
    cache = _cache_from_state(host, pool, stride)
    pb, cb = ft.make_bank(cfg.fmt, H, I, cfg.g, pool), ft.make_bank(cfg.fmt, H, I, cfg.g, cache)
    W = _t(synth.router_weights(cfg.seed, 0, E, H, cfg.router_std))
    x = _t(synth.normal_bf16(synth.stream_key(cfg.seed, "fused-timeout"), (T, H)))
    f = _Fused(ft, T, k, E, H, I, T * k)
    out = torch.full((T, H), 7.0, device=DEV)
    ft.set_wait_limit_ns(1)
    try:
        f(st, cb, pb, 0, E, k, phi, x, W, out)
        torch.cuda.synchronize()
        assert ft.get_status(f.status) == ft.FT_ERR_TIMEOUT
        assert bool((out == 7.0).all())  # no worker saw a plan, so no output row was written
        snap = [t.clone() for t in (st.map, st.slot_owner, st.usage, st.recency, st.step)]
        ft.set_wait_limit_ns(0)
        f(st, cb, pb, 0, E, k, phi, x, W, out)  # sees the status: does nothing
        torch.cuda.synchronize()
        assert bool((out == 7.0).all())
        for a, b in zip(snap, (st.map, st.slot_owner, st.usage, st.recency, st.step)):
            assert torch.equal(a, b)
    finally:
        ft.set_wait_limit_ns(0)
    # recovery: a fresh workspace and status word; the state may hold the
    # timed-out call's resolve, so the reference runs from a copy of it
    f.ws.zero_()
    f.status.zero_()
    ref_state = ft.DeviceCacheState(L, E, S, device=DEV)
    for a, b in [(ref_state.map, st.map), (ref_state.slot_owner, st.slot_owner), (ref_state.usage, st.usage),
                 (ref_state.recency, st.recency), (ref_state.step, st.step)]:
        a.copy_(b)
    ref_cache = cache.clone()
    sep = _Layer(ft, T, k, E, H, I, T * k)
    out_s = torch.empty((T, H), device=DEV)
    sep(ref_state, ft.make_bank(cfg.fmt, H, I, cfg.g, ref_cache), pb, 0, E, k, phi, x, W, out_s)
    f(st, cb, pb, 0, E, k, phi, x, W, out)
    torch.cuda.synchronize()
    assert ft.get_status(f.status) == 0
    assert torch.equal(f.ids, sep.ids) and torch.equal(f.sl, sep.sl)
    assert _states_equal(st, ref_state)
    assert_close(out.cpu().numpy(), out_s.cpu().numpy(), "after recovery", rel_l2=1e-4, max_abs=1e-4, ref_max=None)

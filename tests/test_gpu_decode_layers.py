"""GPU: whole decode layers (route, resolve, fetch, experts) over many steps
and layers on an evolving slot cache, eager and replayed from one CUDA graph
(the programmatic launch chain across layers): outputs, cache bytes and
states bit-identical between the two, and the last layer call within
tolerance of the oracle."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_close, oracle_pairs_output

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def _i32(*shape):
    return torch.empty(shape, dtype=torch.int32, device=DEV)


def _dev_state(ft, host):
    st = ft.DeviceCacheState(host.L, host.E, host.S, device=DEV)
    st.load_from(host)
    return st


def _seeded_host_state(L, E, S, seed, filled=0.5):
    host = oracle.CacheState(L, E, S)
    rng = np.random.default_rng(seed)
    n = min(int(round(filled * S)), L * E)
    if n:
        fids = rng.choice(L * E, n, replace=False)
        host.seed_slots(list(fids), usages=list(rng.integers(0, 50, n)))
    host.step[0] = 60
    return host


# ------------------------------------------------------------ whole layers
def _pool(cfg, L):
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool = torch.zeros((L * cfg.E, stride), dtype=torch.uint8).pin_memory()
    tmp = torch.empty((64, stride), dtype=torch.uint8, device=DEV)  # generated on the device, then copied
    for f0 in range(0, L * cfg.E, 64):
        n = min(64, L * cfg.E - f0)
        synth.bank_blocks_torch(cfg.seed, range(f0, f0 + n), cfg.fmt, cfg.H, cfg.I, cfg.g, tmp[:n],
                                ref_K=cfg.ref_K)
        pool[f0:f0 + n].copy_(tmp[:n])
    torch.cuda.synchronize()
    return pool, stride


def _cache_from_state(host, pool, stride):
    cache = torch.zeros((max(host.S, 1), stride), dtype=torch.uint8, device=DEV)
    for s in range(host.S):
        if host.slot_owner[s] >= 0:
            cache[s].copy_(pool[int(host.slot_owner[s])])
    return cache


class _Layer:
    """One decode layer's buffers: route, resolve, fetch, experts."""

    def __init__(self, ft, T, k, E, H, I, ml):
        self.ft = ft
        self.ids, self.w, self.sl = _i32(T, k), torch.empty((T, k), device=DEV), _i32(T, k)
        self.nf, self.ff, self.fs = torch.zeros(1, dtype=torch.int32, device=DEV), _i32(ml), _i32(ml)
        self.rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=DEV)
        self.ews = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, H, I, E), dtype=torch.uint8, device=DEV)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def __call__(self, st, cache_b, pool_b, layer, E, k, phi, x, W, out):
        ft, T = self.ft, x.shape[0]
        ft.route(x, W, k, self.ids, self.w, self.rws)
        ft.resolve_slots(st, layer, self.ids, phi, self.sl, self.nf, self.ff, self.fs, self.status)
        ft.fetch(pool_b, cache_b, self.nf, self.ff, self.fs, self.status)
        ft.experts_fwd(cache_b, pool_b, layer, E, x, T, k, self.sl, self.ids, self.w, out, self.ews,
                       dev_status=self.status)


@pytest.mark.parametrize("name,T,S,phi", [("tiny", 8, 6, 26214), ("d35b", 1, 48, 65536), ("d35b", 8, 48, 49160)])
def test_layers_eager_graph_and_oracle(cuda_lib, name, T, S, phi):
    ft = cuda_lib
    cfg = synth.get_config(name)
    L, E, k, H, I = 2, cfg.E, cfg.k, cfg.H, cfg.I
    pool, stride = _pool(cfg, L)
    ts_np = synth.tensor_scales(cfg.fmt, H, I, cfg.L * E)
    ts = None if ts_np is None else _t(ts_np)
    host = _seeded_host_state(L, E, S, seed=99, filled=0.5)
    states = [_dev_state(ft, host), _dev_state(ft, host)]
    caches = [_cache_from_state(host, pool, stride) for _ in range(2)]
    pb = ft.make_bank(cfg.fmt, H, I, cfg.g, pool, ts)
    cbs = [ft.make_bank(cfg.fmt, H, I, cfg.g, c, ts) for c in caches]
    Ws = [_t(synth.router_weights(cfg.seed, l, E, H, cfg.router_std, zipf_bias=cfg.zipf)) for l in range(L)]
    layers = [_Layer(ft, T, k, E, H, I, T * k) for _ in range(2)]
    steps = 6
    xs = synth.normal_bf16(synth.stream_key(cfg.seed, "decode-layers", T), (steps, L, T, H))
    if cfg.zipf is not None:
        xs[..., 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
    x_all = _t(xs)
    outs = [torch.empty((steps, L, T, H), dtype=torch.float32, device=DEV) for _ in range(2)]
    for s in range(steps):
        for l in range(L):
            for v in range(2):
                layers[v](states[v], cbs[v], pb, l, E, k, phi, x_all[s, l], Ws[l], outs[v][s, l])
    torch.cuda.synchronize()
    # the last layer call against the oracle (every pair computed, from the cache or the pool):
    # its ids and weights are still in the layer's buffers
    lst = L - 1
    ids, w = layers[0].ids.cpu().numpy(), layers[0].w.cpu().numpy()
    blocks = {lst * E + int(e): pool[lst * E + int(e)].numpy() for e in set(ids.ravel().tolist())}
    ref = oracle_pairs_output(blocks, cfg, ts_np, xs[steps - 1, lst], ids, w, lst)
    assert_close(outs[0][steps - 1, lst].cpu().numpy(), ref, f"{name} T={T} last layer")
    assert ft.get_status(layers[0].status) == 0 and ft.get_status(layers[1].status) == 0
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(caches[0], caches[1])
    for a, b in [(states[0].map, states[1].map), (states[0].slot_owner, states[1].slot_owner),
                 (states[0].usage, states[1].usage), (states[0].recency, states[1].recency),
                 (states[0].step, states[1].step)]:
        assert torch.equal(a, b)
    # two identical histories so far; now history 0 continues from one CUDA graph of
    # all layers, history 1 eagerly
    x_stage = torch.empty((L, T, H), dtype=torch.int16, device=DEV)
    g_out = torch.empty((L, T, H), dtype=torch.float32, device=DEV)
    x_stage.copy_(x_all[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for l in range(L):
                layers[0](states[0], cbs[0], pb, l, E, k, phi, x_stage[l], Ws[l], g_out[l])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    e_out = torch.empty((L, T, H), dtype=torch.float32, device=DEV)
    for s in range(3):
        x_stage.copy_(x_all[(s + 2) % steps])
        g.replay()
        for l in range(L):
            layers[1](states[1], cbs[1], pb, l, E, k, phi, x_stage[l], Ws[l], e_out[l])
        torch.cuda.synchronize()
        assert torch.equal(g_out, e_out), s
    assert torch.equal(caches[0], caches[1])
    assert torch.equal(states[0].usage, states[1].usage) and torch.equal(states[0].map, states[1].map)

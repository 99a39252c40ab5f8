"""GPU: ft_moe_cache_rebuild against the oracle's rebuild (state bit-exact,
moved blocks byte-identical to the pool), a layer call gives the same output
before and after a rebuild, and rebuilds that do not fit are refused without
touching the new arrays."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_close, gapped_tokens, oracle_pairs_output, pool_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENT = -7


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def _history(cfg, L, S, steps, seed):
    """The oracle's cache state after `steps` resolve calls on Zipf-skewed ids."""
    st = oracle.CacheState(L, cfg.E, S)
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, cfg.E + 1) ** 1.1
    p /= p.sum()
    for _ in range(steps):
        layer = int(rng.integers(0, L))
        ids = np.stack([rng.choice(cfg.E, cfg.k, replace=False, p=p) for _ in range(2)]).astype(np.int32)
        oracle.resolve(st, layer, ids, 65536)
    return st


def _device_cache(ft, cfg, host, pool_np):
    """Device state and cache bank holding host's residents (blocks from the pool)."""
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    dev = ft.DeviceCacheState(host.L, host.E, host.S, device=DEV)
    dev.load_from(host)
    cache = torch.zeros((max(host.S, 1), stride), dtype=torch.uint8, device=DEV)
    for s in range(host.S):
        if host.slot_owner[s] >= 0:
            cache[s].copy_(torch.from_numpy(pool_np[host.slot_owner[s]]))
    return dev, cache


def _sentinel_state(ft, L, E, S):
    st = ft.DeviceCacheState(L, E, S, device=DEV)
    for n in ("slot_owner", "map", "usage", "recency", "step"):
        getattr(st, n).fill_(SENT)
    return st


@pytest.mark.parametrize("L,S_old,S_new", [(2, 10, 4), (2, 10, 10), (2, 10, 16), (2, 10, 0), (3, 0, 5),
                                           (3, 24, 7)])
def test_cache_rebuild_matches_oracle(cuda_lib, L, S_old, S_new):
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    E = cfg.E
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool_np = pool_blocks(cfg, range(L * E))
    host = _history(cfg, L, S_old, 40, seed=S_old * 7 + S_new)
    dev_old, cache_old = _device_cache(ft, cfg, host, pool_np)
    old_copy = cache_old.clone()
    dev_new = _sentinel_state(ft, L, E, S_new)
    cache_new = torch.full((max(S_new, 1), stride), 0xAB, dtype=torch.uint8, device=DEV)
    ob = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache_old)
    nb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache_new)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ft.cache_rebuild(dev_old, ob, dev_new, nb, 1 << 40, dev_status=status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == 0
    ref, src = oracle.cache_rebuild(host, S_new)
    assert np.array_equal(dev_new.map.cpu().numpy(), ref.map)
    assert np.array_equal(dev_new.recency.cpu().numpy(), ref.recency)
    assert int(dev_new.step.item()) == int(ref.step[0])
    if S_new:
        assert np.array_equal(dev_new.slot_owner[:S_new].cpu().numpy(), ref.slot_owner)
        assert np.array_equal(dev_new.usage[:S_new].cpu().numpy(), ref.usage)
    c = cache_new.cpu().numpy()
    for d in range(S_new):
        if ref.slot_owner[d] >= 0:
            assert np.array_equal(c[d], pool_np[ref.slot_owner[d]]), d
        else:
            assert (c[d] == 0xAB).all(), d  # an empty new slot is not written
    # the old state and bank are only read
    assert torch.equal(cache_old, old_copy)
    for n in ("map", "recency"):
        assert np.array_equal(getattr(dev_old, n).cpu().numpy(), getattr(host, n))


def test_cache_rebuild_layer_output_unchanged(cuda_lib):
    """The same layer call (resolve -> fetch -> experts with the pool as the
    host path) gives bit-identical outputs on the old cache and on caches
    rebuilt smaller and larger: the cache holds copies of the pool's bytes and
    every pair is computed exactly once from one of them."""
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    L, E, k, T, layer = 2, cfg.E, cfg.k, 8, 1
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool_np = pool_blocks(cfg, range(L * E))
    pool = torch.from_numpy(pool_np).to(DEV)
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool)
    host = _history(cfg, L, 10, 50, seed=11)
    W = synth.router_weights(cfg.seed, layer, E, cfg.H, cfg.router_std, zipf_bias=cfg.zipf)
    x, _ = gapped_tokens(cfg.seed, "rebuild-x", T, cfg.H, W, k, cfg.gap, bias_feature=cfg.zipf is not None)
    ids, w = oracle.route(x, W, k)
    w32 = w.astype(np.float32)

    def layer_call(dev, cache, phi):
        cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache)
        S = dev.S
        sl = torch.empty((T, k), dtype=torch.int32, device=DEV)
        nf = torch.zeros(1, dtype=torch.int32, device=DEV)
        ml = max(min(T * k, S), 1)
        ff = torch.empty(ml, dtype=torch.int32, device=DEV)
        fs = torch.empty(ml, dtype=torch.int32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        ft.resolve_slots(dev, layer, _t(ids), phi, sl, nf, ff, fs, status)
        ft.fetch(pb, cb, nf, ff, fs, status)
        out = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, cfg.H, cfg.I, E), dtype=torch.uint8, device=DEV)
        ft.experts_fwd(cb, pb, layer, E, _t(x), T, k, sl, _t(ids), _t(w32), out, ws, dev_status=status)
        torch.cuda.synchronize()
        assert ft.get_status(status) == 0
        return out.cpu().numpy()

    outs = {}
    for S_new in (None, 3, 10, 25):
        dev, cache = _device_cache(ft, cfg, host, pool_np)
        if S_new is not None:
            dev_n = _sentinel_state(ft, L, E, S_new)
            cache_n = torch.zeros((S_new, stride), dtype=torch.uint8, device=DEV)
            ft.cache_rebuild(dev, ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache), dev_n,
                             ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache_n), 1 << 40)
            dev, cache = dev_n, cache_n
        for phi in (0, 26214, 65536):
            outs[(S_new, phi)] = layer_call(dev, cache, phi)
    base = outs[(None, 65536)]
    for key, o in outs.items():
        assert np.array_equal(o, base), key
    blocks = {f: pool_np[f] for f in range(L * E)}
    ref = oracle_pairs_output(blocks, cfg, None, x, ids, w32, layer, np.ones((T, k), bool))
    assert_close(base, ref, "layer after rebuild")


def test_cache_rebuild_refused_leaves_new_arrays(cuda_lib):
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    L, E = 2, cfg.E
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool_np = pool_blocks(cfg, range(L * E))
    host = _history(cfg, L, 6, 20, seed=3)
    dev_old, cache_old = _device_cache(ft, cfg, host, pool_np)
    ob = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache_old)
    dev_new = _sentinel_state(ft, L, E, 4)
    cache_new = torch.full((4, stride), 0xAB, dtype=torch.uint8, device=DEV)
    nb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache_new)
    cases = [
        dict(new=dev_new, nb=nb, budget=4 * stride),                   # state bytes do not fit
        dict(new=_sentinel_state(ft, L, E + 1, 4), nb=nb, budget=1 << 40),  # another E
        dict(new=dev_new, nb=ob, budget=1 << 40),                      # onto the old bank
        dict(new=_sentinel_state(ft, L, E, 5), nb=nb, budget=1 << 40),  # 5 slots, 4 blocks
    ]
    for c in cases:
        with pytest.raises(ft.FtError) as ei:
            ft.cache_rebuild(dev_old, ob, c["new"], c["nb"], c["budget"])
        assert ei.value.status == ft.FT_ERR_REJECTED
    torch.cuda.synchronize()
    for n in ("slot_owner", "map", "usage", "recency", "step"):
        assert (getattr(dev_new, n) == SENT).all(), n
    assert (cache_new == 0xAB).all()

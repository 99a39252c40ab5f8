"""GPU: the prefill whole-layer buffer -- ft_moe_cache_install against the
oracle's install (bit-exact state), ft_moe_fetch_layer against the pool's
bytes, and the double-buffered prefill pipeline against per-layer prefill on
a fully resident bank (bit-identical outputs) and the oracle."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _random_state(rng, L, E, S, filled):
    st = oracle.CacheState(L, E, S)
    n = min(int(filled * S), L * E)
    fids = rng.choice(L * E, n, replace=False)
    slots = rng.choice(S, n, replace=False)
    for f, s in zip(fids, slots):
        st.slot_owner[s] = f
        st.map[f] = s
        st.usage[s] = int(rng.integers(0, 1000))
    st.step[0] = 1000 + int(rng.integers(0, 50))
    st.recency[:] = rng.integers(-1, 1000, L * E)
    return st


def _same(dev, host):
    S = host.S
    assert np.array_equal(dev.map.cpu().numpy(), host.map)
    assert np.array_equal(dev.recency.cpu().numpy(), host.recency)
    assert int(dev.step.item()) == int(host.step[0])
    assert np.array_equal(dev.slot_owner[:S].cpu().numpy(), host.slot_owner)
    assert np.array_equal(dev.usage[:S].cpu().numpy(), host.usage)


@pytest.mark.parametrize("L,E,S,filled", [(4, 8, 16, 1.0), (3, 16, 40, 0.5), (6, 256, 600, 0.9), (2, 4096, 9000, 0.6),
                                          (43, 256, 512, 1.0)])
def test_cache_install_matches_oracle(cuda_lib, L, E, S, filled):
    ft = cuda_lib
    rng = np.random.default_rng(L * 1000 + E)
    host = _random_state(rng, L, E, S, filled)
    dev = ft.DeviceCacheState(L, E, S, device=DEV)
    dev.load_from(host)
    for it in range(12):
        layer = int(rng.integers(0, L))
        slot0 = int(rng.integers(0, S - E + 1)) if it % 3 else (it // 3 % 2) * E * (S >= 2 * E)
        oracle.cache_install(host, layer, slot0)
        ft.cache_install(dev, layer, slot0)
        torch.cuda.synchronize()
        _same(dev, host)


def test_fetch_layer_copies_the_layer(cuda_lib):
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    L, E = 3, cfg.E
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool = torch.empty((L * E, stride), dtype=torch.uint8).pin_memory()
    synth.bank_blocks_torch(cfg.seed, range(L * E), cfg.fmt, cfg.H, cfg.I, cfg.g, pool, ref_K=cfg.ref_K)
    # a cache with a wider stride than the pool (the copy's pitches differ)
    cache_buf = torch.full((2 * E + 3, stride + 64), 0xAB, dtype=torch.uint8, device=DEV)
    cache = cache_buf[:, :stride]
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache)
    ft.fetch_layer(pb, cb, 2, E, 3)
    ft.fetch_layer(pb, cb, 0, E, 3 + E)
    torch.cuda.synchronize()
    got = cache_buf.cpu()
    assert torch.equal(got[3:3 + E, :stride], pool[2 * E:3 * E])
    assert torch.equal(got[3 + E:3 + 2 * E, :stride], pool[0:E])
    assert (got[:3] == 0xAB).all() and (got[:, stride:] == 0xAB).all()  # nothing else written
    with pytest.raises(ft.FtError):
        ft.fetch_layer(pb, cb, 3, E, 0)  # layer 3's flat ids are not in the pool
    with pytest.raises(ft.FtError):
        ft.fetch_layer(pb, cb, 0, E, E + 4)  # the slots pass the cache


@pytest.mark.parametrize("extra_slots", [5, -13])  # 2E+5 slots: double buffer; E+3: single
def test_prefill_double_buffer_matches_resident_layers(cuda_lib, extra_slots):
    """Prefill over 5 layers through the cache's first slots (the next layer
    copied by the copy engine while this one computes) gives bit for bit the
    outputs of the same calls on a bank holding every layer, leaves the state
    the oracle's install sequence gives, and matches the oracle."""
    import types

    from gpu_helpers import assert_close, oracle_pairs_output
    from quantized_expert_ffn_router_gb300.pipeline import PrefillLayers

    ft = cuda_lib
    FMT = synth.gen.FMT_NVFP4
    H, I, E, k, L, T, seed = 512, 256, 16, 4, 5, 40, 7
    S = 2 * E + extra_slots
    _, stride = synth.block_layout(FMT, H, I, 16)
    full = torch.empty((L * E, stride), dtype=torch.uint8, device=DEV)
    synth.bank_blocks_torch(seed, range(L * E), FMT, H, I, 16, full)
    pool = full.cpu().pin_memory()
    ts_np = synth.tensor_scales(FMT, H, I, L * E)
    ts = torch.from_numpy(ts_np).to(DEV)
    pb = ft.make_bank(FMT, H, I, 16, pool, ts)
    fb = ft.make_bank(FMT, H, I, 16, full, ts)
    xs_np = [synth.normal_bf16(synth.stream_key(seed, "pf-buf-x", l), (T, H)) for l in range(L)]
    xs = [torch.from_numpy(x.view(np.int16)).to(DEV) for x in xs_np]
    Ws = [torch.from_numpy(synth.router_weights(seed, l, E, H, 0.02)).to(DEV) for l in range(L)]
    # reference: the same calls per layer on the bank that holds every layer
    ref = []
    n = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    ids, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=DEV)
    rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=DEV)
    perm, inv, off = torch.empty(n, **i32), torch.empty((T, k), **i32), torch.empty(E + 1, **i32)
    xp, xsc = torch.empty((n, H), dtype=torch.int16, device=DEV), torch.empty(n, dtype=torch.float32, device=DEV)
    pws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=DEV)
    yp = torch.empty((n, H), dtype=torch.int16, device=DEV)
    ews = torch.empty(ft.experts_workspace(ft.FT_PREFILL, T, k, H, I, E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, **i32)
    for l in range(L):
        o = torch.empty((T, H), dtype=torch.int16, device=DEV)
        ft.route(xs[l], Ws[l], k, ids, w, rws)
        ft.permute(ids, E, xs[l], perm, inv, off, xp, pws, dev_status=status, xp_scale=xsc)
        ft.experts_fwd(fb, None, l, E, xp, T, k, torch.arange(l * E, (l + 1) * E, **i32), None, None, yp, ews,
                       mode=ft.FT_PREFILL, offsets=off, dev_status=status, x_scale=xsc)
        ft.combine(yp, inv, w, o)
        ref.append(o)
    # the pipeline, from an empty cache state
    state = ft.DeviceCacheState(L, E, S, device=DEV)
    cache = torch.zeros((S, stride), dtype=torch.uint8, device=DEV)
    cb = ft.make_bank(FMT, H, I, 16, cache, ts)
    pl = PrefillLayers(state, cb, pb, E, k, T, device=DEV)
    assert pl.n_buf == (2 if S >= 2 * E else 1)
    outs = [torch.empty((T, H), dtype=torch.int16, device=DEV) for _ in range(L)]
    pl(list(range(L)), xs, Ws, outs)
    torch.cuda.synchronize()
    assert ft.get_status(status) == 0 and ft.get_status(pl.status) == 0
    for l in range(L):
        assert torch.equal(outs[l], ref[l]), l
    # the state: the oracle's installs in the same order
    host = oracle.CacheState(L, E, S)
    for i in range(L):
        oracle.cache_install(host, i, (i % pl.n_buf) * E)
    _same(state, host)
    for i in range(max(0, L - pl.n_buf), L):
        b = i % pl.n_buf
        assert torch.equal(cache[b * E:(b + 1) * E].cpu(), pool[i * E:(i + 1) * E])
    # the last layer against the oracle on a few tokens, with the pipeline's routing
    cfg = types.SimpleNamespace(E=E, H=H, I=I, fmt=FMT, g=16)
    rows = np.arange(0, T, 5)
    ids_np, w_np = pl.ids.cpu().numpy()[rows], pl.w.cpu().numpy()[rows]
    lst = L - 1
    blocks = {lst * E + int(e): pool[lst * E + int(e)].numpy() for e in set(ids_np.ravel().tolist())}
    oref = oracle_pairs_output(blocks, cfg, ts_np, xs_np[lst][rows], ids_np, w_np, lst)
    got = outs[lst].cpu().numpy().view(np.uint16)[rows]
    assert_close((got.astype(np.uint32) << 16).view(np.float32), oref, "prefill through the layer buffer")

"""GPU: the combined route + resolve call (ft_moe_route_resolve) against
ft_moe_route followed by ft_moe_resolve_slots, over several steps and layers
of an evolving slot cache.  Every output must be equal bit for bit: top-k ids
and weights, slot ids, the fetch count and lists, and the whole cache state.
The shapes cover the one-kernel top-k (T * k <= 32, E <= 512: tiny at four
and eight tokens, d35b at one, flash at E = 512) with fetches, host-path
pairs and an empty cache, and shapes that run the two calls (d35b at eight
tokens, tiny at twenty)."""

import numpy as np
import pytest
import torch

import synth
from test_gpu_decode_layers import _dev_state, _seeded_host_state, _t

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _states_equal(a, b):
    return all(torch.equal(x, y) for x, y in [(a.map, b.map), (a.slot_owner, b.slot_owner), (a.usage, b.usage),
                                              (a.recency, b.recency), (a.step, b.step)])


class _Outs:
    def __init__(self, T, k, ml):
        self.ids = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
        self.w = torch.full((T, k), -7.0, dtype=torch.float32, device=DEV)
        self.sl = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
        self.nf = torch.full((1,), -7, dtype=torch.int32, device=DEV)
        self.ff = torch.full((ml,), -7, dtype=torch.int32, device=DEV)
        self.fs = torch.full((ml,), -7, dtype=torch.int32, device=DEV)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)


CASES = [("tiny", 4, 6, 26214, 2), ("tiny", 8, 6, 65536, 1), ("d35b", 1, 48, 65536, 2), ("d35b", 1, 48, 26214, 2),
         ("d35b", 1, 0, 65536, 1), ("d35b", 8, 48, 65536, 2), ("flash", 1, 64, 65536, 1), ("tiny", 20, 6, 65536, 1)]


@pytest.mark.parametrize("name,T,S,phi,L", CASES)
def test_route_resolve_matches_the_two_calls(cuda_lib, name, T, S, phi, L):
    ft = cuda_lib
    cfg = synth.get_config(name)
    E, k, H = cfg.E, cfg.k, cfg.H
    host = _seeded_host_state(L, E, S, seed=11, filled=0.5)
    st_c, st_s = _dev_state(ft, host), _dev_state(ft, host)
    Ws = [_t(synth.router_weights(cfg.seed, l, E, H, cfg.router_std, zipf_bias=cfg.zipf)) for l in range(L)]
    ml = T * k
    comb, sep = _Outs(T, k, ml), _Outs(T, k, ml)
    rws_c = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=DEV)
    rws_s = torch.zeros_like(rws_c)
    steps = 6
    xs = synth.normal_bf16(synth.stream_key(cfg.seed, "route-resolve", name, T), (steps, L, T, H))
    if cfg.zipf is not None:
        xs[..., 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
    x_all = _t(xs)
    fetched = host_pairs = 0
    for s in range(steps):
        for l in range(L):
            x = x_all[s, l]
            ft.route_resolve(x, Ws[l], k, comb.ids, comb.w, rws_c, st_c, l, phi, comb.sl, comb.nf, comb.ff, comb.fs,
                             dev_status=comb.status)
            ft.route(x, Ws[l], k, sep.ids, sep.w, rws_s)
            ft.resolve_slots(st_s, l, sep.ids, phi, sep.sl, sep.nf, sep.ff, sep.fs, sep.status)
            torch.cuda.synchronize()
            what = f"{name} T={T} S={S} phi={phi} step {s} layer {l}"
            assert torch.equal(comb.ids, sep.ids), what
            assert torch.equal(comb.w, sep.w), what
            assert torch.equal(comb.sl, sep.sl), what
            assert torch.equal(comb.nf, sep.nf), what
            assert torch.equal(comb.ff, sep.ff) and torch.equal(comb.fs, sep.fs), what
            assert _states_equal(st_c, st_s), what
            fetched += int(comb.nf.item())
            host_pairs += int((comb.sl < 0).sum().item())
    assert ft.get_status(comb.status) == 0 and ft.get_status(sep.status) == 0
    # the route workspace's arrival counter is left as the two calls leave it
    assert torch.equal(rws_c[:4], rws_s[:4])
    if S > 0 and phi == 65536:
        assert fetched > 0
    if S == 0 or phi == 26214:
        assert host_pairs > 0


def test_route_resolve_refuses_before_launching(cuda_lib):
    """A bad argument of the resolve half (max_list too small) is refused on
    the one-kernel shapes before the router runs: the top-k outputs keep their
    fill and the state is unchanged."""
    ft = cuda_lib
    cfg = synth.get_config("d35b")
    E, k, H, T = cfg.E, cfg.k, cfg.H, 1
    host = _seeded_host_state(1, E, 48, seed=5)
    st = _dev_state(ft, host)
    snap = [t.clone() for t in (st.map, st.slot_owner, st.usage, st.recency, st.step)]
    o = _Outs(T, k, 2)  # max_list 2 < min(T*k, S) = 8
    rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=DEV)
    W = _t(synth.router_weights(cfg.seed, 0, E, H, cfg.router_std, zipf_bias=cfg.zipf))
    x = _t(synth.normal_bf16(synth.stream_key(cfg.seed, "route-resolve-refuse"), (T, H)))
    with pytest.raises(ft.FtError) as ei:
        ft.route_resolve(x, W, k, o.ids, o.w, rws, st, 0, 65536, o.sl, o.nf, o.ff, o.fs, dev_status=o.status)
    assert ei.value.status == ft.FT_ERR_INVALID
    torch.cuda.synchronize()
    assert bool((o.ids == -7).all()) and bool((o.w == -7.0).all())
    for a, b in zip(snap, (st.map, st.slot_owner, st.usage, st.recency, st.step)):
        assert torch.equal(a, b)

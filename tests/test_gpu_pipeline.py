"""GPU: the decode layer split into its cache and host-path partial sums
(FT_DECODE on the cache, FT_DECODE_HOST on the pool, merged) equals the
single call; the overlapped layer pipeline (host path on a second stream next
to the fetch and the cache GEMV) matches the serial one, also replayed from a
CUDA graph; and the q* calibration measures and derives a valid phi."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_close, gapped_tokens, oracle_pairs_output, pool_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def _layer_inputs(cfg, layer, T, tag):
    W = synth.router_weights(cfg.seed, layer, cfg.E, cfg.H, cfg.router_std, zipf_bias=cfg.zipf)
    x, _ = gapped_tokens(cfg.seed, tag, T, cfg.H, W, cfg.k, cfg.gap, bias_feature=cfg.zipf is not None)
    return W, x


@pytest.mark.parametrize("name,T,cached_frac", [("tiny", 8, 0.5), ("d35b", 1, 0.5), ("d35b", 8, 0.3),
                                                ("flash", 1, 0.6), ("tiny", 4, 0.0), ("tiny", 4, 1.0)])
def test_cache_partial_plus_host_partial_equals_one_call(cuda_lib, name, T, cached_frac):
    ft = cuda_lib
    cfg = synth.get_config(name)
    E, k, layer = cfg.E, cfg.k, 0
    W, x = _layer_inputs(cfg, layer, T, "split")
    ids, w = oracle.route(x, W, k)
    w32 = w.astype(np.float32)
    used = sorted(set(ids.ravel().tolist()))
    rng = np.random.default_rng(T)
    cached = list(rng.choice(used, int(round(cached_frac * len(used))), replace=False))
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    blocks = {e: b for e, b in zip(used, pool_blocks(cfg, used))}
    cache = torch.zeros((max(len(cached), 1), stride), dtype=torch.uint8, device=DEV)
    slot_np = np.full((T, k), -1, np.int32)
    for s, e in enumerate(cached):
        cache[s].copy_(torch.from_numpy(blocks[e]))
        slot_np[ids == e] = s
    pool = torch.zeros((E, stride), dtype=torch.uint8).pin_memory()
    for e in used:
        pool[e].copy_(torch.from_numpy(blocks[e]))
    ts_np = synth.tensor_scales(cfg.fmt, cfg.H, cfg.I, cfg.L * E)
    ts = None if ts_np is None else _t(ts_np)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache, ts)
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool, ts)
    ws = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, cfg.H, cfg.I, E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = {}
    for key, bank, mode in (("full", pb, ft.FT_DECODE), ("cache", None, ft.FT_DECODE), ("host", pb, ft.FT_DECODE_HOST)):
        o = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
        ft.experts_fwd(cb, bank, layer, E, _t(x), T, k, _t(slot_np), _t(ids), _t(w32), o, ws, mode=mode,
                       dev_status=status)
        outs[key] = o
    merged = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    ft.merge_partials(outs["cache"], outs["host"], merged)
    merged32 = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
    ft.merge_partials(outs["cache"], outs["host"], merged32)
    torch.cuda.synchronize()
    assert ft.get_status(status) == 0
    full = outs["full"].cpu().numpy()
    m32 = merged32.cpu().numpy()
    # the same pairs, summed as two partials: equal up to fp32 rounding of the regrouped sum
    assert np.abs(m32 - full).max() <= 1e-5 * max(np.abs(full).max(), 1.0)
    if not cached:
        assert not outs["cache"].any()
    if len(cached) == len(used):
        assert not outs["host"].any()
    ref = oracle_pairs_output({e: blocks[e] for e in used}, cfg, ts_np, x, ids, w32, layer, np.ones((T, k), bool))
    assert_close(m32, ref, f"{name} merged partials")
    assert_close(merged.float().cpu().numpy(), ref, f"{name} merged partials bf16")


def _state_and_banks(ft, cfg, L, S, pool, seed):
    host = oracle.CacheState(L, cfg.E, S)
    rng = np.random.default_rng(seed)
    for _ in range(30):
        ids = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(2)]).astype(np.int32)
        oracle.resolve(host, int(rng.integers(0, L)), ids, 65536)
    st = ft.DeviceCacheState(L, cfg.E, S, device=DEV)
    st.load_from(host)
    cache = torch.zeros((S, pool.shape[1]), dtype=torch.uint8, device=DEV)
    for s in range(S):
        if host.slot_owner[s] >= 0:
            cache[s].copy_(pool[int(host.slot_owner[s])])
    return st, cache


@pytest.mark.parametrize("name,T,S,phi", [("tiny", 8, 6, 26214), ("d35b", 1, 40, 26214), ("d35b", 8, 60, 13107),
                                          ("tiny", 4, 6, 65536)])
def test_overlapped_layer_matches_serial_and_replays(cuda_lib, name, T, S, phi):
    ft = cuda_lib
    from quantized_expert_ffn_router_gb300.pipeline import DecodeLayer

    cfg = synth.get_config(name)
    L, E, k, layer = 2, cfg.E, cfg.k, 1
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    gen = torch.empty((L * E, stride), dtype=torch.uint8, device=DEV)
    synth.bank_blocks_torch(0, range(L * E), cfg.fmt, cfg.H, cfg.I, cfg.g, gen, ref_K=cfg.ref_K)
    pool = gen.cpu().pin_memory()
    del gen
    ts_np = synth.tensor_scales(cfg.fmt, cfg.H, cfg.I, L * E)
    ts = None if ts_np is None else _t(ts_np)
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool, ts)
    W, x = _layer_inputs(cfg, layer, T, "pipe")
    Wd, xd = _t(W), _t(x)
    outs = {}
    for mode in ("serial", "overlapped", "graph"):
        st, cache = _state_and_banks(ft, cfg, L, S, pool, seed=5)
        cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache, ts)
        dl = DecodeLayer(st, cb, pb, E, k, T, device=DEV)
        out = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
        if mode == "graph":
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    dl(layer, xd, Wd, phi, out, overlapped=True)
            torch.cuda.current_stream().wait_stream(side)
            g.replay()
        else:
            dl(layer, xd, Wd, phi, out, overlapped=(mode == "overlapped"))
        torch.cuda.synchronize()
        assert ft.get_status(dl.status) == 0
        outs[mode] = (out.cpu().numpy(), dl.slot_ids.cpu().numpy(), int(dl.num_fetch.item()),
                      st.map.cpu().numpy().copy())
    ser, ovl, gr = outs["serial"], outs["overlapped"], outs["graph"]
    # the same routing, resolution and cache updates in all three
    for o in (ovl, gr):
        assert np.array_equal(o[1], ser[1]) and o[2] == ser[2] and np.array_equal(o[3], ser[3])
        assert np.abs(o[0] - ser[0]).max() <= 1e-5 * max(np.abs(ser[0]).max(), 1.0)
    assert np.array_equal(gr[0], ovl[0])
    if phi < 65536:
        assert (ser[1] == -1).any()  # the host path is exercised
    ids, w = oracle.route(x, W, k)
    used = sorted(set((layer * E + ids).ravel().tolist()))
    blocks = {f: pool[f].numpy() for f in used}
    ref = oracle_pairs_output(blocks, cfg, ts_np, x, ids, w.astype(np.float32), layer, np.ones((T, k), bool))
    assert_close(ovl[0], ref, f"{name} overlapped layer")


def test_calibrate_frac_q16(cuda_lib):
    ft = cuda_lib
    from quantized_expert_ffn_router_gb300.pipeline import calibrate_frac_q16, frac_q16_from_bandwidths

    cfg = synth.get_config("d35b")
    E, k, L = cfg.E, cfg.k, 3
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool = torch.zeros((L * E, stride), dtype=torch.uint8).pin_memory()
    synth.bank_blocks_torch(0, range(L * E), cfg.fmt, cfg.H, cfg.I, cfg.g, pool, ref_K=cfg.ref_K)
    cache = torch.zeros((16, stride), dtype=torch.uint8, device=DEV)
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache)
    r = calibrate_frac_q16(pb, cb, E, k, n_fetch=8, reps=6, device=DEV)
    assert r["status"] == 0
    for key in ("B_P_GBs", "B_H_GBs", "B_P_alone_GBs", "B_H_alone_GBs"):
        assert 1.0 < r[key] < 2000.0, (key, r[key])
    assert 1 <= r["frac_q16"] <= 65536
    assert r["frac_q16"] == frac_q16_from_bandwidths(r["B_P_GBs"], r["B_H_GBs"])
    # the fetch wrote real blocks: the last repetition's experts are in slots 0..7
    print({k2: (round(v, 1) if isinstance(v, float) else v) for k2, v in r.items()})

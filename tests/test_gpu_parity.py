"""GPU parity: every step of the layer through the C ABI against the CPU
oracle on the same seeded inputs.  Integers bit-exact; floats within relative
L2 5e-3 and max-abs 2e-2 (bf16 outputs, fp32 accumulation)."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN
from gpu_helpers import assert_close, bf16_to_f64, gapped_tokens, oracle_pairs_output, pool_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


# ------------------------------------------------------------------- split
def test_split_q16_exhaustive(cuda_lib):
    ft = cuda_lib
    m_max = 512
    ref = oracle.split_q16_grid(m_max, 0, 65536)
    m = torch.arange(m_max + 1, dtype=torch.int32, device=DEV)
    got = torch.empty((65537, m_max + 1), dtype=torch.int32, device=DEV)
    for phi in range(65537):
        ft.split_q16(m, phi, got[phi])
    assert np.array_equal(got.cpu().numpy(), ref)


# ------------------------------------------------------------------- route
@pytest.mark.parametrize("name,T", [("tiny", 8), ("d35b", 1), ("d35b", 8), ("flash", 1), ("flash", 3),
                                    ("prefill", 37), ("d35b", 129), ("flash", 200), ("tiny", 40)])
def test_route_parity(cuda_lib, name, T):
    ft = cuda_lib
    cfg = synth.get_config(name)
    layer = 3 % cfg.L
    W = synth.router_weights(cfg.seed, layer, cfg.E, cfg.H, cfg.router_std, zipf_bias=cfg.zipf)
    x, redraws = gapped_tokens(cfg.seed, f"route-{name}", T, cfg.H, W, cfg.k, cfg.gap,
                               bias_feature=cfg.zipf is not None)
    ids_o, w_o = oracle.route(x, W, cfg.k)
    # one workspace for every call: T <= 16 keeps an arrival counter in the
    # workspace's first 256 bytes, which each call must leave at zero
    ws = torch.zeros(ft.route_workspace(T, cfg.E, cfg.H), dtype=torch.uint8, device=DEV)
    for renorm in (False, True, False):
        ids = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, cfg.k), dtype=torch.float32, device=DEV)
        ft.route(_t(x), _t(W), cfg.k, ids, w, ws, renorm=renorm)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ids_o)
        ref = w_o / w_o.sum(axis=1, keepdims=True) if renorm else w_o
        np.testing.assert_allclose(w.cpu().numpy(), ref, rtol=2e-5, atol=1e-7)
        assert not ws[:256].any()


def test_route_workspace_shared_across_token_counts(cuda_lib):
    """One zero-filled workspace sized for the largest call serves calls of
    every smaller T in any order (the arrival counter has a fixed place), and
    the tiled path (T > 16) may use it in between."""
    ft = cuda_lib
    cfg = synth.get_config("d35b")
    W = synth.router_weights(cfg.seed, 5, cfg.E, cfg.H, cfg.router_std, zipf_bias=cfg.zipf)
    ws = torch.zeros(ft.route_workspace(40, cfg.E, cfg.H), dtype=torch.uint8, device=DEV)
    for T in (8, 1, 16, 40, 1, 3, 8):
        x, _ = gapped_tokens(cfg.seed, f"route-ws-{T}", T, cfg.H, W, cfg.k, cfg.gap, bias_feature=True)
        ids_o, w_o = oracle.route(x, W, cfg.k)
        ids = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, cfg.k), dtype=torch.float32, device=DEV)
        ft.route(_t(x), _t(W), cfg.k, ids, w, ws)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ids_o), T
        np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=2e-5, atol=1e-7)
        assert not ws[:256].any(), T


def test_route_prefill_full_size_sampled(cuda_lib):
    """T = 2048 and 8192 tokens, H 4096, E 256, k 6 (tiled logits kernel): ids
    exact wherever the oracle's top-(k+1) gaps are >= 1e-4 on sampled rows; the
    rest must still be a valid top-k within fp32 rounding."""
    ft = cuda_lib
    cfg = synth.get_config("prefill")
    W = synth.router_weights(cfg.seed, 0, cfg.E, cfg.H, cfg.router_std)
    for T in cfg.tokens:
        x = synth.normal_bf16(synth.stream_key(cfg.seed, "prefill-x", T), (T, cfg.H))
        ids = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, cfg.k), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ft.route_workspace(T, cfg.E, cfg.H), dtype=torch.uint8, device=DEV)
        ft.route(_t(x), _t(W), cfg.k, ids, w, ws)
        torch.cuda.synchronize()
        rows = np.random.default_rng(T).choice(T, 96, replace=False)
        rows[:2] = [0, T - 1]
        ids_o, w_o, lg = oracle.route(x[rows], W, cfg.k, want_logits=True)
        gi = ids.cpu().numpy()[rows]
        gw = w.cpu().numpy()[rows]
        exact = 0
        for r in range(len(rows)):
            top = np.sort(lg[r])[::-1][: cfg.k + 1]
            if np.all(-np.diff(top) >= 1e-4):
                assert np.array_equal(gi[r], ids_o[r]), rows[r]
                np.testing.assert_allclose(gw[r], w_o[r], rtol=2e-5, atol=1e-7)
                exact += 1
            else:
                kth = np.sort(lg[r])[::-1][cfg.k - 1]
                assert np.all(lg[r][gi[r]] >= kth - 1e-5)
        assert exact >= 0.9 * len(rows)


# ----------------------------------------------------------------- resolve
def _dev_state(ft, host):
    st = ft.DeviceCacheState(host.L, host.E, host.S, device=DEV)
    st.load_from(host)
    return st


def _run_resolve(ft, st, layer, ids, phi, max_list, status=None):
    T, k = ids.shape
    sl = torch.empty((T, k), dtype=torch.int32, device=DEV)
    nf = torch.zeros(1, dtype=torch.int32, device=DEV)
    ff = torch.empty(max_list, dtype=torch.int32, device=DEV)
    fs = torch.empty(max_list, dtype=torch.int32, device=DEV)
    ft.resolve_slots(st, layer, _t(ids), phi, sl, nf, ff, fs, status)
    return sl, nf, ff, fs


def _same_state(dev, host):
    S = host.S
    assert np.array_equal(dev.map.cpu().numpy(), host.map)
    assert np.array_equal(dev.recency.cpu().numpy(), host.recency)
    assert int(dev.step.item()) == int(host.step[0])
    if S:
        assert np.array_equal(dev.slot_owner[:S].cpu().numpy(), host.slot_owner)
        assert np.array_equal(dev.usage[:S].cpu().numpy(), host.usage)


def test_resolve_hand_worked_trace(cuda_lib):
    ft = cuda_lib
    g = json.load(open(os.path.join(GOLDEN, "resolve_trace_hand.json")))
    st = ft.DeviceCacheState(g["L"], g["E"], g["S"], device=DEV)
    for c in g["calls"]:
        ids = np.array(c["ids"], np.int32)
        sl, nf, ff, fs = _run_resolve(ft, st, c["layer"], ids, c["phi"], len(c["fetch_fid"]))
        torch.cuda.synchronize()
        assert sl.cpu().tolist() == c["slot_ids"], c["why"]
        assert int(nf.item()) == c["num_fetch"], c["why"]
        assert ff.cpu().tolist() == c["fetch_fid"] and fs.cpu().tolist() == c["fetch_slot"], c["why"]
    f = g["final"]
    assert st.slot_owner.cpu().tolist() == f["slot_owner"] and st.usage.cpu().tolist() == f["usage"]
    assert st.map.cpu().tolist() == f["map"] and st.recency.cpu().tolist() == f["recency"]
    assert int(st.step.item()) == f["step"]


@pytest.mark.parametrize("L,E,S,k,T", [(1, 16, 6, 2, 8), (3, 64, 40, 4, 3), (2, 512, 300, 10, 1),
                                       (4, 256, 0, 8, 2), (1, 256, 256, 8, 8), (2, 40, 79, 6, 8),
                                       (8, 4096, 30000, 8, 4), (40, 256, 2560, 8, 8)])
def test_resolve_random_sequences(cuda_lib, L, E, S, k, T):
    """Random resolve sequences against the oracle.  Caches up to ~24k slots
    run the victim search on a shared-memory copy of the slot state; the
    30000-slot case does not fit and runs it on global memory."""
    ft = cuda_lib
    rng = np.random.default_rng(E * 1000 + S)
    host = oracle.CacheState(L, E, S)
    dev = _dev_state(ft, host)
    phis = [0, 1, 16384, 26214, 32768, 65535, 65536]
    max_list = T * k
    for it in range(200):
        layer = int(rng.integers(0, L))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        phi = phis[it % len(phis)]
        o = oracle.resolve(host, layer, ids, phi, max_list)
        sl, nf, ff, fs = _run_resolve(ft, dev, layer, ids, phi, max_list)
        torch.cuda.synchronize()
        assert np.array_equal(sl.cpu().numpy(), o[0]), it
        assert int(nf.item()) == o[1], it
        assert np.array_equal(ff.cpu().numpy(), o[2]) and np.array_equal(fs.cpu().numpy(), o[3]), it
    _same_state(dev, host)


def test_resolve_large_usage_ranges_radix_path(cuda_lib):
    """Victim selection when usages span many radix digits (large, sparse and
    negative step values): state seeded by hand, compared with the oracle."""
    ft = cuda_lib
    rng = np.random.default_rng(5)
    L, E, S, k, T = 4, 128, 300, 8, 4
    host = oracle.CacheState(L, E, S)
    fids = rng.choice(L * E, S - 20, replace=False)
    host.seed_slots(list(fids), usages=list(rng.integers(-5, 1 << 40, S - 20)))
    host.usage[S - 20:] = -1
    host.step[0] = (1 << 40) + 7
    host.recency[:] = rng.integers(-1, 1 << 40, L * E)
    dev = _dev_state(ft, host)
    for it in range(100):
        layer = int(rng.integers(0, L))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        o = oracle.resolve(host, layer, ids, 65536, T * k)
        sl, nf, ff, fs = _run_resolve(ft, dev, layer, ids, 65536, T * k)
        torch.cuda.synchronize()
        assert np.array_equal(sl.cpu().numpy(), o[0]) and int(nf.item()) == o[1], it
        assert np.array_equal(fs.cpu().numpy(), o[3]), it
    _same_state(dev, host)


def test_resolve_bad_id_leaves_state(cuda_lib):
    ft = cuda_lib
    host = oracle.CacheState(1, 16, 4)
    dev = _dev_state(ft, host)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sl, nf, ff, fs = _run_resolve(ft, dev, 0, np.array([[1, 16]], np.int32), 65536, 2, status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == ft.FT_ERR_BAD_ID
    assert (sl.cpu().numpy() == -1).all() and int(nf.item()) == 0
    _same_state(dev, host)


def test_resolve_sweep_million_steps(cuda_lib):
    """Cache-miss split and exactly-once sweep: 10^6 seeded decode steps over
    (E, k) in {256, 512} x {6, 8, 10}, cache 0/10/50/100% of E, ten frac_q16
    values; every step's outputs bit-exact with the oracle."""
    ft = cuda_lib
    cfg = synth.get_config("sweep")
    combos = [(E, k, f, phi) for (E, k) in cfg.extra["Ek"] for f in cfg.extra["slot_fracs"]
              for phi in cfg.phis]
    per = cfg.extra["total_steps"] // len(combos) + 1
    total = 0
    for ci, (E, k, frac, phi) in enumerate(combos):
        S = int(round(frac * E))
        ids = synth.zipf_history(ci, 1, E, k, per, s=1.1, tag="sweep")[:, 0, :].reshape(per, 1, k)
        host = oracle.CacheState(1, E, S)
        o_sl, o_nf, o_ff, o_fs = oracle.resolve_many(host, 0, ids, phi, k)
        dev = _dev_state(ft, oracle.CacheState(1, E, S))
        d_ids = _t(ids)
        sl = torch.empty((per, 1, k), dtype=torch.int32, device=DEV)
        nf = torch.zeros(per, dtype=torch.int32, device=DEV)
        ff = torch.empty((per, k), dtype=torch.int32, device=DEV)
        fs = torch.empty((per, k), dtype=torch.int32, device=DEV)
        for s in range(per):
            ft.resolve_slots(dev, 0, d_ids[s], phi, sl[s], nf[s:s + 1], ff[s], fs[s])
        torch.cuda.synchronize()
        assert np.array_equal(sl.cpu().numpy(), o_sl), (E, k, S, phi)
        assert np.array_equal(nf.cpu().numpy(), o_nf), (E, k, S, phi)
        assert np.array_equal(ff.cpu().numpy(), o_ff) and np.array_equal(fs.cpu().numpy(), o_fs)
        _same_state(dev, host)
        # exactly once: GPU ids (slot >= 0) and host ids (-1) split every top-k
        got = sl.cpu().numpy()
        assert ((got >= 0) | (got == -1)).all()
        total += per
    assert total >= cfg.extra["total_steps"]


# ------------------------------------------------------------------- fetch
@pytest.mark.parametrize("pinned", [False, True])
def test_fetch_copies_chosen_blocks(cuda_lib, pinned):
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    L, E, S = 2, cfg.E, 5
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    pool_np = pool_blocks(cfg, range(L * E))
    pool = torch.from_numpy(pool_np)
    pool = pool.pin_memory() if pinned else pool.to(DEV)
    cache = torch.zeros((S, stride), dtype=torch.uint8, device=DEV)
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache)
    host = oracle.CacheState(L, E, S)
    dev = _dev_state(ft, host)
    rng = np.random.default_rng(1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for it in range(30):
        layer = int(rng.integers(0, L))
        ids = np.stack([rng.choice(E, cfg.k, replace=False) for _ in range(3)]).astype(np.int32)
        sl, nf, ff, fs = _run_resolve(ft, dev, layer, ids, 65536, 6)
        ft.fetch(pb, cb, nf, ff, fs, status)
        torch.cuda.synchronize()
        owner = dev.slot_owner.cpu().numpy()
        c = cache.cpu().numpy()
        for s in range(S):
            if owner[s] >= 0:
                assert np.array_equal(c[s], pool_np[owner[s]]), (it, s)
    assert ft.get_status(status) == 0


# ---------------------------------------------------------- experts decode
def _decode_case(ft, cfg, T, layer, cached_frac, use_pool, pool_pinned=False, out_bf16=False, seed_tag="dec",
                 ws=None):
    """Route with the oracle, resolve on a partially filled cache, run the
    decode experts and compare with the oracle over the covered pairs."""
    E, k = cfg.E, cfg.k
    W = synth.router_weights(cfg.seed, layer, E, cfg.H, cfg.router_std, zipf_bias=cfg.zipf)
    x, _ = gapped_tokens(cfg.seed, seed_tag, T, cfg.H, W, k, cfg.gap, bias_feature=cfg.zipf is not None)
    ids, w = oracle.route(x, W, k)
    w32 = w.astype(np.float32)
    used = sorted(set(ids.ravel().tolist()))
    rng = np.random.default_rng(T * 7 + layer)
    ncache = int(round(cached_frac * len(used)))
    cached = list(rng.choice(used, ncache, replace=False)) if ncache else []
    S = max(ncache, 1)
    fids = [layer * E + e for e in used]
    blocks = {f: b for f, b in zip(fids, pool_blocks(cfg, fids))}
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    cache = torch.zeros((S, stride), dtype=torch.uint8, device=DEV)
    slot_np = np.full((T, k), -1, np.int32)
    for s, e in enumerate(cached):
        cache[s].copy_(torch.from_numpy(blocks[layer * E + e]))
        slot_np[ids == e] = s
    ts_np = synth.tensor_scales(cfg.fmt, cfg.H, cfg.I, cfg.L * E)
    ts = None if ts_np is None else _t(ts_np)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache, ts)
    pb = None
    if use_pool:
        # a pool bank indexed by flat id up to this layer, holding its used experts
        n = (layer + 1) * E
        pool = torch.zeros((n, stride), dtype=torch.uint8)
        pool = pool.pin_memory() if pool_pinned else pool.to(DEV)
        for f in fids:
            pool[f].copy_(torch.from_numpy(blocks[f]))
        pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool, ts)
    out = torch.empty((T, cfg.H), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=DEV)
    if ws is None:
        ws = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, k, cfg.H, cfg.I, E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ft.experts_fwd(cb, pb, layer, E, _t(x), T, k, _t(slot_np), _t(ids), _t(w32), out, ws, dev_status=status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == 0
    include = np.ones((T, k), bool) if use_pool else (slot_np >= 0)
    ref = oracle_pairs_output(blocks, cfg, ts_np, x, ids, w32, layer, include)
    got = out.float().cpu().numpy()
    return got, ref, x, ids, w32, slot_np, blocks, ts_np


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 8), ("tiny", 12), ("d35b", 1), ("d35b", 3), ("d35b", 8),
                                    ("d35b", 16), ("flash", 1), ("flash", 2), ("flash", 9), ("prefill", 1),
                                    ("prefill", 2)])
def test_experts_decode_all_cached(cuda_lib, name, T):
    """Every batch size up to 16 runs the pair-major kernels (the prefill
    bank's 4096-wide rows at decode: the widest one-row gate/up form)."""
    cfg = synth.get_config(name)
    got, ref, *_ = _decode_case(cuda_lib, cfg, T, layer=1 % cfg.L, cached_frac=1.0, use_pool=False)
    assert_close(got, ref, f"{name} T={T}")


@pytest.mark.parametrize("name", ["tiny", "d35b"])
def test_experts_decode_single_token_reuses_workspace(cuda_lib, name):
    """Consecutive single-token calls on one workspace stay correct (nothing
    of an earlier call leaks into the next)."""
    ft = cuda_lib
    cfg = synth.get_config(name)
    ws = torch.zeros(ft.experts_workspace(ft.FT_DECODE, 1, cfg.k, cfg.H, cfg.I, cfg.E), dtype=torch.uint8,
                     device=DEV)
    for call in range(3):
        got, ref, *_ = _decode_case(ft, cfg, 1, layer=0, cached_frac=1.0, use_pool=False,
                                    seed_tag=f"reuse{call}", ws=ws)
        assert_close(got, ref, f"{name} call {call}")


@pytest.mark.parametrize("name,T", [("tiny", 8), ("d35b", 8), ("d35b", 1), ("flash", 1)])
def test_experts_decode_masked_partial_plus_host_partial(cuda_lib, name, T):
    """Masked mode (no pool): the GPU partial over cached pairs plus the
    oracle's partial over the -1 pairs equals the full output (each pair once)."""
    cfg = synth.get_config(name)
    got, ref_gpu, x, ids, w, slot_np, blocks, ts = _decode_case(cuda_lib, cfg, T, layer=0,
                                                                cached_frac=0.5, use_pool=False)
    assert (slot_np >= 0).any() and (slot_np < 0).any()
    assert_close(got, ref_gpu, f"{name} masked")
    host_part = oracle_pairs_output(blocks, cfg, ts, x, ids, w, 0, slot_np < 0)
    full = oracle_pairs_output(blocks, cfg, ts, x, ids, w, 0, None)
    assert np.allclose(ref_gpu + host_part, full, rtol=1e-12, atol=1e-12)
    assert_close(got + host_part, full, f"{name} merged")


@pytest.mark.parametrize("name,T,pinned", [("tiny", 8, True), ("d35b", 1, True), ("flash", 1, False)])
def test_experts_decode_two_banks(cuda_lib, name, T, pinned):
    """Pairs on the host path read the pool in place (pinned host memory,
    zero-copy) in the same launch as the cached pairs."""
    cfg = synth.get_config(name)
    got, ref, *_ = _decode_case(cuda_lib, cfg, T, layer=0, cached_frac=0.4, use_pool=True,
                                pool_pinned=pinned, out_bf16=True)
    assert_close(got, ref, f"{name} two banks")


@pytest.mark.parametrize("name,T", [("tiny", 2), ("tiny", 10), ("flash", 1)])
def test_experts_decode_duplicate_ids_in_a_token(cuda_lib, name, T):
    """A token may list the same expert more than once: every pair is still
    computed once and weighted separately."""
    ft = cuda_lib
    cfg = synth.get_config(name)
    E, k, layer = cfg.E, cfg.k, 0
    rng = np.random.default_rng(77)
    ids = rng.integers(0, 3, (T, k)).astype(np.int32)  # few experts, many repeats
    w = rng.uniform(0.05, 0.3, (T, k)).astype(np.float32)
    x = synth.normal_bf16(synth.stream_key(5, "dup", T), (T, cfg.H))
    fids = [layer * E + e for e in range(3)]
    blocks = {f: b for f, b in zip(fids, pool_blocks(cfg, fids))}
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    cache = torch.from_numpy(np.stack([blocks[f] for f in fids])).to(DEV)
    ts_np = synth.tensor_scales(cfg.fmt, cfg.H, cfg.I, cfg.L * E)
    ts = None if ts_np is None else _t(ts_np)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache, ts)
    out = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ft.experts_workspace(0, T, k, cfg.H, cfg.I, E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ft.experts_fwd(cb, None, layer, E, _t(x), T, k, _t(ids), _t(ids), _t(w), out, ws, dev_status=status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == 0
    ref = oracle_pairs_output(blocks, cfg, ts_np, x, ids, w, layer)
    assert_close(out.cpu().numpy(), ref, f"{name} duplicates", ref_max=None)


def test_experts_decode_bad_ids_flagged(cuda_lib):
    ft = cuda_lib
    cfg = synth.get_config("tiny")
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    cache = torch.zeros((4, stride), dtype=torch.uint8, device=DEV)
    cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, cache)
    T, k = 2, 2
    x = torch.zeros((T, cfg.H), dtype=torch.int16, device=DEV)
    slot = torch.tensor([[0, 9], [1, -1]], dtype=torch.int32, device=DEV)  # slot 9 outside the bank
    raw = torch.tensor([[0, 1], [2, 99]], dtype=torch.int32, device=DEV)  # id 99 outside E
    w = torch.ones((T, k), dtype=torch.float32, device=DEV)
    out = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
    ws = torch.zeros(ft.experts_workspace(0, T, k, cfg.H, cfg.I, cfg.E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ft.experts_fwd(cb, None, 0, cfg.E, x, T, k, slot, raw, w, out, ws, dev_status=status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == ft.FT_ERR_BAD_ID
    assert torch.isfinite(out).all()


# ---------------------------------------------------------------- permute
@pytest.mark.parametrize("T,k,E,H", [(37, 5, 16, 64), (1, 1, 4, 8), (2048, 6, 256, 512),
                                     (8192, 6, 256, 64), (300, 2, 4096, 16), (513, 8, 7, 24)])
def test_permute_parity(cuda_lib, T, k, E, H):
    ft = cuda_lib
    rng = np.random.default_rng(T + E)
    if E >= k:
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    else:
        ids = rng.integers(0, E, (T, k)).astype(np.int32)
    x = synth.normal_bf16(synth.stream_key(0, "perm", T), (T, H))
    perm_o, inv_o, off_o = oracle.permute(ids, E)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty((T, k), dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    xp = torch.empty((T * k, H), dtype=torch.int16, device=DEV)
    ws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=DEV)
    ft.permute(_t(ids), E, _t(x), perm, inv, off, xp, ws)
    torch.cuda.synchronize()
    assert np.array_equal(perm.cpu().numpy(), perm_o)
    assert np.array_equal(inv.cpu().numpy(), inv_o)
    assert np.array_equal(off.cpu().numpy(), off_o)
    assert np.array_equal(xp.cpu().numpy().view(np.uint16), x[perm_o // k])


def test_permute_all_one_expert_and_bad_id(cuda_lib):
    ft = cuda_lib
    T, k, E = 700, 3, 9
    ids = np.full((T, k), 4, np.int32)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty((T, k), dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=DEV)
    ft.permute(_t(ids), E, None, perm, inv, off, None, ws)
    torch.cuda.synchronize()
    assert perm.cpu().tolist() == list(range(T * k))
    assert off.cpu().tolist() == [0] * 5 + [T * k] * 5
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids[5, 1] = E
    ft.permute(_t(ids), E, None, perm, inv, off, None, ws, dev_status=status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == ft.FT_ERR_BAD_ID


# ---------------------------------------------------------------- combine
@pytest.mark.parametrize("T,k,H,hp", [(5, 3, 64, False), (2048, 6, 4096, True), (1, 1, 8, True)])
def test_combine_parity(cuda_lib, T, k, H, hp):
    ft = cuda_lib
    rng = np.random.default_rng(T * k)
    yp = synth.normal_bf16(synth.stream_key(1, "yp", T), (T * k, H))
    inv = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    w = rng.uniform(0, 0.5, (T, k)).astype(np.float32)
    host = rng.standard_normal((T, H)).astype(np.float32) * 0.3 if hp else None
    out = torch.empty((T, H), dtype=torch.int16, device=DEV)
    ft.combine(_t(yp), _t(inv), _t(w), out, None if host is None else _t(host))
    torch.cuda.synchronize()
    ref = oracle.combine(yp, inv, w, host)
    got = bf16_to_f64(out.cpu().numpy().view(np.uint16))
    assert_close(got, ref, "combine", ref_max=None)

"""GPU: the speculative next-layer prefetch (NVMe-streaming post, "Where the
time actually goes", speculative copies) through the C ABI against the
oracle: the plan kernel bit-exact on the hand-worked trace and on random
resolve/prefetch sequences (state and outputs after every call), and the
speculative decode step, eager and replayed from a CUDA graph, bit-identical
to the plain step and within tolerance of the oracle's layer outputs, its
cache state equal to the oracle's resolve/prefetch sequence."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN
from gpu_helpers import assert_close, gapped_tokens, oracle_pairs_output, pool_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def _dev_state(ft, host):
    st = ft.DeviceCacheState(host.L, host.E, host.S, device=DEV)
    st.load_from(host)
    return st


def _same_state(dev, host, what=""):
    assert np.array_equal(dev.map.cpu().numpy(), host.map), what
    assert np.array_equal(dev.recency.cpu().numpy(), host.recency), what
    assert int(dev.step.item()) == int(host.step[0]), what
    if host.S:
        assert np.array_equal(dev.slot_owner[:host.S].cpu().numpy(), host.slot_owner), what
        assert np.array_equal(dev.usage[:host.S].cpu().numpy(), host.usage), what


def _lists(n):
    i32 = dict(dtype=torch.int32, device=DEV)
    return torch.zeros(1, **i32), torch.empty(n, **i32), torch.empty(n, **i32)


def test_prefetch_hand_worked_trace(cuda_lib):
    ft = cuda_lib
    g = json.load(open(os.path.join(GOLDEN, "prefetch_trace_hand.json")))
    st = ft.DeviceCacheState(g["L"], g["E"], g["S"], device=DEV)
    for c in g["calls"]:
        ids = _t(np.array(c["ids"], np.int32))
        nf, ff, fs = _lists(len(c["fetch_fid"]))
        if c["op"] == "resolve":
            sl = torch.empty_like(ids)
            ft.resolve_slots(st, c["layer"], ids, 0, sl, nf, ff, fs)
            torch.cuda.synchronize()
            assert sl.cpu().tolist() == c["slot_ids"], c["why"]
        else:
            ft.prefetch(st, c["layer"], ids, c["max_prefetch"], nf, ff, fs)
            torch.cuda.synchronize()
        assert int(nf.item()) == c["num"], c["why"]
        assert ff.cpu().tolist() == c["fetch_fid"] and fs.cpu().tolist() == c["fetch_slot"], c["why"]
        if "state" in c:
            assert st.slot_owner.cpu().tolist() == c["state"]["slot_owner"], c["why"]
            assert st.usage.cpu().tolist() == c["state"]["usage"], c["why"]
            assert int(st.step.item()) == c["state"]["step"], c["why"]
    f = g["final"]
    assert st.slot_owner.cpu().tolist() == f["slot_owner"] and st.usage.cpu().tolist() == f["usage"]
    assert st.map.cpu().tolist() == f["map"] and st.recency.cpu().tolist() == f["recency"]
    assert int(st.step.item()) == f["step"]


@pytest.mark.parametrize("L,E,S,k,T", [(3, 16, 6, 2, 4), (4, 64, 40, 4, 3), (2, 512, 300, 10, 1),
                                       (4, 256, 0, 8, 2), (40, 256, 2560, 8, 8), (2, 40, 79, 6, 8),
                                       (8, 4096, 30000, 8, 4)])
def test_prefetch_random_sequences(cuda_lib, L, E, S, k, T):
    """Decode-like sequences (per layer: resolve, then a prefetch of the next
    layer's predicted ids, right or wrong, with caps 0..T*k) against the
    oracle, bit-exact after every call.  The 30000-slot cache runs the victim
    search on global memory, the others on a shared-memory copy."""
    ft = cuda_lib
    rng = np.random.default_rng(E * 7 + S)
    host = oracle.CacheState(L, E, S)
    dev = _dev_state(ft, host)
    n = T * k
    phis = [0, 16384, 26214, 65536]
    for it in range(160):
        layer = it % L
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        o = oracle.resolve(host, layer, ids, phis[it % 4], n)
        sl = torch.empty((T, k), dtype=torch.int32, device=DEV)
        nf, ff, fs = _lists(n)
        ft.resolve_slots(dev, layer, _t(ids), phis[it % 4], sl, nf, ff, fs)
        nxt = (layer + 1) % L
        if it % 4 == 3:
            pred = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        else:  # mostly the ids of a recent call: some predicted experts resident
            pred = ids.copy()
            pred[0, 0] = int(rng.choice([e for e in range(E) if e not in pred[0]]))
        cap = int(rng.integers(0, n + 1)) if it % 5 else n
        po = oracle.prefetch(host, nxt, pred, cap, n)
        pnf, pff, pfs = _lists(n)
        ft.prefetch(dev, nxt, _t(pred), cap, pnf, pff, pfs)
        torch.cuda.synchronize()
        assert np.array_equal(sl.cpu().numpy(), o[0]) and int(nf.item()) == o[1], it
        assert np.array_equal(ff.cpu().numpy(), o[2]) and np.array_equal(fs.cpu().numpy(), o[3]), it
        assert int(pnf.item()) == po[0], it
        assert np.array_equal(pff.cpu().numpy(), po[1]) and np.array_equal(pfs.cpu().numpy(), po[2]), it
        if it % 40 == 39:
            _same_state(dev, host, it)
    _same_state(dev, host)


def test_prefetch_bad_id_leaves_state(cuda_lib):
    ft = cuda_lib
    host = oracle.CacheState(2, 16, 4)
    dev = _dev_state(ft, host)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nf, ff, fs = _lists(2)
    nf.fill_(7)
    ft.prefetch(dev, 1, _t(np.array([[3, 16]], np.int32)), 2, nf, ff, fs, status)
    torch.cuda.synchronize()
    assert ft.get_status(status) == ft.FT_ERR_BAD_ID
    assert int(nf.item()) == 0 and (ff.cpu().numpy() == -1).all()
    _same_state(dev, host)


def _spec_workload(cfg, L, T, steps, tag):
    """Per step and layer: x gapped under its own router and the next layer's
    (so both the route and the speculative route are exact), and the oracle's
    ids for both."""
    Ws = [synth.router_weights(cfg.seed, l, cfg.E, cfg.H, cfg.router_std) for l in range(L)]
    xs, ids, ws, preds = [], [], [], []
    for s in range(steps):
        xs.append([]), ids.append([]), ws.append([]), preds.append([])
        for l in range(L):
            more = (Ws[l + 1],) if l + 1 < L else ()
            x, _ = gapped_tokens(cfg.seed, f"{tag}-{s}-{l}", T, cfg.H, Ws[l], cfg.k, cfg.gap, W_more=more)
            i, w = oracle.route(x, Ws[l], cfg.k)
            xs[s].append(x), ids[s].append(i), ws[s].append(w)
            preds[s].append(oracle.route(x, Ws[l + 1], cfg.k)[0] if l + 1 < L else None)
    return Ws, xs, ids, ws, preds


@pytest.mark.parametrize("T,S", [(1, 10), (4, 10), (4, 3)])
def test_speculative_decode_step(cuda_lib, T, S):
    from quantized_expert_ffn_router_gb300.pipeline import SpeculativeDecode

    ft = cuda_lib
    cfg = synth.get_config("tiny")
    L, E, k, phi = 5, cfg.E, cfg.k, 65536
    steps_eager, steps_graph = 3, 3
    Ws, xs, ids, ws, preds = _spec_workload(cfg, L, T, steps_eager + steps_graph, f"spec{T}-{S}")
    _, stride = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    blocks = pool_blocks(cfg, range(L * E))
    by_fid = {f: blocks[f] for f in range(L * E)}
    pool = torch.from_numpy(blocks).pin_memory()
    pb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, pool)
    caches, pipes = {}, {}
    for name in ("spec", "plain"):
        caches[name] = torch.zeros((S, stride), dtype=torch.uint8, device=DEV)
        cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, caches[name])
        st = ft.DeviceCacheState(L, E, S, device=DEV)
        pipes[name] = SpeculativeDecode(st, cb, pb, E, k, T)
    host = oracle.CacheState(L, E, S)
    xb = torch.empty((L, T, cfg.H), dtype=torch.int16, device=DEV)
    Wd = [_t(W) for W in Ws]
    outs = {n: [torch.empty((T, cfg.H), dtype=torch.float32, device=DEV) for _ in range(L)] for n in pipes}

    def run(name, speculate):
        pipes[name]([xb[l] for l in range(L)], Wd, phi, outs[name], speculate=speculate)

    def check(s):
        torch.cuda.synchronize()
        for l in range(L):
            oracle.resolve(host, l, ids[s][l], phi)
            if l + 1 < L:
                oracle.prefetch(host, l + 1, preds[s][l], T * k)
            a, b = outs["spec"][l].cpu().numpy(), outs["plain"][l].cpu().numpy()
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (s, l)
            ref = oracle_pairs_output(by_fid, cfg, None, xs[s][l], ids[s][l], ws[s][l], l)
            assert_close(a, ref, f"step {s} layer {l}")
        _same_state(pipes["spec"].layer.state, host, f"step {s}")
        assert ft.get_status(pipes["spec"].layer.status) == 0
        # the cached blocks are the pool's
        st = pipes["spec"].layer.state
        owner = st.slot_owner[:S].cpu().numpy()
        for slot in np.nonzero(owner >= 0)[0]:
            assert torch.equal(caches["spec"][slot].cpu(), pool[owner[slot]]), (s, slot)

    for s in range(steps_eager):
        xb.copy_(_t(np.stack(xs[s])))
        run("spec", True)
        run("plain", False)
        check(s)
    # one step of each captured in a CUDA graph, replayed on new inputs
    graphs = {}
    for name, spec in (("spec", True), ("plain", False)):
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            run(name, spec)
        graphs[name] = g
    for s in range(steps_eager, steps_eager + steps_graph):
        xb.copy_(_t(np.stack(xs[s])))
        graphs["spec"].replay()
        graphs["plain"].replay()
        check(s)

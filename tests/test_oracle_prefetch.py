"""Pins for the oracle's speculative next-layer prefetch (CPU only).

The idea is the NVMe-streaming post's ("Where the time actually goes",
speculative copies): layer l+1's router, run on layer l's MoE input, predicts
layer l+1's experts so their copies can start a layer early.  The bookkeeping
is a reading (a fetch ahead of its resolve, with the resolve's choice rules
and two extra exclusions: slots held by predicted hits, and slots held with
usage >= step - 1, which the layer just resolved may still be reading).
"""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def test_prefetch_hand_worked_trace():
    g = json.load(open(os.path.join(GOLDEN, "prefetch_trace_hand.json")))
    st = oracle.CacheState(g["L"], g["E"], g["S"])
    for c in g["calls"]:
        ids = np.array(c["ids"], np.int32)
        if c["op"] == "resolve":
            sl, nf, ff, fs = oracle.resolve(st, c["layer"], ids, 0)
            assert sl.tolist() == c["slot_ids"], c["why"]
        else:
            nf, ff, fs = oracle.prefetch(st, c["layer"], ids, c["max_prefetch"])
        assert nf == c["num"], c["why"]
        assert ff.tolist() == c["fetch_fid"], c["why"]
        assert fs.tolist() == c["fetch_slot"], c["why"]
        if "state" in c:
            assert st.slot_owner.tolist() == c["state"]["slot_owner"], c["why"]
            assert st.usage.tolist() == c["state"]["usage"], c["why"]
            assert int(st.step[0]) == c["state"]["step"], c["why"]
    f = g["final"]
    assert st.slot_owner.tolist() == f["slot_owner"]
    assert st.usage.tolist() == f["usage"]
    assert st.map.tolist() == f["map"]
    assert st.recency.tolist() == f["recency"]
    assert int(st.step[0]) == f["step"]


def _eligible(before, layer, pred):
    """Slots a prefetch may evict, from the definition: not owned by a
    predicted expert that is resident, and not held with usage >= step-1."""
    base = layer * before.E
    now = int(before.step[0])
    out = []
    for s in range(before.S):
        o = int(before.slot_owner[s])
        if o >= 0 and base <= o < base + before.E and o - base in set(pred.ravel().tolist()):
            continue
        if o >= 0 and int(before.usage[s]) >= now - 1:
            continue
        out.append(s)
    return out


def _check_prefetch(before, after, layer, pred, cap, nf, ff, fs):
    E = before.E
    base = layer * E
    U = sorted(set(pred.ravel().tolist()))
    misses = [e for e in U if before.map[base + e] < 0]
    elig = _eligible(before, layer, pred)
    assert nf == min(len(misses), cap, len(elig))
    # brute force: the fetched set is the best nf-subset of the misses by
    # (recency desc, id asc), the victims the best nf-subset of the eligible
    # slots by (usage asc, slot asc), paired in those orders
    best_f = None
    for sub in itertools.combinations(misses, nf):
        key = sorted((-int(before.recency[base + e]), e) for e in sub)
        if best_f is None or key < best_f:
            best_f = key
    best_v = None
    for sub in itertools.combinations(elig, nf):
        key = sorted((int(before.usage[s]), s) for s in sub)
        if best_v is None or key < best_v:
            best_v = key
    assert (ff[:nf] - base).tolist() == ([e for _, e in best_f] if best_f else [])
    assert fs[:nf].tolist() == ([s for _, s in best_v] if best_v else [])
    assert (ff[nf:] == -1).all() and (fs[nf:] == -1).all()
    # state: only the victims change; each now holds its prefetched expert
    now = int(before.step[0])
    for s in range(before.S):
        if s in fs[:nf].tolist():
            i = fs[:nf].tolist().index(s)
            assert after.slot_owner[s] == ff[i] and after.map[ff[i]] == s and after.usage[s] == now
            old = int(before.slot_owner[s])
            if old >= 0:
                assert after.map[old] == -1
        else:
            assert after.slot_owner[s] == before.slot_owner[s] and after.usage[s] == before.usage[s]
    assert np.array_equal(after.recency, before.recency)
    assert int(after.step[0]) == now
    owned = after.slot_owner[after.slot_owner >= 0]
    assert len(set(owned.tolist())) == len(owned)
    for s, o in enumerate(after.slot_owner):
        if o >= 0:
            assert after.map[o] == s
    assert (after.map >= 0).sum() == len(owned)


@pytest.mark.parametrize("S", [0, 1, 3, 6])
def test_prefetch_random_sequences_bruteforce(S):
    """Decode-like sequences: per layer, a prefetch of the next layer's
    predicted ids (right or wrong), then the resolve of the actual ids."""
    rng = np.random.default_rng(300 + S)
    L, E, k = 3, 6, 2
    st = oracle.CacheState(L, E, S)
    for it in range(400):
        layer = it % L
        T = int(rng.integers(1, 3))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        if it % 3:  # mostly right: the predicted ids share experts with the actual ones
            pred = ids.copy()
            pred[0, 0] = (pred[0, 0] + int(rng.integers(0, 2))) % E
            pred[0] = pred[0] if pred[0, 0] != pred[0, 1] else ids[0]
        else:
            pred = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        cap = int(rng.integers(0, 5))
        before = st.copy()
        nf, ff, fs = oracle.prefetch(st, layer, pred, cap)
        _check_prefetch(before, st, layer, pred, cap, nf, ff, fs)
        # the resolve afterwards still covers every pair exactly once
        sl, nfr, _, _ = oracle.resolve(st, layer, ids, 65536)
        for (t, j), s in np.ndenumerate(sl):
            fid = layer * E + int(ids[t, j])
            assert (s >= 0 and st.slot_owner[s] == fid) or (s < 0 and st.map[fid] == -1)


def test_prefetch_right_guess_turns_misses_into_hits():
    """A prediction equal to the actual ids, with room, leaves the resolve
    nothing to fetch: every prefetched expert is a hit, its copy done early."""
    L, E, S, k = 2, 16, 12, 4
    rng = np.random.default_rng(5)
    st = oracle.CacheState(L, E, S)
    spec = st.copy()
    fetched_plain = fetched_spec = 0
    for it in range(60):
        layer = it % L
        ids = rng.choice(E, k, replace=False).astype(np.int32)[None, :]
        _, nf, _, _ = oracle.resolve(st, layer, ids, 0)
        fetched_plain += nf
        oracle.prefetch(spec, layer, ids, k)
        sl, nf2, _, _ = oracle.resolve(spec, layer, ids, 0)
        assert (sl >= 0).all()
        fetched_spec += nf2
        assert nf2 <= nf
    assert fetched_plain > 0 and fetched_spec < fetched_plain


def test_prefetch_zero_cache_and_zero_cap():
    st = oracle.CacheState(2, 8, 0)
    nf, ff, fs = oracle.prefetch(st, 1, np.array([[1, 2]], np.int32), 4)
    assert nf == 0 and (ff == -1).all() and (fs == -1).all()
    st = oracle.CacheState(2, 8, 4)
    before = st.copy()
    nf, _, _ = oracle.prefetch(st, 1, np.array([[1, 2]], np.int32), 0)
    assert nf == 0
    for n in ("slot_owner", "map", "usage", "recency", "step"):
        assert np.array_equal(getattr(st, n), getattr(before, n))


def test_prefetch_rejects_bad_arguments_untouched():
    st = oracle.CacheState(1, 4, 2)
    before = st.copy()
    for pred, cap in (([[0, 4]], 2), ([[-1, 1]], 2), ([[0, 1]], -1)):
        with pytest.raises(ValueError):
            oracle.prefetch(st, 0, np.array(pred, np.int32), cap)
    with pytest.raises(ValueError):
        oracle.prefetch(st, 1, np.array([[0, 1]], np.int32), 2)
    for n in ("slot_owner", "map", "usage", "recency", "step"):
        assert np.array_equal(getattr(st, n), getattr(before, n))

"""The oracle's whole-layer install (the prefill double buffer's bookkeeping)
against a hand-worked example and invariants on random states (CPU only)."""

import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _state_from(g, before):
    st = oracle.CacheState(g["L"], g["E"], g["S"])
    st.slot_owner[:] = before["slot_owner"]
    st.usage[:] = before["usage"]
    st.map[:] = -1
    for s, f in enumerate(before["slot_owner"]):
        if f >= 0:
            st.map[f] = s
    st.step[0] = before["step"]
    st.recency[:] = np.arange(g["L"] * g["E"])
    return st


def test_install_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "cache_install_hand.json")))
    st = _state_from(g, g["before"])
    rec = st.recency.copy()
    oracle.cache_install(st, g["call"]["layer"], g["call"]["slot0"])
    a = g["after"]
    assert st.slot_owner.tolist() == a["slot_owner"], g["why"]
    assert st.usage.tolist() == a["usage"], g["why"]
    assert st.map.tolist() == a["map"], g["why"]
    assert int(st.step[0]) == a["step"]
    assert np.array_equal(st.recency, rec)


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


@pytest.mark.parametrize("L,E,S,filled", [(4, 8, 16, 1.0), (3, 16, 40, 0.5), (6, 32, 64, 0.9), (2, 5, 10, 0.3)])
def test_install_invariants_on_random_states(L, E, S, filled):
    rng = np.random.default_rng(L * 100 + E)
    for it in range(50):
        st = _random_state(rng, L, E, S, filled)
        before = st.copy()
        layer = int(rng.integers(0, L))
        slot0 = int(rng.integers(0, S - E + 1))
        oracle.cache_install(st, layer, slot0)
        rng_slots = set(range(slot0, slot0 + E))
        layer_fids = set(range(layer * E, layer * E + E))
        # the range holds the layer in order, usage = step
        for e in range(E):
            assert st.slot_owner[slot0 + e] == layer * E + e
            assert st.map[layer * E + e] == slot0 + e
            assert st.usage[slot0 + e] == st.step[0]
        # map and owners are inverse; no flat id of the layer outside the range
        for s in range(S):
            f = st.slot_owner[s]
            if f >= 0:
                assert st.map[f] == s
                assert s in rng_slots or f not in layer_fids
        for f in range(L * E):
            if st.map[f] >= 0:
                assert st.slot_owner[st.map[f]] == f
        # slots outside the range: unchanged, except a dropped copy of a layer expert
        for s in set(range(S)) - rng_slots:
            if before.slot_owner[s] in layer_fids:
                assert st.slot_owner[s] == -1 and st.usage[s] == -1
            else:
                assert st.slot_owner[s] == before.slot_owner[s] and st.usage[s] == before.usage[s]
        # evicted owners of the range map to nothing
        for s in rng_slots:
            f = before.slot_owner[s]
            if f >= 0 and f not in layer_fids:
                assert st.map[f] == -1
        assert np.array_equal(st.recency, before.recency) and st.step[0] == before.step[0]


def test_install_then_resolve_hits_the_layer_and_covers_every_pair_once():
    rng = np.random.default_rng(3)
    L, E, S, k = 4, 16, 40, 4
    st = _random_state(rng, L, E, S, 0.8)
    oracle.cache_install(st, 2, 0)
    oracle.cache_install(st, 3, E)
    for layer in (2, 3):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(3)]).astype(np.int32)
        sl, nf, _, _ = oracle.resolve(st, layer, ids, 65536)
        assert nf == 0  # the whole layer is resident: every pair hits
        assert np.array_equal(sl, ids + (layer - 2) * E)


def test_install_rejects_out_of_bounds():
    st = oracle.CacheState(2, 8, 12)
    with pytest.raises(ValueError):
        oracle.cache_install(st, 2, 0)
    with pytest.raises(ValueError):
        oracle.cache_install(st, 0, 5)  # 5 + 8 > 12
    with pytest.raises(ValueError):
        oracle.cache_install(st, 0, -1)

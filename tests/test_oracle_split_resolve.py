"""Pins for the oracle's q* split and slot-cache resolution (CPU only).

split_q16 follows the FreeToken deep-dive, design pattern 2 (Q16 q* split and
its Python reference); resolve follows design patterns 3 and 5 and the
FreeToken paper post, sections 4 and 6.
"""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


# ----------------------------------------------------------------- split ----
def _brute_split(m_max: int, phis: np.ndarray) -> np.ndarray:
    """argmin over every f in 0..m of max(f*(65536-phi), (m-f)*phi), first
    minimum (the smaller f), for each m <= m_max and phi in phis (> 0)."""
    phis = phis.astype(np.int64)[None, :]
    out = np.empty((m_max + 1, phis.shape[1]), np.int64)
    for m in range(m_max + 1):
        f = np.arange(m + 1, dtype=np.int64)[:, None]
        cost = np.maximum(f * (65536 - phis), (m - f) * phis)
        out[m] = np.argmin(cost, axis=0)
    return out


def test_split_hand_worked_golden():
    g = json.load(open(os.path.join(GOLDEN, "split_q16_hand.json")))
    for c in g["cases"]:
        assert oracle.split_q16(c["m"], c["phi"]) == c["fetch"], c


def test_split_bruteforce_all_m_grid_phi():
    rng = np.random.default_rng(1)
    special = [1, 2, 3, 255, 256, 257, 16383, 16384, 16385, 26214, 27306, 27307,
               32767, 32768, 32769, 49152, 65534, 65535, 65536]
    phis = np.unique(np.concatenate([special, rng.integers(1, 65537, 400)]))
    brute = _brute_split(512, phis)
    L = oracle.lib()
    got = np.array([[L.orc_split_q16(m, int(p)) for p in phis] for m in range(513)])
    bad = np.argwhere(got != brute)
    assert bad.size == 0, [(int(m), int(phis[j]), int(got[m, j]), int(brute[m, j]))
                           for m, j in bad[:10]]


def test_split_bruteforce_small_m_every_phi():
    phis = np.arange(1, 65537)
    brute = _brute_split(24, phis)
    L = oracle.lib()
    for m in range(25):
        got = np.fromiter((L.orc_split_q16(m, int(p)) for p in phis), np.int64, len(phis))
        assert np.array_equal(got, brute[m]), m


def test_split_continuous_limit_and_edges():
    # q* ~ m * B_P / B_H (FreeToken paper post, section 6): within one of the
    # continuous optimum, monotone in phi, and all-fetch at phi = 65536.
    for m in range(0, 300, 7):
        prev = -1
        for phi in range(1, 65537, 997):
            f = oracle.split_q16(m, phi)
            assert abs(f - m * phi / 65536) <= 1.0
            assert 0 <= f <= m
            assert f >= prev
            prev = f
        assert oracle.split_q16(m, 65536) == m
        assert oracle.split_q16(m, 0) == m  # no cap at phi = 0


def test_split_remainder_closed_form():
    # cost(f) = max(f*(65536-phi), (m-f)*phi) falls until the crossing
    # f* = m*phi/65536 and rises after it, so the minimum is at lo = floor(f*)
    # or lo + 1.  Writing m*phi = 65536*lo + r, lo + 1 is strictly cheaper
    # exactly when (lo+1)*(65536-phi) < (m-lo)*phi, i.e. when r + phi > 65536.
    # The oracle tries every f; this closed form must agree over the whole
    # domain of the Q16 rule for m <= 512.
    grid = oracle.split_q16_grid(512, 1, 65536)  # [phi - 1, m]
    phi = np.arange(1, 65537, dtype=np.int64)[:, None]
    m = np.arange(513, dtype=np.int64)[None, :]
    prod = m * phi
    closed = (prod >> 16) + ((prod & 0xFFFF) + phi > 65536)
    assert np.array_equal(grid, closed)


# --------------------------------------------------------------- resolve ----
def test_resolve_hand_worked_trace():
    g = json.load(open(os.path.join(GOLDEN, "resolve_trace_hand.json")))
    st = oracle.CacheState(g["L"], g["E"], g["S"])
    for c in g["calls"]:
        ids = np.array(c["ids"], np.int32)
        sl, nf, ff, fs = oracle.resolve(st, c["layer"], ids, c["phi"])
        assert sl.tolist() == c["slot_ids"], c["why"]
        assert nf == c["num_fetch"], c["why"]
        assert ff.tolist() == c["fetch_fid"], c["why"]
        assert fs.tolist() == c["fetch_slot"], c["why"]
    f = g["final"]
    assert st.slot_owner.tolist() == f["slot_owner"]
    assert st.usage.tolist() == f["usage"]
    assert st.map.tolist() == f["map"]
    assert st.recency.tolist() == f["recency"]
    assert int(st.step[0]) == f["step"]


def _check_invariants(before, after, layer, ids, phi, sl, nf, ff, fs):
    E, S = before.E, before.S
    base = layer * E
    U = sorted(set(ids.ravel().tolist()))
    hits = [e for e in U if before.map[base + e] >= 0]
    misses = [e for e in U if before.map[base + e] < 0]
    m = len(misses)
    assert nf == min(oracle.split_q16(m, phi), S - len(hits))
    # exactly once: every pair is a slot that owns its expert, or -1
    for (t, j), s in np.ndenumerate(sl):
        fid = base + int(ids[t, j])
        if s >= 0:
            assert after.slot_owner[s] == fid and after.map[fid] == s
        else:
            assert after.map[fid] == -1
    # the host path holds exactly the misses that were not fetched
    host = {int(e) for e, s in zip(ids.ravel(), sl.ravel()) if s < 0}
    assert len(host) == m - nf
    # fetched list: distinct misses into distinct, previously non-hit slots
    got_f = ff[:nf].tolist()
    got_s = fs[:nf].tolist()
    assert len(set(got_f)) == nf and len(set(got_s)) == nf
    hit_slots = {int(before.map[base + e]) for e in hits}
    assert not (set(got_s) & hit_slots)
    assert all(f - base in misses for f in got_f)
    assert (ff[nf:] == -1).all() and (fs[nf:] == -1).all()
    # the map and the owners stay a bijection
    owned = after.slot_owner[after.slot_owner >= 0]
    assert len(set(owned.tolist())) == len(owned)
    for s, o in enumerate(after.slot_owner):
        if o >= 0:
            assert after.map[o] == s
    assert (after.map >= 0).sum() == len(owned)
    assert int(after.step[0]) == int(before.step[0]) + 1


def _brute_victims(before, layer, ids, nf):
    """Every nf-subset of the non-hit slots; the one whose sorted (usage, slot)
    keys are lexicographically smallest."""
    base = layer * before.E
    hit_slots = {int(before.map[base + e]) for e in set(ids.ravel().tolist())
                 if before.map[base + e] >= 0}
    cand = [s for s in range(before.S) if s not in hit_slots]
    best = None
    for sub in itertools.combinations(cand, nf):
        key = sorted((int(before.usage[s]), s) for s in sub)
        if best is None or key < best:
            best = key
    return [s for _, s in best] if best else []


@pytest.mark.parametrize("S", [0, 1, 3, 5])
def test_resolve_random_tiny_states_bruteforce_victims(S):
    rng = np.random.default_rng(100 + S)
    L, E, k = 2, 6, 2
    st = oracle.CacheState(L, E, S)
    phis = [0, 1, 20000, 32768, 65535, 65536]
    for it in range(300):
        layer = int(rng.integers(0, L))
        T = int(rng.integers(1, 4))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        phi = phis[it % len(phis)]
        before = st.copy()
        sl, nf, ff, fs = oracle.resolve(st, layer, ids, phi)
        _check_invariants(before, st, layer, ids, phi, sl, nf, ff, fs)
        assert fs[:nf].tolist() == _brute_victims(before, layer, ids, nf)
        # fetched misses: the nf most recent misses (ties to the lower id),
        # found by brute force over every nf-subset
        base = layer * E
        misses = [e for e in sorted(set(ids.ravel().tolist())) if before.map[base + e] < 0]
        best = None
        for sub in itertools.combinations(misses, nf):
            key = sorted((-int(before.recency[base + e]), e) for e in sub)
            if best is None or key < best:
                best = key
        assert (ff[:nf] - base).tolist() == ([e for _, e in best] if best else [])


def test_resolve_zero_and_full_cache():
    E, k = 32, 4
    rng = np.random.default_rng(7)
    empty = oracle.CacheState(1, E, 0)
    full = oracle.CacheState(1, E, E)
    for it in range(50):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(2)]).astype(np.int32)
        sl, nf, _, _ = oracle.resolve(empty, 0, ids, 65536)
        assert nf == 0 and (sl == -1).all()
        sl, nf, _, _ = oracle.resolve(full, 0, ids, 65536)
        assert (sl >= 0).all()  # a full-size cache fetches every miss
    # after every expert has been seen, a 100% cache has no misses at all
    ids = np.arange(E, dtype=np.int32).reshape(-1, k)
    oracle.resolve(full, 0, ids, 65536)
    for it in range(20):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(2)]).astype(np.int32)
        _, nf, _, _ = oracle.resolve(full, 0, ids, 0)
        assert nf == 0


def test_resolve_rejects_bad_ids_untouched():
    st = oracle.CacheState(1, 4, 2)
    before = st.copy()
    with pytest.raises(ValueError):
        oracle.resolve(st, 0, np.array([[0, 4]], np.int32), 65536)
    with pytest.raises(ValueError):
        oracle.resolve(st, 0, np.array([[-1, 1]], np.int32), 65536)
    with pytest.raises(ValueError):
        oracle.resolve(st, 0, np.array([[0, 1]], np.int32), 65537)
    assert np.array_equal(st.usage, before.usage) and int(st.step[0]) == 0


# ------------------------------------------------------------ cache rebuild
def _random_state(rng, L, E, S, steps, phi=65536):
    st = oracle.CacheState(L, E, S)
    for _ in range(steps):
        layer = int(rng.integers(0, L))
        T, k = int(rng.integers(1, 4)), int(rng.integers(1, min(E, 4) + 1))
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        oracle.resolve(st, layer, ids, phi)
    return st


@pytest.mark.parametrize("S_old,S_new", [(0, 4), (6, 0), (6, 3), (6, 6), (6, 11), (12, 5), (30, 17)])
def test_cache_rebuild_keeps_most_recently_used(S_old, S_new):
    """Properties that hold whatever the order of the work: the kept count, no
    dropped resident used later than a kept one, map = inverse of owner,
    usage carried with its expert, recency and step unchanged."""
    rng = np.random.default_rng(S_old * 31 + S_new)
    for trial in range(20):
        st = _random_state(rng, 3, 12, S_old, int(rng.integers(0, 40)))
        before = st.copy()
        new, src = oracle.cache_rebuild(st, S_new)
        for n in ("slot_owner", "map", "usage", "recency", "step"):  # the old state is only read
            assert np.array_equal(getattr(st, n), getattr(before, n))
        resident = [s for s in range(S_old) if st.slot_owner[s] >= 0]
        kept = [d for d in range(S_new) if new.slot_owner[d] >= 0]
        assert len(kept) == min(len(resident), S_new)
        assert kept == list(range(len(kept)))  # packed into the first slots
        moved = {int(src[d]) for d in kept}
        assert moved <= set(resident) and len(moved) == len(kept)
        for d in kept:
            s = int(src[d])
            assert new.slot_owner[d] == st.slot_owner[s] and new.usage[d] == st.usage[s]
        dropped = [s for s in resident if s not in moved]
        if kept and dropped:
            assert min(new.usage[d] for d in kept) >= max(st.usage[s] for s in dropped)
        assert all(new.usage[d] >= new.usage[d + 1] for d in range(len(kept) - 1))
        inv = np.full(st.L * st.E, -1, np.int32)
        for d in kept:
            inv[new.slot_owner[d]] = d
        assert np.array_equal(new.map, inv)
        assert all(new.usage[d] == -1 and src[d] == -1 for d in range(len(kept), S_new))
        assert np.array_equal(new.recency, st.recency) and new.step[0] == st.step[0]


def test_cache_rebuild_then_resolve_still_covers_every_pair_once():
    """After a rebuild to any size, resolve keeps its exactly-once rule: every
    (token, rank) pair lands on the slot of its expert or on -1, never on a
    slot holding another expert."""
    rng = np.random.default_rng(5)
    st = _random_state(rng, 2, 16, 10, 60)
    for S_new in (0, 3, 10, 20):
        new, _ = oracle.cache_rebuild(st, S_new)
        for _ in range(15):
            layer = int(rng.integers(0, 2))
            ids = np.stack([rng.choice(16, 4, replace=False) for _ in range(3)]).astype(np.int32)
            sl, nf, ff, fs = oracle.resolve(new, layer, ids, int(rng.integers(0, 65537)))
            for (t, j), s in np.ndenumerate(sl):
                assert s == -1 or new.slot_owner[s] == layer * 16 + ids[t, j]


def test_cache_rebuild_rejects_bad_owner():
    st = oracle.CacheState(1, 4, 3)
    st.slot_owner[1] = 9  # outside L*E
    st.usage[1] = 0
    with pytest.raises(ValueError):
        oracle.cache_rebuild(st, 2)

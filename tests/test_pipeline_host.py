"""The q* calibration rule on the host: phi = B_P / B_H in Q16, checked
against the pages' statement of the split (the optimal fetch count is
q* = m * B_P / B_H, the two branches taking equal time) through the oracle's
split, and the limiting cases the pages name (CPU only)."""

import numpy as np
import pytest

import oracle
from quantized_expert_ffn_router_gb300.pipeline import frac_q16_from_bandwidths


@pytest.mark.parametrize("b_p,b_h", [(28.6, 60.0), (28.6, 200.0), (200.0, 210.0), (5.0, 400.0), (63.9, 64.0)])
def test_split_with_calibrated_phi_is_q_star(b_p, b_h):
    phi = frac_q16_from_bandwidths(b_p, b_h)
    ms = np.arange(0, 513)
    got = oracle.split_q16_many(ms, phi)
    q_star = ms * b_p / b_h
    assert (np.abs(got - q_star) <= 1.0 + 1e-9).all()
    # the chosen q minimises the slower branch (per expert byte): fill q / B_P
    # against host (m - q) / (B_H - B_P), the residual host bandwidth while
    # the link is busy; brute force over every q in 0..m
    for m in (1, 7, 64, 333, 512):
        q = np.arange(m + 1)
        cost = np.maximum(q / b_p, (m - q) / (b_h - b_p))
        best = np.flatnonzero(cost <= cost.min() * (1 + 1e-12))
        assert np.min(np.abs(best - got[m])) <= 1, (m, got[m], best)


def test_fast_link_fetches_everything_slow_link_little():
    # B_P >= B_H: every miss is worth copying (q* -> m)
    assert frac_q16_from_bandwidths(100.0, 100.0) == 65536
    assert frac_q16_from_bandwidths(150.0, 100.0) == 65536
    assert oracle.split_q16(300, 65536) == 300
    # a slow link next to ample host bandwidth leaves most misses on the host
    phi = frac_q16_from_bandwidths(10.0, 1000.0)
    assert oracle.split_q16(300, phi) <= 4
    # never 0, which the split reads as "no cap"
    assert frac_q16_from_bandwidths(1e-12, 1e6) == 1
    with pytest.raises(ValueError):
        frac_q16_from_bandwidths(0.0, 1.0)


def test_speculative_decode_needs_a_pool():
    # the speculative copies come from the pool; refused before any device work
    from quantized_expert_ffn_router_gb300.pipeline import SpeculativeDecode

    with pytest.raises(ValueError):
        SpeculativeDecode(None, None, None, 8, 2, 1)


# ------------------------------------------------- validate before destroy
class _Allocs:
    """torch.full on the CPU that raises torch.cuda.OutOfMemoryError on the
    n-th allocation (the injected failure)."""

    def __init__(self, fail_at=None):
        self.n, self.fail_at = 0, fail_at

    def __call__(self, shape, dtype, fill):
        import torch

        self.n += 1
        if self.fail_at is not None and self.n == self.fail_at:
            raise torch.cuda.OutOfMemoryError("injected: allocation failed")
        return torch.full(shape, fill, dtype=dtype)


def _old_cache():
    import torch

    import quantized_expert_ffn_router_gb300 as ft

    st = ft.DeviceCacheState(2, 8, 4, device="cpu")
    st.slot_owner.copy_(torch.tensor([3, 9, -1, 12], dtype=torch.int32))
    st.usage.copy_(torch.tensor([5, 7, -1, 2], dtype=torch.int64))
    st.map[3], st.map[9], st.map[12] = 0, 1, 3
    st.step.fill_(8)
    n, stride = ft.block_bytes(0, 256, 128, 32)
    cache = torch.arange(4 * n, dtype=torch.int64).remainder(251).to(torch.uint8).reshape(4, n)
    return st, cache, n


def _snapshot(st, cache):
    return [t.clone() for t in (st.slot_owner, st.map, st.usage, st.recency, st.step, cache)]


@pytest.mark.parametrize("fail_at", [1, 2, 3, 4, 5, 6])
def test_resize_cache_allocation_failure_leaves_old_cache(fail_at):
    """Any of the six allocations of a resize (five state arrays and the bank)
    failing raises before the library is called; the running cache is as it
    was."""
    import torch

    from quantized_expert_ffn_router_gb300.pipeline import resize_cache

    st, cache, n = _old_cache()
    before = _snapshot(st, cache)
    calls = []
    with pytest.raises(torch.cuda.OutOfMemoryError):
        resize_cache(st, cache, 0, 256, 128, 32, 6, 1 << 30, alloc=_Allocs(fail_at),
                     rebuild=lambda *a, **k: calls.append(a))
    assert calls == []
    for a, b in zip(before, _snapshot(st, cache)):
        assert torch.equal(a, b)


def test_resize_cache_refused_rebuild_leaves_old_cache():
    """A rebuild the library refuses (here: over budget) propagates its
    FT_ERR_REJECTED; the old state and bank are untouched."""
    import torch

    import quantized_expert_ffn_router_gb300 as ft
    from quantized_expert_ffn_router_gb300.pipeline import resize_cache

    st, cache, n = _old_cache()
    before = _snapshot(st, cache)

    def refuse(old_state, old_bank, new_state, new_bank, budget, **kw):
        assert new_state.S == 6 and new_bank.n_blocks == 6 and new_bank.stride == n
        assert old_bank.base == cache.data_ptr()
        raise ft.FtError(ft.FT_ERR_REJECTED, "over budget")

    with pytest.raises(ft.FtError) as ei:
        resize_cache(st, cache, 0, 256, 128, 32, 6, 100, alloc=_Allocs(), rebuild=refuse)
    assert ei.value.status == ft.FT_ERR_REJECTED
    for a, b in zip(before, _snapshot(st, cache)):
        assert torch.equal(a, b)


def test_resize_cache_allocates_everything_before_the_rebuild():
    """All six allocations happen before the library call, which receives the
    new buffers; the new objects are returned."""
    from quantized_expert_ffn_router_gb300.pipeline import resize_cache

    st, cache, n = _old_cache()
    allocs = _Allocs()
    seen = []

    def rebuild(old_state, old_bank, new_state, new_bank, budget, **kw):
        seen.append((allocs.n, new_state.S, new_bank.n_blocks, budget))

    new_state, new_cache, new_bank = resize_cache(st, cache, 0, 256, 128, 32, 3, 12345, alloc=allocs,
                                                  rebuild=rebuild)
    assert seen == [(6, 3, 3, 12345)]
    assert new_state.S == 3 and tuple(new_cache.shape) == (3, n) and new_bank.base == new_cache.data_ptr()

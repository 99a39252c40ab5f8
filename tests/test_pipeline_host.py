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

"""Shared helpers of the GPU parity tests: tolerance checks, seeded inputs with
no near-ties in the router, expert banks on the device."""

from __future__ import annotations

import numpy as np

import oracle
import synth

REL_L2 = 5e-3   # relative L2 bound on bf16 / fp32 outputs
MAX_ABS = 2e-2  # max-abs bound


def assert_close(got, ref, what="", rel_l2=REL_L2, max_abs=MAX_ABS, ref_max=4.0):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if ref_max is not None:
        assert np.abs(ref).max() < ref_max, f"{what}: oracle max |y| {np.abs(ref).max():.3g} >= {ref_max}"
    den = max(np.linalg.norm(ref), 1e-30)
    rel = np.linalg.norm(got - ref) / den
    mab = np.abs(got - ref).max() if got.size else 0.0
    assert rel <= rel_l2 and mab <= max_abs, f"{what}: rel L2 {rel:.3g}, max abs {mab:.3g}"
    return rel, mab


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gapped_tokens(seed: int, tag: str, T: int, H: int, W: np.ndarray, k: int, gap: float,
                  bias_feature: bool = False, max_tries: int = 64, W_more=()):
    """x [T,H] bf16 rows, each redrawn (seeded) until the oracle's sorted logits
    at ranks 1..k+1 differ pairwise by >= gap, under W and under every router
    in W_more.  Returns (x, redraw count)."""
    x = np.empty((T, H), np.uint16)
    redraws = 0
    for t in range(T):
        for a in range(max_tries):
            row = synth.normal_bf16(synth.stream_key(seed, tag, t, a), (1, H))
            if bias_feature:
                row[0, 0] = synth.bf16_bits(np.array([1.0], np.float32))[0]
            ok = True
            for Wr in (W, *W_more):
                _, _, lg = oracle.route(row, Wr, k, want_logits=True)
                top = np.sort(lg[0])[::-1][: k + 1]
                ok = ok and bool(np.all(-np.diff(top) >= gap))
            if ok:
                break
            redraws += 1
        else:
            raise RuntimeError("could not draw a gapped row")
        x[t] = row[0]
    return x, redraws


def pool_blocks(cfg, fids) -> np.ndarray:
    return np.stack([synth.bank_block_np(cfg.seed, int(f), cfg.fmt, cfg.H, cfg.I, cfg.g, cfg.ref_K)
                     for f in fids])


def oracle_pairs_output(blocks_by_fid: dict, cfg, tscales, x_bf16, ids, w, layer, include=None):
    """Reference layer output sum_j w * expert(fid)(x) over included pairs (fp64)."""
    T, k = ids.shape
    xv = bf16_to_f64(x_bf16)
    out = np.zeros((T, cfg.H))
    for t in range(T):
        for j in range(k):
            if include is not None and not include[t, j]:
                continue
            fid = layer * cfg.E + int(ids[t, j])
            ts = None if tscales is None else tscales[fid]
            y = oracle.expert(blocks_by_fid[fid], cfg.fmt, cfg.H, cfg.I, cfg.g, xv[t], ts)
            out[t] += float(np.float32(w[t, j])) * y
    return out

"""Pins for the oracle's number formats, routing, experts, permute and combine.

Sources: the NVMe-streaming post ("Why this model": three 2560x640 NVFP4
matrices per expert; engine step 1: the 2,764,800-byte expert block), the
Edge0 summary ("What it is": 1.77 MB per int4 expert, 453 MB per layer;
"How it works": down(silu(gate x) * up x) against a dequantised reference),
and the FreeToken paper post, section 2 (router on the GPU) and section 6
(exact partial-sum merge).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN

INT4, NVFP4 = oracle.FMT_INT4, oracle.FMT_NVFP4


# --------------------------------------------------------------- formats ----
def test_e2m1_codes_match_ocp_definition():
    vals = json.load(open(os.path.join(GOLDEN, "e2m1_ocp.json")))["values"]
    for code, v in enumerate(vals):
        got = oracle.e2m1_value(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), code


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], c
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_fp16_and_bf16_all_codes():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref16 = h.view(np.float16).astype(np.float64)
    L = oracle.lib()
    got16 = np.array([L.orc_fp16_value(int(v)) for v in h])
    same = (got16 == ref16) | (np.isnan(got16) & np.isnan(ref16))
    assert same.all()
    refb = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    gotb = np.array([L.orc_bf16_value(int(v)) for v in h])
    sameb = (gotb == refb) | (np.isnan(gotb) & np.isnan(refb))
    assert sameb.all()


def test_block_sizes_match_pages():
    # NVMe post, engine step 1: one NVFP4 expert = 2,764,800 bytes = 675 pages of 4 KiB
    off, tot = oracle.block_layout(NVFP4, 2560, 640, 16)
    assert tot == 2_764_800 and tot == 675 * 4096
    assert off[3] == 3 * 819_200  # three 2560x640 matrices of 4-bit codes
    # Edge0: 1.77 MB per int4 expert, 453 MB per 256-expert layer (group 32, fp16 scales)
    _, tot32 = oracle.block_layout(INT4, 2048, 512, 32)
    assert tot32 == 1_769_472 and round(tot32 / 1e6, 2) == 1.77
    assert round(256 * tot32 / 1e6) == 453
    # the 35B-shaped layer with group 64 and the tiny layer
    assert oracle.block_layout(INT4, 2048, 512, 64)[1] == 1_671_168
    assert oracle.block_layout(INT4, 256, 128, 32)[1] == 55_296
    # the generator's layout agrees with the oracle's
    for fmt, H, I, g in [(INT4, 256, 128, 32), (INT4, 2048, 512, 64), (NVFP4, 2560, 640, 16),
                         (NVFP4, 4096, 2048, 16)]:
        assert tuple(synth.block_layout(fmt, H, I, g)[0]) == tuple(oracle.block_layout(fmt, H, I, g)[0])
        assert synth.block_layout(fmt, H, I, g)[1] == oracle.block_layout(fmt, H, I, g)[1]


def _encode_block(fmt, H, I, g, Gq, Uq, Dq, Gs, Us, Ds):
    """Pack code matrices and scale-code matrices into one block (test helper)."""
    def pack(q):
        q = q.astype(np.uint8).ravel()
        return (q[0::2] | (q[1::2] << 4)).astype(np.uint8)

    parts = [pack(Gq), pack(Uq), pack(Dq)]
    if fmt == INT4:
        parts += [np.asarray(s, np.float16).ravel().view(np.uint8) for s in (Gs, Us, Ds)]
    else:
        parts += [np.asarray(s, np.uint8).ravel() for s in (Gs, Us, Ds)]
    blk = np.concatenate(parts)
    assert blk.size == oracle.block_layout(fmt, H, I, g)[1]
    return blk


def test_int4_dequant_round_trip_and_nibble_order():
    H, I, g = 64, 32, 32
    rng = np.random.default_rng(3)
    q = [rng.integers(0, 16, (I, H)), rng.integers(0, 16, (I, H)), rng.integers(0, 16, (H, I))]
    s = [rng.uniform(0.5, 2, (I, H // g)).astype(np.float16),
         rng.uniform(0.5, 2, (I, H // g)).astype(np.float16),
         rng.uniform(0.5, 2, (H, I // g)).astype(np.float16)]
    blk = _encode_block(INT4, H, I, g, *q, *s)
    for which in range(3):
        W = oracle.dequant(blk, INT4, H, I, g, which)
        scale = np.repeat(s[which].astype(np.float64), g, axis=1)
        assert np.array_equal(W, (q[which] - 8) * scale)
    # low nibble is the even K index
    W = oracle.dequant(blk, INT4, H, I, g, 0)
    b0 = int(blk[0])
    s00 = float(s[0][0, 0])
    assert W[0, 0] == ((b0 & 15) - 8) * s00 and W[0, 1] == ((b0 >> 4) - 8) * s00


def test_nvfp4_dequant_definition():
    H, I = 32, 16
    rng = np.random.default_rng(4)
    q = [rng.integers(0, 16, (I, H)), rng.integers(0, 16, (I, H)), rng.integers(0, 16, (H, I))]
    sc = [rng.integers(0x30, 0x50, (I, H // 16)), rng.integers(0x30, 0x50, (I, H // 16)),
          rng.integers(0x30, 0x50, (H, I // 16))]
    blk = _encode_block(NVFP4, H, I, 16, *q, *sc)
    e2m1 = np.array(json.load(open(os.path.join(GOLDEN, "e2m1_ocp.json")))["values"])
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for which in range(3):
        W = oracle.dequant(blk, NVFP4, H, I, 16, which, tensor_scale=0.25)
        ref = e2m1[q[which]] * np.repeat(e4m3[sc[which]], 16, axis=1) * 0.25
        assert np.array_equal(W, ref)


# ---------------------------------------------------------------- experts ---
def _onehot_int4(H, I, g, gi, ga, gq, ui, ua, uq, dr, di, dq, s=1.0):
    """Blocks whose dequantised matrices are all zero except one entry each."""
    Gq = np.full((I, H), 8); Uq = np.full((I, H), 8); Dq = np.full((H, I), 8)
    Gq[gi, ga] = gq; Uq[ui, ua] = uq; Dq[dr, di] = dq
    sc = lambda r, c: np.full((r, c), s, np.float16)
    return _encode_block(INT4, H, I, g, Gq, Uq, Dq, sc(I, H // g), sc(I, H // g), sc(H, I // g))


def silu(v):
    return v / (1 + math.exp(-v))


def test_expert_closed_form_single_paths():
    H, I, g = 64, 32, 32
    x = np.linspace(-1.5, 2.0, H)
    # gate row 5 reads x[7], up row 5 reads x[9], down row 3 reads h[5]
    blk = _onehot_int4(H, I, g, 5, 7, 11, 5, 9, 2, 3, 5, 14)
    y = oracle.expert(blk, INT4, H, I, g, x)
    want = np.zeros(H)
    want[3] = (14 - 8) * silu((11 - 8) * x[7]) * ((2 - 8) * x[9])
    assert np.allclose(y, want, rtol=1e-15, atol=0)
    # gate and up on different rows: the product vanishes (h = silu(g) * u per row)
    blk = _onehot_int4(H, I, g, 5, 7, 11, 6, 9, 2, 3, 5, 14)
    assert np.all(oracle.expert(blk, INT4, H, I, g, x) == 0)
    # down reading a row of h that is zero gives zero
    blk = _onehot_int4(H, I, g, 5, 7, 11, 5, 9, 2, 3, 4, 14)
    assert np.all(oracle.expert(blk, INT4, H, I, g, x) == 0)


def test_expert_nvfp4_closed_form_with_tensor_scales():
    H, I = 32, 16
    Gq = np.zeros((I, H), int); Uq = np.zeros((I, H), int); Dq = np.zeros((H, I), int)
    Gq[2, 17] = 0x5   # +3.0
    Uq[2, 30] = 0xC   # -2.0
    Dq[9, 2] = 0x7    # +6.0
    sg = np.full((I, H // 16), 0x38); su = np.full((I, H // 16), 0x40); sd = np.full((H, I // 16), 0x30)
    blk = _encode_block(NVFP4, H, I, 16, Gq, Uq, Dq, sg, su, sd)
    x = np.linspace(-1, 1, H)
    ts = np.array([0.5, 0.25, 2.0], np.float32)
    y = oracle.expert(blk, NVFP4, H, I, 16, x, ts)
    # e4m3 0x38 = 1.0, 0x40 = 2.0, 0x30 = 0.5
    gv = 3.0 * 1.0 * 0.5 * x[17]
    uv = -2.0 * 2.0 * 0.25 * x[30]
    want = np.zeros(H)
    want[9] = 6.0 * 0.5 * 2.0 * silu(gv) * uv
    assert np.allclose(y, want, rtol=1e-15, atol=0)


def test_expert_matches_dense_dequantised_reference():
    # Edge0 "How it works": every path is compared with the dequantised reference.
    H, I, g = 256, 128, 32
    blk = synth.bank_block_np(5, 3, INT4, H, I, g)
    x = np.random.default_rng(0).standard_normal(H)
    G = oracle.dequant(blk, INT4, H, I, g, 0)
    U = oracle.dequant(blk, INT4, H, I, g, 1)
    D = oracle.dequant(blk, INT4, H, I, g, 2)
    gg, uu = G @ x, U @ x
    ref = D @ (gg / (1 + np.exp(-gg)) * uu)
    assert np.allclose(oracle.expert(blk, INT4, H, I, g, x), ref, rtol=1e-12, atol=1e-12)


def _tiny_pool(cfg, n):
    off, tot = synth.block_layout(cfg.fmt, cfg.H, cfg.I, cfg.g)
    return np.stack([synth.bank_block_np(cfg.seed, f, cfg.fmt, cfg.H, cfg.I, cfg.g, cfg.ref_K)
                     for f in range(n)]), tot


def test_partial_sum_merge_is_exact_and_cache_invariant():
    # FreeToken paper post, section 6: GPU and CPU partial sums add exactly;
    # deep-dive design pattern 3: each pair is computed exactly once.
    cfg = synth.get_config("tiny")
    pool, stride = _tiny_pool(cfg, cfg.E)
    x = synth.normal_bf16(synth.stream_key(0, "x"), (cfg.tokens[0], cfg.H))
    rng = np.random.default_rng(9)
    ids = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(cfg.tokens[0])]).astype(np.int32)
    w = rng.uniform(0.1, 0.5, ids.shape).astype(np.float32)
    full = oracle.moe_experts(pool, stride, None, cfg.fmt, cfg.H, cfg.I, cfg.g, 0, cfg.E, x, ids, w)
    for trial in range(5):
        mask = rng.integers(0, 2, ids.shape).astype(np.uint8)
        a = oracle.moe_experts(pool, stride, None, cfg.fmt, cfg.H, cfg.I, cfg.g, 0, cfg.E, x, ids, w, mask)
        b = oracle.moe_experts(pool, stride, None, cfg.fmt, cfg.H, cfg.I, cfg.g, 0, cfg.E, x, ids, w, 1 - mask)
        assert np.allclose(a + b, full, rtol=1e-13, atol=1e-13)
    # linear in the gate weights, zero with zero weights
    z = oracle.moe_experts(pool, stride, None, cfg.fmt, cfg.H, cfg.I, cfg.g, 0, cfg.E, x, ids, 0 * w)
    assert np.all(z == 0)
    two = oracle.moe_experts(pool, stride, None, cfg.fmt, cfg.H, cfg.I, cfg.g, 0, cfg.E, x, ids, 2 * w)
    assert np.allclose(two, 2 * full, rtol=1e-14, atol=0)
    # the tiny layer's recipe keeps outputs O(1) (max |y| < 4)
    assert np.abs(full).max() < 4


# ----------------------------------------------------------------- route ----
def test_route_constructed_logits_and_ties():
    H, E, k = 8, 6, 3
    W = np.zeros((E, H), np.float32)
    # logits = 2 * x0 * c_e with x0 = 1: c = [0.1, 0.9, 0.5, 0.9, -1, 0.3]
    c = [0.1, 0.9, 0.5, 0.9, -1.0, 0.3]
    W[:, 0] = np.array(c, np.float32) * 2
    x = synth.bf16_bits(np.array([[1.0] + [0.0] * (H - 1)], np.float32))
    ids, w, lg = oracle.route(x, W, k, want_logits=True)
    assert ids.tolist() == [[1, 3, 2]]  # the tie between experts 1 and 3 goes to the lower id
    lf = np.array(c, np.float64) * 2
    lf = np.asarray(np.float32(np.array(c, np.float32) * 2), np.float64)
    p = np.exp(lf - lf.max()) / np.exp(lf - lf.max()).sum()
    assert np.allclose(w[0], p[[1, 3, 2]], rtol=1e-14)
    ids_r, w_r = oracle.route(x, W, k, renorm=True)
    assert np.isclose(w_r.sum(), 1.0, rtol=1e-15)


def test_route_two_experts_is_a_sigmoid():
    rng = np.random.default_rng(2)
    H = 16
    W = rng.standard_normal((2, H)).astype(np.float32)
    x = synth.bf16_bits(rng.standard_normal((5, H)).astype(np.float32))
    ids, w, lg = oracle.route(x, W, 2, want_logits=True)
    d = lg[:, 0] - lg[:, 1]
    p0 = 1 / (1 + np.exp(-d))
    top = np.where(d >= 0, p0, 1 - p0)
    assert np.allclose(w[:, 0], top, rtol=1e-13)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-14)


def test_route_relabelling_equivariance_and_logit_order():
    rng = np.random.default_rng(5)
    T, H, E, k = 12, 64, 32, 6
    W = (rng.standard_normal((E, H)) * 0.2).astype(np.float32)
    x = synth.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids, w, lg = oracle.route(x, W, k, want_logits=True)
    # top-k of the softmax is the top-k of the logits (numpy ordering, ties to lower id)
    order = np.lexsort((np.tile(np.arange(E), (T, 1)), -lg), axis=1)[:, :k]
    assert np.array_equal(ids, order)
    # the logits themselves: x . W^T in fp64 from the decoded inputs
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.allclose(lg, xv @ W.astype(np.float64).T, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(E)
    ids2, w2 = oracle.route(x, W[perm], k)
    assert np.array_equal(perm[ids2], ids)
    assert np.allclose(w2, w, rtol=1e-14)


# ---------------------------------------------------------------- permute ---
def test_permute_is_the_stable_sort_by_expert():
    rng = np.random.default_rng(11)
    T, k, E = 37, 5, 16
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    perm, inv, off = oracle.permute(ids, E)
    ref = np.argsort(ids.ravel(), kind="stable")
    assert np.array_equal(perm, ref)
    assert np.array_equal(inv.ravel()[perm], np.arange(T * k))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(ids.ravel(), minlength=E))]))
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert (ids.ravel()[seg] == e).all() and (np.diff(seg) > 0).all()


def test_permute_degenerate():
    perm, inv, off = oracle.permute(np.zeros((0, 3), np.int32), 4)
    assert perm.size == 0 and off.tolist() == [0] * 5
    perm, inv, off = oracle.permute(np.full((4, 1), 2, np.int32), 4)
    assert perm.tolist() == [0, 1, 2, 3] and off.tolist() == [0, 0, 0, 4, 4]


# ---------------------------------------------------------------- combine ---
def test_combine_one_hot_and_linear():
    rng = np.random.default_rng(12)
    T, k, H = 6, 3, 16
    yp_f = rng.standard_normal((T * k, H)).astype(np.float32)
    yp = synth.bf16_bits(yp_f)
    ypv = torch.from_numpy(yp.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    inv = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    w = np.zeros((T, k), np.float32)
    w[:, 1] = 1.0
    out = oracle.combine(yp, inv, w)
    assert np.array_equal(out, ypv[inv[:, 1]])
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    hp = rng.standard_normal((T, H)).astype(np.float32)
    out = oracle.combine(yp, inv, w, hp)
    want = hp.astype(np.float64) + sum(w[:, j:j + 1].astype(np.float64) * ypv[inv[:, j]] for j in range(k))
    assert np.allclose(out, want, rtol=1e-14, atol=1e-14)


def test_grouped_rows_match_per_pair_experts():
    cfg = synth.get_config("tiny")
    pool, stride = _tiny_pool(cfg, cfg.E)
    rng = np.random.default_rng(13)
    T = 5
    ids = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    x = synth.normal_bf16(synth.stream_key(0, "xg"), (T, cfg.H))
    perm, inv, off = oracle.permute(ids, cfg.E)
    rows = np.arange(T * cfg.k, dtype=np.int32)
    yp = oracle.grouped_rows(pool, stride, None, cfg.fmt, cfg.H, cfg.I, cfg.g, 0, cfg.E, x, perm,
                             cfg.k, off, rows)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for pos in range(T * cfg.k):
        t, j = divmod(int(perm[pos]), cfg.k)
        y = oracle.expert(pool[ids[t, j]], cfg.fmt, cfg.H, cfg.I, cfg.g, xv[t])
        assert np.array_equal(yp[pos], y)


def test_expert_batch_equals_single_calls():
    cfg = synth.get_config("tiny")
    blk = synth.bank_block_np(1, 2, cfg.fmt, cfg.H, cfg.I, cfg.g)
    X = np.random.default_rng(4).standard_normal((3, cfg.H))
    Y = oracle.expert_batch(blk, cfg.fmt, cfg.H, cfg.I, cfg.g, X)
    for r in range(3):
        assert np.array_equal(Y[r], oracle.expert(blk, cfg.fmt, cfg.H, cfg.I, cfg.g, X[r]))

"""GPU parity of the prefill path: route -> permute (f16 gather) -> grouped
SwiGLU experts on tcgen05 -> combine, against the CPU oracle."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMT = synth.gen.FMT_NVFP4


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def _run_prefill(ft, H, I, E, k, ids, x, layer=0, seed=0, bank=None, slot_of=None):
    """Permute + grouped experts on the GPU; returns (yp bf16 bits, perm, offsets, bank)."""
    T = ids.shape[0]
    n = T * k
    _, stride = synth.block_layout(FMT, H, I, 16)
    if bank is None:
        bank = torch.empty((E, stride), dtype=torch.uint8, device=DEV)
        synth.bank_blocks_torch(seed, range(layer * E, (layer + 1) * E), FMT, H, I, 16, bank)
    if slot_of is None:
        slot_of = np.arange(E, dtype=np.int32)
    ts = _t(synth.tensor_scales(FMT, H, I, (layer + 1) * E))
    cb = ft.make_bank(FMT, H, I, 16, bank, ts)
    perm = torch.empty(n, dtype=torch.int32, device=DEV)
    inv = torch.empty((T, k), dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    xp = torch.empty((n, H), dtype=torch.int16, device=DEV)
    xs = torch.empty(n, dtype=torch.float32, device=DEV)
    pws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d_ids = _t(ids)
    ft.permute(d_ids, E, _t(x), perm, inv, off, xp, pws, dev_status=status, xp_scale=xs)
    yp = torch.empty((n, H), dtype=torch.int16, device=DEV)
    ews = torch.empty(ft.experts_workspace(ft.FT_PREFILL, T, k, H, I, E), dtype=torch.uint8, device=DEV)
    ft.experts_fwd(cb, None, layer, E, xp, T, k, _t(slot_of), None, None, yp, ews, mode=ft.FT_PREFILL,
                   offsets=off, dev_status=status, x_scale=xs)
    torch.cuda.synchronize()
    assert ft.get_status(status) == 0
    return yp, perm, inv, off, bank, ts


def _oracle_rows(bank_np_by_e, H, I, E, layer, x, perm, k, offsets, rows, ts_np):
    """Oracle Yp for the given permuted rows, grouped by expert (one dequant each)."""
    xv = bf16_to_f64(x)
    out = np.empty((len(rows), H))
    ex = np.searchsorted(offsets, rows, side="right") - 1
    for e in np.unique(ex):
        sel = np.nonzero(ex == e)[0]
        X = xv[perm[rows[sel]] // k]
        out[sel] = oracle.expert_batch(bank_np_by_e(e), FMT, H, I, 16, X, ts_np[layer * E + e])
    return out


@pytest.mark.parametrize("H", [256, 768, 2048, 3072, 4096, 264])  # warp(s) per token; 264: per pair
def test_permute_f16_gather_is_exact(H):
    import quantized_expert_ffn_router_gb300 as ft

    ft.load()
    T, k, E = 64, 3, 8
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    xf[5] *= 3e5     # a row beyond the f16 range gets a power-of-two prescale
    xf[6] *= 1e-3
    x = synth.bf16_bits(xf)
    n = T * k
    perm = torch.empty(n, dtype=torch.int32, device=DEV)
    inv = torch.empty((T, k), dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    xp = torch.empty((n, H), dtype=torch.int16, device=DEV)
    xs = torch.empty(n, dtype=torch.float32, device=DEV)
    ws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=DEV)
    ft.permute(_t(ids), E, _t(x), perm, inv, off, xp, ws, xp_scale=xs)
    torch.cuda.synchronize()
    p = perm.cpu().numpy()
    s_np = xs.cpu().numpy()[:, None]
    vals = xp.cpu().numpy().view(np.float16).astype(np.float64) * s_np
    ref = bf16_to_f64(x)[p // k]
    normal = np.abs(ref / s_np) >= 2.0 ** -14  # f16 normal range: exact
    assert np.array_equal(vals[normal], ref[normal])
    assert (np.abs(vals - ref) <= 2.0 ** -25 * s_np).all()  # subnormal: within half an f16 ulp
    s = xs.cpu().numpy()
    assert (s[p // k == 5] > 1).all() and (s[p // k != 5] == 1).all()
    assert (np.log2(s) == np.round(np.log2(s))).all()


@pytest.mark.parametrize("H,I,E,k,T", [(512, 256, 8, 2, 40), (256, 512, 3, 2, 300), (768, 256, 16, 4, 33)])
def test_prefill_experts_small(cuda_lib, H, I, E, k, T):
    """Every permuted row against the oracle: ragged segments, empty experts,
    segments longer than one 256-token pass."""
    ft = cuda_lib
    rng = np.random.default_rng(H + I + T)
    p = np.array([0.5, 0.3] + [0.2 / max(E - 2, 1)] * (E - 2))[:E]
    p = p / p.sum()
    ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    x = synth.normal_bf16(synth.stream_key(0, "pf-x", H, T), (T, H))
    yp, perm, inv, off, bank, ts = _run_prefill(ft, H, I, E, k, ids, x)
    bank_np = bank.cpu().numpy()
    for e in range(E):  # the device bank holds the generator's bytes
        assert np.array_equal(bank_np[e], synth.bank_block_np(0, e, FMT, H, I, 16))
    offsets = off.cpu().numpy()
    assert np.array_equal(offsets, oracle.permute(ids, E)[2])
    rows = np.arange(T * k)
    ref = _oracle_rows(lambda e: bank_np[e], H, I, E, 0, x, perm.cpu().numpy(), k, offsets, rows,
                       synth.tensor_scales(FMT, H, I, E))
    got = bf16_to_f64(yp.cpu().numpy().view(np.uint16))
    assert_close(got, ref, f"prefill rows {H}x{I}")


@pytest.mark.parametrize("E,k,T", [(400, 4, 100), (160, 4, 4000)])
def test_prefill_experts_many_items(cuda_lib, E, k, T):
    """More (row tile, expert) work items than SMs, so each persistent CTA
    walks several and its rings run on from one item to the next: 400
    experts of which most are empty (short segments, token tiles inside the A
    stages), and 160 experts of ~100 rows (mean above 96: the separate token
    ring).  Sampled permuted rows against the oracle."""
    ft = cuda_lib
    H, I = 256, 256
    rng = np.random.default_rng(E + T)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    x = synth.normal_bf16(synth.stream_key(0, "pf-items", E, T), (T, H))
    yp, perm, inv, off, bank, ts = _run_prefill(ft, H, I, E, k, ids, x, seed=3)
    bank_np = bank.cpu().numpy()
    offsets = off.cpu().numpy()
    assert np.array_equal(offsets, oracle.permute(ids, E)[2])
    n = T * k
    rows = np.unique(np.concatenate([rng.choice(n, min(n, 600), replace=False), [0, n - 1]]))
    ref = _oracle_rows(lambda e: bank_np[e], H, I, E, 0, x, perm.cpu().numpy(), k, offsets, rows,
                       synth.tensor_scales(FMT, H, I, E))
    got = bf16_to_f64(yp.cpu().numpy().view(np.uint16))[rows]
    assert_close(got, ref, f"prefill {E} experts, {T} tokens")


@pytest.mark.parametrize("T", [2048, 8192])
def test_prefill_full_layer_sampled(cuda_lib, T):
    """The whole-layer prefill shape (H 4096, I 2048, 256 experts, top-6) at
    both prompt lengths the benchmark times: route on the GPU, permute, grouped
    experts and combine; every row of four sampled experts (the largest, the
    smallest active one and two fixed ones) checked against the oracle, and
    the combine on sampled tokens."""
    ft = cuda_lib
    cfg = synth.get_config("prefill")
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    W = synth.router_weights(cfg.seed, 0, E, H, cfg.router_std)
    x = synth.normal_bf16(synth.stream_key(cfg.seed, "prefill-x", T), (T, H))
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=DEV)
    ft.route(_t(x), _t(W), k, ids, w, rws)
    torch.cuda.synchronize()
    ids_np = ids.cpu().numpy()
    yp, perm, inv, off, bank, ts = _run_prefill(ft, H, I, E, k, ids_np, x, seed=cfg.seed)
    offsets = off.cpu().numpy()
    counts = np.diff(offsets)
    assert (counts > 0).sum() >= 0.9 * E  # nearly every expert is active
    perm_np = perm.cpu().numpy()
    experts = [int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 10 ** 9))), 17, 200]
    blocks = {}
    for e in experts:
        blk = synth.bank_block_np(cfg.seed, e, FMT, H, I, 16)
        assert np.array_equal(bank[e].cpu().numpy(), blk)
        blocks[e] = blk
    rows = np.concatenate([np.arange(offsets[e], offsets[e + 1]) for e in experts])
    ref = _oracle_rows(lambda e: blocks[e], H, I, E, 0, x, perm_np, k, offsets, rows,
                       synth.tensor_scales(FMT, H, I, E))
    got = bf16_to_f64(yp.cpu().numpy().view(np.uint16)[rows])
    assert_close(got, ref, "prefill full-size rows")
    # combine: out[t] = sum_j w[t,j] Yp[inv[t,j]] for sampled tokens
    out = torch.empty((T, H), dtype=torch.int16, device=DEV)
    ft.combine(yp, inv, w, out)
    torch.cuda.synchronize()
    toks = np.array([0, 5, 1000, T // 2 + 3, T - 1])
    inv_np = inv.cpu().numpy()
    ref_c = oracle.combine(yp.cpu().numpy().view(np.uint16), inv_np[toks], w.cpu().numpy()[toks])
    got_c = bf16_to_f64(out.cpu().numpy().view(np.uint16)[toks])
    assert_close(got_c, ref_c, "prefill combine", ref_max=None)


@pytest.mark.parametrize("T", [2048, 8192])
def test_prefill_repeats_are_identical(cuda_lib, T):
    """The grouped experts call is deterministic: at the whole-layer prefill
    shape, twelve calls on the same permuted batch give byte-identical Hp
    (gate/up output) and Yp.  At 8192 tokens (192-token segments, passes of
    256) a ring stage released before its shared-memory loads had returned
    once let the refilling TMA change a few weight rows of a tile in most
    calls; this catches that class of race."""
    ft = cuda_lib
    cfg = synth.get_config("prefill")
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    n = T * k
    W = synth.router_weights(cfg.seed, 0, E, H, cfg.router_std)
    x = synth.normal_bf16(synth.stream_key(cfg.seed, "prefill-x", T), (T, H))
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    rws = torch.zeros(ft.route_workspace(T, E, H), dtype=torch.uint8, device=DEV)
    ft.route(_t(x), _t(W), k, ids, w, rws)
    torch.cuda.synchronize()
    _, perm, inv, off, bank, ts = _run_prefill(ft, H, I, E, k, ids.cpu().numpy(), x, seed=cfg.seed)
    cb = ft.make_bank(FMT, H, I, 16, bank, ts)
    xp = torch.empty((n, H), dtype=torch.int16, device=DEV)
    xs = torch.empty(n, dtype=torch.float32, device=DEV)
    pws = torch.empty(ft.permute_workspace(T, k, E), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ft.permute(ids, E, _t(x), perm, inv, off, xp, pws, dev_status=status, xp_scale=xs)
    slot = torch.arange(E, dtype=torch.int32, device=DEV)
    yp = torch.empty((n, H), dtype=torch.int16, device=DEV)
    ews = torch.empty(ft.experts_workspace(ft.FT_PREFILL, T, k, H, I, E), dtype=torch.uint8, device=DEV)
    hp0 = yp0 = None
    for rep in range(12):
        ft.experts_fwd(cb, None, 0, E, xp, T, k, slot, None, None, yp, ews, mode=ft.FT_PREFILL, offsets=off,
                       dev_status=status, x_scale=xs)
        torch.cuda.synchronize()
        assert ft.get_status(status) == 0
        hp = ews[: n * I * 2].clone()
        if hp0 is None:
            hp0, yp0 = hp, yp.clone()
        n_hp = int((hp != hp0).sum())
        n_yp = int((yp != yp0).any(dim=1).sum())
        assert n_hp == 0 and n_yp == 0, f"call {rep}: {n_hp} Hp bytes and {n_yp} Yp rows differ from the first call"

"""Input recipes: expert banks, activations, router weights, routing histories.

Expert block layout (the format both sides read): gate | up | down |
gate_scale | up_scale | down_scale, gate/up [I, H] and down [H, I] row-major
with K contiguous, two 4-bit codes per byte (low nibble = even K index).
int4 blocks carry fp16 scales per g elements of K; NVFP4 blocks carry E4M3
codes per 16 elements of K (the fp32 per-tensor scales live outside the block).
"""

from __future__ import annotations

import math

import numpy as np

from .rng import stream_key, u64_stream_np, uniform01_np

FMT_INT4 = 0
FMT_NVFP4 = 1

# E4M3 codes whose values lie in [1, 4]: 0x38 (1.0) .. 0x48 (4.0).
E4M3_CODE_LO = 0x38
E4M3_CODE_COUNT = 17


def block_layout(fmt: int, H: int, I: int, g: int):
    """Byte offsets of the six parts and the block size."""
    blk, sb = (g, 2) if fmt == FMT_INT4 else (16, 1)
    gate = I * H // 2
    down = H * I // 2
    gs = I * (H // blk) * sb
    ds = H * (I // blk) * sb
    off = [0, gate, 2 * gate, 2 * gate + down]
    off += [off[3] + gs, off[3] + 2 * gs]
    return off, off[5] + ds


def _scale_counts(fmt, H, I, g):
    blk = g if fmt == FMT_INT4 else 16
    return I * (H // blk), H * (I // blk)  # per gate (= per up), down


def int4_scale_params(H: int, I: int, ref_K):
    """(lo, hi, factor_gate_up, factor_down): fp16 scales ~ U(lo, hi) * factor.

    With ref_K None the factors are 1 (the tiny layer's recipe); otherwise each
    matrix's scales are multiplied by sqrt(ref_K / K), K its reduction length,
    which keeps activations O(1) as the fan-in grows."""
    if ref_K is None:
        return 0.005, 0.02, 1.0, 1.0
    return 0.005, 0.02, math.sqrt(ref_K / H), math.sqrt(ref_K / I)


def nvfp4_tensor_scales(H: int, I: int):
    """fp32 per-tensor scales (gate, up, down) = 1 / (2.93 * 2.5 * sqrt(K)).

    2.93 is the RMS of a uniformly drawn E2M1 code and 2.5 the mean of the
    block-scale values drawn from [1, 4]; the product keeps outputs O(1)."""
    f = lambda K: np.float32(1.0 / (2.93 * 2.5 * math.sqrt(K)))
    return np.array([f(H), f(H), f(I)], np.float32)


def tensor_scales(fmt: int, H: int, I: int, n_fids: int):
    """[n_fids, 3] fp32 per-tensor scales (NVFP4), or None for int4."""
    if fmt != FMT_NVFP4:
        return None
    return np.tile(nvfp4_tensor_scales(H, I), (n_fids, 1))


def bank_block_np(seed: int, fid: int, fmt: int, H: int, I: int, g: int = 16,
                  ref_K=None) -> np.ndarray:
    """One expert block (uint8) for flat id `fid`."""
    off, total = block_layout(fmt, H, I, g)
    out = np.empty(total, np.uint8)
    nib = off[3]
    words = (nib + 7) // 8
    z = u64_stream_np(stream_key(seed, "nib", fid), 0, words)
    out[:nib] = z.view(np.uint8)[:nib]
    n_gu, n_d = _scale_counts(fmt, H, I, g)
    n_s = 2 * n_gu + n_d
    zs = u64_stream_np(stream_key(seed, "scale", fid), 0, n_s)
    if fmt == FMT_INT4:
        lo, hi, f_gu, f_d = int4_scale_params(H, I, ref_K)
        u = (zs >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
        s = u * np.float32(hi - lo)
        s = s + np.float32(lo)
        fac = np.empty(n_s, np.float32)
        fac[: 2 * n_gu] = np.float32(f_gu)
        fac[2 * n_gu:] = np.float32(f_d)
        s = s * fac
        out[nib:] = s.astype(np.float16).view(np.uint8)
    else:
        codes = E4M3_CODE_LO + ((zs >> np.uint64(33)) % np.uint64(E4M3_CODE_COUNT))
        out[nib:] = codes.astype(np.uint8)
    return out


def bank_blocks_torch(seed: int, fids, fmt: int, H: int, I: int, g: int, out, ref_K=None,
                      chunk: int = 32):
    """Fill out[i] (uint8 torch tensor [n, >= block bytes], any device) with the
    block of fids[i]; bit-identical to bank_block_np."""
    import torch

    from .rng import u64_stream_torch_keys

    off, total = block_layout(fmt, H, I, g)
    nib = off[3]
    words = (nib + 7) // 8
    n_gu, n_d = _scale_counts(fmt, H, I, g)
    n_s = 2 * n_gu + n_d
    dev = out.device
    fids = [int(f) for f in fids]
    if fmt == FMT_INT4:
        lo, hi, f_gu, f_d = int4_scale_params(H, I, ref_K)
        fac = torch.empty(n_s, dtype=torch.float32, device=dev)
        fac[: 2 * n_gu] = float(np.float32(f_gu))
        fac[2 * n_gu:] = float(np.float32(f_d))
    for c0 in range(0, len(fids), chunk):
        sub = fids[c0:c0 + chunk]
        rows = out[c0:c0 + len(sub)]
        z = u64_stream_torch_keys([stream_key(seed, "nib", f) for f in sub], words, device=dev)
        rows[:, :nib] = z.view(torch.uint8).view(len(sub), words * 8)[:, :nib]
        zs = u64_stream_torch_keys([stream_key(seed, "scale", f) for f in sub], n_s, device=dev)
        if fmt == FMT_INT4:
            u = ((zs >> 40) & ((1 << 24) - 1)).to(torch.float32) * (2.0 ** -24)
            s = u * float(np.float32(hi - lo))
            s = s + float(np.float32(lo))
            s = s * fac[None, :]
            rows[:, nib:total] = s.to(torch.float16).view(torch.uint8).view(len(sub), 2 * n_s)
        else:
            codes = E4M3_CODE_LO + ((zs >> 33) & ((1 << 31) - 1)) % E4M3_CODE_COUNT
            rows[:, nib:total] = codes.to(torch.uint8)
    return out


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (data encoding)."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    rnd = ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((b + rnd) >> np.uint64(16)).astype(np.uint16)


def normal_f64(key: int, count: int) -> np.ndarray:
    """count standard normals (Box-Muller on pairs of 53-bit uniforms)."""
    n2 = (count + 1) // 2
    u = uniform01_np(key, 0, 2 * n2)
    u1 = 1.0 - u[0::2]  # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * n2)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:count]


def normal_f32(key: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return (normal_f64(key, n) * std).astype(np.float32).reshape(shape)


def normal_bf16(key: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) values encoded as bf16 bit patterns (uint16)."""
    return _f32_to_bf16_bits(normal_f32(key, shape, std)).reshape(shape)


def bf16_bits(values) -> np.ndarray:
    return _f32_to_bf16_bits(np.asarray(values, np.float32))


def zipf_probs(E: int, s: float = 1.1) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    return p / p.sum()


def layer_rank_perm(seed: int, layer: int, E: int) -> np.ndarray:
    """perm[rank] = expert id: which expert holds popularity rank r in a layer."""
    keys = u64_stream_np(stream_key(seed, "rankperm", layer), 0, E)
    return np.argsort(keys, kind="stable").astype(np.int32)


def zipf_history(seed: int, L: int, E: int, k: int, steps: int, s: float = 1.1,
                 tag: str = "history", layers=None) -> np.ndarray:
    """ids[step, layer, k]: k distinct experts per (step, layer), ranks drawn
    from Zipf(s) over 1..E and mapped through the layer's rank permutation."""
    cdf = np.cumsum(zipf_probs(E, s))
    cdf[-1] = 1.0
    layers = list(range(L)) if layers is None else list(layers)
    out = np.empty((steps, len(layers), k), np.int32)
    C = max(8 * k, 64)
    for li, l in enumerate(layers):
        perm = layer_rank_perm(seed, l, E)
        u = uniform01_np(stream_key(seed, tag, l), 0, steps * C).reshape(steps, C)
        cand = perm[np.searchsorted(cdf, u, side="right").clip(0, E - 1)]
        first = np.ones_like(cand, dtype=bool)
        for c in range(1, C):
            first[:, c] = ~np.any(cand[:, :c] == cand[:, c:c + 1], axis=1)
        cnt = np.cumsum(first, axis=1)
        take = first & (cnt <= k)
        good = cnt[:, -1] >= k
        out[good, li] = cand[good][take[good]].reshape(-1, k)
        for st in np.nonzero(~good)[0]:
            # vanishingly rare: top up with the lowest unused ids
            have = list(dict.fromkeys(cand[st].tolist()))
            have = (have + [e for e in range(E) if e not in have])[:k]
            out[st, li] = have
    return out


def router_weights(seed: int, layer: int, E: int, H: int, std: float = 0.02,
                   zipf_bias: float | None = None) -> np.ndarray:
    """W_router [E, H] fp32 ~ N(0, std^2).  With zipf_bias = s, column 0 holds
    log p_Zipf(s)(rank of expert e in this layer): paired with inputs whose
    feature 0 is 1.0 (a bias feature), routing then favours the layer's
    popular experts the way a Zipf(s) history does."""
    W = normal_f32(stream_key(seed, "router", layer), (E, H), std)
    if zipf_bias is not None:
        perm = layer_rank_perm(seed, layer, E)
        logp = np.log(zipf_probs(E, zipf_bias))
        col = np.empty(E, np.float64)
        col[perm] = logp
        W[:, 0] = col.astype(np.float32)
    return W

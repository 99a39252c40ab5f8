"""The C-ABI library builds, loads, exports every symbol include/ft_moe.h
declares, agrees with the oracle on the block layout, and rejects bad
arguments on the host before any CUDA call (CPU only)."""

import ctypes
import os
import re

import pytest

import oracle
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "ft_moe.h")


@pytest.fixture(scope="module")
def ft():
    from quantized_expert_ffn_router_gb300 import build as b

    b.build()
    import quantized_expert_ffn_router_gb300 as ft

    ft.load()
    return ft


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ft_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(ft):
    names = _declared()
    assert len(names) >= 15
    lib = ctypes.CDLL(ft.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps every one of them
    assert set(names) == set(ft._SIGS)


def test_block_layout_agrees_with_oracle(ft):
    for fmt, H, I, g in [(0, 256, 128, 32), (0, 2048, 512, 64), (0, 2048, 512, 32),
                         (1, 2560, 640, 16), (1, 4096, 2048, 16)]:
        n, off = ft.block_bytes(fmt, H, I, g)
        ooff, on = oracle.block_layout(fmt, H, I, g)
        assert n == on and off == ooff
    assert ft.block_bytes(0, 2048, 512, 48)[0] == 0  # unsupported group
    assert ft.block_bytes(1, 2560, 640, 32)[0] == 0  # NVFP4 blocks are 16 wide


def test_host_validation_without_gpu(ft):
    lib = ft.load()
    V = ctypes.c_void_p
    dummy = V(16)
    # split: frac_q16 outside [0, 65536]
    assert lib.ft_moe_split_q16(dummy, 4, 65537, dummy, None) == ft.FT_ERR_INVALID
    assert lib.ft_moe_split_q16(dummy, -1, 100, dummy, None) == ft.FT_ERR_INVALID
    assert "frac_q16" in ft.load().ft_last_error().decode() or True
    # route: k outside [1, min(E, 32)]
    assert lib.ft_moe_route(dummy, 1, 64, dummy, 8, 0, 0, dummy, dummy, dummy, 1 << 20, None) == ft.FT_ERR_INVALID
    assert lib.ft_moe_route(dummy, 1, 64, dummy, 8, 9, 0, dummy, dummy, dummy, 1 << 20, None) == ft.FT_ERR_INVALID
    assert lib.ft_moe_route(dummy, 1, 60, dummy, 8, 2, 0, dummy, dummy, dummy, 1 << 20, None) == ft.FT_ERR_INVALID
    # resolve: layer out of range, frac out of range, short fetch list
    st = ft.FtCacheState(2, 8, 4, dummy, dummy, dummy, dummy, dummy)
    args = lambda layer, phi, ml: (ctypes.byref(st), layer, dummy, 1, 2, phi, dummy, dummy, dummy,
                                   dummy, ml, None, None)
    assert lib.ft_moe_resolve_slots(*args(2, 100, 4)) == ft.FT_ERR_INVALID
    assert lib.ft_moe_resolve_slots(*args(0, -1, 4)) == ft.FT_ERR_INVALID
    assert lib.ft_moe_resolve_slots(*args(0, 100, 1)) == ft.FT_ERR_INVALID
    # route + resolve: on a one-kernel shape (T*k <= 32, E <= 512, the state's E) a bad
    # resolve argument (a short fetch list) is refused before anything runs; on a
    # two-call shape (k = 0 is outside the one-kernel limits) the route's check refuses
    rr = lambda T, k, ml: (dummy, T, 64, dummy, 8, k, 0, dummy, dummy, dummy, 1 << 20, ctypes.byref(st), 0, 100,
                           dummy, dummy, dummy, dummy, ml, None, None)
    assert lib.ft_moe_route_resolve(*rr(1, 2, 1)) == ft.FT_ERR_INVALID
    assert "max_list" in ft.load().ft_last_error().decode()
    assert lib.ft_moe_route_resolve(*rr(20, 0, 64)) == ft.FT_ERR_INVALID
    # prefetch: negative cap, layer out of range, short fetch list
    pargs = lambda layer, cap, ml: (ctypes.byref(st), layer, dummy, 1, 2, cap, dummy, dummy, dummy, ml,
                                    None, None)
    assert lib.ft_moe_prefetch(*pargs(0, -1, 4)) == ft.FT_ERR_INVALID
    assert lib.ft_moe_prefetch(*pargs(2, 2, 4)) == ft.FT_ERR_INVALID
    assert lib.ft_moe_prefetch(*pargs(0, 2, 1)) == ft.FT_ERR_INVALID
    # experts: unsupported bank format / misaligned base
    bad = ft.FtBank(0, 2048, 512, 48, dummy, 1 << 21, 4, None)
    assert lib.ft_moe_experts_fwd(ctypes.byref(bad), None, 0, 8, dummy, None, 1, dummy, dummy, dummy, 2, 0,
                                  None, dummy, 0, dummy, 1 << 20, None, None) == ft.FT_ERR_UNSUPPORTED
    mis = ft.FtBank(0, 256, 128, 32, V(8), 55296, 4, None)
    assert lib.ft_moe_experts_fwd(ctypes.byref(mis), None, 0, 8, dummy, None, 1, dummy, dummy, dummy, 2, 0,
                                  None, dummy, 0, dummy, 1 << 20, None, None) == ft.FT_ERR_INVALID
    nvfp4_no_scale = ft.FtBank(1, 2560, 640, 16, dummy, 2764800, 4, None)
    assert lib.ft_moe_fetch(ctypes.byref(nvfp4_no_scale), ctypes.byref(nvfp4_no_scale), dummy, dummy,
                            dummy, 1, None, None) == ft.FT_ERR_INVALID
    # decode limits: too many pairs
    ok = ft.FtBank(0, 256, 128, 32, dummy, 55296, 4, None)
    assert lib.ft_moe_experts_fwd(ctypes.byref(ok), None, 0, 16, dummy, None, 200, dummy, dummy, dummy, 2, 0,
                                  None, dummy, 0, dummy, 1 << 30, None, None) == ft.FT_ERR_INVALID
    # permute / combine shapes
    assert lib.ft_moe_permute(dummy, 4, 2, 5000, None, 0, dummy, dummy, dummy, None, 0, None, dummy,
                              1 << 20, None, None) == ft.FT_ERR_INVALID
    assert lib.ft_moe_permute(dummy, 4, 2, 8, dummy, 16, dummy, dummy, dummy, dummy, 1, None, dummy,
                              1 << 20, None, None) == ft.FT_ERR_INVALID  # f16 gather without xp_scale
    assert lib.ft_moe_combine(dummy, dummy, dummy, 4, 2, 12, None, dummy, None) == ft.FT_ERR_INVALID
    assert ft.load().ft_status_string(ft.FT_ERR_BAD_ID).decode() == "expert id out of range"



def test_cache_rebuild_refusals_without_gpu(ft):
    """Every refusal is decided on the host, before anything is enqueued."""
    lib = ft.load()
    V = ctypes.c_void_p
    stride = 55296  # tiny int4 block
    old_bank = ft.FtBank(0, 256, 128, 32, V(1 << 20), stride, 8, None)
    new_bank = ft.FtBank(0, 256, 128, 32, V(1 << 30), stride, 8, None)

    def state(L, E, S, base):
        return ft.FtCacheState(L, E, S, V(base), V(base + 0x1000), V(base + 0x2000), V(base + 0x3000),
                               V(base + 0x4000))

    old = state(2, 16, 8, 1 << 24)
    big = 1 << 40

    def rebuild(new, nb=new_bank, budget=big, ob=old_bank):
        return lib.ft_moe_cache_rebuild(ctypes.byref(old), ctypes.byref(ob), ctypes.byref(new), ctypes.byref(nb),
                                        budget, None, None)

    assert rebuild(state(2, 32, 4, 1 << 28)) == ft.FT_ERR_REJECTED  # another model's E
    assert rebuild(state(3, 16, 4, 1 << 28)) == ft.FT_ERR_REJECTED  # another L
    other = ft.FtBank(0, 256, 128, 64, V(1 << 30), 53248, 8, None)
    assert ft.block_bytes(0, 256, 128, 64)[0] <= 53248
    assert rebuild(state(2, 16, 4, 1 << 28), nb=other) == ft.FT_ERR_REJECTED  # another group size
    assert rebuild(state(2, 16, 9, 1 << 28)) == ft.FT_ERR_REJECTED  # 9 slots, 8 blocks in the bank
    assert rebuild(state(2, 16, 4, 1 << 28), budget=4 * stride) == ft.FT_ERR_REJECTED  # state bytes too
    assert rebuild(state(2, 16, 4, 1 << 28), nb=old_bank) == ft.FT_ERR_REJECTED  # the old bank itself
    assert rebuild(state(2, 16, 4, (1 << 24) + 0x2000)) == ft.FT_ERR_REJECTED  # aliases the old arrays
    assert rebuild(state(2, 16, 4, 1 << 28), budget=4 * stride) == ft.FT_ERR_REJECTED
    assert "budget" in lib.ft_last_error().decode()
    # malformed calls are invalid, not refused
    assert rebuild(state(2, 16, -1, 1 << 28)) == ft.FT_ERR_INVALID
    assert lib.ft_moe_cache_rebuild(None, ctypes.byref(old_bank), None, ctypes.byref(new_bank), big, None,
                                    None) == ft.FT_ERR_INVALID
    assert lib.ft_status_string(ft.FT_ERR_REJECTED).decode() == "cache rebuild rejected"


def test_binding_fails_loudly_without_library(tmp_path):
    import quantized_expert_ffn_router_gb300 as ftmod

    saved = ftmod._lib
    ftmod._lib = None
    try:
        with pytest.raises(ftmod.FtError):
            ftmod.load(str(tmp_path / "missing.so"))
    finally:
        ftmod._lib = saved

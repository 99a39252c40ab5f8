"""Python binding of libft_moe.so, the routed quantized expert-FFN MoE layer
for GB300 (sm_103a).

Argument marshalling only: every function passes torch tensors' data pointers
and the current CUDA stream straight to the C ABI declared in
include/ft_moe.h, and raises FtError on a non-zero status.  There is no
fallback: if the shared library is missing or fails to load, load() raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libft_moe.so")

(FT_OK, FT_ERR_INVALID, FT_ERR_UNSUPPORTED, FT_ERR_CUDA, FT_ERR_TIMEOUT, FT_ERR_BAD_ID, FT_ERR_RANGE,
 FT_ERR_REJECTED) = range(8)
FT_INT4, FT_NVFP4 = 0, 1
FT_DECODE, FT_PREFILL, FT_DECODE_HOST = 0, 1, 2
FT_OUT_F32, FT_OUT_BF16 = 0, 1
FT_XP_BF16, FT_XP_F16 = 0, 1

_lib = None


class FtError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"ft_moe status {status}: {message}")
        self.status = status


class FtBank(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("group", ctypes.c_int32), ("base", ctypes.c_void_p), ("stride", ctypes.c_uint64),
                ("n_blocks", ctypes.c_int64), ("tensor_scale", ctypes.c_void_p)]


class FtCacheState(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("E", ctypes.c_int32), ("S", ctypes.c_int32),
                ("slot_owner", ctypes.c_void_p), ("map", ctypes.c_void_p),
                ("usage", ctypes.c_void_p), ("recency", ctypes.c_void_p), ("step", ctypes.c_void_p)]


_V, _I32, _I64, _U64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
_SIGS = {
    "ft_version": (ctypes.c_char_p, []),
    "ft_status_string": (ctypes.c_char_p, [_I32]),
    "ft_last_error": (ctypes.c_char_p, []),
    "ft_block_bytes": (_U64, [_I32, _I32, _I32, _I32, _V]),
    "ft_moe_get_status": (_I32, [_V, _V]),
    "ft_moe_route_workspace": (_SZ, [_I32, _I32, _I32]),
    "ft_moe_route": (_I32, [_V, _I32, _I32, _V, _I32, _I32, _I32, _V, _V, _V, _SZ, _V]),
    "ft_moe_split_q16": (_I32, [_V, _I32, _I32, _V, _V]),
    "ft_moe_resolve_slots": (_I32, [_V, _I32, _V, _I32, _I32, _I32, _V, _V, _V, _V, _I32, _V, _V]),
    "ft_moe_route_resolve": (_I32, [_V, _I32, _I32, _V, _I32, _I32, _I32, _V, _V, _V, _SZ, _V, _I32, _I32, _V, _V,
                                    _V, _V, _I32, _V, _V]),
    "ft_moe_prefetch": (_I32, [_V, _I32, _V, _I32, _I32, _I32, _V, _V, _V, _I32, _V, _V]),
    "ft_moe_fetch": (_I32, [_V, _V, _V, _V, _V, _I32, _V, _V]),
    "ft_moe_fetch_layer": (_I32, [_V, _V, _I32, _I32, _I32, _V]),
    "ft_moe_cache_install": (_I32, [_V, _I32, _I32, _V]),
    "ft_moe_cache_rebuild": (_I32, [_V, _V, _V, _V, _U64, _V, _V]),
    "ft_moe_experts_workspace": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "ft_moe_experts_fwd": (_I32, [_V, _V, _I32, _I32, _V, _V, _I32, _V, _V, _V, _I32, _I32, _V, _V,
                                  _I32, _V, _SZ, _V, _V]),
    "ft_moe_experts_decode_static": (_I32, [_V, _V, _I32, _I32, _V, _I32, _V, _V, _V, _I32, _V, _I32,
                                            _V, _V]),
    "ft_moe_permute_workspace": (_SZ, [_I32, _I32, _I32]),
    "ft_moe_permute": (_I32, [_V, _I32, _I32, _I32, _V, _I32, _V, _V, _V, _V, _I32, _V, _V, _SZ, _V,
                              _V]),
    "ft_moe_combine": (_I32, [_V, _V, _V, _I32, _I32, _I32, _V, _V, _V]),
    "ft_moe_merge_partials": (_I32, [_V, _V, _I64, _V, _I32, _V]),
    "ft_moe_decode_layer_workspace": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "ft_moe_decode_layer": (_I32, [_V, _I32, _V, _I32, _I32, _V, _I32, _I32, _V, _V, _V, _V, _V, _V, _V, _V,
                                   _I32, _V, _I32, _V, _SZ, _V, _V]),
    "ft_set_wait_limit_ns": (_I32, [_U64]),
}


def load(path: str | None = None):
    """Load libft_moe.so (in-tree).  Raises if it is missing or incomplete."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FtError(FT_ERR_UNSUPPORTED,
                      f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)  # AttributeError if a declared symbol is not exported
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if isinstance(stream, int):  # a raw cudaStream_t handle (0: the legacy default stream)
        return ctypes.c_void_p(stream)
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int):
    if status != FT_OK:
        raise FtError(status, _lib.ft_last_error().decode())


def version() -> str:
    return load().ft_version().decode()


def block_bytes(fmt: int, H: int, I: int, group: int):
    off = (ctypes.c_uint64 * 6)()
    n = load().ft_block_bytes(fmt, H, I, group, off)
    return int(n), [int(v) for v in off]


def make_bank(fmt: int, H: int, I: int, group: int, blocks, tensor_scale=None) -> FtBank:
    """blocks: uint8 tensor [n_blocks, stride] (device or pinned host)."""
    n, stride = int(blocks.shape[0]), int(blocks.stride(0)) * blocks.element_size()
    return FtBank(fmt, H, I, group, ctypes.c_void_p(blocks.data_ptr()), stride, n,
                  None if tensor_scale is None else ctypes.c_void_p(tensor_scale.data_ptr()))


class DeviceCacheState:
    """The slot-cache state as device tensors plus its ft_cache_state view."""

    def __init__(self, L: int, E: int, S: int, device="cuda", recency_init: int = -1, alloc=None):
        """alloc(shape, dtype, fill) -> tensor, default torch.full on `device`."""
        import torch

        if alloc is None:
            def alloc(shape, dtype, fill):
                return torch.full(shape, fill, dtype=dtype, device=device)
        self.L, self.E, self.S = L, E, S
        self.slot_owner = alloc((max(S, 1),), torch.int32, -1)
        self.map = alloc((L * E,), torch.int32, -1)
        self.usage = alloc((max(S, 1),), torch.int64, -1)
        self.recency = alloc((L * E,), torch.int64, recency_init)
        self.step = alloc((1,), torch.int64, 0)

    def struct(self) -> FtCacheState:
        return FtCacheState(self.L, self.E, self.S, _ptr(self.slot_owner), _ptr(self.map),
                            _ptr(self.usage), _ptr(self.recency), _ptr(self.step))

    def load_from(self, host):
        """Copy a host state (numpy arrays with the same fields) to the device."""
        import torch

        S = self.S
        if S:
            self.slot_owner[:S].copy_(torch.from_numpy(host.slot_owner))
            self.usage[:S].copy_(torch.from_numpy(host.usage))
        self.map.copy_(torch.from_numpy(host.map))
        self.recency.copy_(torch.from_numpy(host.recency))
        self.step.copy_(torch.from_numpy(host.step))


# ------------------------------------------------------------------ entries
def route_workspace(T: int, E: int, H: int) -> int:
    return int(load().ft_moe_route_workspace(T, E, H))


def route(x, w_router, k: int, topk_ids, topk_w, ws, renorm: bool = False, stream=None):
    T, H = x.shape
    E = w_router.shape[0]
    _check(load().ft_moe_route(_ptr(x), T, H, _ptr(w_router), E, k, int(bool(renorm)), _ptr(topk_ids),
                               _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def split_q16(num_missing, frac_q16: int, num_fetch, stream=None):
    _check(load().ft_moe_split_q16(_ptr(num_missing), num_missing.numel(), int(frac_q16),
                                   _ptr(num_fetch), _stream(stream)))


def resolve_slots(state: DeviceCacheState, layer: int, topk_ids, frac_q16: int, slot_ids, num_fetch,
                  fetch_fid, fetch_slot, dev_status=None, stream=None):
    T, k = topk_ids.shape
    st = state.struct()
    _check(load().ft_moe_resolve_slots(ctypes.byref(st), layer, _ptr(topk_ids), T, k, int(frac_q16),
                                       _ptr(slot_ids), _ptr(num_fetch), _ptr(fetch_fid),
                                       _ptr(fetch_slot), fetch_fid.numel(), _ptr(dev_status),
                                       _stream(stream)))


def route_resolve(x, w_router, k: int, topk_ids, topk_w, ws, state: DeviceCacheState, layer: int, frac_q16: int,
                  slot_ids, num_fetch, fetch_fid, fetch_slot, dev_status=None, renorm: bool = False, stream=None):
    """route() then resolve_slots() as one C call (ft_moe_route_resolve):
    the same outputs, with the top-k taken inside the resolve kernel."""
    T, H = x.shape
    E = w_router.shape[0]
    st = state.struct()
    _check(load().ft_moe_route_resolve(_ptr(x), T, H, _ptr(w_router), E, k, int(bool(renorm)), _ptr(topk_ids),
                                       _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(st),
                                       layer, int(frac_q16), _ptr(slot_ids), _ptr(num_fetch), _ptr(fetch_fid),
                                       _ptr(fetch_slot), fetch_fid.numel(), _ptr(dev_status), _stream(stream)))


def prefetch(state: DeviceCacheState, layer: int, pred_ids, max_prefetch: int, num_fetch, fetch_fid,
             fetch_slot, dev_status=None, stream=None):
    """Plan a speculative fetch of `layer`'s predicted ids (ft_moe_prefetch);
    the copy itself is fetch() with the same list."""
    T, k = pred_ids.shape
    st = state.struct()
    _check(load().ft_moe_prefetch(ctypes.byref(st), layer, _ptr(pred_ids), T, k, int(max_prefetch),
                                  _ptr(num_fetch), _ptr(fetch_fid), _ptr(fetch_slot), fetch_fid.numel(),
                                  _ptr(dev_status), _stream(stream)))


def fetch(pool: FtBank, cache: FtBank, num_fetch, fetch_fid, fetch_slot, dev_status=None, stream=None):
    _check(load().ft_moe_fetch(ctypes.byref(pool), ctypes.byref(cache), _ptr(num_fetch),
                               _ptr(fetch_fid), _ptr(fetch_slot), fetch_fid.numel(),
                               _ptr(dev_status), _stream(stream)))


def fetch_layer(pool: FtBank, cache: FtBank, layer: int, E: int, slot0: int, stream=None):
    """Copy layer `layer`'s E expert blocks from the pool into cache slots slot0.. (copy engine)."""
    _check(load().ft_moe_fetch_layer(ctypes.byref(pool), ctypes.byref(cache), layer, E, slot0, _stream(stream)))


def cache_install(state: DeviceCacheState, layer: int, slot0: int, stream=None):
    """Record layer `layer`'s experts as resident in slots slot0..slot0+E-1."""
    st = state.struct()
    _check(load().ft_moe_cache_install(ctypes.byref(st), layer, slot0, _stream(stream)))


def cache_rebuild(old_state, old_cache: FtBank, new_state, new_cache: FtBank, budget_bytes: int,
                  dev_status=None, stream=None):
    """Rebuild the slot cache into new_state / new_cache (see ft_moe_cache_rebuild).
    The states are DeviceCacheState objects or FtCacheState structs.  Raises
    FtError with status FT_ERR_REJECTED when the rebuild does not fit."""
    so = old_state.struct() if hasattr(old_state, "struct") else old_state
    sn = new_state.struct() if hasattr(new_state, "struct") else new_state
    _check(load().ft_moe_cache_rebuild(ctypes.byref(so), ctypes.byref(old_cache), ctypes.byref(sn),
                                       ctypes.byref(new_cache), int(budget_bytes), _ptr(dev_status),
                                       _stream(stream)))


def experts_workspace(mode: int, T: int, k: int, H: int, I: int, E: int) -> int:
    return int(load().ft_moe_experts_workspace(mode, T, k, H, I, E))


def experts_fwd(cache: FtBank, pool, layer: int, E: int, x, T: int, k: int, slot_ids, raw_ids, topk_w,
                out, ws, mode: int = FT_DECODE, offsets=None, dev_status=None, stream=None, x_scale=None):
    import torch

    out_dtype = FT_OUT_BF16 if out.dtype in (torch.bfloat16, torch.int16, torch.uint16) else FT_OUT_F32
    _check(load().ft_moe_experts_fwd(ctypes.byref(cache), None if pool is None else ctypes.byref(pool),
                                     layer, E, _ptr(x), _ptr(x_scale), T, _ptr(slot_ids), _ptr(raw_ids),
                                     _ptr(topk_w), k, mode, _ptr(offsets), _ptr(out), out_dtype,
                                     _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
                                     _stream(stream)))


def experts_decode_static(cache: FtBank, pool, layer: int, E: int, x, T: int, k: int, slot_ids, raw_ids,
                          topk_w, out, dev_status=None, stream=None):
    """Decode experts with the library's own 1 MiB device scratch: for callers
    that cannot allocate a workspace (inside a stream capture, under another
    framework's memory pool).  Calls share the scratch: do not overlap them."""
    import torch

    out_dtype = FT_OUT_BF16 if out.dtype in (torch.bfloat16, torch.int16, torch.uint16) else FT_OUT_F32
    _check(load().ft_moe_experts_decode_static(ctypes.byref(cache), None if pool is None else ctypes.byref(pool),
                                               layer, E, _ptr(x), T, _ptr(slot_ids), _ptr(raw_ids),
                                               _ptr(topk_w), k, _ptr(out), out_dtype, _ptr(dev_status),
                                               _stream(stream)))


def permute_workspace(T: int, k: int, E: int) -> int:
    return int(load().ft_moe_permute_workspace(T, k, E))


def permute(topk_ids, E: int, x, perm, inv, offsets, xp, ws, dev_status=None, stream=None,
            xp_scale=None):
    """xp_scale given: xp is written as f16 with per-row power-of-two factors."""
    T, k = topk_ids.shape
    H = 0 if x is None else x.shape[1]
    fmt = FT_XP_BF16 if xp_scale is None else FT_XP_F16
    _check(load().ft_moe_permute(_ptr(topk_ids), T, k, E, _ptr(x), H, _ptr(perm), _ptr(inv),
                                 _ptr(offsets), _ptr(xp), fmt, _ptr(xp_scale), _ptr(ws),
                                 ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream)))


def combine(yp, inv, topk_w, out, host_partial=None, stream=None):
    T, k = inv.shape
    H = out.shape[1]
    _check(load().ft_moe_combine(_ptr(yp), _ptr(inv), _ptr(topk_w), T, k, H, _ptr(host_partial),
                                 _ptr(out), _stream(stream)))


def get_status(dev_status) -> int:
    v = ctypes.c_int32(0)
    _check(load().ft_moe_get_status(_ptr(dev_status), ctypes.byref(v)))
    return int(v.value)


def merge_partials(a, b, out, stream=None):
    """out = a + b (fp32 partial sums; out fp32 or bf16)."""
    out_dtype = FT_OUT_BF16 if out.dtype.itemsize == 2 else FT_OUT_F32
    _check(load().ft_moe_merge_partials(_ptr(a), _ptr(b), a.numel(), _ptr(out), out_dtype, _stream(stream)))


def decode_layer_workspace(T: int, k: int, H: int, I: int, E: int) -> int:
    return int(load().ft_moe_decode_layer_workspace(T, k, H, I, E))


def decode_layer(x, w_router, k: int, state: DeviceCacheState, layer: int, frac_q16: int, cache: FtBank,
                 pool: FtBank, topk_ids, topk_w, slot_ids, num_fetch, fetch_fid, fetch_slot, out, ws,
                 renorm: bool = False, dev_status=None, stream=None):
    """One decode layer call in one kernel (ft_moe_decode_layer): route, resolve,
    fetch, experts and combine, with the separate calls' results."""
    import torch

    T = x.shape[0]
    out_dtype = FT_OUT_BF16 if out.dtype in (torch.bfloat16, torch.int16, torch.uint16) else FT_OUT_F32
    st = state.struct()
    _check(load().ft_moe_decode_layer(_ptr(x), T, _ptr(w_router), k, int(bool(renorm)), ctypes.byref(st), layer,
                                      int(frac_q16), ctypes.byref(cache), ctypes.byref(pool), _ptr(topk_ids),
                                      _ptr(topk_w), _ptr(slot_ids), _ptr(num_fetch), _ptr(fetch_fid),
                                      _ptr(fetch_slot), fetch_fid.numel(), _ptr(out), out_dtype, _ptr(ws),
                                      ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream)))


def set_wait_limit_ns(ns: int):
    """Limit of the kernels' bounded waits launched from now on (0: the 2 s default)."""
    _check(load().ft_set_wait_limit_ns(int(ns)))

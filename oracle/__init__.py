"""CPU oracle for the routed, quantized expert-FFN MoE layer.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its binding) never does.  The arithmetic lives in
``ft_oracle.cpp`` (plain single-threaded C++, fp64); this module only builds it
with g++ and marshals numpy arrays through ctypes.

Parity status per function (what pins it is in the "not gpu" tests):
  split_q16        pinned: brute-force argmin of the cost over every f.
  route            pinned: hand-built logits, softmax closed forms, expert
                   relabelling equivariance.
  resolve          pinned: hand-worked trace, brute-force victim order on tiny
                   states, exactly-once and cache-size invariants.  The choice
                   of WHICH misses are fetched follows a reading (recency
                   descending, ties to the lower id); that ordering is
                   parity unpinned beyond the hand-worked trace.
  dequant          pinned: all E2M1 / E4M3 / fp16 / bf16 codes against their
                   definitions and library decoders; the pages' block sizes.
  expert, layer    pinned: closed forms on one-hot quantised matrices.
  permute          pinned: numpy stable argsort, segment invariants.
  combine          pinned: one-hot weights, linearity.
  cache_rebuild    pinned: invariants, brute force on small states.
  cache_install    pinned: a hand-worked example, invariants on random states.
  prefetch         pinned: a hand-worked trace, brute force over the fetched
                   and victim sets on tiny states, invariants.  Which
                   predicted misses come first when slots run short follows
                   the resolve's reading (recency descending, lower id).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ft_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libft_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_INT4 = 0
FMT_NVFP4 = 1


def build(force: bool = False) -> str:
    """Compile ft_oracle.cpp into libft_oracle.so beside it (g++, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            c = ctypes
            L.orc_bf16_value.restype = c.c_double
            L.orc_bf16_value.argtypes = [c.c_uint16]
            L.orc_fp16_value.restype = c.c_double
            L.orc_fp16_value.argtypes = [c.c_uint16]
            L.orc_e2m1_value.restype = c.c_double
            L.orc_e2m1_value.argtypes = [c.c_int]
            L.orc_e4m3_value.restype = c.c_double
            L.orc_e4m3_value.argtypes = [c.c_int]
            L.orc_block_layout.restype = c.c_int
            L.orc_block_layout.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int,
                                           _P(c.c_uint64), _P(c.c_uint64)]
            L.orc_dequant.restype = c.c_int
            L.orc_dequant.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_int,
                                      c.c_int, c.c_double, c.c_void_p]
            L.orc_split_q16.restype = c.c_int32
            L.orc_split_q16.argtypes = [c.c_int32, c.c_int32]
            L.orc_split_q16_grid.restype = None
            L.orc_split_q16_grid.argtypes = [c.c_int32, c.c_int32, c.c_int32, c.c_void_p]
            L.orc_resolve_many.restype = c.c_int
            L.orc_resolve_many.argtypes = ([c.c_int] * 3 + [c.c_void_p] * 5 + [c.c_int, c.c_void_p,
                                           c.c_int, c.c_int, c.c_int32, c.c_int] + [c.c_void_p] * 4
                                           + [c.c_int])
            L.orc_prefetch.restype = c.c_int
            L.orc_prefetch.argtypes = ([c.c_int] * 3 + [c.c_void_p] * 5 + [c.c_int, c.c_void_p,
                                       c.c_int, c.c_int, c.c_int32] + [c.c_void_p] * 3 + [c.c_int])
            L.orc_cache_install.restype = c.c_int
            L.orc_cache_install.argtypes = [c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
                                            c.c_void_p, c.c_int, c.c_int]
            L.orc_cache_rebuild.restype = c.c_int
            L.orc_cache_rebuild.argtypes = [c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_int,
                                            c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p]
            L.orc_route.restype = None
            L.orc_route.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_void_p, c.c_int,
                                    c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p]
            L.orc_resolve.restype = c.c_int
            L.orc_resolve.argtypes = ([c.c_int] * 3 + [c.c_void_p] * 5 + [c.c_int, c.c_void_p,
                                      c.c_int, c.c_int, c.c_int32] + [c.c_void_p] * 4 + [c.c_int])
            L.orc_permute.restype = c.c_int
            L.orc_permute.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int,
                                      c.c_void_p, c.c_void_p, c.c_void_p]
            L.orc_expert.restype = c.c_int
            L.orc_expert.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_int,
                                     c.c_void_p, c.c_void_p, c.c_void_p]
            L.orc_expert_batch.restype = c.c_int
            L.orc_expert_batch.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_int,
                                           c.c_void_p, c.c_void_p, c.c_int, c.c_void_p]
            L.orc_moe_experts.restype = c.c_int
            L.orc_moe_experts.argtypes = [c.c_void_p, c.c_uint64, c.c_void_p, c.c_int, c.c_int,
                                          c.c_int, c.c_int, c.c_int, c.c_int, c.c_void_p,
                                          c.c_int, c.c_void_p, c.c_void_p, c.c_int,
                                          c.c_void_p, c.c_void_p]
            L.orc_grouped_rows.restype = c.c_int
            L.orc_grouped_rows.argtypes = [c.c_void_p, c.c_uint64, c.c_void_p, c.c_int, c.c_int,
                                           c.c_int, c.c_int, c.c_int, c.c_int, c.c_void_p,
                                           c.c_void_p, c.c_int, c.c_void_p, c.c_void_p,
                                           c.c_int, c.c_void_p]
            L.orc_combine.restype = None
            L.orc_combine.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_int, c.c_int,
                                      c.c_int, c.c_void_p, c.c_void_p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# ------------------------------------------------------------------ formats
def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits))


def fp16_value(bits: int) -> float:
    return lib().orc_fp16_value(int(bits))


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def block_layout(fmt: int, H: int, I: int, g: int):
    """(offsets of gate, up, down, gate_scale, up_scale, down_scale; total bytes)."""
    off = (ctypes.c_uint64 * 6)()
    tot = ctypes.c_uint64()
    rc = lib().orc_block_layout(fmt, H, I, g, off, ctypes.byref(tot))
    if rc != 0:
        raise ValueError("unsupported block shape")
    return [int(v) for v in off], int(tot.value)


def dequant(block: np.ndarray, fmt: int, H: int, I: int, g: int, which: int,
            tensor_scale: float = 1.0) -> np.ndarray:
    block = _c(block, np.uint8)
    rows, K = (H, I) if which == 2 else (I, H)
    out = np.empty((rows, K), np.float64)
    rc = lib().orc_dequant(_ptr(block), fmt, H, I, g, which, float(tensor_scale), _ptr(out))
    if rc != 0:
        raise ValueError("bad dequant arguments")
    return out


# -------------------------------------------------------------------- split
def split_q16(m: int, phi: int) -> int:
    return int(lib().orc_split_q16(int(m), int(phi)))


def split_q16_many(ms, phi: int) -> np.ndarray:
    L = lib()
    return np.array([L.orc_split_q16(int(m), int(phi)) for m in np.asarray(ms).ravel()],
                    np.int32).reshape(np.shape(ms))


def split_q16_grid(m_max: int, phi_lo: int, phi_hi: int) -> np.ndarray:
    """[phi_hi - phi_lo + 1, m_max + 1] table of the rule."""
    out = np.empty((phi_hi - phi_lo + 1, m_max + 1), np.int32)
    lib().orc_split_q16_grid(m_max, phi_lo, phi_hi, _ptr(out))
    return out


# -------------------------------------------------------------------- route
def route(x_bf16: np.ndarray, W: np.ndarray, k: int, renorm: bool = False,
          want_logits: bool = False):
    x = _c(x_bf16, np.uint16)
    W = _c(W, np.float32)
    T, H = x.shape
    E = W.shape[0]
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lg = np.empty((T, E), np.float64) if want_logits else None
    lib().orc_route(_ptr(x), T, H, _ptr(W), E, k, int(bool(renorm)), _ptr(ids), _ptr(w), _ptr(lg))
    return (ids, w, lg) if want_logits else (ids, w)


# ------------------------------------------------------------------ resolve
class CacheState:
    """Host copy of the slot-cache state (numpy arrays, mutated in place)."""

    def __init__(self, L: int, E: int, S: int, recency_init: int = -1):
        self.L, self.E, self.S = L, E, S
        self.slot_owner = np.full(S, -1, np.int32)
        self.map = np.full(L * E, -1, np.int32)
        self.usage = np.full(S, -1, np.int64)
        self.recency = np.full(L * E, recency_init, np.int64)
        self.step = np.zeros(1, np.int64)

    def copy(self) -> "CacheState":
        c = CacheState.__new__(CacheState)
        c.L, c.E, c.S = self.L, self.E, self.S
        for n in ("slot_owner", "map", "usage", "recency", "step"):
            setattr(c, n, getattr(self, n).copy())
        return c

    def seed_slots(self, fids, usages=None):
        """Place the given flat ids in slots 0.. in order (a seeded cache)."""
        for s, fid in enumerate(fids):
            self.slot_owner[s] = fid
            self.map[fid] = s
            self.usage[s] = 0 if usages is None else usages[s]


def resolve(st: CacheState, layer: int, ids: np.ndarray, phi: int, max_list: int | None = None):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    n = T * k
    if max_list is None:
        max_list = n
    slot_ids = np.empty((T, k), np.int32)
    nf = np.zeros(1, np.int32)
    ff = np.empty(max_list, np.int32)
    fs = np.empty(max_list, np.int32)
    rc = lib().orc_resolve(st.L, st.E, st.S, _ptr(st.slot_owner), _ptr(st.map), _ptr(st.usage),
                           _ptr(st.recency), _ptr(st.step), layer, _ptr(ids), T, k, int(phi),
                           _ptr(slot_ids), _ptr(nf), _ptr(ff), _ptr(fs), max_list)
    if rc != 0:
        raise ValueError("orc_resolve rejected its arguments")
    return slot_ids, int(nf[0]), ff, fs


def resolve_many(st: CacheState, layer: int, ids: np.ndarray, phi: int, max_list: int):
    """ids [steps, T, k]; returns slot_ids [steps, T, k], num_fetch [steps],
    fetch_fid / fetch_slot [steps, max_list]."""
    ids = _c(ids, np.int32)
    steps, T, k = ids.shape
    sl = np.empty_like(ids)
    nf = np.empty(steps, np.int32)
    ff = np.empty((steps, max_list), np.int32)
    fs = np.empty((steps, max_list), np.int32)
    rc = lib().orc_resolve_many(st.L, st.E, st.S, _ptr(st.slot_owner), _ptr(st.map), _ptr(st.usage),
                                _ptr(st.recency), _ptr(st.step), layer, _ptr(ids), T, k, int(phi),
                                steps, _ptr(sl), _ptr(nf), _ptr(ff), _ptr(fs), max_list)
    if rc != 0:
        raise ValueError("orc_resolve_many rejected its arguments")
    return sl, nf, ff, fs


def prefetch(st: CacheState, layer: int, pred_ids: np.ndarray, max_prefetch: int,
             max_list: int | None = None):
    """A speculative fetch of `layer`'s predicted experts, one layer ahead of
    its resolve (see orc_prefetch); mutates st.  Returns (num, fetch_fid,
    fetch_slot)."""
    pred = _c(pred_ids, np.int32)
    T, k = pred.shape
    if max_list is None:
        max_list = T * k
    nf = np.zeros(1, np.int32)
    ff = np.empty(max_list, np.int32)
    fs = np.empty(max_list, np.int32)
    rc = lib().orc_prefetch(st.L, st.E, st.S, _ptr(st.slot_owner), _ptr(st.map), _ptr(st.usage),
                            _ptr(st.recency), _ptr(st.step), layer, _ptr(pred), T, k, int(max_prefetch),
                            _ptr(nf), _ptr(ff), _ptr(fs), max_list)
    if rc != 0:
        raise ValueError("orc_prefetch rejected its arguments")
    return int(nf[0]), ff, fs


# ------------------------------------------------------------------ permute
def cache_rebuild(st: CacheState, S_new: int):
    """The slot cache rebuilt at S_new slots (see orc_cache_rebuild): returns
    (new CacheState, src_of_new [S_new] = old slot moved to each new slot or -1)."""
    new = CacheState(st.L, st.E, S_new)
    src = np.full(S_new, -1, np.int32)
    rc = lib().orc_cache_rebuild(st.L, st.E, st.S, _ptr(_c(st.slot_owner, np.int32)),
                                 _ptr(_c(st.usage, np.int64)), S_new, _ptr(new.slot_owner), _ptr(new.map),
                                 _ptr(new.usage), _ptr(src))
    if rc != 0:
        raise ValueError("orc_cache_rebuild: an owner is outside [0, L*E)")
    new.recency[:] = st.recency
    new.step[:] = st.step
    return new, src


def cache_install(st: CacheState, layer: int, slot0: int):
    """Install all E experts of `layer` in slots slot0..slot0+E-1, in place
    (see orc_cache_install)."""
    rc = lib().orc_cache_install(st.L, st.E, st.S, _ptr(st.slot_owner), _ptr(st.map), _ptr(st.usage),
                                 _ptr(st.step), int(layer), int(slot0))
    if rc != 0:
        raise ValueError("orc_cache_install: layer or slot range out of bounds")


def permute(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    n = T * k
    perm = np.empty(n, np.int32)
    inv = np.empty((T, k), np.int32)
    off = np.empty(E + 1, np.int32)
    rc = lib().orc_permute(_ptr(ids), T, k, E, _ptr(perm), _ptr(inv), _ptr(off))
    if rc != 0:
        raise ValueError("expert id out of range")
    return perm, inv, off


# ------------------------------------------------------------------ experts
def expert(block: np.ndarray, fmt: int, H: int, I: int, g: int, x: np.ndarray,
           tscale3=None) -> np.ndarray:
    block = _c(block, np.uint8)
    x = _c(x, np.float64)
    ts = None if tscale3 is None else _c(tscale3, np.float32)
    y = np.empty(H, np.float64)
    rc = lib().orc_expert(_ptr(block), fmt, H, I, g, _ptr(ts), _ptr(x), _ptr(y))
    if rc != 0:
        raise ValueError("bad expert arguments")
    return y


def expert_batch(block: np.ndarray, fmt: int, H: int, I: int, g: int, X: np.ndarray,
                 tscale3=None) -> np.ndarray:
    """expert(x) for every row of X [n, H] (fp64), one dequantisation."""
    block = _c(block, np.uint8)
    X = _c(X, np.float64)
    ts = None if tscale3 is None else _c(tscale3, np.float32)
    Y = np.empty_like(X)
    rc = lib().orc_expert_batch(_ptr(block), fmt, H, I, g, _ptr(ts), _ptr(X), X.shape[0], _ptr(Y))
    if rc != 0:
        raise ValueError("bad expert_batch arguments")
    return Y


def moe_experts(pool: np.ndarray, stride: int, tscales, fmt: int, H: int, I: int, g: int,
                layer: int, E: int, x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray,
                include=None) -> np.ndarray:
    """Full-precision routed output over the pool (see orc_moe_experts)."""
    pool = np.ascontiguousarray(pool).view(np.uint8)
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    ts = None if tscales is None else _c(tscales, np.float32)
    inc = None if include is None else _c(include, np.uint8)
    T, k = ids.shape
    out = np.empty((T, H), np.float64)
    rc = lib().orc_moe_experts(_ptr(pool), stride, _ptr(ts), fmt, H, I, g, layer, E, _ptr(x),
                               T, _ptr(ids), _ptr(w), k, _ptr(inc), _ptr(out))
    if rc != 0:
        raise ValueError("bad moe_experts arguments")
    return out


def grouped_rows(pool: np.ndarray, stride: int, tscales, fmt: int, H: int, I: int, g: int,
                 layer: int, E: int, x_bf16: np.ndarray, perm: np.ndarray, k: int,
                 offsets: np.ndarray, rows) -> np.ndarray:
    pool = np.ascontiguousarray(pool).view(np.uint8)
    x = _c(x_bf16, np.uint16)
    perm = _c(perm, np.int32)
    offsets = _c(offsets, np.int32)
    rows = _c(rows, np.int32)
    ts = None if tscales is None else _c(tscales, np.float32)
    out = np.empty((len(rows), H), np.float64)
    rc = lib().orc_grouped_rows(_ptr(pool), stride, _ptr(ts), fmt, H, I, g, layer, E, _ptr(x),
                                _ptr(perm), k, _ptr(offsets), _ptr(rows), len(rows), _ptr(out))
    if rc != 0:
        raise ValueError("bad grouped_rows arguments")
    return out


def combine(yp_bf16: np.ndarray, inv: np.ndarray, w: np.ndarray, host_partial=None) -> np.ndarray:
    yp = _c(yp_bf16, np.uint16)
    inv = _c(inv, np.int32)
    w = _c(w, np.float32)
    T, k = inv.shape
    H = yp.shape[1]
    hp = None if host_partial is None else _c(host_partial, np.float32)
    out = np.empty((T, H), np.float64)
    lib().orc_combine(_ptr(yp), _ptr(inv), _ptr(w), T, k, H, _ptr(hp), _ptr(out))
    return out

"""The decode experts entry point that allocates nothing.

Callers inside a stream capture or under another framework's memory pool
cannot pass a workspace; ft_moe_experts_decode_static uses a scratch array the
library owns instead.  Its results must match ft_moe_experts_fwd with a
caller workspace and the CPU oracle, call after call (the shared scratch
keeps the previous call's contents).  This file is collected last on purpose."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import assert_close, oracle_pairs_output, pool_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(cfg, T, seed):
    rng = np.random.default_rng(seed)
    E, k = cfg.E, cfg.k
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    used = sorted(set(ids.ravel().tolist()))
    slot = {e: s for s, e in enumerate(used)}
    slots = np.vectorize(slot.get)(ids).astype(np.int32)
    blocks_np = pool_blocks(cfg, used)
    blocks = torch.from_numpy(blocks_np).to(DEV)
    w = rng.uniform(0.05, 0.3, (T, k)).astype(np.float32)
    x = synth.normal_bf16(synth.stream_key(seed, "noalloc-x"), (T, cfg.H))
    by_fid = {int(e): blocks_np[i] for i, e in enumerate(used)}  # layer 0: flat id = expert id
    return ids, slots, blocks, w, x, by_fid


@pytest.mark.parametrize("name,T", [("d35b", 1), ("flash", 1), ("tiny", 8)])
def test_static_scratch_matches_workspace_call_twice(cuda_lib, name, T):
    ft = cuda_lib
    cfg = synth.get_config(name)
    ts_np = synth.tensor_scales(cfg.fmt, cfg.H, cfg.I, cfg.L * cfg.E)
    ts = None if ts_np is None else torch.from_numpy(ts_np).to(DEV)
    for call in range(2):  # two calls in a row with different inputs
        ids, slots, blocks, w, x, by_fid = _case(cfg, T, 100 + call)
        cb = ft.make_bank(cfg.fmt, cfg.H, cfg.I, cfg.g, blocks, ts)
        args = [torch.from_numpy(a).to(DEV) for a in (x.view(np.int16), slots, ids, w)]
        ref = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
        ws = torch.zeros(ft.experts_workspace(ft.FT_DECODE, T, cfg.k, cfg.H, cfg.I, cfg.E),
                         dtype=torch.uint8, device=DEV)
        ft.experts_fwd(cb, None, 0, cfg.E, args[0], T, cfg.k, args[1], args[2], args[3], ref, ws)
        got = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        ft.experts_decode_static(cb, None, 0, cfg.E, args[0], T, cfg.k, args[1], args[2], args[3], got,
                                 dev_status=status)
        torch.cuda.synchronize()
        assert ft.get_status(status) == 0
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), f"{name} static call {call}", ref_max=None)
        # and both against the oracle
        oref = oracle_pairs_output(by_fid, cfg, ts_np, x, ids, w, 0)
        assert_close(got.cpu().numpy(), oref, f"{name} static call {call} vs oracle")


def test_static_scratch_rejects_oversize(cuda_lib):
    """T*k*I*4 above the 1 MiB scratch is refused before anything runs."""
    ft = cuda_lib
    H, I, g, E, T, k = 256, 4096, 32, 16, 16, 8  # 128 pairs x 4096 x 4 B = 2 MiB
    _, stride = synth.block_layout(0, H, I, g)
    cb = ft.make_bank(0, H, I, g, torch.zeros((1, stride), dtype=torch.uint8, device=DEV))
    z = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    with pytest.raises(ft.FtError) as ei:
        ft.experts_decode_static(cb, None, 0, E, torch.zeros((T, H), dtype=torch.int16, device=DEV),
                                 T, k, z, z, z.float(), torch.empty((T, H), device=DEV))
    assert ei.value.status == ft.FT_ERR_INVALID and "static scratch" in str(ei.value)

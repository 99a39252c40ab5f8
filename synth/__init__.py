"""Seeded synthetic inputs for the routed, quantized expert-FFN layer.

This package holds only random-number plumbing and input recipes: no step of
the layer's arithmetic lives here.  Both the CPU oracle's tests and the CUDA
path's tests and benchmark draw their inputs from it, so both sides see the
same bytes.

Every random quantity comes from a counter-based SplitMix64 stream
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014): value i of stream `key` is mix64(key + (i+1) * GOLDEN).  The
integer streams have two implementations, numpy (host) and torch int64
(device, for multi-GB expert banks); the tests check they agree bit for bit.
"""

from .rng import GOLDEN, mix64_np, stream_key, u64_stream_np, u64_stream_torch  # noqa: F401
from .gen import (  # noqa: F401
    block_layout,
    bank_block_np,
    bank_blocks_torch,
    tensor_scales,
    normal_bf16,
    normal_f32,
    bf16_bits,
    router_weights,
    zipf_history,
    zipf_probs,
    layer_rank_perm,
)
from .configs import CONFIGS, get_config  # noqa: F401

"""The five synthetic workloads of the routed, quantized expert-FFN layer.

Shapes follow the source pages' models: a 35B-A3B-class decode layer (int4,
40 layers x 256 experts, top-8), a Flash-Next-class NVFP4 decode layer
(48 x 512, top-10, 2560x640 experts), a DeepSeek-V4-Flash-class prefill layer
(43 x 256, top-6), a tiny parity layer and the cache-split sweep.
"""

from __future__ import annotations

from dataclasses import dataclass, field

FMT_INT4 = 0
FMT_NVFP4 = 1


@dataclass(frozen=True)
class LayerConfig:
    name: str
    L: int
    H: int
    I: int
    E: int
    k: int
    fmt: int
    g: int
    tokens: tuple
    slots: int
    phis: tuple
    ref_K: int | None = None
    router_std: float = 0.02
    zipf: float | None = None
    history_steps: int = 0
    gap: float = 1e-4
    seed: int = 0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_fids(self) -> int:
        return self.L * self.E


TINY = LayerConfig(
    name="tiny", L=1, H=256, I=128, E=16, k=2, fmt=FMT_INT4, g=32, tokens=(8,), slots=6,
    phis=(26214,), ref_K=None, note="tiny int4 g32 layer, 6 seeded slots")

D35B = LayerConfig(
    name="d35b", L=40, H=2048, I=512, E=256, k=8, fmt=FMT_INT4, g=64, tokens=(1, 8),
    slots=2560, phis=(65536, 26214), ref_K=256, zipf=1.1, history_steps=4096,
    note="35B-A3B-shaped int4 g64 decode, cache 25% of (layer, expert) pairs")

FLASH = LayerConfig(
    name="flash", L=48, H=2560, I=640, E=512, k=10, fmt=FMT_NVFP4, g=16, tokens=(1,),
    slots=48 * 512, phis=(65536,), gap=1e-3, extra={"steps": 256},
    note="Flash-Next-shaped NVFP4 decode, every expert resident")

PREFILL = LayerConfig(
    name="prefill", L=43, H=4096, I=2048, E=256, k=6, fmt=FMT_NVFP4, g=16, tokens=(2048, 8192),
    slots=2 * 256, phis=(65536,), note="whole-layer prefill, two NVFP4 layer banks alternating")

SWEEP = LayerConfig(
    name="sweep", L=1, H=0, I=0, E=256, k=8, fmt=FMT_INT4, g=0, tokens=(1,), slots=0,
    phis=(0, 1, 16384, 26214, 27306, 27307, 32768, 49152, 65535, 65536), zipf=1.1,
    extra={"Ek": [(256, 6), (256, 8), (256, 10), (512, 6), (512, 8), (512, 10)],
           "slot_fracs": [0.0, 0.10, 0.50, 1.00], "total_steps": 1_000_000},
    note="cache-miss split and exactly-once sweep")

CONFIGS = {c.name: c for c in (TINY, D35B, FLASH, PREFILL, SWEEP)}


def get_config(name: str) -> LayerConfig:
    return CONFIGS[name]

"""Layer shapes of the synthetic workloads and the generator's stream kinds.

The shapes follow the models the DGPP pages serve (page 4 forum post 1,
quantisation table; page 1 README performance table): an NVFP4 routed-expert
layer with an FP8 block-128 shared expert, an MXFP4 layer, and an int4 g64
layer with an int8 g64 shared expert, each at decode batch sizes, plus an
NVFP4 prefill layer with a skewed router.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

# Format enumerators; the values match the C ABI's moe_format.
FMT_NVFP4 = 1
FMT_MXFP4 = 2
FMT_INT4_G64 = 3
FMT_INT8_G64 = 4
FMT_FP8_B128 = 5
FMT_INT4_G128 = 6   # AutoRound / GPTQ layout: unsigned nibbles with zero point 8, FP16 scale per 128

FMT_NAMES = {FMT_NVFP4: "nvfp4", FMT_MXFP4: "mxfp4", FMT_INT4_G64: "int4_g64", FMT_INT8_G64: "int8_g64",
             FMT_FP8_B128: "fp8_b128", FMT_INT4_G128: "int4_g128"}

# Generator stream kinds (part of the stream key, see qmoe_synth.c).
KIND_ROUTER = 1
KIND_ZIPF = 2
KIND_ROUTED = 3   # proj 0 = gate, 1 = up, 2 = down
KIND_SHARED = 4   # proj 0 = gate, 1 = up, 2 = down
KIND_TOKENS = 5   # expert field = batch index

WEIGHT_SIGMA = 0.02


@dataclass(frozen=True)
class LayerConfig:
    name: str
    fmt: int
    H: int          # hidden size
    E: int          # routed experts
    k: int          # top-k
    I: int          # routed expert intermediate size
    shared_fmt: int = 0   # 0 = no shared expert
    shared_I: int = 0
    batches: Tuple[int, ...] = (1,)
    zipf_s: float = 0.0   # > 0: router bias -s*ln(rank) (prefill load skew)

    def with_(self, **kw) -> "LayerConfig":
        d = self.__dict__.copy()
        d.update(kw)
        return LayerConfig(**d)


CONFIGS = {
    "tiny_nvfp4": LayerConfig("tiny_nvfp4", FMT_NVFP4, H=256, E=8, k=2, I=128, batches=(1,)),
    "decode_nvfp4": LayerConfig("decode_nvfp4", FMT_NVFP4, H=2048, E=512, k=10, I=512,
                                shared_fmt=FMT_FP8_B128, shared_I=512, batches=(1, 4, 8)),
    "decode_mxfp4": LayerConfig("decode_mxfp4", FMT_MXFP4, H=4096, E=256, k=8, I=2048, batches=(1, 8)),
    "decode_int4": LayerConfig("decode_int4", FMT_INT4_G64, H=6144, E=256, k=8, I=2048,
                               shared_fmt=FMT_INT8_G64, shared_I=2048, batches=(8,)),
    "prefill_nvfp4": LayerConfig("prefill_nvfp4", FMT_NVFP4, H=2048, E=512, k=10, I=512, batches=(4096,),
                                 zipf_s=1.1),
}


def get(name: str) -> LayerConfig:
    return CONFIGS[name]

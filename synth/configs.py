"""Workload registry: shapes, dtypes and value distributions of the layer configurations.

Shapes follow the model families the pages use: the 350M / 1.3B MoE NLG models with 128
experts per FFN and the PR-MoE residual layer (DeepSpeed-MoE review, "MoE based NLG Model
Architecture" and "PR-MoE"), and the 2.4B+MoE-128 model with hidden size 3584
(DeepSpeed-MoE Inference wiki, "성능: 딥 MoE에서의 확장" table).  FFN width is 4x hidden.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    d: int
    f: int
    E: int
    k: int
    cf: float
    dtype: str                      # "f32" or "f16": activations and expert weights
    residual: bool = False
    f_res: int = 0
    tok_sigma: float = 1.0          # tokens ~ N(0, tok_sigma^2)
    w_sigma: float = 0.02           # weights ~ N(0, w_sigma^2)
    zipf: float | None = None       # Zipf exponent of the expert-load skew, None = uniform
    T_list: tuple = field(default_factory=tuple)

    def at(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


CONFIGS = {
    # tiny fp32 parity layer
    "tiny_fp32": LayerConfig("tiny_fp32", d=64, f=256, E=4, k=1, cf=1.0, dtype="f32",
                             tok_sigma=0.02, T_list=(128,)),
    # 350M+MoE-128 layer, decode to prefill
    "moe350m_e128": LayerConfig("moe350m_e128", d=1024, f=4096, E=128, k=1, cf=1.25, dtype="f16",
                                T_list=(1, 8, 64, 512, 4096)),
    # 1.3B+MoE-128 layer with Zipf(1.1) expert load, cf 1.0 and 2.0
    "moe1p3b_e128_zipf": LayerConfig("moe1p3b_e128_zipf", d=2048, f=8192, E=128, k=1, cf=1.0,
                                     dtype="f16", zipf=1.1, T_list=(16, 256, 8192)),
    # PR-MoE residual layer: dense MLP (f_res 8192) + one routed expert, shallow / deep setting
    "prmoe_e64": LayerConfig("prmoe_e64", d=2048, f=8192, E=64, k=1, cf=1.0, dtype="f16",
                             residual=True, f_res=8192, T_list=(64, 2048)),
    "prmoe_e128": LayerConfig("prmoe_e128", d=2048, f=8192, E=128, k=1, cf=1.0, dtype="f16",
                              residual=True, f_res=8192, T_list=(64, 2048)),
    # Top2-MoE at the PR-MoE layer's shape (d 2048, f 8192, E 64 / 128): two routed experts in
    # place of one routed expert plus the dense MLP, the comparison of the DeepSpeed-MoE review,
    # "Phenomenon2"
    "top2_e64": LayerConfig("top2_e64", d=2048, f=8192, E=64, k=2, cf=1.0, dtype="f16",
                            T_list=(64, 2048)),
    "top2_e128": LayerConfig("top2_e128", d=2048, f=8192, E=128, k=2, cf=1.0, dtype="f16",
                             T_list=(64, 2048)),
    # small PR-MoE layers for the stack parity test (dropless, so tokens do not interact);
    # weights ~ N(0, 1/d) keep activations of order one through the chain
    "tiny_prmoe_e8": LayerConfig("tiny_prmoe_e8", d=256, f=512, E=8, k=1, cf=float("inf"),
                                 dtype="f16", residual=True, f_res=512, w_sigma=0.0625,
                                 T_list=(64,)),
    "tiny_prmoe_e16": LayerConfig("tiny_prmoe_e16", d=256, f=512, E=16, k=1, cf=float("inf"),
                                  dtype="f16", residual=True, f_res=512, w_sigma=0.0625,
                                  T_list=(64,)),
    # 2.4B+MoE-128 layer, top-2 with normalised gate weights, uniform and Zipf(1.2) load
    "moe2p4b_e128_top2": LayerConfig("moe2p4b_e128_top2", d=3584, f=14336, E=128, k=2, cf=1.25,
                                     dtype="f16", T_list=(1, 32, 1024, 16384)),
    "moe2p4b_e128_top2_zipf": LayerConfig("moe2p4b_e128_top2_zipf", d=3584, f=14336, E=128, k=2,
                                          cf=1.25, dtype="f16", zipf=1.2,
                                          T_list=(1, 32, 1024, 16384)),
}


# Pyramid stacks (DeepSpeed-MoE review, "PR-MoE: Pyramid-Residual-MoE for Smaller Model Size
# and Fast Inference": more experts in the last layers, an MLP beside every MoE module).  The
# pages give neither the depth nor the split; the reading here: 12 MoE layers, the last two
# with twice the experts, as in a 24-layer model with an MoE FFN in every other layer.
STACKS = {
    "prmoe_pyramid_12": ("prmoe_e64",) * 10 + ("prmoe_e128",) * 2,
    "tiny_pyramid_3": ("tiny_prmoe_e8", "tiny_prmoe_e8", "tiny_prmoe_e16"),
}


def layer_seed(seed: int, layer: int) -> int:
    """Seed of one layer's weights in a stack: distinct weights per layer."""
    return seed * 1000 + 7919 * (layer + 1)


def workload(name: str, T: int | None = None, **overrides) -> tuple[LayerConfig, int]:
    cfg = CONFIGS[name]
    if overrides:
        cfg = cfg.at(**overrides)
    return cfg, (T if T is not None else cfg.T_list[-1])

"""Seeded synthetic inputs for the decoder-only Transformer forward pass.

This module is shared by the CPU oracle and the CUDA path.  It holds the
five model shapes and the random draws (weights and token ids) and nothing
of the method's arithmetic: no norm, projection, rotation or attention.

Shapes follow the tutorial pages on building a decoder-only Transformer
from scratch: the toy character model (d_model 64, 4 heads, 2 layers, a
23-symbol vocabulary) of "Chapter 4: Implement a Transformer from Scratch"
and of the CS336 Transformer walkthrough, the GPT-2-small width with the
SwiGLU d_ff = 2048 and 2752 of the CS336 walkthrough's FLOP-accounting
section, and a long-context and a grouped-query shape.

Every draw uses ``numpy.random.Generator(PCG64(seed))`` in float32, in a
fixed tensor order.  bf16 configurations round the float32 draws to the
nearest bf16 value (ties to even) and keep them as float32 arrays whose
values are exactly representable in bf16, so both sides see the same
numbers.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "ModelConfig", "CONFIGS", "get_config", "round_to_bf16", "bf16_bits",
    "make_weights", "make_tokens", "zipf_tokens", "LAYER_KEYS",
    "GPT2_CONFIGS", "GPT2_LAYER_KEYS", "make_gpt2_weights",
]


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    vocab: int
    d_model: int
    n_head: int
    n_kv_head: int
    n_layer: int
    d_ff: int
    batch: int
    seq: int
    mode: str                 # "fp32" or "bf16": storage type of weights/activations
    rope_theta: float = 10000.0
    norm_eps: float = 1e-5
    weight_seed: int = 0
    token_seed: int = 0
    token_dist: str = "uniform"   # "uniform" or "zipf1.1"
    out_proj_std: float = 0.02    # std of Wo and W2
    std: float = 0.02             # std of every other weight

    @property
    def d_head(self) -> int:
        return self.d_model // self.n_head

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def replace(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": ModelConfig("tiny", 23, 64, 4, 4, 2, 176, 4, 64, "fp32",
                        weight_seed=1000, token_seed=2000),
    "small": ModelConfig("small", 10000, 512, 16, 16, 4, 1344, 32, 256, "bf16",
                         weight_seed=1001, token_seed=2001),
    "gpt2s": ModelConfig("gpt2s", 50257, 768, 12, 12, 12, 2048, 8, 1024, "bf16",
                         weight_seed=1002, token_seed=2002, token_dist="zipf1.1"),
    "long": ModelConfig("long", 32000, 1024, 16, 16, 4, 2752, 1, 8192, "bf16",
                        weight_seed=1003, token_seed=2003),
    "gqa": ModelConfig("gqa", 32000, 2048, 16, 4, 8, 5632, 4, 2048, "bf16",
                       weight_seed=1004, token_seed=2004,
                       out_proj_std=0.02 / math.sqrt(2 * 8)),
}


def get_config(name: str) -> ModelConfig:
    return CONFIGS[name]


# Per-layer weight names, in draw order.  Shapes are (out_features, in_features).
LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w1", "w3", "w2")


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 array -> float32 array holding the nearest bf16 values."""
    return (bf16_bits(a).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _shapes(cfg: ModelConfig):
    D, dh = cfg.d_model, cfg.d_head
    Dq, Dkv = cfg.n_head * dh, cfg.n_kv_head * dh
    return {
        "attn_norm": (D,), "wq": (Dq, D), "wk": (Dkv, D), "wv": (Dkv, D),
        "wo": (D, Dq), "ffn_norm": (D,), "w1": (cfg.d_ff, D),
        "w3": (cfg.d_ff, D), "w2": (D, cfg.d_ff),
    }


def make_weights(cfg: ModelConfig, gains: str = "ones", seed: int | None = None) -> dict:
    """Draw every weight of ``cfg`` from its seed.

    Returns ``{"embed": [V,D], "layers": [ {key: array} ... ], "final_norm": [D],
    "lm_head": [V,D]}`` as float32 arrays (bf16-exact values in bf16 mode).
    ``gains="ones"`` sets every RMSNorm gain to 1; ``gains="random"`` draws them
    from U(0.5, 1.5) with a second generator (seed + 7919) so that the matrix
    draws are the same in both cases.
    """
    rng = np.random.Generator(np.random.PCG64(cfg.weight_seed if seed is None else seed))
    grng = np.random.Generator(np.random.PCG64((cfg.weight_seed if seed is None else seed) + 7919))
    rnd = round_to_bf16 if cfg.mode == "bf16" else (lambda a: a)
    D, V = cfg.d_model, cfg.vocab

    def normal(shape, std):
        return rnd(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))

    def gain(n):
        if gains == "ones":
            return np.ones(n, dtype=np.float32)
        return grng.uniform(0.5, 1.5, n).astype(np.float32)

    w = {"embed": normal((V, D), cfg.std), "layers": []}
    shapes = _shapes(cfg)
    for _ in range(cfg.n_layer):
        layer = {}
        for key in LAYER_KEYS:
            if key.endswith("norm"):
                layer[key] = gain(D)
            else:
                std = cfg.out_proj_std if key in ("wo", "w2") else cfg.std
                layer[key] = normal(shapes[key], std)
        w["layers"].append(layer)
    w["final_norm"] = gain(D)
    w["lm_head"] = normal((V, D), cfg.std)
    return w


def zipf_tokens(rng: np.random.Generator, vocab: int, n: int, s: float = 1.1) -> np.ndarray:
    """Token ids with P(id = r-1) proportional to r**-s over the finite vocabulary,
    drawn by inverse CDF on a precomputed table."""
    r = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(r ** -s)
    cdf /= cdf[-1]
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int32)


def make_tokens(cfg: ModelConfig, batch: int | None = None, seq: int | None = None,
                seed: int | None = None) -> np.ndarray:
    """int32 token ids [B, S] from the config's token seed and distribution."""
    B = cfg.batch if batch is None else batch
    S = cfg.seq if seq is None else seq
    rng = np.random.Generator(np.random.PCG64(cfg.token_seed if seed is None else seed))
    if cfg.token_dist == "zipf1.1":
        t = zipf_tokens(rng, cfg.vocab, B * S)
    else:
        t = rng.integers(0, cfg.vocab, B * S, dtype=np.int64).astype(np.int32)
    return t.reshape(B, S)


# ---------------------------------------------------------------- GPT-2-style family
# The second model family of the pages: absolute positions added to the token
# embedding, LayerNorm with a shift, biased linears, a 4 x d_model GELU MLP, an
# optionally tied and biased LM head.  Shapes: the toy character model of
# "Chapter 4: Implement a Transformer from Scratch" (d_model 64, 4 heads, 2
# layers, hidden 256) and the GPT-2-small width (768, 12 heads, 12 layers, 3072).
GPT2_CONFIGS = {
    "gpt2_tiny": ModelConfig("gpt2_tiny", 23, 64, 4, 4, 2, 256, 4, 64, "fp32",
                             weight_seed=1100, token_seed=2100),
    "gpt2_small": ModelConfig("gpt2_small", 50257, 768, 12, 12, 12, 3072, 8, 1024, "bf16",
                              weight_seed=1101, token_seed=2101, token_dist="zipf1.1"),
}

# Per-layer names in draw order: LayerNorm gain/shift, fused [Wq; Wk; Wv] and its
# bias, output projection and bias, LayerNorm 2, MLP up (fc) and down (fc2).
GPT2_LAYER_KEYS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_proj", "b_proj",
                   "ln2_g", "ln2_b", "w_fc", "b_fc", "w_fc2", "b_fc2")


def make_gpt2_weights(cfg: ModelConfig, pos: str = "learned", lm_bias: bool = False,
                      tied: bool = False, max_seq: int | None = None,
                      seed: int | None = None) -> dict:
    """Draw every weight of the GPT-2-style model ``cfg`` from its seed.

    Returns ``{"embed": [V,D], "pos": [max_seq,D] or None, "layers": [...],
    "lnf_g", "lnf_b": [D], "lm_head": [V,D] (the embed array itself when tied),
    "lm_bias": [V] or None}``.  Matrices (and the learned position table) are
    N(0, std) (bf16-exact in bf16 mode); LayerNorm gains U(0.5, 1.5), shifts and
    biases N(0, 0.02) in float32 from a second generator (seed + 7919)."""
    base = cfg.weight_seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(base))
    grng = np.random.Generator(np.random.PCG64(base + 7919))
    rnd = round_to_bf16 if cfg.mode == "bf16" else (lambda a: a)
    D, V, F, dh = cfg.d_model, cfg.vocab, cfg.d_ff, cfg.d_head
    Nqkv = (cfg.n_head + 2 * cfg.n_kv_head) * dh
    T = cfg.seq if max_seq is None else max_seq

    def normal(shape, std):
        return rnd(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))

    def small(n):
        return (grng.standard_normal(n, dtype=np.float32) * np.float32(0.02)).astype(np.float32)

    def gain(n):
        return grng.uniform(0.5, 1.5, n).astype(np.float32)

    w = {"embed": normal((V, D), cfg.std)}
    w["pos"] = normal((T, D), cfg.std) if pos == "learned" else None
    shapes = {"w_qkv": (Nqkv, D), "w_proj": (D, cfg.n_head * dh), "w_fc": (F, D), "w_fc2": (D, F)}
    vecs = {"b_qkv": Nqkv, "b_proj": D, "b_fc": F, "b_fc2": D}
    w["layers"] = []
    for _ in range(cfg.n_layer):
        layer = {}
        for key in GPT2_LAYER_KEYS:
            if key.endswith("_g"):
                layer[key] = gain(D)
            elif key.startswith("ln"):
                layer[key] = small(D)
            elif key.startswith("b_"):
                layer[key] = small(vecs[key])
            else:
                std = cfg.out_proj_std if key in ("w_proj", "w_fc2") else cfg.std
                layer[key] = normal(shapes[key], std)
        w["layers"].append(layer)
    w["lnf_g"] = gain(D)
    w["lnf_b"] = small(D)
    w["lm_head"] = w["embed"] if tied else normal((V, D), cfg.std)
    w["lm_bias"] = small(V) if lm_bias else None
    return w

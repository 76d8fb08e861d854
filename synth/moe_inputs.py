"""Seeded synthetic workloads for the fine-grained MoE layer.

Shapes follow the NanoColibri MoE described in "Una carrera de relevos con GPUs
alquiladas entrenó el MoE de 2.7B de NanoColibri por $200" (and its zh / ar
translations), opening section, architecture paragraph: hidden width 1024, 64
routed experts of width 512, top-2, one shared expert of width 2048.  The pages
print no data, so every tensor is drawn here:

* x ~ N(0, 1); routed and shared expert weights ~ N(0, 0.02) (std);
* router weight ~ N(0, 1/sqrt(d)) (std), kept in fp32;
* bias ~ U(-0.01, 0.01) (zero for the tiny case); gamma = 1e-3;
* the skewed case adds ln p_e to expert e's logit, p a Zipf(s=1.2) law.

Every draw is an fp32 sample from ``numpy.random.default_rng`` seeded with
``SeedSequence([seed, case, layer, tensor])``; tensors stored as bf16 are the
round-to-nearest-even bf16 of that sample, carried as uint16 bit patterns so
that the oracle and the GPU read identical bytes.  Nothing in this module is
part of the layer's arithmetic: it only produces inputs.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Case numbers used in the seed: they are fixed so that stored fixtures and
# bench runs stay reproducible.
_CASE_ID = {"tiny": 0, "nano": 1, "skew": 2, "decode": 3, "stack": 4, "attn": 5, "attn_tiny": 6}
_TENSOR_ID = {
    "x": 0, "w_router": 1, "bias": 2, "w_gate": 3, "w_up": 4, "w_down": 5,
    "s_gate": 6, "s_up": 7, "s_down": 8, "dout": 9,
    "w_q": 10, "w_k": 11, "w_v": 12, "w_o": 13,
}


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Sizes of one MoE layer: T tokens, hidden d, E experts of width f, shared width F, top-k."""

    T: int
    d: int
    E: int
    f: int
    F: int
    k: int
    renorm: bool = True          # renormalise gates over the k winners
    x_dtype: str = "bf16"        # "bf16" or "f32"
    w_format: str = "bf16"       # routed expert weights: "bf16" or "int4"
    bias_init: str = "uniform"   # "uniform" U(-0.01, 0.01) or "zero"
    gamma: float = 1e-3
    skew_zipf_s: float = 0.0     # > 0 adds ln Zipf(s) logit offsets
    steps: int = 1
    layers: int = 1

    def replace(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


CONFIGS: dict[str, LayerShape] = {
    # 0: correctness-only tiny layer, fp32 activations, bias 0.
    "tiny": LayerShape(T=64, d=64, E=8, f=32, F=128, k=2, x_dtype="f32", bias_init="zero"),
    # 1: Nano-shaped layer forward (batch 4 x seq 2048 tokens).
    "nano": LayerShape(T=8192, d=1024, E=64, f=512, F=2048, k=2),
    # 2: skewed-load stress, 50 forward + bias-update steps.
    "skew": LayerShape(T=8192, d=1024, E=64, f=512, F=2048, k=2, skew_zipf_s=1.2, steps=50),
    # 3: top-1 serving decode with int4 routed experts (T in {1, 8, 64}).
    "decode": LayerShape(T=64, d=1024, E=64, f=512, F=2048, k=1, renorm=False, w_format="int4"),
    # 4: 23 consecutive Nano layers with a residual add.
    "stack": LayerShape(T=8192, d=1024, E=64, f=512, F=2048, k=2, layers=23),
}


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 samples to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    # Finite inputs only: the sum below stays inside 32 bits for every finite fp32.
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Expand bf16 bit patterns to the fp32 values they encode (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, case: str, layer: int, tensor: str) -> np.random.Generator:
    ss = np.random.SeedSequence([seed, _CASE_ID[case], layer, _TENSOR_ID[tensor]])
    return np.random.default_rng(ss)


def _normal(seed, case, layer, tensor, shape, std) -> np.ndarray:
    g = _rng(seed, case, layer, tensor)
    out = g.standard_normal(size=shape, dtype=np.float32)
    out *= np.float32(std)
    return out


def make_tokens(shape: LayerShape, case: str, seed: int = 0) -> np.ndarray:
    """Token activations x[T][d]: fp32 array for x_dtype 'f32', else bf16 bits (uint16)."""
    x = _normal(seed, case, 0, "x", (shape.T, shape.d), 1.0)
    return x if shape.x_dtype == "f32" else bf16_bits_from_f32(x)


def make_output_grad(shape: LayerShape, case: str, seed: int = 0) -> np.ndarray:
    """Gradient of a loss with respect to the layer output, dout[T][d] ~ N(0, 1), bf16 bits."""
    return bf16_bits_from_f32(_normal(seed, case, 0, "dout", (shape.T, shape.d), 1.0))


def zipf_logit_offset(E: int, s: float) -> np.ndarray:
    """ln p_e for p_e proportional to (e+1)^-s, expert 0 the most popular (fp32)."""
    w = np.array([(e + 1) ** (-s) for e in range(E)], dtype=np.float64)
    return np.log(w / w.sum()).astype(np.float32)


def make_layer(shape: LayerShape, case: str, seed: int = 0, layer: int = 0,
               with_tokens: bool = True) -> dict:
    """All inputs of one MoE layer as host numpy arrays.

    Keys: x (see make_tokens), w_router f32[E][d], bias f32[E], logit_offset f32[E] or None,
    w_gate / w_up bf16 bits [E][f][d], w_down bf16 bits [E][d][f], s_gate / s_up bf16 bits
    [F][d], s_down bf16 bits [d][F], gamma (python float).  Weights are bf16 in every case;
    the int4 case quantises these bf16 values.
    """
    T, d, E, f, F = shape.T, shape.d, shape.E, shape.f, shape.F
    out: dict = {}
    if with_tokens:
        out["x"] = make_tokens(shape, case, seed)
    out["w_router"] = _normal(seed, case, layer, "w_router", (E, d), 1.0 / math.sqrt(d))
    if shape.bias_init == "zero":
        out["bias"] = np.zeros(E, dtype=np.float32)
    else:
        g = _rng(seed, case, layer, "bias")
        out["bias"] = g.uniform(-0.01, 0.01, size=E).astype(np.float32)
    out["logit_offset"] = zipf_logit_offset(E, shape.skew_zipf_s) if shape.skew_zipf_s > 0 else None
    out["w_gate"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_gate", (E, f, d), 0.02))
    out["w_up"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_up", (E, f, d), 0.02))
    out["w_down"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_down", (E, d, f), 0.02))
    out["s_gate"] = bf16_bits_from_f32(_normal(seed, case, layer, "s_gate", (F, d), 0.02))
    out["s_up"] = bf16_bits_from_f32(_normal(seed, case, layer, "s_up", (F, d), 0.02))
    out["s_down"] = bf16_bits_from_f32(_normal(seed, case, layer, "s_down", (d, F), 0.02))
    out["gamma"] = shape.gamma
    return out


@dataclasses.dataclass(frozen=True)
class AttnShape:
    """Sizes of one attention block: batch x seq tokens, hidden d, n_head query heads sharing
    n_kv_head key/value heads (grouped-query attention), head width head_dim."""

    batch: int
    seq: int
    d: int
    n_head: int
    n_kv_head: int
    head_dim: int = 128
    eps: float = 1e-6

    @property
    def T(self) -> int:
        return self.batch * self.seq

    def replace(self, **kw) -> "AttnShape":
        return dataclasses.replace(self, **kw)


ATTN_CONFIGS: dict[str, AttnShape] = {
    # The Nano model's attention (hidden 1024, 4x GQA, head width 128), batch 4 x seq 2048.
    "attn": AttnShape(batch=4, seq=2048, d=1024, n_head=8, n_kv_head=2),
    # Small, ragged sequences (not a multiple of the 128-token tile), one key/value head.
    "attn_tiny": AttnShape(batch=2, seq=200, d=512, n_head=4, n_kv_head=1),
}


def make_attention(shape: AttnShape, case: str, seed: int = 0, layer: int = 0) -> dict:
    """Inputs of one attention block: x bf16 bits [T][d] ~ N(0, 1), w_q [H*hd][d], w_k, w_v
    [Hkv*hd][d], w_o [d][H*hd] bf16 bits ~ N(0, 0.02)."""
    hd = shape.head_dim
    out = {"x": bf16_bits_from_f32(_normal(seed, case, layer, "x", (shape.T, shape.d), 1.0))}
    out["w_q"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_q", (shape.n_head * hd, shape.d), 0.02))
    out["w_k"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_k", (shape.n_kv_head * hd, shape.d), 0.02))
    out["w_v"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_v", (shape.n_kv_head * hd, shape.d), 0.02))
    out["w_o"] = bf16_bits_from_f32(_normal(seed, case, layer, "w_o", (shape.d, shape.n_head * hd), 0.02))
    return out

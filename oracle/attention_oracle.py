"""Oracle for the GQA attention block with per-head QK-norm.

TEST INFRASTRUCTURE.  A plain, slow CPU restatement of what the GPU path computes.
Only the tests, the package's smoke check and the bench's CPU baseline may import it;
the library never calls it.  It shares no code with the CUDA path.

Source of the method.  "Una carrera de relevos con GPUs alquiladas entrenó el MoE de
2.7B de NanoColibri por $200" (the same article in Chinese and Arabic), opening
section, architecture paragraph: the model's attention is grouped-query attention
with four query heads per key/value head ("4x GQA") and a normalisation of the queries
and keys of every head ("per-head QK-norm").  Nothing else about the block is stated.

Readings where the article is silent (each is also listed in the design notes):

* head width 128, so the hidden width 1024 gives 8 query heads and 2 key/value heads;
* QK-norm is an RMS normalisation over each head's 128 values, without a learned
  scale: u / sqrt(mean(u^2) + eps) with eps = 1e-6, applied to q and k (not v);
* scores q.k / sqrt(head width), causal (a token sees itself and earlier tokens of its
  own sequence), softmax over the keys;
* no positional encoding (the article names none);
* out = x + o W_o^T (residual add; the block without it is the same minus x);
* projections without biases; token rows are batch-major: row b * S + s.

Precision: fp64, with the values the GPU stores in bf16 (the projected q, k, v, the
normalised q and k, the attention output o) rounded to bf16 where it stores them
(`round_stored`).  Parity pins: tests/test_oracle_pins.py (PyTorch CPU scaled-dot-
product attention and rms_norm on the same inputs, closed forms, causality, the GQA
grouping).
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import round_to_bf16


def rms_norm_heads(u: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """u / sqrt(mean(u^2) + eps) over the last axis (one head's values)."""
    u = np.asarray(u, dtype=np.float64)
    return u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True) + eps)


def gqa_attention(x, w_q, w_k, w_v, w_o, batch: int, seq: int, n_head: int, n_kv_head: int,
                  head_dim: int = 128, eps: float = 1e-6, residual: bool = True,
                  round_stored: bool = True) -> dict:
    """One attention block: projections, per-head QK-norm, causal GQA, output projection.

    x [batch*seq][d]; w_q [n_head*head_dim][d]; w_k, w_v [n_kv_head*head_dim][d];
    w_o [d][n_head*head_dim] (all real values).  Query head h reads key/value head
    h // (n_head // n_kv_head).  Returns q, k, v (after the norm for q, k), o and out.
    """
    x = np.asarray(x, dtype=np.float64)
    T = batch * seq
    assert x.shape[0] == T and n_head % n_kv_head == 0
    group = n_head // n_kv_head
    rnd = round_to_bf16 if round_stored else (lambda a: a)
    q = rnd(x @ np.asarray(w_q, np.float64).T).reshape(T, n_head, head_dim)
    k = rnd(x @ np.asarray(w_k, np.float64).T).reshape(T, n_kv_head, head_dim)
    v = rnd(x @ np.asarray(w_v, np.float64).T).reshape(T, n_kv_head, head_dim)
    qn = rnd(rms_norm_heads(q, eps))
    kn = rnd(rms_norm_heads(k, eps))
    o = np.zeros((T, n_head, head_dim), dtype=np.float64)
    scale = 1.0 / np.sqrt(head_dim)
    causal = np.tril(np.ones((seq, seq), dtype=bool))
    for b in range(batch):
        rows = slice(b * seq, (b + 1) * seq)
        for h in range(n_head):
            g = h // group
            s = (qn[rows, h, :] @ kn[rows, g, :].T) * scale
            s = np.where(causal, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            o[rows, h, :] = p @ v[rows, g, :]
    o = rnd(o).reshape(T, n_head * head_dim)
    out = o @ np.asarray(w_o, np.float64).T
    if residual:
        out = out + x
    return dict(q=qn, k=kn, v=v, o=o, out=out)

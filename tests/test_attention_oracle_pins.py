"""Pins of the attention oracle (oracle/attention_oracle.py) against things other than
itself: PyTorch's CPU rms_norm and scaled-dot-product attention with grouped key/value
heads (library routines) on the same inputs, closed forms, causality, the grouping of
query heads, and the scale invariance the QK-norm gives.

The relay article ("Una carrera de relevos con GPUs alquiladas...", architecture
paragraph) states only 4x grouped-query attention with a per-head QK-norm; the other
readings (head width, RMS norm without learned scale, causal softmax, no positional
encoding, residual) are the oracle's and are listed there.
"""
import numpy as np
import pytest
import torch

from oracle import attention_oracle as A
from oracle.moe_oracle import bf16_value_from_bits
from synth import ATTN_CONFIGS, make_attention


def _inputs(shape, case="attn_tiny", seed=0):
    h = make_attention(shape, case, seed)
    return {k: bf16_value_from_bits(v) for k, v in h.items()}


def _torch_reference(s, P, residual=True):
    x = torch.from_numpy(P["x"])
    T, hd = s.T, s.head_dim
    q = (x @ torch.from_numpy(P["w_q"]).T).reshape(s.batch, s.seq, s.n_head, hd).transpose(1, 2)
    k = (x @ torch.from_numpy(P["w_k"]).T).reshape(s.batch, s.seq, s.n_kv_head, hd).transpose(1, 2)
    v = (x @ torch.from_numpy(P["w_v"]).T).reshape(s.batch, s.seq, s.n_kv_head, hd).transpose(1, 2)
    q = torch.nn.functional.rms_norm(q, (hd,), eps=s.eps)
    k = torch.nn.functional.rms_norm(k, (hd,), eps=s.eps)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    o = o.transpose(1, 2).reshape(T, s.n_head * hd)
    out = o @ torch.from_numpy(P["w_o"]).T
    return (out + x if residual else out).numpy(), o.numpy()


@pytest.mark.parametrize("shape", [ATTN_CONFIGS["attn_tiny"],
                                   ATTN_CONFIGS["attn_tiny"].replace(batch=1, seq=37, n_head=8, n_kv_head=2,
                                                                     d=256, head_dim=32)])
def test_attention_matches_torch_sdpa_with_grouped_heads(shape):
    P = _inputs(shape)
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], shape.batch, shape.seq, shape.n_head,
                        shape.n_kv_head, shape.head_dim, shape.eps, residual=True, round_stored=False)
    want, o = _torch_reference(shape, P)
    assert np.allclose(r["o"], o, rtol=1e-10, atol=1e-12)
    assert np.allclose(r["out"], want, rtol=1e-10, atol=1e-12)


def test_zero_queries_attend_uniformly_over_the_prefix():
    # q = 0 -> the norm gives 0 -> every score 0: token t averages v over positions <= t.
    s = ATTN_CONFIGS["attn_tiny"].replace(batch=1, seq=9)
    P = _inputs(s)
    P["w_q"] = np.zeros_like(P["w_q"])
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head,
                        residual=False, round_stored=False)
    v = (P["x"] @ P["w_v"].T).reshape(s.T, s.n_kv_head, s.head_dim)
    for t in range(s.seq):
        want = v[:t + 1].mean(axis=0)  # one key/value head shared by all query heads
        for h in range(s.n_head):
            assert np.allclose(r["o"][t, h * 128:(h + 1) * 128], want[0], rtol=1e-12, atol=1e-12)


def test_first_token_output_is_its_own_value():
    s = ATTN_CONFIGS["attn_tiny"]
    P = _inputs(s)
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head,
                        residual=False, round_stored=False)
    v = (P["x"] @ P["w_v"].T).reshape(s.T, s.n_kv_head, s.head_dim)
    for b in range(s.batch):
        t = b * s.seq  # first token of each sequence sees only itself
        for h in range(s.n_head):
            assert np.allclose(r["o"][t, h * 128:(h + 1) * 128], v[t, 0], rtol=1e-12, atol=1e-12)


def test_causality_and_sequence_independence():
    s = ATTN_CONFIGS["attn_tiny"].replace(seq=50)
    P = _inputs(s)
    base = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head,
                           s.n_kv_head, round_stored=False)["out"]
    x2 = P["x"].copy()
    x2[30:50] += 1.0        # later tokens of sequence 0
    x2[50 + 10] -= 2.0      # a token of sequence 1
    r2 = A.gqa_attention(x2, P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head,
                         round_stored=False)["out"]
    assert np.array_equal(r2[:30], base[:30])          # earlier tokens of sequence 0 unchanged
    assert np.array_equal(r2[50:60], base[50:60])      # sequence 1 before the change unchanged
    assert not np.allclose(r2[30:50], base[30:50]) and not np.allclose(r2[60:], base[60:])


def test_grouped_heads_share_keys_and_values():
    # Query heads 0 and 1 with equal projection rows give equal outputs (same group);
    # changing the key projection of group 1 changes only heads 4..7.
    s = ATTN_CONFIGS["attn_tiny"].replace(batch=1, seq=40, d=256, n_head=8, n_kv_head=2, head_dim=32)
    P = _inputs(s)
    hd = s.head_dim
    P["w_q"][hd:2 * hd] = P["w_q"][:hd]
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head,
                        hd, residual=False, round_stored=False)
    assert np.array_equal(r["o"][:, :hd], r["o"][:, hd:2 * hd])
    wk = P["w_k"].copy()
    wk[hd:] *= -1.5
    r2 = A.gqa_attention(P["x"], P["w_q"], wk, P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head, hd,
                         residual=False, round_stored=False)
    assert np.array_equal(r2["o"][:, :4 * hd], r["o"][:, :4 * hd])
    assert not np.allclose(r2["o"][:, 4 * hd:], r["o"][:, 4 * hd:])


def test_qk_norm_removes_the_scale_of_queries_and_keys():
    # Scaling W_q and W_k by positive constants changes q and k but not their RMS-normed
    # directions (up to eps), so the output is unchanged; scaling W_v scales the output.
    # With eps = 0 the invariance is exact (up to rounding); with eps = 1e-6 it holds up
    # to the eps term (q and k have mean squares near 0.2 here).
    s = ATTN_CONFIGS["attn_tiny"].replace(batch=1, seq=60)
    P = _inputs(s)
    kw = dict(batch=s.batch, seq=s.seq, n_head=s.n_head, n_kv_head=s.n_kv_head, residual=False, round_stored=False)
    r0 = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], eps=0.0, **kw)
    r0s = A.gqa_attention(P["x"], 3.0 * P["w_q"], 0.5 * P["w_k"], P["w_v"], P["w_o"], eps=0.0, **kw)
    assert np.allclose(r0s["out"], r0["out"], rtol=1e-10, atol=1e-12)
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], **kw)
    r2 = A.gqa_attention(P["x"], 3.0 * P["w_q"], 0.5 * P["w_k"], P["w_v"], P["w_o"], **kw)
    assert np.abs(r2["out"] - r["out"]).max() <= 1e-4 * np.abs(r["out"]).max()
    r3 = A.gqa_attention(P["x"], P["w_q"], P["w_k"], 2.0 * P["w_v"], P["w_o"], **kw)
    assert np.allclose(r3["out"], 2.0 * r["out"], rtol=1e-12, atol=1e-12)
    # The normed rows have RMS 1 (eps aside).
    rms = np.sqrt(np.mean(r["q"] ** 2, axis=-1))
    assert np.allclose(rms, 1.0, atol=1e-5)

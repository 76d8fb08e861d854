"""GPU parity of the attention block (4x grouped-query attention with per-head QK-norm,
relay article, architecture paragraph) against oracle/attention_oracle.py, through the
C ABI.

moe_attention_core (the tcgen05 attention kernel alone) is fed the oracle's own
normalised q, k and v (bf16), so it is checked in isolation; moe_attention_fwd (the
projections on the tensor cores, the QK-norm kernel, the attention kernel, the output
projection with the residual) is checked end to end.  The head groupings (1, 2, 4 and 8
query heads per key/value head) reach every cluster size of the kernel (key and value
tiles shared by 1, 2 or 4 CTAs through multicast copies).  Tolerance: the bf16 bound of
gpu_util (2e-2 relative L2 plus an element-wise bound).
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from gpu_util import assert_close_bf16, bf16_to_np, bf64
from oracle import attention_oracle as A
from synth import ATTN_CONFIGS, bf16_bits_from_f32, make_attention
from aux_loss_free_gb300.layer import to_device_bf16

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    yield
    assert M.moe_device_status() == 0


def _ms(s):
    return M.make_attn_shape(s.batch, s.seq, s.d, s.n_head, s.n_kv_head, s.head_dim, s.eps)


CORE_CASES = [
    ATTN_CONFIGS["attn_tiny"],                                            # ragged: 200 = 128 + 72
    ATTN_CONFIGS["attn_tiny"].replace(batch=3, seq=128, n_head=8, n_kv_head=2, d=1024),
    ATTN_CONFIGS["attn_tiny"].replace(batch=1, seq=1),                    # one token
    ATTN_CONFIGS["attn_tiny"].replace(batch=2, seq=129, n_head=2, n_kv_head=2, d=256),  # no grouping
    ATTN_CONFIGS["attn_tiny"].replace(batch=1, seq=700, n_head=8, n_kv_head=1, d=1024),  # one shared head
    ATTN_CONFIGS["attn_tiny"].replace(batch=2, seq=260, n_head=4, n_kv_head=2, d=512),   # pairs of heads
]


@pytest.mark.parametrize("s", CORE_CASES, ids=[f"B{c.batch}-S{c.seq}-H{c.n_head}-G{c.n_kv_head}" for c in CORE_CASES])
def test_attention_core_matches_oracle(s):
    P = {k: bf64(v) for k, v in make_attention(s, "attn_tiny").items()}
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head,
                        s.head_dim, s.eps, residual=False, round_stored=True)
    qkv = np.concatenate([r["q"].reshape(s.T, -1), r["k"].reshape(s.T, -1), r["v"].reshape(s.T, -1)], axis=1)
    qkv_bits = bf16_bits_from_f32(qkv.astype(np.float32))  # the values are bf16 already: exact
    o = torch.empty(s.T, s.n_head * s.head_dim, dtype=torch.bfloat16, device=DEV)
    M.moe_attention_core(_ms(s), to_device_bf16(qkv_bits, DEV), o)
    torch.cuda.synchronize()
    assert_close_bf16(bf16_to_np(o), r["o"], "attention output")


BLOCK_CASES = [ATTN_CONFIGS["attn_tiny"],
               ATTN_CONFIGS["attn_tiny"].replace(batch=2, seq=300, d=1024, n_head=8, n_kv_head=2)]


@pytest.mark.parametrize("s", BLOCK_CASES, ids=[f"B{c.batch}-S{c.seq}-d{c.d}" for c in BLOCK_CASES])
@pytest.mark.parametrize("residual", [True, False])
def test_attention_block_matches_oracle(s, residual):
    H = make_attention(s, "attn_tiny")
    P = {k: bf64(v) for k, v in H.items()}
    r = A.gqa_attention(P["x"], P["w_q"], P["w_k"], P["w_v"], P["w_o"], s.batch, s.seq, s.n_head, s.n_kv_head,
                        s.head_dim, s.eps, residual=residual, round_stored=True)
    ms = _ms(s)
    w_qkv = np.concatenate([H["w_q"], H["w_k"], H["w_v"]], axis=0)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(M.moe_attention_workspace_size(ms), dtype=torch.uint8, device=DEV)
    M.moe_attention_fwd(ms, to_device_bf16(H["x"], DEV), to_device_bf16(w_qkv, DEV), to_device_bf16(H["w_o"], DEV),
                        residual, out, ws)
    torch.cuda.synchronize()
    assert_close_bf16(bf16_to_np(out), r["out"], "attention block out")


def test_attention_block_nano_size_first_sequence():
    """The Nano block (batch 4 x seq 2048, d 1024, 8 query heads on 2 key/value heads):
    sequences are independent, so the first one (2048 tokens, every query tile and head)
    is checked against the oracle run on it alone."""
    s = ATTN_CONFIGS["attn"]
    H = make_attention(s, "attn")
    ms = _ms(s)
    w_qkv = np.concatenate([H["w_q"], H["w_k"], H["w_v"]], axis=0)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(M.moe_attention_workspace_size(ms), dtype=torch.uint8, device=DEV)
    M.moe_attention_fwd(ms, to_device_bf16(H["x"], DEV), to_device_bf16(w_qkv, DEV), to_device_bf16(H["w_o"], DEV),
                        True, out, ws)
    torch.cuda.synchronize()
    rows = slice(0, s.seq)
    r = A.gqa_attention(bf64(H["x"][rows]), bf64(H["w_q"]), bf64(H["w_k"]), bf64(H["w_v"]), bf64(H["w_o"]), 1,
                        s.seq, s.n_head, s.n_kv_head, s.head_dim, s.eps, residual=True, round_stored=True)
    assert_close_bf16(bf16_to_np(out)[rows], r["out"], "Nano attention block, sequence 0")

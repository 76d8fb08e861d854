"""Top-1 int4 serving in one persistent launch (at most 8 tokens), on the
GPU through the C ABI, against the oracle.

Relay article, opening section (int4 experts, sigmoid-plus-bias router, shared expert)
and section "Entrenamiento por relevos", top-2 paragraph (serving with one expert per
token).  The fused launch does the router, the selection, the bias update, the balance
statistics, the shared expert, the int4 routed experts and the combine; the library's
stage profiler shows which path a call took.  Checked: selection, gates, loads, bias
and balance bit for bit (the oracle's top-k fed the GPU's fp32 scores), the output
within the bf16 tolerance of the oracle run on its own dequantised weights, and the
same call through the multi-launch path (forced by asking for the permutation) giving
the same routing and an output within tolerance of it.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import LayerOnDevice, to_device_tokens
from gpu_util import assert_close_bf16, bf16_to_np, bf64, tokens64
from oracle import moe_oracle as O
from synth import CONFIGS, make_layer, make_tokens

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    yield
    assert M.moe_device_status() == 0


def _dequant(bits3d):
    """The oracle's own int4 round trip of bf16 weights [G][rows][K]."""
    G, R, K = bits3d.shape
    packed, scale, _ = O.quantize_int4_g32(bf64(bits3d.reshape(-1, K)).astype(np.float32))
    return O.dequantize_int4_g32(packed, scale).reshape(G, R, K)


def _run(s, host, x_bits, res_bits, update_bias, want_perm=False):
    """One forward; returns the device outputs and the stages the profiler saw."""
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(x_bits, DEV)
    res = to_device_tokens(res_bits, DEV) if res_bits is not None else None
    T, E, k = s.T, s.E, s.k
    scores = torch.empty(T, E, dtype=torch.float32, device=DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, k, dtype=torch.float32, device=DEV)
    load = torch.full((E,), -5, dtype=torch.int32, device=DEV)
    bal = torch.zeros(M.BALANCE_BYTES, dtype=torch.uint8, device=DEV)
    extra = {}
    if want_perm:
        extra = dict(offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
                     perm_tok=torch.empty(T * k, dtype=torch.int32, device=DEV),
                     inv_pos=torch.empty(T, k, dtype=torch.int32, device=DEV))
    dbg = M.make_debug(scores=scores, idx=idx, gate=gate, load=load, balance=bal, **extra)
    out = torch.empty(T, s.d, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    M.moe_profile_start(4)
    layer.forward(x, out, update_bias=update_bias, residual=res, debug=dbg)
    torch.cuda.synchronize()
    _, stage_calls = M.moe_profile_stop(per_stage_calls=True)
    return dict(scores=scores.cpu().numpy(), idx=idx.cpu().numpy(), gate=gate.cpu().numpy(),
                load=load.cpu().numpy(), balance=M.balance_from_bytes(bal), out=bf16_to_np(out),
                bias=layer.bias.cpu().numpy(), stages={n for n, c in stage_calls.items() if c})


def _check_against_oracle(s, host, x_bits, res_bits, update_bias, got, what):
    ref = O.layer_forward(tokens64(x_bits), host["w_router"], host["bias"], _dequant(host["w_gate"]),
                          _dequant(host["w_up"]), _dequant(host["w_down"]), bf64(host["s_gate"]),
                          bf64(host["s_up"]), bf64(host["s_down"]), k=s.k, renorm=s.renorm, gamma=s.gamma,
                          scores_f32=got["scores"],
                          residual=bf64(res_bits) if res_bits is not None else None)
    assert np.abs(got["scores"] - O.router_scores(tokens64(x_bits), host["w_router"])).max() <= 1e-5, what
    assert np.array_equal(got["idx"], ref["idx"]), what
    assert np.abs(got["gate"] - ref["gate"]).max() <= 1e-6, what
    ld = O.expert_load(ref["idx"], s.E)
    assert np.array_equal(got["load"], ld), what
    want_bias = O.bias_update(host["bias"], ld, s.T * s.k, s.gamma) if update_bias else host["bias"]
    assert np.array_equal(got["bias"].view(np.uint32), want_bias.view(np.uint32)), what
    want_bal = O.balance_stats(ld, s.E)
    for key in ("pairs", "max_load", "min_load", "dead_experts"):
        assert got["balance"][key] == want_bal[key], (what, key)
    for key in ("max_over_mean", "min_over_mean", "dead_fraction"):
        assert np.float32(got["balance"][key]).view(np.uint32) == np.float32(want_bal[key]).view(np.uint32)
    assert_close_bf16(got["out"], ref["out"], what)


# (T, k, renorm, residual, update_bias): 1 to 8 tokens, top-1 with the raw score as the
# gate (int4 layers serve one expert per token); with and without the residual and the
# bias update.
CASES = [(1, 1, False, False, False), (1, 1, False, True, True), (2, 1, False, True, True),
         (5, 1, False, False, True), (7, 1, False, True, False), (8, 1, False, True, True)]


@pytest.mark.parametrize("T,k,renorm,residual,update_bias", CASES,
                         ids=[f"T{c[0]}-k{c[1]}{'-renorm' if c[2] else ''}{'-res' if c[3] else ''}"
                              f"{'-bias' if c[4] else ''}" for c in CASES])
def test_fused_serving_matches_oracle(T, k, renorm, residual, update_bias):
    s = CONFIGS["decode"].replace(T=T, k=k, renorm=renorm)
    host = make_layer(s, "decode")
    res_bits = make_tokens(s, "decode", seed=11) if residual else None
    got = _run(s, host, host["x"], res_bits, update_bias)
    assert "serve_fused" in got["stages"], got["stages"]
    _check_against_oracle(s, host, host["x"], res_bits, update_bias, got, f"fused T={T} k={k}")


@pytest.mark.parametrize("T", [2, 8])
def test_fused_serving_with_every_token_on_the_same_expert(T):
    """A zero router: every score is exactly 1/2 and, with a zero bias, every key ties,
    so all tokens pick expert 0 (ties to the lower index) and the one routed expert
    serves every pair in one pass."""
    k = 1
    s = CONFIGS["decode"].replace(T=T)
    host = make_layer(s, "decode")
    host["bias"] = np.zeros(s.E, np.float32)
    host["w_router"] = np.zeros_like(host["w_router"])
    got = _run(s, host, host["x"], None, True)
    assert "serve_fused" in got["stages"]
    assert (got["idx"] == np.arange(k)[None, :]).all()
    assert (got["scores"] == 0.5).all()
    _check_against_oracle(s, host, host["x"], None, True, got, f"fused, one expert T={T}")


@pytest.mark.parametrize("T", [1, 3, 8])
def test_fused_serving_equals_the_multi_launch_path(T):
    s = CONFIGS["decode"].replace(T=T)
    host = make_layer(s, "decode")
    res_bits = make_tokens(s, "decode", seed=13)
    fused = _run(s, host, host["x"], res_bits, True)
    multi = _run(s, host, host["x"], res_bits, True, want_perm=True)
    assert "serve_fused" in fused["stages"] and "serve_fused" not in multi["stages"]
    for key in ("idx", "load"):
        assert np.array_equal(fused[key], multi[key]), key
    assert np.array_equal(fused["bias"].view(np.uint32), multi["bias"].view(np.uint32))
    assert np.abs(fused["scores"] - multi["scores"]).max() <= 1e-5
    assert_close_bf16(fused["out"], multi["out"].astype(np.float64), "fused vs multi-launch")

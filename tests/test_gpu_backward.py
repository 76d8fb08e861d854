"""GPU parity of the layer backward (moe_layer_bwd) against the oracle's layer_backward.

The forward runs first on the GPU (its routing state is what the backward consumes);
the oracle selects with the GPU's fp32 scores, and its expert choice must agree
exactly.  Every gradient is compared within the bf16 tolerance of gpu_util: bf16
operands and intermediates with fp32 accumulation, fp32 weight gradients.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import (LayerGrads, LayerOnDevice, SavedForward, layer_backward,
                                       to_device_bf16, to_device_tokens)
from gpu_util import assert_close_bf16, assert_close_grad, bf16_to_np, bf64
from oracle import moe_oracle as O
from synth import CONFIGS, make_layer, make_output_grad

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    yield
    assert M.moe_device_status() == 0


def _deinterleave(w, width):
    """[G][2*width][d] rows interleaved in blocks of moe_gate_up_block(width) -> (gate, up)."""
    b = M.moe_gate_up_block(width)
    G, _, d = w.shape
    v = w.reshape(G, width // b, 2, b, d)
    return v[:, :, 0].reshape(G, width, d), v[:, :, 1].reshape(G, width, d)


def _forward(s, host, residual):
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    saved = SavedForward(s.T, s.E, s.k, DEV)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=False, residual=x if residual else None, debug=saved.debug)
    return layer, x, saved


def _check_shared(s, got, ref_dsg, ref_dsu, ref_dsd):
    g, u = _deinterleave(got.ds_gate_up.cpu().numpy()[None].astype(np.float64), s.F)
    assert_close_grad(g[0], ref_dsg, "dS_gate")
    assert_close_grad(u[0], ref_dsu, "dS_up")
    assert_close_grad(got.ds_down.cpu().numpy(), ref_dsd, "dS_down")


BWD_CASES = [
    ("small", dict(T=200, d=256, E=8, f=128, F=256, k=2), False),
    ("nano widths", dict(T=512), False),
    ("top-1 renormalised (zero router gradient)", dict(T=300, d=256, E=16, f=128, F=0, k=1), False),
    ("top-4 raw gates", dict(T=100, d=512, E=32, f=256, F=128, k=4, renorm=False), False),
    ("most experts empty", dict(T=5, d=256, E=16, f=128, F=128, k=2), False),
    ("residual, ragged", dict(T=333, d=384, E=24, f=384, F=640, k=3), True),
]


@pytest.mark.parametrize("what,kw,residual", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_layer_bwd_matches_oracle(what, kw, residual):
    s = CONFIGS["nano"].replace(**kw)
    host = make_layer(s, "nano")
    dout_bits = make_output_grad(s, "nano")
    layer, x, saved = _forward(s, host, residual)
    dout = to_device_bf16(dout_bits, DEV)
    grads = LayerGrads(layer, want_dgate=True)
    layer_backward(layer, x, saved, dout, grads, residual=residual)
    torch.cuda.synchronize()
    sc = saved.scores.cpu().numpy()
    ref = O.layer_backward(bf64(host["x"]), host["w_router"], host["bias"], bf64(host["w_gate"]),
                           bf64(host["w_up"]), bf64(host["w_down"]),
                           bf64(host["s_gate"]) if s.F else None, bf64(host["s_up"]) if s.F else None,
                           bf64(host["s_down"]) if s.F else None, bf64(dout_bits), s.k,
                           renorm=s.renorm, logit_offset=host["logit_offset"], scores_f32=sc,
                           residual=residual)
    assert np.array_equal(saved.idx.cpu().numpy(), ref["idx"])
    assert_close_bf16(grads.dgate.cpu().numpy(), ref["dgate"], "dgate")
    assert_close_bf16(bf16_to_np(grads.dx), ref["dx"], "dx")
    if s.k > 1 or not s.renorm:
        assert_close_grad(grads.dw_router.cpu().numpy(), ref["dw_router"], "dW_router")
    else:  # one renormalised gate is the constant 1: no gradient reaches the router
        assert not grads.dw_router.cpu().numpy().any()
    g, u = _deinterleave(grads.dw_gate_up.cpu().numpy().astype(np.float64), s.f)
    used = np.unique(ref["idx"])
    for e in range(s.E):
        if e in used:
            assert_close_grad(g[e], ref["dw_gate"][e], f"dW_gate[{e}]")
            assert_close_grad(u[e], ref["dw_up"][e], f"dW_up[{e}]")
            assert_close_grad(grads.dw_down[e].cpu().numpy(), ref["dw_down"][e], f"dW_down[{e}]")
        else:  # an expert without tokens gets an exact zero gradient
            assert not g[e].any() and not u[e].any() and not grads.dw_down[e].cpu().numpy().any()
    if s.F:
        _check_shared(s, grads, ref["ds_gate"], ref["ds_up"], ref["ds_down"])


def test_layer_bwd_full_nano_sampled():
    """The Nano layer at 8192 tokens, in the launch configuration the bench times.

    The oracle's per-pair loop is too slow for every token, so the routed gradients
    are checked on a sample: every token routed to three experts (their weight
    gradients, router rows, and those tokens' dx and dgate are then complete); the
    shared expert's weight gradients are checked over all tokens.
    """
    s = CONFIGS["nano"]
    host = make_layer(s, "nano")
    dout_bits = make_output_grad(s, "nano")
    layer, x, saved = _forward(s, host, False)
    dout = to_device_bf16(dout_bits, DEV)
    grads = LayerGrads(layer, want_dgate=True)
    layer_backward(layer, x, saved, dout, grads)
    torch.cuda.synchronize()
    idx = saved.idx.cpu().numpy()
    sc = saved.scores.cpu().numpy()
    experts = [0, 37, 63]
    toks = np.nonzero(np.isin(idx, experts).any(axis=1))[0]
    assert toks.size > 100
    x64 = bf64(host["x"])
    d64 = bf64(dout_bits)
    sg, su, sd = bf64(host["s_gate"]), bf64(host["s_up"]), bf64(host["s_down"])
    ref = O.layer_backward(x64[toks], host["w_router"], host["bias"], bf64(host["w_gate"]),
                           bf64(host["w_up"]), bf64(host["w_down"]), sg, su, sd, d64[toks], s.k,
                           renorm=s.renorm, scores_f32=sc[toks], idx=idx[toks])
    assert_close_bf16(bf16_to_np(grads.dx)[toks], ref["dx"], "dx (sampled tokens)")
    assert_close_bf16(grads.dgate.cpu().numpy()[toks], ref["dgate"], "dgate (sampled tokens)")
    g, u = _deinterleave(grads.dw_gate_up.cpu().numpy().astype(np.float64), s.f)
    dwr = grads.dw_router.cpu().numpy()
    for e in experts:
        assert_close_grad(g[e], ref["dw_gate"][e], f"dW_gate[{e}]")
        assert_close_grad(u[e], ref["dw_up"][e], f"dW_up[{e}]")
        assert_close_grad(grads.dw_down[e].cpu().numpy(), ref["dw_down"][e], f"dW_down[{e}]")
        assert_close_grad(dwr[e], ref["dw_router"][e], f"dW_router[{e}]")
    _, dsg, dsu, dsd = O.shared_expert_backward(x64, sg, su, sd, d64)
    _check_shared(s, grads, dsg, dsu, dsd)
    # Properties at full size: finite everywhere, and the expert weight gradients of
    # every expert are nonzero (each receives tokens at this size).
    assert torch.isfinite(grads.dw_gate_up).all() and torch.isfinite(grads.dw_down).all()
    assert torch.isfinite(grads.dx.float()).all()
    assert (grads.dw_down.abs().sum(dim=(1, 2)) > 0).all()


def test_layer_bwd_rejects_unsupported_shapes():
    s = CONFIGS["nano"].replace(T=64, f=96, F=0)  # f not a multiple of 128
    ms = M.make_shape(s.T, s.d, s.E, s.f, s.F, s.k)
    assert M.moe_layer_bwd_workspace_size(ms) == 0
    s2 = CONFIGS["tiny"]  # fp32 tokens
    ms2 = M.make_shape(s2.T, s2.d, s2.E, s2.f, s2.F, s2.k, x_dtype=M.MOE_X_F32)
    assert M.moe_layer_bwd_workspace_size(ms2) == 0

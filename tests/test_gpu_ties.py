"""Exact ties in the selection key on the GPU, through the C ABI.

The tie rule (equal keys fl32(score + bias) go to the lower expert index, and the k
winners are listed by descending key, lower index first) is this build's reading; the
relay article's architecture paragraph only names top-k routing on a sigmoid-plus-bias
router.  Random inputs almost never tie in fp32, so these cases build ties on purpose:

* x = 0: every logit is 0 and every score exactly 0.5; with bias 0 the winners are
  experts 0..k-1 and the renormalised gates exactly 1/k; with biases on a dyadic grid
  the keys 0.5 + b are exact and the winners follow the bias, ties to the lower index;
* a "grid" router: tokens with entries in {-1, 0, 1} on a few dimensions, router rows
  drawn from four patterns with entries in {0, +-0.5, 1}, so every logit is a small
  exact dyadic number in any summation order, many experts share a logit (equal scores
  within a kernel), and biases from {0, +-2^-9} tie keys again.

Each case is routed to a chosen kernel: the tensor-core router (bf16 x, T >= 128, E in
{16, 32, 48, 64, 80}), the cluster router (T <= 256 otherwise) or the SIMT router (the
rest).  Indices and loads are compared bit for bit with the oracle's top-k fed the
GPU's fp32 scores; gates within 1e-6.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import LayerOnDevice, to_device_tokens
from gpu_util import assert_close_bf16, bf16_to_np, bf64, tokens64
from oracle import moe_oracle as O
from synth import CONFIGS, bf16_bits_from_f32, make_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    yield
    assert M.moe_device_status() == 0


def _tie_inputs(kind, T, d, E, x_dtype, seed):
    """(x as bf16 bits or fp32, w_router fp32, bias fp32) with exactly tied keys."""
    rng = np.random.default_rng(seed)
    x = np.zeros((T, d), np.float32)
    wr = np.zeros((E, d), np.float32)
    if kind == "zero":
        bias = np.zeros(E, np.float32)
    elif kind == "zero_grid_bias":
        bias = (rng.integers(-2, 3, E) * 2.0 ** -9).astype(np.float32)
    else:  # "grid"
        x[:, :4] = rng.integers(-1, 2, (T, 4))
        patterns = rng.choice(np.array([0.0, 0.5, -0.5, 1.0], np.float32), size=(4, 4))
        wr[:, :4] = patterns[rng.integers(0, 4, E)]
        bias = (rng.integers(-1, 2, E) * 2.0 ** -9).astype(np.float32)
    xin = x if x_dtype == "f32" else bf16_bits_from_f32(x)
    return xin, wr, bias


# (kernel, T, E, k, x dtype): the dispatch rules above pick the kernel.
ROUTER_CASES = [
    ("tensor-core", 512, 64, 2, "bf16"),
    ("tensor-core", 384, 64, 8, "bf16"),
    ("tensor-core", 200, 16, 4, "bf16"),
    ("cluster", 100, 64, 2, "bf16"),
    ("cluster", 256, 256, 8, "bf16"),
    ("cluster", 77, 64, 3, "f32"),
    ("simt", 1000, 256, 8, "bf16"),
    ("simt", 600, 64, 2, "f32"),
    ("simt", 300, 40, 5, "bf16"),
]


@pytest.mark.parametrize("kind", ["zero", "zero_grid_bias", "grid"])
@pytest.mark.parametrize("kernel,T,E,k,xd", ROUTER_CASES, ids=[f"{c[0]}-T{c[1]}-E{c[2]}-k{c[3]}-{c[4]}"
                                                                for c in ROUTER_CASES])
def test_router_exact_ties_go_to_lower_index(kernel, T, E, k, xd, kind):
    d = 1024
    xin, wr, bias = _tie_inputs(kind, T, d, E, xd, seed=T + E + k)
    ms = M.make_shape(T, d, E, 32, 0, k, x_dtype=M.MOE_X_F32 if xd == "f32" else M.MOE_X_BF16)
    tc = M.moe_route_workspace_size(ms) > 0
    assert tc == (kernel == "tensor-core")
    x = to_device_tokens(xin, DEV)
    scores = torch.empty(T, E, dtype=torch.float32, device=DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, k, dtype=torch.float32, device=DEV)
    load = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    nws = M.moe_route_workspace_size(ms)
    ws = torch.empty(nws, dtype=torch.uint8, device=DEV) if nws else None
    M.moe_route(ms, x, torch.from_numpy(wr).to(DEV), None, torch.from_numpy(bias).to(DEV), scores, idx,
                gate, load, ws)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref_s = O.router_scores(tokens64(xin), wr)
    assert np.abs(sc - ref_s).max() <= 1e-5
    keys = O.selection_keys(sc, bias)
    # The case really has ties among the k + 1 largest keys (at the selection boundary,
    # or inside the winners, where they decide the output order) for most tokens.
    srt = -np.sort(-keys, axis=1)[:, :k + 1]
    tied = (srt[:, 1:] == srt[:, :-1]).any(axis=1)
    assert tied.mean() > 0.5, tied.mean()
    ref_idx = O.topk_select(sc, bias, k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.abs(gate.cpu().numpy() - O.gate_weights(sc.astype(np.float64), ref_idx, True)).max() <= 1e-6
    assert np.array_equal(load.cpu().numpy(), O.expert_load(ref_idx, E))
    if kind.startswith("zero"):
        assert (sc == 0.5).all()  # sigmoid(0) is exactly 1/2
        want = np.array(sorted(range(E), key=lambda e: (-float(np.float32(0.5) + bias[e]), e))[:k])
        assert (idx.cpu().numpy() == want[None, :]).all()
        assert (gate.cpu().numpy() == np.float32(1.0 / k)).all()


@pytest.mark.parametrize("kind,T", [("zero", 1024), ("grid", 2048), ("zero_grid_bias", 300)])
def test_layer_exact_ties_match_oracle(kind, T):
    """The whole layer on tie-built routing: selection, permutation and bias bit for bit,
    output within tolerance (x = 0 gives an exactly zero output, every pair on the
    lowest experts)."""
    s = CONFIGS["nano"].replace(T=T)
    host = make_layer(s.replace(T=1), "nano", with_tokens=False)
    xin, wr, bias = _tie_inputs(kind, T, s.d, s.E, "bf16", seed=T)
    host.update(x=xin, w_router=wr, bias=bias, logit_offset=None)
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(xin, DEV)
    scores = torch.empty(T, s.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(T, s.k, dtype=torch.int32, device=DEV)
    load = torch.empty(s.E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(s.E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * s.k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T, s.k, dtype=torch.int32, device=DEV)
    out = torch.empty(T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=True, debug=M.make_debug(scores=scores, idx=idx, load=load, offsets=offsets,
                                                               perm_tok=perm, inv_pos=inv))
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref = O.layer_forward(tokens64(xin), wr, bias, bf64(host["w_gate"]), bf64(host["w_up"]), bf64(host["w_down"]),
                          bf64(host["s_gate"]), bf64(host["s_up"]), bf64(host["s_down"]), k=s.k,
                          gamma=host["gamma"], scores_f32=sc)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(load.cpu().numpy(), ref["load"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(perm.cpu().numpy(), ref["perm_tok"])
    assert np.array_equal(inv.cpu().numpy(), ref["inv_pos"])
    assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), ref["bias"].view(np.uint32))
    got = bf16_to_np(out)
    if kind == "zero":
        assert (ref["idx"] == np.array([[0, 1]])).all() and (got == 0).all()
    else:
        assert_close_bf16(got, ref["out"], "layer out on tied routing")

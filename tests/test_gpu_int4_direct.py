"""Top-1 int4 serving above 8 tokens without the permutation: the routed experts on the
tensor cores straight from the routing result, on the GPU through the C ABI, against
the oracle.

Relay article, opening section (int4 experts, sigmoid-plus-bias router, shared expert)
and section "Entrenamiento por relevos", top-2 paragraph (serving with one expert per
token).  The cases reach every branch of the routed kernels: an expert with one pair,
experts with more than 8 pairs (several passes over the MMA's 8 columns, the last one
ragged), every pair on one expert, and shapes where a warp's share of the inputs ends
inside its register chunk.  Checked: selection and loads bit for bit, the bias update
bit for bit, the output within the bf16 tolerance of the oracle run on its own
dequantised weights.
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


def _check(s, host, residual):
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    res_bits = make_tokens(s, "decode", seed=5) if residual else None
    res = to_device_tokens(res_bits, DEV) if residual else None
    scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    load = torch.empty(s.E, dtype=torch.int32, device=DEV)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=True, residual=res, debug=M.make_debug(scores=scores, idx=idx, load=load))
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref = O.layer_forward(tokens64(host["x"]), host["w_router"], host["bias"], _dequant(host["w_gate"]),
                          _dequant(host["w_up"]), _dequant(host["w_down"]), bf64(host["s_gate"]),
                          bf64(host["s_up"]), bf64(host["s_down"]), k=1, renorm=False, gamma=s.gamma,
                          scores_f32=sc, logit_offset=host.get("logit_offset"),
                          residual=bf64(res_bits) if residual else None)
    got_idx = idx.cpu().numpy()
    assert np.array_equal(got_idx, ref["idx"])
    ld = O.expert_load(ref["idx"], s.E)
    assert np.array_equal(load.cpu().numpy(), ld)
    want_bias = O.bias_update(host["bias"], ld, s.T * s.k, s.gamma)
    assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), want_bias.view(np.uint32))
    assert_close_bf16(bf16_to_np(out), ref["out"], f"int4 direct T={s.T} d={s.d} f={s.f}")
    return ld


# (T, extra shape fields, residual)
CASES = [
    (9, {}, False),
    (40, {}, True),
    (64, {}, True),
    (64, dict(skew_zipf_s=1.2), False),
    (64, dict(d=512, f=256, F=512), True),
    # with a shared expert and d = 256 (the skinny shared-expert kernels want d a multiple
    # of 512) the layer takes the permutation path instead: checked here all the same
    (24, dict(d=256, f=128, F=256, E=16), False),
    # no shared expert: the CUDA-core kernels where the tensor-core ones do not apply
    # (d = 192: gate/up and down; f = 128: the down projection)
    (24, dict(d=192, f=128, F=0, E=16), True),
    (40, dict(d=256, f=128, F=0, E=16), False),
]


@pytest.mark.parametrize("T,kw,residual", CASES,
                         ids=[f"T{c[0]}" + "".join(f"-{k}{v}" for k, v in c[1].items()) +
                              ("-res" if c[2] else "") for c in CASES])
def test_int4_direct_serving_matches_oracle(T, kw, residual):
    s = CONFIGS["decode"].replace(T=T, **kw)
    host = make_layer(s, "decode")
    ld = _check(s, host, residual)
    if "skew_zipf_s" in kw:
        assert ld.max() > 8  # several passes over the MMA's columns for one expert


@pytest.mark.parametrize("T", [20, 64])
def test_int4_direct_serving_every_pair_on_one_expert(T):
    """A zero router and a zero bias: every key ties, every token takes expert 0, and
    that expert's rows serve all T pairs in ceil(T / 8) passes."""
    s = CONFIGS["decode"].replace(T=T)
    host = make_layer(s, "decode")
    host["bias"] = np.zeros(s.E, np.float32)
    host["w_router"] = np.zeros_like(host["w_router"])
    ld = _check(s, host, False)
    assert ld[0] == T

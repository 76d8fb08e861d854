"""Expert-balance statistics and the bias update from summed loads, on the GPU.

The relay's dashboard tracks expert balance and the top-2 paragraph reports a low
dead-expert fraction (relay article, section "Entrenamiento por relevos"); the library
computes max/mean, min/mean and the dead fraction on the device (moe_load_balance, or
moe_layer_fwd's debug output, fused into the permutation's first block).  Compared bit
for bit with oracle.balance_stats.  The skewed 50-step trajectory checks the fused
output on every step (tests/test_gpu_parity.py).
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import LayerOnDevice, to_device_tokens
from oracle import moe_oracle as O
from synth import CONFIGS, make_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    yield
    assert M.moe_device_status() == 0


def assert_balance_equal(got: dict, want: dict, what=""):
    for key in ("pairs", "max_load", "min_load", "dead_experts"):
        assert got[key] == want[key], (what, key, got[key], want[key])
    for key in ("max_over_mean", "min_over_mean", "dead_fraction"):
        g = np.float32(got[key]).view(np.uint32)
        w = np.float32(want[key]).view(np.uint32)
        assert g == w, (what, key, got[key], want[key])


def test_load_balance_matches_oracle_bitwise():
    rng = np.random.default_rng(8)
    buf = torch.zeros(M.BALANCE_BYTES, dtype=torch.uint8, device=DEV)
    cases = [np.zeros(64, np.int32), np.full(64, 256, np.int32), np.array([7], np.int32)]
    for E in (1, 3, 8, 40, 64, 255, 256):
        for _ in range(5):
            ld = rng.integers(0, 3000, E).astype(np.int32)
            ld[rng.random(E) < 0.25] = 0
            cases.append(ld)
    cases.append(np.array([16384] + [0] * 63, np.int32))
    for ld in cases:
        M.moe_load_balance(len(ld), torch.from_numpy(ld).to(DEV), buf)
        got = M.balance_from_bytes(buf)
        assert_balance_equal(got, O.balance_stats(ld, len(ld)), str(ld[:4]))


def test_bias_update_takes_global_tokens_times_k_from_summed_loads():
    """MOE_TK_FROM_LOAD: the kernel sums the loads itself; equal to the update with the
    true global T*k passed in, bit for bit, for loads that do not divide evenly."""
    rng = np.random.default_rng(9)
    for E, tk in ((64, 194), (16, 97 * 2), (256, 70001 * 4), (8, 5)):
        ld = np.bincount(rng.integers(0, E, tk), minlength=E).astype(np.int32)
        bias = rng.uniform(-0.05, 0.05, E).astype(np.float32)
        b = torch.from_numpy(bias).to(DEV)
        M.moe_bias_update(E, M.MOE_TK_FROM_LOAD, torch.from_numpy(ld).to(DEV), 1e-3, b)
        torch.cuda.synchronize()
        want = O.bias_update(bias, ld, int(ld.sum()), 1e-3)
        assert np.array_equal(b.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("T", [3, 64, 200])
def test_serving_path_balance_output(T):
    """The top-1 int4 serving path (no permutation up to 64 pairs, the permutation
    beyond): the fused balance output equals the oracle's statistics of its loads."""
    s = CONFIGS["decode"].replace(T=T)
    host = make_layer(s, "decode")
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    scores = torch.empty(T, s.E, dtype=torch.float32, device=DEV)
    buf = torch.zeros(M.BALANCE_BYTES, dtype=torch.uint8, device=DEV)
    out = torch.empty(T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=False, debug=M.make_debug(scores=scores, balance=buf))
    torch.cuda.synchronize()
    idx = O.topk_select(scores.cpu().numpy(), host["bias"], s.k)
    assert_balance_equal(M.balance_from_bytes(buf), O.balance_stats(O.expert_load(idx, s.E), s.E))
    assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), host["bias"].view(np.uint32))


@pytest.mark.parametrize("T", [300, 3000])
def test_layer_balance_output(T):
    """The bf16 layer (one stream below 1024 tokens, the second stream above)."""
    s = CONFIGS["nano"].replace(T=T)
    host = make_layer(s, "nano")
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    scores = torch.empty(T, s.E, dtype=torch.float32, device=DEV)
    load = torch.empty(s.E, dtype=torch.int32, device=DEV)
    buf = torch.zeros(M.BALANCE_BYTES, dtype=torch.uint8, device=DEV)
    out = torch.empty(T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=True, debug=M.make_debug(scores=scores, load=load, balance=buf))
    torch.cuda.synchronize()
    ld = O.expert_load(O.topk_select(scores.cpu().numpy(), host["bias"], s.k), s.E)
    assert np.array_equal(load.cpu().numpy(), ld)
    assert_balance_equal(M.balance_from_bytes(buf), O.balance_stats(ld, s.E))

"""GPU parity of the int4 expert residency cache (moe_layer_fwd_cached).

Each serving step runs the layer through the cache and again with every expert
resident (moe_layer_fwd): the outputs must be identical, bit for bit (the same int4
weights, read from a slot instead of their home position, by the same kernels: the
single serving launch up to 8 tokens, the multi-launch path above), and so must the
routing.  After every step the cache's slot table, stamps and counters must equal the
oracle's least-recently-used policy (oracle/expert_cache.py) run on the same routing
results.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import ExpertCache, LayerOnDevice, to_device_tokens
from oracle import expert_cache as OC
from synth import CONFIGS, make_layer, make_tokens

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    yield
    assert M.moe_device_status() == 0


CASES = [
    # at most 8 pairs: the single serving launch (plan and fill inside it); Zipf-skewed routing
    ("direct, skewed", dict(T=8, skew_zipf_s=1.2), 12, 40),
    ("direct, one token", dict(T=1, skew_zipf_s=1.2), 3, 30),
    # 9 to 64 pairs: the permutation-free path (router of small CTAs, tensor-core int4
    # kernels reading the experts from their slots)
    ("direct, 32 tokens", dict(T=32, skew_zipf_s=1.2), 40, 12),
    # more pairs: the permutation path (active experts); more experts than slots
    ("permuted", dict(T=100, E=160, d=256, f=128, F=256, skew_zipf_s=0.8), 120, 12),
]


@pytest.mark.parametrize("what,kw,slots,steps", CASES, ids=[c[0] for c in CASES])
def test_cached_layer_matches_resident_and_oracle(what, kw, slots, steps):
    s = CONFIGS["decode"].replace(**kw)
    host = make_layer(s, "decode", with_tokens=False)
    layer = LayerOnDevice(s, host, DEV)
    cache = ExpertCache(layer, slots)
    expert_bytes = sum(int(t.numel() * t.element_size()) // s.E for t in cache.host.values())
    seen = []
    state = OC.lru_cache_state(s.E, slots)
    tot = dict(hits=0, misses=0, evictions=0)
    for step in range(steps):
        x = to_device_tokens(make_tokens(s, "decode", seed=1000 + step), DEV)
        idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
        idx_r = torch.empty_like(idx)
        out_c = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
        out_r = torch.empty_like(out_c)
        cache.forward(x, out_c, debug=M.make_debug(idx=idx))
        layer.forward(x, out_r, update_bias=False, debug=M.make_debug(idx=idx_r))
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_r), f"step {step}"
        assert torch.equal(out_c.view(torch.int16), out_r.view(torch.int16)), f"step {step}"
        ids = idx.cpu().numpy()
        seen.append(ids)
        state, h, m, ev, _ = OC.lru_cache_step(state, ids)
        tot["hits"] += h
        tot["misses"] += m
        tot["evictions"] += ev
        stats, se, es, sp = cache.read()
        assert np.array_equal(se, state[0]) and np.array_equal(es, state[1]) and np.array_equal(sp, state[2])
        assert stats["steps"] == step + 1 and stats["overflow"] == 0
        assert (stats["hits"], stats["misses"], stats["evictions"]) == (tot["hits"], tot["misses"], tot["evictions"])
        assert stats["bytes"] == tot["misses"] * expert_bytes
    if what.startswith("direct, skewed"):
        assert tot["hits"] > 0 and tot["evictions"] > 0  # the case exercises both


def test_cache_rejects_too_few_slots_and_other_formats():
    s = CONFIGS["decode"].replace(T=8)
    ms = M.make_shape(s.T, s.d, s.E, s.f, s.F, s.k, renorm=s.renorm, w_format=M.MOE_W_INT4_G32)
    assert M.moe_expert_cache_bytes(ms, 7) == 0     # a step can use 8 experts
    assert M.moe_expert_cache_bytes(ms, 8) > 0
    assert M.moe_expert_cache_bytes(ms, 257) == 0
    mb = M.make_shape(s.T, s.d, s.E, s.f, s.F, s.k, renorm=s.renorm)  # bf16 weights
    assert M.moe_expert_cache_bytes(mb, 16) == 0

"""Pins of the oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against brute force, a closed form, a special
case that reduces to a library routine, an invariant the method fixes, or the
hand-worked example in tests/golden/.  A plausible slip (dropped term, wrong sign,
transposed operand, wrong index) fails at least one of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import CONFIGS, f32_from_bf16_bits, make_layer


def _bf(b):
    return f32_from_bf16_bits(b).astype(np.float64)


# ---------------------------------------------------------------- top-k selection

def _brute_force_topk(keys_row, k):
    """Best k-subset: maximise the descending key vector, then the smallest index set."""
    E = len(keys_row)
    best = None
    for subset in itertools.combinations(range(E), k):
        vec = tuple(sorted((float(keys_row[e]) for e in subset), reverse=True))
        rank = (tuple(-v for v in vec), subset)
        if best is None or rank < best[0]:
            best = (rank, subset)
    chosen = best[1]
    return sorted(chosen, key=lambda e: (-float(keys_row[e]), e))


@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_matches_brute_force_with_ties(k):
    rng = np.random.default_rng(11)
    E, T = 8, 200
    # Few distinct values so that ties are everywhere.
    scores = rng.choice(np.array([0.25, 0.5, 0.625, 0.75], np.float32), size=(T, E))
    bias = rng.choice(np.array([0.0, 0.125, -0.125], np.float32), size=E)
    idx = O.topk_select(scores, bias, k)
    keys = scores + bias[None, :]
    for t in range(T):
        assert list(idx[t]) == _brute_force_topk(keys[t], k)


def test_topk_tiny_workload_matches_brute_force():
    s = CONFIGS["tiny"]
    L = make_layer(s, "tiny")
    sc = O.router_scores(L["x"], L["w_router"]).astype(np.float32)
    idx = O.topk_select(sc, L["bias"], 2)
    keys = O.selection_keys(sc, L["bias"])
    for t in range(s.T):
        assert list(idx[t]) == _brute_force_topk(keys[t], 2)


def test_topk_matches_stable_argsort_library():
    rng = np.random.default_rng(3)
    scores = rng.random((300, 64)).astype(np.float32)
    bias = (rng.random(64).astype(np.float32) - 0.5) * np.float32(0.02)
    keys = (scores + bias).astype(np.float32)
    lib = np.argsort(-keys, axis=1, kind="stable")[:, :2]
    assert np.array_equal(O.topk_select(scores, bias, 2), lib)


def test_topk_all_equal_keys_picks_lowest_indices():
    scores = np.full((5, 8), 0.5, np.float32)
    idx = O.topk_select(scores, np.zeros(8, np.float32), 2)
    assert (idx == np.array([0, 1])).all()


def test_top1_is_first_argmax():
    rng = np.random.default_rng(5)
    scores = rng.choice(np.array([0.1, 0.2, 0.3], np.float32), size=(100, 16))
    idx = O.topk_select(scores, np.zeros(16, np.float32), 1)
    assert np.array_equal(idx[:, 0], np.argmax(scores, axis=1))


def test_bias_steers_selection_only():
    # A bias that flips the winner must not enter the gate: gates use the raw score.
    scores = np.array([[0.6, 0.5, 0.1]], np.float32)
    bias = np.array([0.0, 0.2, 0.0], np.float32)
    idx = O.topk_select(scores, bias, 1)
    assert idx[0, 0] == 1
    g = O.gate_weights(scores, idx, renorm=False)
    assert g[0, 0] == np.float64(np.float32(0.5))


# ---------------------------------------------------------------- router scores

def test_sigmoid_closed_forms_and_orientation():
    # W_r is a non-symmetric permutation: logit_e = x[sigma(e)].  With x = ln 3 at the
    # position expert 2 reads and -ln 3 where expert 0 reads, the scores are 3/4 and 1/4.
    d, E = 4, 4
    sigma = [3, 0, 1, 2]
    W = np.zeros((E, d), np.float32)
    for e in range(E):
        W[e, sigma[e]] = 1.0
    x = np.zeros((1, d))
    x[0, 1] = math.log(3.0)   # expert 2 reads x[1]
    x[0, 3] = -math.log(3.0)  # expert 0 reads x[3]
    s = O.router_scores(x, W)
    assert s[0, 2] == pytest.approx(0.75, abs=1e-15)
    assert s[0, 0] == pytest.approx(0.25, abs=1e-15)
    assert s[0, 1] == 0.5 and s[0, 3] == 0.5
    off = np.array([0.0, math.log(3.0), 0.0, 0.0])
    assert O.router_scores(np.zeros((1, d)), W, off)[0, 1] == pytest.approx(0.75, abs=1e-15)


def test_zero_tokens_give_half_scores_and_lowest_pair():
    E, d = 8, 64
    W = np.random.default_rng(0).standard_normal((E, d)).astype(np.float32)
    s = O.router_scores(np.zeros((3, d)), W)
    assert (s == 0.5).all()
    idx = O.topk_select(s.astype(np.float32), np.zeros(E, np.float32), 2)
    assert (idx == [0, 1]).all()
    assert (O.gate_weights(s, idx, True) == 0.5).all()


def test_router_matches_torch_library():
    s = CONFIGS["tiny"]
    L = make_layer(s, "tiny")
    ref = torch.sigmoid(torch.from_numpy(L["x"]).double() @ torch.from_numpy(L["w_router"]).double().T)
    assert np.allclose(O.router_scores(L["x"], L["w_router"]), ref.numpy(), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- gates and loads

def test_gate_renorm_properties():
    rng = np.random.default_rng(8)
    s = rng.random((50, 16))
    idx = O.topk_select(s.astype(np.float32), np.zeros(16, np.float32), 2)
    g = O.gate_weights(s, idx, True)
    assert np.allclose(g.sum(axis=1), 1.0, atol=1e-15)
    g1 = O.gate_weights(s, O.topk_select(s.astype(np.float32), np.zeros(16, np.float32), 1), True)
    assert (g1 == 1.0).all()          # top-1 with renormalisation: constant weight
    g_off = O.gate_weights(s, idx, False)
    assert np.array_equal(g_off, np.take_along_axis(s, idx, axis=1))


def test_load_matches_bincount_and_sums():
    rng = np.random.default_rng(2)
    idx = np.stack([rng.permutation(64)[:2] for _ in range(1000)])
    load = O.expert_load(idx, 64)
    assert load.sum() == 2000
    assert np.array_equal(load, np.bincount(idx.ravel(), minlength=64))


# ---------------------------------------------------------------- permutation

def test_permutation_invariants_and_library_sort():
    rng = np.random.default_rng(4)
    T, E, k = 500, 16, 2
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    offsets, perm_tok, inv_pos = O.stable_permutation(idx, E)
    load = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(load)]))
    assert sorted(perm_tok.tolist()) == sorted(np.repeat(np.arange(T), k).tolist())
    assert sorted(inv_pos.ravel().tolist()) == list(range(T * k))        # bijection
    for t in range(T):
        for j in range(k):
            p = inv_pos[t, j]
            assert perm_tok[p] == t
            assert offsets[idx[t, j]] <= p < offsets[idx[t, j] + 1]
    for e in range(E):
        blk = perm_tok[offsets[e]:offsets[e + 1]]
        assert (np.diff(blk) > 0).all()                                   # ascending tokens
    order = np.argsort(idx.ravel(), kind="stable")                        # library stable sort
    assert np.array_equal(perm_tok, order // k)
    assert np.array_equal(inv_pos.ravel()[order], np.arange(T * k))


# ---------------------------------------------------------------- bias update

def _nearest_f32(q: Fraction) -> np.float32:
    """Nearest fp32 to an exact rational, found by bracketing (ties to even)."""
    c = np.float32(float(q))
    lo, hi = np.nextafter(c, np.float32(-np.inf)), np.nextafter(c, np.float32(np.inf))
    cands = sorted([lo, c, hi], key=lambda v: (abs(Fraction(float(v)) - q),
                                               int(np.array(v).view(np.uint32)) & 1))
    return cands[0]


def test_bias_update_bitwise_nearest_and_direction():
    rng = np.random.default_rng(6)
    E, T, k = 64, 8192, 2
    bias = rng.uniform(-0.01, 0.01, E).astype(np.float32)
    bias[:4] = [0.0, 1.0, -1.0, 0.125]
    load = rng.integers(0, 600, E)
    load[4] = T * k // E                            # exactly on target: unchanged
    new = O.bias_update(bias, load, T * k, 1e-3)
    g = Fraction(float(np.float32(1e-3)))
    for e in range(E):
        target_minus = Fraction(T * k, E) - int(load[e])
        if target_minus == 0:
            assert new[e] == bias[e]
            continue
        step = g if target_minus > 0 else -g       # under-loaded experts go up
        want = _nearest_f32(Fraction(float(bias[e])) + step)
        assert new[e].view(np.uint32) == want.view(np.uint32), e


def test_bias_update_balanced_loads_leave_bias_unchanged():
    bias = np.linspace(-0.01, 0.01, 8).astype(np.float32)
    new = O.bias_update(bias, np.full(8, 16), 64 * 2, 1e-3)
    assert np.array_equal(new.view(np.uint32), bias.view(np.uint32))


def test_bias_update_replicas_equal_full_batch():
    s = CONFIGS["tiny"].replace(T=96)
    rng = np.random.default_rng(9)
    sc = rng.random((s.T, s.E)).astype(np.float32)
    bias = np.zeros(s.E, np.float32)
    idx = O.topk_select(sc, bias, s.k)
    full = O.bias_update(bias, O.expert_load(idx, s.E), s.T * s.k, 1e-3)
    for n in (2, 3, 4):
        shards = np.array_split(np.arange(s.T), n)
        load = sum(O.expert_load(O.topk_select(sc[sh], bias, s.k), s.E) for sh in shards)
        assert np.array_equal(O.bias_update(bias, load, s.T * s.k, 1e-3).view(np.uint32),
                              full.view(np.uint32))


# ---------------------------------------------------------------- hand-worked fixture

def test_golden_route_permute_bias(golden_dir):
    G = json.load(open(os.path.join(golden_dir, "route_permute_bias_worked.json")))
    s = np.array(G["scores"], np.float32)
    b = np.array(G["bias"], np.float32)
    idx = O.topk_select(s, b, G["k"])
    assert idx.tolist() == G["idx"]
    g = O.gate_weights(s.astype(np.float64), idx, True)
    for t in range(G["T"]):
        for j in range(G["k"]):
            num, den = G["gate_num_den"][t][j]
            assert g[t, j] == pytest.approx(num / den, abs=1e-15)
    load = O.expert_load(idx, G["E"])
    assert load.tolist() == G["load"]
    off, perm, inv = O.stable_permutation(idx, G["E"])
    assert off.tolist() == G["offsets"] and perm.tolist() == G["perm_tok"]
    assert inv.tolist() == G["inv_pos"]
    nb = O.bias_update(b, load, G["T"] * G["k"], G["gamma"])
    for e, sg in enumerate(G["bias_sign"]):
        assert np.sign(float(nb[e]) - float(b[e])) == sg


# ---------------------------------------------------------------- bf16 rounding

def test_round_to_bf16_against_torch_and_ties():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(20000) * 3).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(v.astype(np.float64)), lib)
    assert O.round_to_bf16(np.array([1 + 2 ** -8]))[0] == 1.0                  # tie -> even
    assert O.round_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6      # tie -> even
    assert O.round_to_bf16(np.array([1 + 2 ** -8 + 2 ** -20]))[0] == 1 + 2 ** -7


# ---------------------------------------------------------------- expert FFN

def test_swiglu_structured_weights_closed_form():
    # d = f = 5, W_gate = diag(c), W_up = I, W_down a permutation sigma (rows pick hidden
    # units).  Then y_i = silu(c_s x_s) * x_s with s = sigma(i): this fixes which matrix
    # gets the activation and the orientation of each matrix.
    n = 5
    c = np.array([0.5, -1.0, 2.0, 0.25, 1.5])
    sigma = [2, 4, 0, 1, 3]
    Wg = np.diag(c)
    Wu = np.eye(n)
    Wd = np.zeros((n, n))
    for i in range(n):
        Wd[i, sigma[i]] = 1.0
    x = np.array([[0.3, -0.7, 1.1, 2.0, -1.5]])
    y = O.swiglu_ffn(x, Wg, Wu, Wd, round_hidden=False)
    for i in range(n):
        s_ = sigma[i]
        a = c[s_] * x[0, s_]
        assert y[0, i] == pytest.approx(a / (1 + math.exp(-a)) * x[0, s_], abs=1e-15)
    # Swapping gate and up changes the result (the activation is on the gate only).
    y_sw = O.swiglu_ffn(x, Wu, Wg, Wd, round_hidden=False)
    assert not np.allclose(y, y_sw)


def test_dense_swiglu_matches_torch_library():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((33, 64))
    Wg, Wu = rng.standard_normal((2, 48, 64)) * 0.1
    Wd = rng.standard_normal((64, 48)) * 0.1
    tx = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(tx @ torch.from_numpy(Wg).T) * (tx @ torch.from_numpy(Wu).T)) \
        @ torch.from_numpy(Wd).T
    assert np.allclose(O.swiglu_ffn(x, Wg, Wu, Wd, round_hidden=False), ref.numpy(), atol=1e-12)


def _tiny_layer(**override):
    s = CONFIGS["tiny"]
    L = make_layer(s, "tiny")
    P = dict(x=L["x"].astype(np.float64), w_router=L["w_router"], bias=L["bias"],
             w_gate=_bf(L["w_gate"]), w_up=_bf(L["w_up"]), w_down=_bf(L["w_down"]),
             s_gate=_bf(L["s_gate"]), s_up=_bf(L["s_up"]), s_down=_bf(L["s_down"]),
             k=s.k, x_is_bf16=False)
    P.update(override)
    return s, P


def test_layer_equals_per_token_dense_mixture():
    # Independent formulation without any permutation: for each token, run the shared
    # expert and each selected expert directly and add them with the gates.
    s, P = _tiny_layer()
    r = O.layer_forward(**P)
    xb = O.round_to_bf16(P["x"])
    for t in range(s.T):
        want = O.swiglu_ffn(xb[t:t + 1], P["s_gate"], P["s_up"], P["s_down"])[0]
        for j in range(s.k):
            e = r["idx"][t, j]
            want = want + r["gate"][t, j] * O.swiglu_ffn(xb[t:t + 1], P["w_gate"][e], P["w_up"][e],
                                                        P["w_down"][e])[0]
        assert np.allclose(r["out"][t], want, rtol=0, atol=1e-14)


def test_layer_zero_weights_isolate_the_two_branches():
    s, P = _tiny_layer()
    r_full = O.layer_forward(**P)
    r_no_shared = O.layer_forward(**dict(P, s_down=np.zeros_like(P["s_down"])))
    r_no_routed = O.layer_forward(**dict(P, w_down=np.zeros_like(P["w_down"])))
    assert np.allclose(r_no_routed["out"], r_full["shared"], atol=0)
    routed = r_full["out"] - r_full["shared"]
    assert np.allclose(r_no_shared["out"], routed, atol=1e-15)
    # The routed branch is linear in W_down.
    r2 = O.layer_forward(**dict(P, s_down=np.zeros_like(P["s_down"]), w_down=2 * P["w_down"]))
    assert np.allclose(r2["out"], 2 * r_no_shared["out"], atol=1e-15)


def test_layer_invariants_tiny():
    s, P = _tiny_layer()
    r = O.layer_forward(**P)
    assert r["load"].sum() == s.T * s.k
    for t in range(s.T):
        assert len(set(r["idx"][t].tolist())) == s.k
    assert np.allclose(r["gate"].sum(axis=1), 1.0, atol=1e-12)
    assert set(np.abs(r["bias"] - P["bias"]).tolist()) <= {0.0, float(np.float32(1e-3))}


# ---------------------------------------------------------------- int4 container

def test_int4_exact_codes_and_nibble_order():
    s = np.float32(0.0625)                       # exactly representable in fp16
    q = np.array([1, -1, 7, -7, 0, 3, -4, 2] * 4, dtype=np.float32)
    w = (q * s)[None, :]
    packed, scale, codes = O.quantize_int4_g32(w)
    assert scale.view(np.float16)[0, 0] == np.float16(s)
    assert np.array_equal(codes[0], q.astype(np.int8))
    assert packed[0, 0] == 0xF1 and packed[0, 1] == 0x97     # (1, -1) and (7, -7)
    assert np.array_equal(O.dequantize_int4_g32(packed, scale), w.astype(np.float64))


def test_int4_roundtrip_error_bound_and_zero_group():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3, 32:64] = 0.0
    packed, scale, codes = O.quantize_int4_g32(w)
    deq = O.dequantize_int4_g32(packed, scale)
    sc = np.repeat(O.fp16_value_from_bits(scale), 32, axis=1)
    # |w - q*s| <= s/2 inside the range, plus the fp16 rounding of the scale at the edge.
    assert (np.abs(deq - w) <= sc / 2 + np.abs(w) * 2 ** -10 + 1e-12).all()
    assert (codes[3, 32:64] == 0).all() and O.fp16_value_from_bits(scale)[3, 1] == 0.0
    assert codes.max() <= 7 and codes.min() >= -7


# ---------------------------------------------------------------- backward

def _bwd_case(seed, T=6, d=16, E=5, f=8, F=12, k=2):
    """Small random layer in fp64 with a selection held fixed (top-k of its own
    scores); the scores are kept away from ties so the selection is stable."""
    rng = np.random.default_rng(seed)
    P = dict(x=rng.standard_normal((T, d)), w_router=rng.standard_normal((E, d)) * 0.4,
             bias=np.zeros(E, np.float32), w_gate=rng.standard_normal((E, f, d)) * 0.3,
             w_up=rng.standard_normal((E, f, d)) * 0.3, w_down=rng.standard_normal((E, d, f)) * 0.3,
             s_gate=rng.standard_normal((F, d)) * 0.3, s_up=rng.standard_normal((F, d)) * 0.3,
             s_down=rng.standard_normal((d, F)) * 0.3, dout=rng.standard_normal((T, d)))
    sc = O.router_scores(P["x"], P["w_router"])
    P["idx"] = O.topk_select(sc.astype(np.float32), P["bias"], k)
    return P


def _torch_layer(P, k, renorm, residual):
    """The layer written densely in PyTorch (CPU, fp64), selection fixed to P['idx'];
    autograd supplies every gradient independently of the oracle's chain rule."""
    t = {n: torch.tensor(P[n], dtype=torch.float64, requires_grad=True)
         for n in ("x", "w_router", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")}
    idx = torch.tensor(P["idx"].astype(np.int64))
    s = torch.sigmoid(t["x"] @ t["w_router"].T)
    ssel = torch.gather(s, 1, idx)
    g = ssel / ssel.sum(dim=1, keepdim=True) if renorm else ssel
    out = torch.zeros_like(t["x"])
    for j in range(k):
        e = idx[:, j]
        a = torch.einsum("tfd,td->tf", t["w_gate"][e], t["x"])
        b = torch.einsum("tfd,td->tf", t["w_up"][e], t["x"])
        h = torch.nn.functional.silu(a) * b
        y = torch.einsum("tdf,tf->td", t["w_down"][e], h)
        out = out + g[:, j:j + 1] * y
    hs = torch.nn.functional.silu(t["x"] @ t["s_gate"].T) * (t["x"] @ t["s_up"].T)
    out = out + hs @ t["s_down"].T
    if residual:
        out = out + t["x"]
    (out * torch.tensor(P["dout"])).sum().backward()
    return {n: v.grad.numpy() for n, v in t.items()}


@pytest.mark.parametrize("renorm,residual,k", [(True, False, 2), (False, True, 1), (True, True, 3)])
def test_backward_matches_torch_autograd(renorm, residual, k):
    P = _bwd_case(11 + k, k=k)
    ref = _torch_layer(P, k, renorm, residual)
    g = O.layer_backward(P["x"], P["w_router"], P["bias"], P["w_gate"], P["w_up"], P["w_down"],
                         P["s_gate"], P["s_up"], P["s_down"], P["dout"], k=k, renorm=renorm,
                         residual=residual, idx=P["idx"], exact_gates=True, round_hidden=False)
    pairs = {"x": "dx", "w_router": "dw_router", "w_gate": "dw_gate", "w_up": "dw_up",
             "w_down": "dw_down", "s_gate": "ds_gate", "s_up": "ds_up", "s_down": "ds_down"}
    for n, m in pairs.items():
        assert np.allclose(g[m], ref[n], rtol=1e-10, atol=1e-12), n


def test_backward_directional_finite_differences():
    """d/de <dout, out(theta + e v)> at e = 0 equals <grad, v> for random directions,
    from the oracle's own forward (selection fixed, exact gates, H not rounded)."""
    P = _bwd_case(5)
    k = 2

    def loss(**over):
        Q = dict(P, **over)
        r = O.layer_forward(Q["x"], Q["w_router"], Q["bias"], Q["w_gate"], Q["w_up"], Q["w_down"],
                            Q["s_gate"], Q["s_up"], Q["s_down"], k=k, renorm=True, idx=P["idx"],
                            exact_gates=True, round_hidden=False)
        return float((r["out"] * P["dout"]).sum())

    g = O.layer_backward(P["x"], P["w_router"], P["bias"], P["w_gate"], P["w_up"], P["w_down"],
                         P["s_gate"], P["s_up"], P["s_down"], P["dout"], k=k, renorm=True,
                         idx=P["idx"], exact_gates=True, round_hidden=False)
    rng = np.random.default_rng(99)
    eps = 1e-6
    for n, m in (("x", "dx"), ("w_router", "dw_router"), ("w_gate", "dw_gate"), ("w_up", "dw_up"),
                 ("w_down", "dw_down"), ("s_gate", "ds_gate"), ("s_up", "ds_up"), ("s_down", "ds_down")):
        v = rng.standard_normal(P[n].shape)
        fd = (loss(**{n: P[n] + eps * v}) - loss(**{n: P[n] - eps * v})) / (2 * eps)
        assert abs(fd - float((g[m] * v).sum())) <= 1e-6 * max(1.0, abs(fd)), n


def test_backward_gate_gradient_special_cases():
    """Top-1 with renormalisation: the gate is the constant 1, so no gradient reaches
    the router (the top-2 paragraph's reason for top-2); without renormalisation the
    gate is the score and the router gradient is dgate * s (1 - s)."""
    P = _bwd_case(3, k=1)
    g = O.layer_backward(P["x"], P["w_router"], P["bias"], P["w_gate"], P["w_up"], P["w_down"],
                         P["s_gate"], P["s_up"], P["s_down"], P["dout"], k=1, renorm=True,
                         idx=P["idx"], exact_gates=True)
    assert np.all(g["gate"] == 1.0) and np.all(g["dz"] == 0.0) and np.all(g["dw_router"] == 0.0)
    g2 = O.layer_backward(P["x"], P["w_router"], P["bias"], P["w_gate"], P["w_up"], P["w_down"],
                          P["s_gate"], P["s_up"], P["s_down"], P["dout"], k=1, renorm=False,
                          idx=P["idx"], exact_gates=True)
    sc = O.router_scores(P["x"], P["w_router"])
    for t in range(P["x"].shape[0]):
        e = int(P["idx"][t, 0])
        assert np.isclose(g2["dz"][t, e], g2["dgate"][t, 0] * sc[t, e] * (1 - sc[t, e]), rtol=1e-12)


# ----------------------------------------------------------------- expert cache (LRU)

def test_expert_cache_worked_example():
    """The least-recently-used reading, worked by hand on a 6-expert, 3-slot cache."""
    import json
    import os
    from oracle import expert_cache as C
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "expert_cache_lru_worked.json")))
    state = C.lru_cache_state(g["E"], g["slots"])
    for st in g["steps"]:
        state, h, m, ev, jobs = C.lru_cache_step(state, np.array(st["idx"]))
        assert (h, m, ev) == (st["hits"], st["misses"], st["evictions"])
        assert [list(j) for j in jobs] == st["jobs"]
        assert state[0].tolist() == st["slot_expert"] and state[2].tolist() == st["stamp"]
    assert state[1].tolist() == g["final_expert_slot"]
    with pytest.raises(C.CacheCapacityError):
        C.lru_cache_step(state, np.array(g["overflow_step_idx"]))


def test_expert_cache_invariants_and_textbook_cases():
    from oracle import expert_cache as C
    rng = np.random.default_rng(0)
    E, slots = 16, 6
    steps = [rng.choice(E, size=rng.integers(1, 4), replace=False) for _ in range(300)]
    r = C.lru_cache_run(E, slots, steps)
    state = C.lru_cache_state(E, slots)
    for s, idx in enumerate(steps):
        state, h, m, ev, jobs = C.lru_cache_step(state, idx)
        used = set(int(e) for e in idx)
        assert h + m == len(used)
        slot_expert, expert_slot = state[0], state[1]
        assert all(expert_slot[e] >= 0 and slot_expert[expert_slot[e]] == e for e in used)
        assert all(slot_expert[expert_slot[e]] == e for e in range(E) if expert_slot[e] >= 0)
        assert all(expert_slot[slot_expert[c]] == c for c in range(slots) if slot_expert[c] >= 0)
        assert (h, m, ev) == (r["hits"][s], r["misses"][s], r["evictions"][s])
    # Enough slots for every expert: one miss per first touch, never an eviction.
    r2 = C.lru_cache_run(E, E, steps)
    assert sum(r2["misses"]) == len(set(int(e) for st in steps for e in st)) and sum(r2["evictions"]) == 0
    # Cycling one expert per step over slots + 1 experts: LRU misses every time.
    cyc = [np.array([s % (slots + 1)]) for s in range(50)]
    r3 = C.lru_cache_run(E, slots, cyc)
    assert all(m == 1 for m in r3["misses"])
    # A working set that fits: misses only on the first pass.
    ws = [np.array([s % slots]) for s in range(60)]
    r4 = C.lru_cache_run(E, slots, ws)
    assert sum(r4["misses"]) == slots and all(m == 0 for m in r4["misses"][slots:])


# ---------------------------------------------------------------- combine residual


def test_golden_combine_with_and_without_residual(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "combine_residual_worked.json")))
    Y, sh = np.array(g["Y"]), np.array(g["shared"])
    inv, gate, res = np.array(g["inv_pos"]), np.array(g["gate"]), np.array(g["residual"])
    assert np.array_equal(O.combine(Y, sh, inv, gate), np.array(g["out_without_residual"]))
    assert np.array_equal(O.combine(Y, sh, inv, gate, residual=res), np.array(g["out_with_residual"]))


def test_combine_residual_is_added_once():
    # Dyadic values on a coarse grid: every sum below is exact in fp64, so the residual
    # must appear exactly once (a dropped or doubled residual fails the equality).
    rng = np.random.default_rng(11)
    T, k, d = 16, 3, 8
    Y = rng.integers(-64, 64, (T * k, d)) / 8.0
    sh = rng.integers(-64, 64, (T, d)) / 8.0
    res = rng.integers(-64, 64, (T, d)) / 8.0
    inv = rng.permutation(T * k).reshape(T, k)
    gate = rng.integers(1, 8, (T, k)) / 8.0
    base = O.combine(Y, sh, inv, gate)
    with_res = O.combine(Y, sh, inv, gate, residual=res)
    assert np.array_equal(with_res - res, base)
    assert not np.array_equal(with_res, base)


def test_layer_with_residual_equals_per_token_dense_mixture_plus_x():
    s, P = _tiny_layer()
    xb = O.round_to_bf16(P["x"])
    r = O.layer_forward(**P, residual=xb)
    r0 = O.layer_forward(**P)
    for t in range(s.T):
        want = xb[t] + O.swiglu_ffn(xb[t:t + 1], P["s_gate"], P["s_up"], P["s_down"])[0]
        for j in range(s.k):
            e = r["idx"][t, j]
            want = want + r["gate"][t, j] * O.swiglu_ffn(xb[t:t + 1], P["w_gate"][e], P["w_up"][e],
                                                        P["w_down"][e])[0]
        assert np.allclose(r["out"][t], want, rtol=0, atol=1e-13)
    assert np.allclose(r["out"] - xb, r0["out"], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- balance statistics


def test_golden_balance_stats(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "balance_worked.json")))
    for c in g["cases"]:
        got = O.balance_stats(c["load"], len(c["load"]))
        for key in ("pairs", "max_load", "min_load", "dead_experts"):
            assert got[key] == c[key], (c["load"], key)
        for key in ("max_over_mean", "min_over_mean", "dead_fraction"):
            bits = int(np.float32(got[key]).view(np.uint32))
            assert bits == int(c[key + "_bits"], 16), (c["load"], key, hex(bits))


def test_nearest_f32_against_correctly_rounded_division():
    # Python's int / int is the correctly rounded fp64 quotient (a library routine);
    # rounding that to fp32 gives the nearest fp32 whenever the denominator is below
    # 2^28 (the exact quotient cannot lie within half an fp64 ulp of an fp32 rounding
    # boundary without being one).  Also exact cases and ties.
    rng = np.random.default_rng(3)
    for _ in range(20000):
        a = int(rng.integers(0, 1 << 40))
        b = int(rng.integers(1, 1 << 27))
        assert O.nearest_f32(a, b) == np.float32(a / b), (a, b)
    assert O.nearest_f32(7, 7) == np.float32(1.0)
    # 1 + 2^-24 is halfway between 1 and the next fp32: ties to the even significand (1).
    assert O.nearest_f32((1 << 24) + 1, 1 << 24) == np.float32(1.0)
    # 1 + 3 * 2^-24 is halfway between 1 + 2^-23 and 1 + 2^-22: ties to even (1 + 2^-22).
    assert O.nearest_f32((1 << 24) + 3, 1 << 24) == np.float32(1.0 + 2.0 ** -22)


def test_balance_stats_properties():
    rng = np.random.default_rng(5)
    for E in (1, 3, 8, 64, 256):
        for _ in range(20):
            load = rng.integers(0, 50, E)
            load[rng.random(E) < 0.3] = 0
            st = O.balance_stats(load, E)
            assert st["pairs"] == int(load.sum())
            assert st["max_load"] == int(load.max()) and st["min_load"] == int(load.min())
            assert st["dead_experts"] == int((load == 0).sum())
            if st["pairs"]:
                assert st["min_over_mean"] <= 1.0 <= st["max_over_mean"] <= E
                # Within half an fp32 ulp of the exact ratio.
                exact = st["max_load"] * E / st["pairs"]
                assert abs(float(st["max_over_mean"]) - exact) <= np.spacing(np.float32(exact)) / 2 * 1.0000001
    # Every pair on one expert: max/mean = E, every other expert dead.
    st = O.balance_stats([0, 0, 12, 0], 4)
    assert st["max_over_mean"] == 4.0 and st["dead_fraction"] == 0.75 and st["min_over_mean"] == 0.0

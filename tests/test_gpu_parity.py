"""GPU parity: every step of the CUDA path against the oracle, through the C ABI.

Routing indices, loads, offsets, permutation and bias are compared bit for bit;
scores within 1e-5 absolute, gates within 1e-6, expert and layer outputs within the
bf16 tolerance of gpu_util (2e-2 relative L2 plus an element-wise bound).  The
oracle's top-k is fed the GPU's own fp32 scores, as the parity contract asks.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import LayerOnDevice, to_device_bf16, to_device_tokens
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


def _shape(name, **kw):
    return CONFIGS[name].replace(**kw)


def _ms(s, x_dtype=None):
    xd = x_dtype or s.x_dtype
    return M.make_shape(s.T, s.d, s.E, s.f, s.F, s.k, renorm=s.renorm,
                        x_dtype=M.MOE_X_F32 if xd == "f32" else M.MOE_X_BF16)


ROUTE_CASES = [
    ("tiny", {}),
    ("nano", {}),
    ("skew", {}),
    ("nano", {"T": 1000}),                       # ragged: not a multiple of 32
    ("nano", {"T": 1, "k": 1, "renorm": False}),  # serving shape
    ("nano", {"T": 333, "k": 1}),                 # top-1 with renorm: gates are exactly 1
    ("nano", {"T": 257, "E": 16, "k": 3}),
    ("nano", {"T": 130, "E": 256, "k": 8}),
    ("tiny", {"T": 77, "E": 40, "k": 5}),
]


@pytest.mark.parametrize("name,kw", ROUTE_CASES)
def test_route_matches_oracle(name, kw):
    s = _shape(name, **kw)
    host = make_layer(s.replace(f=32, F=32), name)  # routing does not read the FFN weights
    ms = _ms(s)
    x = to_device_tokens(host["x"], DEV)
    wr = torch.from_numpy(host["w_router"]).to(DEV)
    bias = torch.from_numpy(host["bias"]).to(DEV)
    lo = None if host["logit_offset"] is None else torch.from_numpy(host["logit_offset"]).to(DEV)
    scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(s.T, s.k, dtype=torch.float32, device=DEV)
    load = torch.full((s.E,), -7, dtype=torch.int32, device=DEV)
    nws = M.moe_route_workspace_size(ms)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=DEV) if nws else None
    M.moe_route(ms, x, wr, lo, bias, scores, idx, gate, load, ws)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref_s = O.router_scores(tokens64(host["x"]), host["w_router"], host["logit_offset"])
    assert np.abs(sc - ref_s).max() <= 1e-5
    ref_idx = O.topk_select(sc, host["bias"], s.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    ref_g = O.gate_weights(sc.astype(np.float64), ref_idx, s.renorm)
    assert np.abs(gate.cpu().numpy() - ref_g).max() <= 1e-6
    if s.k == 1 and s.renorm:
        assert (gate.cpu().numpy() == 1.0).all()
    assert np.array_equal(load.cpu().numpy(), O.expert_load(ref_idx, s.E))
    # Secondary check with the oracle's own fp64 scores: equal except at near-ties.
    keys = O.selection_keys(ref_s.astype(np.float32), host["bias"])
    srt = -np.sort(-keys, axis=1)
    clear = (srt[:, s.k - 1] - srt[:, s.k]) >= 1e-6 if s.k < s.E else np.ones(s.T, bool)
    own = O.topk_select(ref_s.astype(np.float32), host["bias"], s.k)
    assert np.array_equal(own[clear], ref_idx[clear])


def _random_idx(T, E, k, seed, skew=False):
    rng = np.random.default_rng(seed)
    p = None
    if skew:
        w = 1.0 / (np.arange(E) + 1.0) ** 1.5
        p = w / w.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


PERM_CASES = [(64, 8, 2, False), (8192, 64, 2, False), (8192, 64, 2, True), (1, 64, 1, False),
              (1000, 64, 2, True), (8192, 256, 4, False), (5000, 3, 3, False), (70000, 64, 2, True)]


@pytest.mark.parametrize("T,E,k,skew", PERM_CASES)
def test_permute_matches_oracle(T, E, k, skew):
    idx_np = _random_idx(T, E, k, seed=T + E + k, skew=skew)
    ms = M.make_shape(T, 64, E, 32, 0, k)
    idx = torch.from_numpy(idx_np).to(DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T, k, dtype=torch.int32, device=DEV)
    ws = torch.empty(M.moe_permute_workspace_size(ms), dtype=torch.uint8, device=DEV)
    ws.fill_(0xAB)  # garbage: the call must not depend on workspace contents
    M.moe_permute(ms, idx, offsets, perm, inv, ws)
    torch.cuda.synchronize()
    o_off, o_perm, o_inv = O.stable_permutation(idx_np, E)
    assert np.array_equal(offsets.cpu().numpy(), o_off)
    assert np.array_equal(perm.cpu().numpy(), o_perm)
    assert np.array_equal(inv.cpu().numpy(), o_inv)


def test_bias_update_bitwise():
    rng = np.random.default_rng(0)
    for E, Tk in ((64, 16384), (8, 128), (256, 1 << 20), (64, 16384 * 3)):
        bias = rng.uniform(-0.05, 0.05, E).astype(np.float32)
        bias[0] = 0.0
        load = rng.integers(0, 2 * Tk // E + 1, E).astype(np.int32)
        load[1] = Tk // E
        b = torch.from_numpy(bias).to(DEV)
        M.moe_bias_update(E, Tk, torch.from_numpy(load).to(DEV), 1e-3, b)
        torch.cuda.synchronize()
        want = O.bias_update(bias, load, Tk, 1e-3)
        assert np.array_equal(b.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_pack_gate_up_layout():
    rng = np.random.default_rng(1)
    for G, width, d in ((3, 512, 128), (1, 2048, 64), (2, 32, 64), (2, 96, 64)):
        wg = rng.integers(0, 65535, (G, width, d), dtype=np.uint16)
        wu = rng.integers(0, 65535, (G, width, d), dtype=np.uint16)
        out = torch.empty(G, 2 * width, d, dtype=torch.bfloat16, device=DEV)
        M.moe_pack_gate_up(G, width, d, to_device_bf16(wg, DEV), to_device_bf16(wu, DEV), out)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        b = M.moe_gate_up_block(width)
        for g in range(G):
            for blk in range(width // b):
                assert np.array_equal(got[g, 2 * blk * b:(2 * blk + 1) * b], wg[g, blk * b:(blk + 1) * b])
                assert np.array_equal(got[g, (2 * blk + 1) * b:(2 * blk + 2) * b], wu[g, blk * b:(blk + 1) * b])


def test_quantize_int4_bitexact():
    s = CONFIGS["decode"]
    host = make_layer(s.replace(E=4), "decode")
    for key in ("w_gate", "w_down"):
        w = host[key].reshape(-1, host[key].shape[-1])
        q = torch.empty(w.shape[0], w.shape[1] // 2, dtype=torch.uint8, device=DEV)
        sc = torch.empty(w.shape[0], w.shape[1] // 32, dtype=torch.int16, device=DEV)
        M.moe_quantize_int4(w.shape[0], w.shape[1], to_device_bf16(w, DEV), q, sc)
        packed, scale, _ = O.quantize_int4_g32(bf64(w).astype(np.float32))
        assert np.array_equal(q.cpu().numpy(), packed)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), scale)


def _oracle_layer(s, host, gpu_scores, residual=None):
    xv = tokens64(host["x"])
    return O.layer_forward(xv, host["w_router"], host["bias"], bf64(host["w_gate"]),
                           bf64(host["w_up"]), bf64(host["w_down"]),
                           bf64(host["s_gate"]) if s.F else None, bf64(host["s_up"]) if s.F else None,
                           bf64(host["s_down"]) if s.F else None, k=s.k, renorm=s.renorm,
                           logit_offset=host["logit_offset"], gamma=host["gamma"],
                           scores_f32=gpu_scores, residual=residual,
                           x_is_bf16=host["x"].dtype == np.uint16)


FFN_CASES = [("tiny", {}), ("nano", {"T": 1000}), ("nano", {"T": 300, "F": 0}),
             ("tiny", {"x_dtype": "bf16"})]


@pytest.mark.parametrize("name,kw", FFN_CASES)
def test_expert_ffn_and_combine_match_oracle(name, kw):
    s = _shape(name, **kw)
    host = make_layer(s, name)
    layer = LayerOnDevice(s, host, DEV)
    ms = layer.shape
    x = to_device_tokens(host["x"], DEV)
    # Routing from the oracle (its own scores), so this test isolates the FFN.
    sc = O.router_scores(tokens64(host["x"]), host["w_router"]).astype(np.float32)
    ref = _oracle_layer(s, host, sc)
    offsets = torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV)
    perm = torch.from_numpy(ref["perm_tok"].astype(np.int32)).to(DEV)
    inv = torch.from_numpy(ref["inv_pos"].astype(np.int32)).to(DEV)
    gate = torch.from_numpy(ref["gate"].astype(np.float32)).to(DEV)
    y = torch.empty(s.T * s.k, s.d, dtype=torch.bfloat16, device=DEV)
    sh = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV) if s.F else None
    ws = torch.empty(M.moe_expert_ffn_workspace_size(ms), dtype=torch.uint8, device=DEV)
    M.moe_expert_ffn(ms, x, offsets, perm, layer.weights, y, sh, ws)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    M.moe_combine(ms, y, sh, inv, gate, None, out)
    torch.cuda.synchronize()
    assert_close_bf16(bf16_to_np(y), ref["Y"], "y_perm")
    if s.F:
        assert_close_bf16(bf16_to_np(sh), ref["shared"], "shared_out")
    assert_close_bf16(bf16_to_np(out), ref["out"], "combine")


LAYER_CASES = [("tiny", {}), ("nano", {}), ("skew", {}), ("nano", {"T": 1000}),
               ("nano", {"T": 77, "F": 0}), ("nano", {"T": 1, "k": 1, "renorm": False}),
               ("tiny", {"T": 200, "E": 16, "k": 4, "f": 64, "F": 96}),
               ("nano", {"T": 4096, "E": 256, "k": 8, "f": 128, "F": 0}),
               ("nano", {"T": 3000}),                                # second stream, ragged tiles
               ("nano", {"T": 2500, "d": 512, "f": 256, "F": 1024})]  # second stream, other widths


@pytest.mark.parametrize("name,kw", LAYER_CASES)
@pytest.mark.parametrize("with_residual", [False, True])
def test_layer_fwd_matches_oracle(name, kw, with_residual):
    if with_residual and name not in ("tiny", "nano"):
        pytest.skip("residual covered on the base shapes")
    s = _shape(name, **kw)
    host = make_layer(s, name)
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    res_np = None
    res = None
    if with_residual:
        rng = np.random.default_rng(5)
        from synth import bf16_bits_from_f32
        res_bits = bf16_bits_from_f32(rng.standard_normal((s.T, s.d)).astype(np.float32))
        res = to_device_bf16(res_bits, DEV)
        res_np = bf64(res_bits)
    scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    load = torch.empty(s.E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(s.E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(s.T * s.k, dtype=torch.int32, device=DEV)
    inv = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    dbg = M.make_debug(scores=scores, idx=idx, load=load, offsets=offsets, perm_tok=perm, inv_pos=inv)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=True, residual=res, debug=dbg)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref = _oracle_layer(s, host, sc, residual=res_np)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(load.cpu().numpy(), ref["load"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(perm.cpu().numpy(), ref["perm_tok"])
    assert np.array_equal(inv.cpu().numpy(), ref["inv_pos"])
    assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), ref["bias"].view(np.uint32))
    assert_close_bf16(bf16_to_np(out), ref["out"], "layer out")


def test_skewed_bias_trajectory_bitexact():
    """50 forward + bias-update steps on the Zipf-skewed router: the GPU's bias after
    every step equals the oracle's, the fused balance statistics equal the oracle's
    (bit for bit), and the max/mean load falls from its start."""
    s = CONFIGS["skew"]
    host = make_layer(s, "skew")
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
    load = torch.empty(s.E, dtype=torch.int32, device=DEV)
    bal = torch.zeros(M.BALANCE_BYTES, dtype=torch.uint8, device=DEV)
    dbg = M.make_debug(scores=scores, load=load, balance=bal)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    bias = host["bias"].copy()
    ratios = []
    for step in range(s.steps):
        layer.forward(x, out, update_bias=True, debug=dbg)
        torch.cuda.synchronize()
        sc = scores.cpu().numpy()
        idx = O.topk_select(sc, bias, s.k)
        ld = O.expert_load(idx, s.E)
        assert np.array_equal(load.cpu().numpy(), ld), step
        # The fused balance output (max/mean, min/mean, dead fraction) of every step.
        got, want = M.balance_from_bytes(bal), O.balance_stats(ld, s.E)
        for key in want:
            assert np.float64(got[key]) == np.float64(want[key]), (step, key)
        bias = O.bias_update(bias, ld, s.T * s.k, s.gamma)
        assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), bias.view(np.uint32)), step
        ratios.append(ld.max() / ld.mean())
    assert ratios[0] > 10.0          # the workload is skewed as specified
    assert ratios[-1] < ratios[0]    # and the balancing pulls it back


def _dequant_oracle(bits3d):
    """Oracle int4 round trip of bf16 weights [G][rows][K] (its own quantiser)."""
    G, R, K = bits3d.shape
    packed, scale, _ = O.quantize_int4_g32(bf64(bits3d.reshape(-1, K)).astype(np.float32))
    return O.dequantize_int4_g32(packed, scale).reshape(G, R, K)


@pytest.mark.parametrize("T", [1, 8, 64, 200])
def test_int4_top1_serving_layer_matches_oracle(T):
    """Top-1 serving with int4 routed experts (dequantised inside the kernels) and the
    bf16 shared expert: routing bit-exact, gate = raw score, output within tolerance
    of the oracle run on the oracle's own dequantised weights; no bias update."""
    s = CONFIGS["decode"].replace(T=T)
    host = make_layer(s, "decode")
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(s.T, s.k, dtype=torch.float32, device=DEV)
    dbg = M.make_debug(scores=scores, idx=idx, gate=gate)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=False, debug=dbg)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ref = O.layer_forward(tokens64(host["x"]), host["w_router"], host["bias"],
                          _dequant_oracle(host["w_gate"]), _dequant_oracle(host["w_up"]),
                          _dequant_oracle(host["w_down"]), bf64(host["s_gate"]), bf64(host["s_up"]),
                          bf64(host["s_down"]), k=1, renorm=False, scores_f32=sc)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.abs(gate.cpu().numpy() - ref["gate"]).max() <= 1e-6
    assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), host["bias"].view(np.uint32))
    assert_close_bf16(bf16_to_np(out), ref["out"], "int4 serving out")


@pytest.mark.gpu
@pytest.mark.parametrize("T", [3, 64])
def test_int4_serving_without_permutation_bias_update_and_residual(T):
    """The serving path that skips the permutation (at most 64 token-expert pairs, no
    permutation outputs requested): loads bit-exact, the bias update applied from
    them bit for bit, and the output with a residual within tolerance."""
    s = CONFIGS["decode"].replace(T=T)
    host = make_layer(s, "decode")
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    res_bits = make_tokens(s, "decode", seed=7)
    res = to_device_tokens(res_bits, DEV)
    scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
    load = torch.empty(s.E, dtype=torch.int32, device=DEV)
    dbg = M.make_debug(scores=scores, idx=idx, load=load)
    out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
    layer.forward(x, out, update_bias=True, residual=res, debug=dbg)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    res_np = bf64(res_bits)
    ref = O.layer_forward(tokens64(host["x"]), host["w_router"], host["bias"],
                          _dequant_oracle(host["w_gate"]), _dequant_oracle(host["w_up"]),
                          _dequant_oracle(host["w_down"]), bf64(host["s_gate"]), bf64(host["s_up"]),
                          bf64(host["s_down"]), k=1, renorm=False, gamma=s.gamma, scores_f32=sc,
                          residual=res_np)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(load.cpu().numpy(), O.expert_load(ref["idx"], s.E))
    want_bias = O.bias_update(host["bias"], O.expert_load(ref["idx"], s.E), s.T * s.k, s.gamma)
    assert np.array_equal(layer.bias.cpu().numpy().view(np.uint32), want_bias.view(np.uint32))
    assert_close_bf16(bf16_to_np(out), ref["out"], "int4 serving out with residual")


def test_stack_23_layers_with_residual():
    """Config 4: 23 Nano layers, x_{l+1} = x_l + MoE_l(x_l) in bf16, each layer with its
    own weights and bias update.  Every layer's routing, loads and updated bias are
    checked bit for bit; the outputs of 64 sampled tokens are checked at layers 0, 11
    and 22 against the oracle fed that layer's GPU input (tokens are independent
    within a layer, so a sample is exact to check)."""
    s = CONFIGS["stack"]
    x = to_device_tokens(make_layer(s.replace(f=32, F=32), "stack")["x"], DEV)
    acts = [x]
    layers, hosts, dbgs = [], [], []
    for l in range(s.layers):
        host = make_layer(s, "stack", layer=l, with_tokens=False)
        layer = LayerOnDevice(s, host, DEV)
        scores = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
        load = torch.empty(s.E, dtype=torch.int32, device=DEV)
        out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
        layer.forward(acts[-1], out, update_bias=True, residual=acts[-1],
                      debug=M.make_debug(scores=scores, load=load))
        acts.append(out)
        dbgs.append((scores, load))
        # Keep host weights only for the layers whose outputs are checked.
        hosts.append(host if l in (0, 11, s.layers - 1) else {"bias": host["bias"]})
        layers.append(layer)
    torch.cuda.synchronize()
    rng = np.random.default_rng(23)
    sample = np.sort(rng.choice(s.T, 64, replace=False))
    for l in range(s.layers):
        sc = dbgs[l][0].cpu().numpy()
        idx = O.topk_select(sc, hosts[l]["bias"], s.k)
        ld = O.expert_load(idx, s.E)
        assert np.array_equal(dbgs[l][1].cpu().numpy(), ld), l
        want_b = O.bias_update(hosts[l]["bias"], ld, s.T * s.k, s.gamma)
        assert np.array_equal(layers[l].bias.cpu().numpy().view(np.uint32), want_b.view(np.uint32)), l
        if "w_gate" not in hosts[l]:
            continue
        H = hosts[l]
        xin = bf16_to_np(acts[l])[sample]
        gidx = idx[sample]
        gate = O.gate_weights(sc[sample].astype(np.float64), gidx, True)
        want = xin.copy()
        for i in range(len(sample)):
            row = xin[i:i + 1]
            y = O.swiglu_ffn(row, bf64(H["s_gate"]), bf64(H["s_up"]), bf64(H["s_down"]))[0]
            for j in range(s.k):
                e = gidx[i, j]
                y = y + gate[i, j] * O.swiglu_ffn(row, bf64(H["w_gate"][e]), bf64(H["w_up"][e]),
                                                  bf64(H["w_down"][e]))[0]
            want[i] += y
        assert_close_bf16(bf16_to_np(acts[l + 1])[sample], want, f"stack layer {l}")


def test_expert_ffn_outputs_only_16_byte_aligned():
    """The ABI promises 16-byte alignment only: outputs offset by 16 bytes from a
    32-byte boundary take the 128-bit store path and must give the same result."""
    s = CONFIGS["nano"].replace(T=512)
    host = make_layer(s, "nano")
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    sc = O.router_scores(tokens64(host["x"]), host["w_router"]).astype(np.float32)
    ref = _oracle_layer(s, host, sc)
    offsets = torch.from_numpy(ref["offsets"].astype(np.int32)).to(DEV)
    perm = torch.from_numpy(ref["perm_tok"].astype(np.int32)).to(DEV)
    ybuf = torch.empty(s.T * s.k * s.d + 8, dtype=torch.bfloat16, device=DEV)
    sbuf = torch.empty(s.T * s.d + 8, dtype=torch.bfloat16, device=DEV)
    y = ybuf[8:].view(s.T * s.k, s.d)     # 16 bytes past the allocation's start
    sh = sbuf[8:].view(s.T, s.d)
    assert y.data_ptr() % 32 == 16 and sh.data_ptr() % 32 == 16
    ws = torch.empty(M.moe_expert_ffn_workspace_size(layer.shape), dtype=torch.uint8, device=DEV)
    M.moe_expert_ffn(layer.shape, x, offsets, perm, layer.weights, y, sh, ws)
    torch.cuda.synchronize()
    assert_close_bf16(bf16_to_np(y), ref["Y"], "y_perm (16-byte aligned)")
    assert_close_bf16(bf16_to_np(sh), ref["shared"], "shared_out (16-byte aligned)")
    obuf = torch.empty(s.T * s.d + 8, dtype=torch.bfloat16, device=DEV)
    out = obuf[8:].view(s.T, s.d)
    inv = torch.from_numpy(ref["inv_pos"].astype(np.int32)).to(DEV)
    gate = torch.from_numpy(ref["gate"].astype(np.float32)).to(DEV)
    M.moe_combine(layer.shape, y, sh, inv, gate, None, out)
    torch.cuda.synchronize()
    assert_close_bf16(bf16_to_np(out), ref["out"], "combine (16-byte aligned)")

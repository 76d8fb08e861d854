"""Oracle for the fine-grained MoE layer forward and its aux-loss-free bias update.

TEST INFRASTRUCTURE.  This module is a plain, slow CPU restatement of what the GPU
path computes.  Only the tests, the package's smoke check and the bench's CPU
baseline may import it; the library never calls it and never falls back to it.
It shares no code with the CUDA path and imports nothing from it.

Source of the method.  "Una carrera de relevos con GPUs alquiladas entrenó el MoE de
2.7B de NanoColibri por $200" (the same article in Chinese and Arabic), referred to
below as *the relay article*:

* opening section, architecture paragraph: 64 routed experts of width 512 with
  top-2 routing, an always-resident shared expert of width 2048, a sigmoid-plus-bias
  router, and DeepSeek-V3 balancing that moves each layer's expert bias by gamma
  times the sign of (target - load);
* section "Entrenamiento por relevos", fourth paragraph (the top-2 lesson): at
  top_k = 1 the routed weight collapses to a constant, so gates are renormalised
  over the k winners; serving runs one expert per token;
* opening section, second paragraph: experts ship in an int4 container.

Readings where the article is silent (each is also listed in the design notes):

* activation: SwiGLU, three matrices per expert (gate, up, down);
* target load: the mean T*k/E, compared through the integer sign of T*k - E*load;
  sign(0) = 0;
* the bias only selects experts; gates use the unbiased sigmoid scores;
* ties in the selection key go to the lower expert index; the k winners are listed
  by descending key, lower index first;
* the shared expert is added with weight 1;
* H (the SwiGLU hidden activation) is stored in bf16 between the two GEMMs;
* int4: symmetric, groups of 32 along the input dimension, fp16 scale
  max|w|/7, codes rint(w/scale) clamped to [-7, 7], low nibble = even index.

Precision: fp64 everywhere except the selection key fl32(s + b) and the bias update
fl32(b + gamma*sign), whose fp32 rounding is part of the definition, and the int4
quantiser, whose code decisions are taken in fp32 as the GPU takes them.

Parity pins: every function here is checked in tests/test_oracle_pins.py against
something other than itself: brute force (top-k over all subsets), closed forms
(structured SwiGLU weights, sigmoid through a one-hot router, exact rational bias
rounding), library routines (PyTorch SwiGLU, sigmoid and autograd, stable sort,
bincount), hand-worked fixtures (tests/golden/) and, for the whole layer, an
independent per-token dense mixture with no permutation.  The pages print no worked
example of the layer's values, so no pin is a printed number.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Number formats used by the definition (own implementations).
# ---------------------------------------------------------------------------


def bf16_value_from_bits(bits: np.ndarray) -> np.ndarray:
    """Value (fp64) of bf16 bit patterns: the 16 bits are the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round real values to the nearest bf16 value (8 significant bits), ties to even.

    Written from the format's definition: v = m * 2^e with 0.5 <= |m| < 1, keep 8
    significant bits of m.  Values in this workload are far from bf16's range limits.
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def fp16_value_from_bits(bits: np.ndarray) -> np.ndarray:
    """Value (fp64) of IEEE binary16 bit patterns."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------------------------------
# Router: logits, sigmoid scores, biased top-k, gates, loads.
# ---------------------------------------------------------------------------


def router_scores(x: np.ndarray, w_router: np.ndarray, logit_offset=None) -> np.ndarray:
    """Sigmoid router scores s[t][e] = 1 / (1 + exp(-(x_t . w_e + o_e))) in fp64.

    Relay article, architecture paragraph ("sigmoid-plus-bias router").  x is the
    exact token values (fp32 or bf16-valued), w_router fp32 [E][d]; logit_offset is
    an optional per-expert additive term used by the skewed workload.
    """
    z = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T
    if logit_offset is not None:
        z = z + np.asarray(logit_offset, dtype=np.float64)[None, :]
    return 1.0 / (1.0 + np.exp(-z))


def selection_keys(scores_f32: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Selection key fl32(s + b) (one fp32 addition); the bias steers selection only."""
    s = np.asarray(scores_f32, dtype=np.float32)
    b = np.asarray(bias, dtype=np.float32)
    return (s + b[None, :]).astype(np.float32)


def topk_select(scores_f32: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """idx[t][j]: the k experts of largest key per token, by (key desc, index asc).

    Relay article, architecture paragraph (top-k routing on sigmoid plus bias); the
    tie rule (lower index wins) is this build's reading.
    """
    keys = selection_keys(scores_f32, bias)
    T, E = keys.shape
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        row = keys[t]
        order = sorted(range(E), key=lambda e: (-float(row[e]), e))
        idx[t, :] = order[:k]
    return idx


def gate_weights(scores: np.ndarray, idx: np.ndarray, renorm: bool) -> np.ndarray:
    """Gate g[t][j] from the unbiased score of each winner.

    With renorm, g_j = s_j / sum over the k winners (relay article, top-2 lesson:
    at top_k = 1 this is the constant 1); without it g_j = s_j.
    """
    s = np.asarray(scores, dtype=np.float64)
    T, k = idx.shape
    g = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        picked = [s[t, idx[t, j]] for j in range(k)]
        denom = sum(picked) if renorm else 1.0
        for j in range(k):
            g[t, j] = picked[j] / denom
    return g


def expert_load(idx: np.ndarray, E: int) -> np.ndarray:
    """load[e] = number of (token, slot) pairs routed to expert e."""
    load = np.zeros(E, dtype=np.int64)
    for e in np.asarray(idx).ravel():
        load[int(e)] += 1
    return load


# ---------------------------------------------------------------------------
# Token permutation (stable counting sort by expert).
# ---------------------------------------------------------------------------


def stable_permutation(idx: np.ndarray, E: int):
    """Group the (t, j) pairs by expert, tokens ascending inside each expert.

    Returns offsets[E+1] (start row of each expert's block), perm_tok[T*k] (source
    token of each row) and inv_pos[T][k] (row that holds pair (t, j)).
    """
    T, k = idx.shape
    buckets = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            buckets[int(idx[t, j])].append((t, j))
    offsets = np.zeros(E + 1, dtype=np.int64)
    perm_tok = np.empty(T * k, dtype=np.int64)
    inv_pos = np.empty((T, k), dtype=np.int64)
    row = 0
    for e in range(E):
        offsets[e] = row
        for (t, j) in buckets[e]:
            perm_tok[row] = t
            inv_pos[t, j] = row
            row += 1
    offsets[E] = row
    return offsets, perm_tok, inv_pos


# ---------------------------------------------------------------------------
# Expert FFNs.
# ---------------------------------------------------------------------------


def silu(a: np.ndarray) -> np.ndarray:
    """silu(a) = a / (1 + exp(-a)).  For a below about -709, exp(-a) overflows to inf
    and the quotient is the correct limit -0.0 (the overflow warning is silenced)."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu_ffn(xb: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray,
               round_hidden: bool = True) -> np.ndarray:
    """y = (silu(x Wg^T) * (x Wu^T)) Wd^T in fp64, H rounded to bf16 when stored so.

    xb [n][d], w_gate / w_up [f][d], w_down [d][f], all as real values.
    """
    g = xb @ w_gate.T
    u = xb @ w_up.T
    h = silu(g) * u
    if round_hidden:
        h = round_to_bf16(h)
    return h @ w_down.T


def routed_experts(xb: np.ndarray, offsets, perm_tok, w_gate, w_up, w_down,
                   round_hidden: bool = True) -> np.ndarray:
    """Y[p] for every permuted row p: expert e's FFN applied to token perm_tok[p]."""
    E = len(offsets) - 1
    d = xb.shape[1]
    Y = np.zeros((len(perm_tok), d), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        rows = xb[perm_tok[lo:hi]]
        Y[lo:hi] = swiglu_ffn(rows, w_gate[e], w_up[e], w_down[e], round_hidden)
    return Y


def combine(Y: np.ndarray, shared: np.ndarray, inv_pos: np.ndarray, gate: np.ndarray,
            residual=None) -> np.ndarray:
    """out[t] = residual[t] + shared[t] + sum_j g[t][j] * Y[inv_pos[t][j]] (fp64)."""
    T, k = inv_pos.shape
    out = np.array(shared, dtype=np.float64, copy=True)
    if residual is not None:
        out += np.asarray(residual, dtype=np.float64)
    for j in range(k):
        out += gate[:, j:j + 1] * Y[inv_pos[:, j]]
    return out


# ---------------------------------------------------------------------------
# Aux-loss-free bias update.
# ---------------------------------------------------------------------------


def bias_update(bias: np.ndarray, load: np.ndarray, tokens_times_k: int, gamma: float) -> np.ndarray:
    """b_e <- fl32(b_e + gamma * sign(T*k/E - load_e)), with sign(0) = 0.

    Relay article, architecture paragraph (DeepSeek-V3 recipe: nudge each expert's bias
    by gamma times the sign of target minus load).  The target is the mean load T*k/E;
    the sign is taken on the integer T*k - E*load_e so no rounding enters it.
    tokens_times_k is the global T*k when loads were summed over replicas.
    """
    b = np.asarray(bias, dtype=np.float32)
    E = b.shape[0]
    g32 = np.float32(gamma)
    out = np.empty(E, dtype=np.float32)
    for e in range(E):
        diff = int(tokens_times_k) - E * int(load[e])
        sgn = (diff > 0) - (diff < 0)
        step = np.float32(sgn) * g32          # exactly +gamma, -gamma or 0
        out[e] = np.float32(b[e] + step)      # one fp32 addition, nearest-even
    return out


def nearest_f32(num: int, den: int) -> np.float32:
    """The fp32 value nearest to the exact rational num / den (ties to even), den > 0.

    Exact arithmetic: the quotient is scaled by a power of two so that its integer part
    has 25 to 26 bits, the 24-bit significand is chosen by integer rounding (ties to the
    even significand), and the power of two is put back.  Plain integers only.
    """
    if num == 0:
        return np.float32(0.0)
    if num < 0:
        return -nearest_f32(-num, den)
    # num / den = q * 2^e with 2^23 <= q < 2^24 after rounding.
    e = num.bit_length() - den.bit_length() - 24
    while True:
        n, d = (num, den << e) if e >= 0 else (num << -e, den)
        if n >= d << 24:
            e += 1
        elif n < d << 23:
            e -= 1
        else:
            break
    q, r = divmod(n, d)
    if 2 * r > d or (2 * r == d and q % 2 == 1):
        q += 1
    return np.float32(np.ldexp(np.float64(q), e))  # q <= 2^24: exact in fp64 and fp32


def balance_stats(load, E: int) -> dict:
    """Expert-balance statistics of one routing result (per-expert loads).

    Relay article, section "Entrenamiento por relevos": the relay's dashboard tracks
    expert balance, and the top-2 paragraph says the fraction of dead experts stayed
    low.  The pages define neither; this build's reading: the mean load is pairs / E
    with pairs = sum of the loads; max/mean = max_load * E / pairs, min/mean likewise;
    an expert is dead when its load is 0, dead fraction = dead / E.  Each ratio is the
    fp32 value nearest to the exact rational (0 when pairs is 0).
    """
    load = [int(v) for v in np.asarray(load).ravel()]
    assert len(load) == E
    pairs = sum(load)
    mx, mn = max(load), min(load)
    dead = sum(1 for v in load if v == 0)
    return dict(pairs=pairs, max_load=mx, min_load=mn, dead_experts=dead,
                max_over_mean=nearest_f32(mx * E, pairs) if pairs else np.float32(0.0),
                min_over_mean=nearest_f32(mn * E, pairs) if pairs else np.float32(0.0),
                dead_fraction=nearest_f32(dead, E))


# ---------------------------------------------------------------------------
# int4 container (symmetric, group 32 along the input dimension, fp16 scales).
# ---------------------------------------------------------------------------


def quantize_int4_g32(w: np.ndarray):
    """Quantise rows of w [rows][K] (fp32 values) to int4 codes with fp16 group scales.

    Relay article, opening section (int4 container).  Per group of 32 consecutive input
    elements: scale = fp16(fl32(max|w| / 7)); q = clamp(rint(fl32(w / scale)), -7, 7),
    ties to even, q = 0 where scale = 0.  Returns (packed uint8 [rows][K/2] with the even
    index in the low nibble, scale bits uint16 [rows][K/32], codes int8 [rows][K]).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, K = w.shape
    groups = w.reshape(rows, K // 32, 32)
    amax = np.abs(groups).max(axis=2)
    scale32 = (amax / np.float32(7.0)).astype(np.float32)
    scale16 = scale32.astype(np.float16)
    s = scale16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s > 0, groups / np.where(s > 0, s, np.float32(1)), np.float32(0))
    q = np.clip(np.rint(ratio.astype(np.float32)), -7, 7).astype(np.int8).reshape(rows, K)
    nib = (q.astype(np.int16) & 0xF).astype(np.uint8)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale16.view(np.uint16), q


def dequantize_int4_g32(packed: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """w = q * scale in fp64 from packed nibbles (two's complement) and fp16 scales."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    lo = (packed & 0xF).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    q = np.empty((rows, 2 * half), dtype=np.float64)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    s = fp16_value_from_bits(scale_bits)
    return q * np.repeat(s, 32, axis=1)


# ---------------------------------------------------------------------------
# Whole layer.
# ---------------------------------------------------------------------------


def layer_forward(x, w_router, bias, w_gate, w_up, w_down, s_gate, s_up, s_down, k: int,
                  renorm: bool = True, logit_offset=None, gamma: float = 1e-3,
                  scores_f32=None, residual=None, x_is_bf16: bool = True,
                  idx=None, exact_gates: bool = False, round_hidden: bool = True):
    """One MoE layer forward plus the bias update, all in the order the method states.

    Token values x and all weights are given as real values (fp64 arrays).  If
    scores_f32 is given (the GPU's fp32 sigmoid scores), selection uses it, as the
    parity contract prescribes; else the oracle's own scores rounded to fp32.
    The expert FFNs read x rounded to bf16 when x is fp32 (x_is_bf16 False).
    """
    x = np.asarray(x, dtype=np.float64)
    E = w_router.shape[0]
    T = x.shape[0]
    scores = router_scores(x, w_router, logit_offset)
    sel_scores = scores.astype(np.float32) if scores_f32 is None else np.asarray(scores_f32, np.float32)
    if idx is None:
        idx = topk_select(sel_scores, bias, k)
    # exact_gates: gates from the fp64 scores (a smooth function of x and W_r, for
    # derivative checks with the selection held fixed through idx).
    gate = gate_weights(scores if exact_gates else sel_scores.astype(np.float64), idx, renorm)
    load = expert_load(idx, E)
    offsets, perm_tok, inv_pos = stable_permutation(idx, E)
    xb = x if x_is_bf16 else round_to_bf16(x)
    Y = routed_experts(xb, offsets, perm_tok, w_gate, w_up, w_down, round_hidden)
    if s_gate is not None and s_gate.shape[0] > 0:
        shared = swiglu_ffn(xb, s_gate, s_up, s_down, round_hidden)
    else:
        shared = np.zeros_like(xb)
    out = combine(Y, shared, inv_pos, gate, residual)
    new_bias = bias_update(bias, load, T * k, gamma)
    return dict(scores=scores, idx=idx, gate=gate, load=load, offsets=offsets,
                perm_tok=perm_tok, inv_pos=inv_pos, Y=Y, shared=shared, out=out,
                bias=new_bias)


def shared_expert_backward(xb, s_gate, s_up, s_down, dout, round_hidden: bool = True):
    """Gradients through the shared expert, out_t += Sd (silu(Sg x_t) * (Su x_t)), gate 1.

    Relay article, architecture paragraph (the always-resident shared expert); the
    chain rule as for one routed pair in layer_backward.  Returns (dx, dS_gate, dS_up,
    dS_down) for all tokens at once, fp64.
    """
    xb = np.asarray(xb, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    a = xb @ s_gate.T
    b = xb @ s_up.T
    sa = silu(a)
    h = sa * b
    if round_hidden:
        h = round_to_bf16(h)
    dh = dout @ s_down
    sig = 1.0 / (1.0 + np.exp(-a))
    da = dh * b * (sig * (1.0 + a * (1.0 - sig)))
    db = dh * sa
    dx = da @ s_gate + db @ s_up
    return dx, da.T @ xb, db.T @ xb, dout.T @ h


def layer_backward(x, w_router, bias, w_gate, w_up, w_down, s_gate, s_up, s_down, dout, k: int,
                   renorm: bool = True, logit_offset=None, scores_f32=None,
                   residual: bool = False, x_is_bf16: bool = True, idx=None,
                   exact_gates: bool = False, round_hidden: bool = True):
    """Gradients of the layer output (as layer_forward computes it) given dout = dL/dout.

    The relay article states the forward (architecture paragraph, top-2 paragraph) and
    nothing about its derivatives; these are the chain rule through that forward:

    * the selection (biased top-k) is piecewise constant: no gradient flows through
      the choice of experts, and the bias gets none (it moves by the balancing rule);
    * pair (t, j) with expert e = idx[t][j] and gate g: y = Wd_e h, h = silu(a) * b,
      a = Wg_e x_t, b = Wu_e x_t, out_t += g y;  so dy = g dout_t, dg = <dout_t, y>,
      dh = Wd_e^T dy, da = dh * b * silu'(a), db = dh * silu(a),
      dx_t += Wg_e^T da + Wu_e^T db, dWd_e += dy h^T, dWg_e += da x_t^T, dWu_e += db x_t^T;
    * the shared expert likewise with g = 1;
    * gates: renormalised, g_j = s_j / S with S = sum of the winners' scores, so
      ds_j = (dg_j - sum_i dg_i g_i) / S; raw, ds_j = dg_j; then dz_j = ds_j s_j (1 - s_j)
      for the logit z = x W_r^T (+ offset): dx_t += sum_j dz_j W_r[e_j],
      dW_r[e_j] += dz_j x_t;
    * with a residual (out = x + MoE(x)), dx += dout.

    h is taken as stored in bf16 when round_hidden (as in the forward); its rounding is
    passed through unchanged.  Selection uses scores_f32 (the GPU's scores) when given,
    as in layer_forward; idx and exact_gates as there.  All arithmetic in fp64.
    """
    x = np.asarray(x, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    E, d = w_router.shape
    T = x.shape[0]
    scores = router_scores(x, w_router, logit_offset)
    sel_scores = scores.astype(np.float32) if scores_f32 is None else np.asarray(scores_f32, np.float32)
    if idx is None:
        idx = topk_select(sel_scores, bias, k)
    s_used = scores if exact_gates else sel_scores.astype(np.float64)
    gate = gate_weights(s_used, idx, renorm)
    xb = x if x_is_bf16 else round_to_bf16(x)
    dx = np.zeros_like(x)
    dwg = np.zeros_like(w_gate, dtype=np.float64)
    dwu = np.zeros_like(w_up, dtype=np.float64)
    dwd = np.zeros_like(w_down, dtype=np.float64)
    dgate = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            xt = xb[t]
            a = w_gate[e] @ xt
            b = w_up[e] @ xt
            sa = silu(a)
            h = sa * b
            if round_hidden:
                h = round_to_bf16(h)
            y = w_down[e] @ h
            dgate[t, j] = dout[t] @ y
            dy = gate[t, j] * dout[t]
            dh = w_down[e].T @ dy
            sig = 1.0 / (1.0 + np.exp(-a))
            da = dh * b * (sig * (1.0 + a * (1.0 - sig)))  # silu'(a) = s + a s (1 - s)
            db = dh * sa
            dx[t] += w_gate[e].T @ da + w_up[e].T @ db
            dwd[e] += np.outer(dy, h)
            dwg[e] += np.outer(da, xt)
            dwu[e] += np.outer(db, xt)
    if s_gate is not None and s_gate.shape[0] > 0:
        dxs, dsg, dsu, dsd = shared_expert_backward(xb, s_gate, s_up, s_down, dout, round_hidden)
        dx += dxs
    else:
        dsg = dsu = dsd = None
    # Router: through the gates' scores.
    dz = np.zeros((T, E), dtype=np.float64)
    for t in range(T):
        sel = [int(e) for e in idx[t]]
        st = np.array([s_used[t, e] for e in sel])
        if renorm:
            S = st.sum()
            dsel = (dgate[t] - (dgate[t] * gate[t]).sum()) / S
        else:
            dsel = dgate[t].copy()
        for j, e in enumerate(sel):
            dz[t, e] += dsel[j] * st[j] * (1.0 - st[j])
    dx += dz @ w_router
    dwr = dz.T @ x
    if residual:
        dx += dout
    return dict(idx=idx, gate=gate, dgate=dgate, dz=dz, dx=dx, dw_gate=dwg, dw_up=dwu,
                dw_down=dwd, ds_gate=dsg, ds_up=dsu, ds_down=dsd, dw_router=dwr)

"""Expert parallelism on one GPU: N ranks emulated in one process (ep_forward_emulated).

Each rank routes its consecutive token shard, sends the rows of other ranks' experts
to them, runs its own experts over what it receives and combines what comes back.  The
routing, the permutation, each expert's rows and their order are then those of the
single-GPU layer over the whole batch, and every row's arithmetic is the same, so the
outputs and the bias after the update must equal moe_layer_fwd's bit for bit.  The
outputs are also checked against the oracle directly (fed the GPU's scores) and the
bias trajectory against the oracle's, for every world size, with equal and unequal
token shards.  The regrouping kernel is checked against its definition
(tests/ep_util.py) on its own.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.ep import EPRank, ep_forward_emulated
from aux_loss_free_gb300.layer import LayerOnDevice, to_device_tokens
from ep_util import regroup_reference
from gpu_util import assert_close_bf16, bf16_to_np, bf64
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


@pytest.mark.parametrize("world,counts_seed", [(1, 0), (2, 1), (4, 2), (8, 3)])
def test_regroup_matches_definition(world, counts_seed):
    el = 64 // world
    rng = np.random.default_rng(counts_seed)
    counts = rng.integers(0, 40, size=(world, el)).astype(np.int32)
    counts[rng.random(counts.shape) < 0.2] = 0  # empty runs
    perm_ref, inv_ref, off_ref = regroup_reference(counts)
    rows = int(counts.sum())
    c = torch.from_numpy(counts).to(DEV)
    perm = torch.full((rows,), -1, dtype=torch.int32, device=DEV)
    inv = torch.full((rows,), -1, dtype=torch.int32, device=DEV)
    off = torch.full((el + 1,), -1, dtype=torch.int32, device=DEV)
    M.moe_ep_regroup(world, el, c, perm, inv, off)
    torch.cuda.synchronize()
    assert np.array_equal(perm.cpu().numpy(), perm_ref)
    assert np.array_equal(inv.cpu().numpy(), inv_ref)
    assert np.array_equal(off.cpu().numpy(), off_ref)


def test_gather_rows():
    rng = np.random.default_rng(7)
    src = torch.from_numpy(rng.integers(0, 1 << 16, size=(300, 256), dtype=np.int64).astype(np.int16)).to(DEV)
    index = torch.from_numpy(rng.integers(0, 300, size=517).astype(np.int32)).to(DEV)
    dst = torch.empty(517, 256, dtype=torch.int16, device=DEV)
    M.moe_gather_rows(517, 256, src, index, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[index.long()])


EP_CASES = [
    # world, layer shape (T is the whole batch, split into consecutive shards by
    # np.array_split: equal shards when world divides T)
    (2, dict(T=1024, d=256, E=16, f=128, F=256, k=2)),
    (4, dict(T=2048, d=512, E=32, f=256, F=512, k=2)),
    (4, dict(T=8192)),                                   # the Nano layer, 16 experts per rank
    (8, dict(T=2048, d=256, E=64, f=128, F=256, k=2, skew_zipf_s=1.2)),  # skewed: some ranks get little
    (2, dict(T=1001, d=256, E=16, f=128, F=256, k=2)),   # unequal shards: 501 and 500 tokens
    (8, dict(T=8192)),                                   # the Nano layer, 8 experts per rank
]


def _oracle_sample(s, host, x_bits, scores, bias, rows):
    """The oracle layer output of the token rows `rows` (routing is per token, so a
    subset with its own scores is exact to check), fed the GPU's fp32 scores."""
    return O.layer_forward(bf64(x_bits[rows]), host["w_router"], bias, bf64(host["w_gate"]), bf64(host["w_up"]),
                           bf64(host["w_down"]), bf64(host["s_gate"]), bf64(host["s_up"]), bf64(host["s_down"]),
                           k=s.k, renorm=s.renorm, logit_offset=host["logit_offset"], gamma=s.gamma,
                           scores_f32=scores[rows])["out"]


@pytest.mark.parametrize("world,kw", EP_CASES, ids=[f"w{w}-{kw.get('T')}" for w, kw in EP_CASES])
def test_emulated_expert_parallel_equals_single_gpu_and_oracle(world, kw):
    case = "skew" if kw.get("skew_zipf_s") else "nano"
    s = CONFIGS["nano"].replace(**kw)
    host = make_layer(s, case)
    layer = LayerOnDevice(s, host, DEV)
    x = to_device_tokens(host["x"], DEV)
    shards = np.array_split(np.arange(s.T), world)
    bounds = [(int(sh[0]), int(sh[-1]) + 1) for sh in shards]
    ranks = [EPRank(s, host, hi - lo, r, world, DEV) for r, (lo, hi) in enumerate(bounds)]
    bias = host["bias"].copy()
    for step in range(3):  # the bias moves each step, and the routing with it
        idx_ref = torch.empty(s.T, s.k, dtype=torch.int32, device=DEV)
        sc_ref = torch.empty(s.T, s.E, dtype=torch.float32, device=DEV)
        out_ref = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=DEV)
        layer.forward(x, out_ref, update_bias=True, debug=M.make_debug(idx=idx_ref, scores=sc_ref))
        outs = [torch.empty(hi - lo, s.d, dtype=torch.bfloat16, device=DEV) for lo, hi in bounds]
        ep_forward_emulated(ranks, [x[lo:hi] for lo, hi in bounds], outs)
        torch.cuda.synchronize()
        got = torch.cat(outs)
        assert torch.equal(got.view(torch.int16), out_ref.view(torch.int16)), f"step {step}"
        for r in ranks:
            assert torch.equal(r.bias.view(torch.int32), layer.bias.view(torch.int32)), f"step {step}"
        sc = sc_ref.cpu().numpy()
        ld = O.expert_load(O.topk_select(sc, bias, s.k), s.E)
        bias = O.bias_update(bias, ld, s.T * s.k, s.gamma)
        assert np.array_equal(ranks[0].bias.cpu().numpy().view(np.uint32), bias.view(np.uint32)), f"step {step}"
        if step == 0:
            # The expert-parallel output itself against the oracle: every token of the
            # small cases, a sample of 256 tokens of the Nano-sized ones.
            rows = np.arange(s.T) if s.T * s.d <= 2048 * 512 else \
                np.sort(np.random.default_rng(world).choice(s.T, 256, replace=False))
            ref = _oracle_sample(s, host, host["x"], sc, host["bias"], rows)
            assert_close_bf16(bf16_to_np(got)[rows], ref, f"expert-parallel out, {world} ranks")

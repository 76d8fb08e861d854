"""Two CPU ranks (gloo) run the data-parallel balancing step on their token shards.

Each rank routes its shard with the oracle, the loads are summed with the package's
allreduce_load, and each rank applies the bias update with the global T*k that the
package's global_tokens_times_k takes from the summed loads.  The batch (97 tokens)
does not split evenly (shards of 49 and 48), so world * (local T*k) would be wrong for
both ranks.  Every rank must end with the bias that the single-process full batch
gives, bit for bit, and each shard's routing must equal the full batch's routing of
those tokens.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from aux_loss_free_gb300.dp import allreduce_load, global_tokens_times_k
from oracle import moe_oracle as O
from synth import CONFIGS, make_layer


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape():
    return CONFIGS["tiny"].replace(T=97, E=16)  # shards of 49 and 48 tokens


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s = _shape()
        L = make_layer(s, "tiny")
        shard = np.array_split(np.arange(s.T), world)[rank]
        scores = O.router_scores(L["x"][shard], L["w_router"]).astype(np.float32)
        bias = L["bias"] + np.float32(0.004) * np.arange(s.E, dtype=np.float32)
        idx = O.topk_select(scores, bias, s.k)
        load = torch.from_numpy(O.expert_load(idx, s.E).astype(np.int32))
        n = allreduce_load(load)
        tk = global_tokens_times_k(load)
        assert tk == s.T * s.k != n * len(shard) * s.k
        new_bias = O.bias_update(bias, load.numpy(), tk, s.gamma)
        np.save(os.path.join(out_dir, f"bias_{rank}.npy"), new_bias)
        np.save(os.path.join(out_dir, f"idx_{rank}.npy"), idx)
        np.save(os.path.join(out_dir, f"load_{rank}.npy"), load.numpy())
        assert n == world
    finally:
        dist.destroy_process_group()


def test_two_rank_bias_update_equals_full_batch(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    s = _shape()
    L = make_layer(s, "tiny")
    bias = L["bias"] + np.float32(0.004) * np.arange(s.E, dtype=np.float32)
    scores = O.router_scores(L["x"], L["w_router"]).astype(np.float32)
    idx = O.topk_select(scores, bias, s.k)
    load = O.expert_load(idx, s.E)
    want = O.bias_update(bias, load, s.T * s.k, s.gamma)
    shards = np.array_split(np.arange(s.T), world)
    # The case can tell the formulas apart: world * (a shard's T*k) moves some bias
    # differently from the global T*k (an expert's E * load equals a wrong target).
    wrong = [O.bias_update(bias, load, world * len(sh) * s.k, s.gamma) for sh in shards]
    assert any(not np.array_equal(w.view(np.uint32), want.view(np.uint32)) for w in wrong)
    for r in range(world):
        got = np.load(tmp_path / f"bias_{r}.npy")
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        assert np.array_equal(np.load(tmp_path / f"load_{r}.npy"), load)
        assert np.array_equal(np.load(tmp_path / f"idx_{r}.npy"), idx[shards[r]])


# ---------------------------------------------------------------- expert parallelism

class _OracleRank:
    """The phases of aux_loss_free_gb300.ep.EPRank computed by the oracle (fp64, on
    the CPU), so that the exchange logic of ep.ep_forward -- the per-owner counts, the
    split sizes, the order rows arrive and go back in -- runs over gloo ranks."""

    def __init__(self, s, host, shard, rank, world, bias):
        from ep_util import regroup_reference
        self.regroup = regroup_reference
        self.spec, self.world, self.el, self.t = s, world, s.E // world, len(shard)
        self.bias, self.host = bias.copy(), host
        bf = O.bf16_value_from_bits
        e0 = rank * self.el
        self.wg, self.wu, self.wd = (bf(host[n])[e0:e0 + self.el] for n in ("w_gate", "w_up", "w_down"))
        self.sg, self.su, self.sd = (bf(host[n]) for n in ("s_gate", "s_up", "s_down"))

    def dispatch(self, x):
        s = self.spec
        xn = x.numpy()
        scores = O.router_scores(xn, self.host["w_router"]).astype(np.float32)
        idx = O.topk_select(scores, self.bias, s.k)
        gate = O.gate_weights(scores, idx, s.renorm)
        load = torch.from_numpy(O.expert_load(idx, s.E).astype(np.int32))
        _, perm_tok, inv_pos = O.stable_permutation(idx, s.E)
        return dict(idx=idx, gate=gate, load=load, inv_pos=inv_pos, xp=x[torch.from_numpy(np.asarray(perm_tok))],
                    counts=load.view(self.world, self.el))

    def experts(self, recv_x, recv_counts):
        perm, inv, offsets = self.regroup(recv_counts.numpy())
        xg = recv_x.numpy()[perm]
        yg = np.zeros_like(xg)
        for e in range(self.el):
            r = slice(offsets[e], offsets[e + 1])
            yg[r] = O.swiglu_ffn(xg[r], self.wg[e], self.wu[e], self.wd[e])
        return torch.from_numpy(yg[inv])

    def combine(self, st, x, y_back, out, residual=None):
        shared = O.swiglu_ffn(x.numpy(), self.sg, self.su, self.sd)
        out[:] = torch.from_numpy(O.combine(y_back.numpy(), shared, st["inv_pos"], st["gate"]))
        return out

    def bias_update(self, load, tokens_times_k):
        self.bias = O.bias_update(self.bias, load.numpy(), tokens_times_k, self.spec.gamma)


def _ep_shape():
    return CONFIGS["tiny"].replace(T=97, E=16)  # unequal shards: 49 and 48 tokens


def _ep_rank_main(rank, world, port, out_dir):
    from aux_loss_free_gb300.ep import ep_forward
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s = _ep_shape()
        host = make_layer(s, "tiny")
        shard = np.array_split(np.arange(s.T), world)[rank]
        bias = host["bias"] + np.float32(0.004) * np.arange(s.E, dtype=np.float32)
        r = _OracleRank(s, host, shard, rank, world, bias)
        x = torch.from_numpy(O.round_to_bf16(host["x"][shard].astype(np.float64)))
        out = torch.empty(len(shard), s.d, dtype=torch.float64)
        ep_forward(r, x, out)
        np.save(os.path.join(out_dir, f"ep_out_{rank}.npy"), out.numpy())
        np.save(os.path.join(out_dir, f"ep_bias_{rank}.npy"), r.bias)
    finally:
        dist.destroy_process_group()


def test_expert_parallel_exchange_equals_full_batch(tmp_path):
    """Two gloo ranks, 8 experts each: ep.ep_forward's dispatch and return must put
    every row where the single-process layer has it, and both ranks must end with the
    full batch's bias update."""
    world = 2
    mp.spawn(_ep_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    s = _ep_shape()
    host = make_layer(s, "tiny")
    bias = host["bias"] + np.float32(0.004) * np.arange(s.E, dtype=np.float32)
    bf = O.bf16_value_from_bits
    xb = O.round_to_bf16(host["x"].astype(np.float64))
    ref = O.layer_forward(xb, host["w_router"], bias, bf(host["w_gate"]), bf(host["w_up"]), bf(host["w_down"]),
                          bf(host["s_gate"]), bf(host["s_up"]), bf(host["s_down"]), k=s.k, gamma=s.gamma)
    got = np.concatenate([np.load(tmp_path / f"ep_out_{r}.npy") for r in range(world)])
    assert np.allclose(got, ref["out"], rtol=1e-12, atol=1e-12)
    for r in range(world):
        assert np.array_equal(np.load(tmp_path / f"ep_bias_{r}.npy").view(np.uint32), ref["bias"].view(np.uint32))

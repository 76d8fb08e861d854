"""Two CPU ranks (gloo) run the data-parallel balancing step on their token shards.

Each rank routes its shard with the oracle, the loads are summed with the package's
allreduce_load, and each rank applies the bias update with the global T*k.  Every
rank must end with the bias that the single-process full batch gives, bit for bit,
and each shard's routing must equal the full batch's routing of those tokens.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from aux_loss_free_gb300.dp import allreduce_load
from oracle import moe_oracle as O
from synth import CONFIGS, make_layer


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape():
    return CONFIGS["tiny"].replace(T=96, E=16)


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
        new_bias = O.bias_update(bias, load.numpy(), n * len(shard) * s.k, s.gamma)  # global T*k
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
    for r in range(world):
        got = np.load(tmp_path / f"bias_{r}.npy")
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        assert np.array_equal(np.load(tmp_path / f"load_{r}.npy"), load)
        assert np.array_equal(np.load(tmp_path / f"idx_{r}.npy"), idx[shards[r]])

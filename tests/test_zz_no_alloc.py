"""moe_permute_noalloc against moe_permute, on the GPU, through the C ABI.

The no-workspace variant exists for callers that cannot give the library device
memory (a plugin in a framework that owns the memory pool, a serving loop with a
fixed device-memory budget, code about to be captured into a CUDA graph).  It must
produce exactly what the workspace version produces.  Two calls in a row with
different routings check that the shared static scratch, which keeps the previous
call's contents, is cleared where it must be.  This file sorts last so that a run
stopping at the first failure has already run every other test; it also passes on
its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    w = 1.0 / (np.arange(E) + 1.0) ** 1.2
    return np.stack([rng.choice(E, size=k, replace=False, p=w / w.sum())
                     for _ in range(T)]).astype(np.int32)


def _with_workspace(ms, idx, T, E, k):
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T, k, dtype=torch.int32, device=DEV)
    ws = torch.empty(M.moe_permute_workspace_size(ms), dtype=torch.uint8, device=DEV)
    M.moe_permute(ms, idx, off, perm, inv, ws)
    return off, perm, inv


def _without_workspace(ms, idx, T, E, k):
    off = torch.full((E + 1,), -1, dtype=torch.int32, device=DEV)
    perm = torch.full((T * k,), -1, dtype=torch.int32, device=DEV)
    inv = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    M.moe_permute_noalloc(ms, idx, off, perm, inv)
    return off, perm, inv


@pytest.mark.parametrize("T,E,k", [(8192, 64, 2), (1000, 16, 3), (70000, 256, 4)])
def test_noalloc_permute_equals_workspace_permute_twice(T, E, k):
    assert torch.cuda.is_available(), "this test needs a CUDA device"
    M.load_library()
    ms = M.make_shape(T, 1024, E, 512, 0, k)
    for call, seed in enumerate((T, T + 1)):  # two calls in a row, different routings
        idx = torch.from_numpy(_routing(T, E, k, seed)).to(DEV)
        ref = _with_workspace(ms, idx, T, E, k)
        got = _without_workspace(ms, idx, T, E, k)
        torch.cuda.synchronize()
        for name, a, b in zip(("offsets", "perm_tok", "inv_pos"), got, ref):
            assert torch.equal(a, b), f"call {call}: {name} differs"
    assert M.moe_device_status() == 0

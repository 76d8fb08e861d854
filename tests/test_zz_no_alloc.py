"""moe_permute_noalloc on the GPU, through the C ABI.

The no-workspace variant serves callers that cannot give the library device memory
for scratch: a plugin inside a framework that owns the device memory pool and hands out
no scratch, or a serving loop whose device-memory budget was fixed at start-up.  It
must produce exactly what the workspace version produces, and what the oracle's
definitional counting sort produces.  Two calls in a row with different routings check
that the shared static scratch, which keeps the previous call's contents, is cleared
where it must be.  An expert id outside [0, E) is skipped by the kernels' own bounds
checks and reported through the device status word.  This file sorts last so that a
run stopping at the first failure has already run every other test; it also passes on
its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from oracle import moe_oracle as O

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
        idx_np = _routing(T, E, k, seed)
        idx = torch.from_numpy(idx_np).to(DEV)
        ref = _with_workspace(ms, idx, T, E, k)
        got = _without_workspace(ms, idx, T, E, k)
        torch.cuda.synchronize()
        for name, a, b in zip(("offsets", "perm_tok", "inv_pos"), got, ref):
            assert torch.equal(a, b), f"call {call}: {name} differs"
        if T <= 8192:  # the oracle's definitional loop, directly
            o_off, o_perm, o_inv = O.stable_permutation(idx_np, E)
            for name, a, b in zip(("offsets", "perm_tok", "inv_pos"), got, (o_off, o_perm, o_inv)):
                assert np.array_equal(a.cpu().numpy(), b), f"call {call}: {name} differs from the oracle"
    assert M.moe_device_status() == 0


def test_noalloc_permute_reports_an_expert_id_out_of_range():
    """One id equal to E: not counted, not ranked (the kernels check every id before
    using it as an index), MOE_ERR_DEVICE in the status word, which the read clears; the
    next call with valid ids is exact again."""
    M.load_library()
    T, E, k = 256, 16, 2
    ms = M.make_shape(T, 1024, E, 512, 0, k)
    assert M.moe_device_status() == 0
    idx_np = _routing(T, E, k, 4)
    bad = idx_np.copy()
    bad[17, 1] = E
    _without_workspace(ms, torch.from_numpy(bad).to(DEV), T, E, k)
    assert M.moe_device_status() == 6  # MOE_ERR_DEVICE
    assert M.moe_device_status() == 0  # cleared by the read
    got = _without_workspace(ms, torch.from_numpy(idx_np).to(DEV), T, E, k)
    torch.cuda.synchronize()
    o_off, o_perm, o_inv = O.stable_permutation(idx_np, E)
    for a, b in zip(got, (o_off, o_perm, o_inv)):
        assert np.array_equal(a.cpu().numpy(), b)
    assert M.moe_device_status() == 0

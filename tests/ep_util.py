"""The grouping of received rows that moe_ep_regroup computes, written from its
definition: rows arrive source by source, each source's rows by local expert; grouped,
local expert e's rows are the sources' runs for e in source order."""
import numpy as np


def regroup_reference(counts):
    """counts [world][E_local] -> (perm [rows], inv [rows], offsets [E_local + 1])."""
    counts = np.asarray(counts, dtype=np.int64)
    world, el = counts.shape
    received = []  # (source, expert, j) of each received row, in arrival order
    for s in range(world):
        for e in range(el):
            received += [(s, e, j) for j in range(counts[s, e])]
    grouped = sorted(range(len(received)), key=lambda i: (received[i][1], received[i][0], received[i][2]))
    perm = np.array(grouped, dtype=np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    offsets = np.concatenate([[0], np.cumsum(counts.sum(axis=0))])
    return perm, inv, offsets

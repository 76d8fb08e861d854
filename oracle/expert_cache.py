"""Oracle of the GPU-side int4 expert residency cache (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline may use this module;
the library's product path never imports it.

The relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B
de NanoColibri por $200"), opening section, second paragraph, streams the int4 experts
from NVMe through an LRU cache under a memory budget, and its top-2 paragraph notes
that the routing skew left after balancing is what such a cache likes.  The GPU
analogue kept here: every expert's int4 weights live in host memory, the GPU holds
`slots` of them, and each serving step brings in the experts its routing uses.  The
pages fix no policy details; this is the plain reading taken (least recently used):

* the experts a step uses are the distinct values of its routing result, taken in
  ascending order;
* first every used expert that is resident is a hit and its slot is stamped with the
  step number (so that nothing the step uses can be evicted by it);
* then each used expert that is not resident, in ascending order, is a miss: it takes
  the slot with the smallest stamp among the slots not stamped in this step (an empty
  slot has stamp -1, so empty slots go first), ties to the lowest slot index; the
  expert that held the slot (if any) is evicted; the slot is stamped;
* a step that uses more distinct experts than there are slots cannot be served.
"""
from __future__ import annotations

import numpy as np


class CacheCapacityError(ValueError):
    pass


def lru_cache_state(E: int, slots: int):
    """Empty cache: (slot_expert[slots], expert_slot[E], stamp[slots], step)."""
    return (np.full(slots, -1, np.int64), np.full(E, -1, np.int64), np.full(slots, -1, np.int64), 0)


def lru_cache_step(state, idx):
    """One serving step with routing result idx (any shape of expert ids).

    Returns (new_state, hits, misses, evictions, jobs) where jobs lists the (expert,
    slot) copies the step needs, in the order the misses were served."""
    slot_expert, expert_slot, stamp, step = (state[0].copy(), state[1].copy(), state[2].copy(), state[3])
    used = sorted(set(int(e) for e in np.asarray(idx).ravel()))
    hits = misses = evictions = 0
    missing = []
    for e in used:
        if expert_slot[e] >= 0:
            stamp[expert_slot[e]] = step
            hits += 1
        else:
            missing.append(e)
    jobs = []
    for e in missing:
        best = -1
        for c in range(len(stamp)):
            if stamp[c] < step and (best < 0 or stamp[c] < stamp[best]):
                best = c
        if best < 0:
            raise CacheCapacityError(f"step {step} uses {len(used)} experts, more than {len(stamp)} slots")
        if slot_expert[best] >= 0:
            expert_slot[slot_expert[best]] = -1
            evictions += 1
        slot_expert[best] = e
        expert_slot[e] = best
        stamp[best] = step
        misses += 1
        jobs.append((e, best))
    return (slot_expert, expert_slot, stamp, step + 1), hits, misses, evictions, jobs


def lru_cache_run(E: int, slots: int, idx_per_step):
    """Run a sequence of steps from an empty cache.

    Returns dict(state=final state, hits=[...], misses=[...], evictions=[...],
    jobs=[[(e, slot), ...], ...]) with one entry per step."""
    state = lru_cache_state(E, slots)
    out = dict(hits=[], misses=[], evictions=[], jobs=[])
    for idx in idx_per_step:
        state, h, m, ev, jobs = lru_cache_step(state, idx)
        out["hits"].append(h)
        out["misses"].append(m)
        out["evictions"].append(ev)
        out["jobs"].append(jobs)
    out["state"] = state
    return out

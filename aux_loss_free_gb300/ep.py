"""Expert parallelism for the MoE layer: each rank owns E / world consecutive routed
experts and a copy of the router, the bias and the shared expert.

Relay article, top-2 paragraph: the imbalance left after aux-loss-free balancing is
what expert parallelism meets; the balancing keeps the per-expert (so per-rank) row
counts close to even.  Architecture paragraph: the bias update uses the global load,
the one exchange the method itself needs.

One forward of a rank (every step in the library's kernels; the exchanges are
torch.distributed all-to-alls, or in-process copies when one GPU emulates the ranks):
  1. dispatch: route and permute the rank's tokens (moe_route, moe_permute) and gather
     their rows in permuted order (moe_gather_rows).  Rows are sorted by expert, so the
     rows for each owner rank are one contiguous run; the per-expert loads give the
     counts;
  2. exchange: counts per (owner, local expert), then the rows;
  3. experts: the owner groups the received rows by local expert (moe_ep_regroup), runs
     the grouped expert FFN over them (moe_expert_ffn, its E / world experts) and puts
     the outputs back in received order (moe_gather_rows with the inverse);
  4. exchange back;
  5. combine: the shared expert over the rank's tokens (moe_expert_ffn as one group of
     all tokens) and moe_combine;
  6. the loads summed over ranks, and the same bias update on every rank
     (moe_bias_update with the global T*k).
With consecutive token shards per rank, each expert's rows reach it in global token
order, so the outputs equal the single-GPU layer's bit for bit.
"""
from __future__ import annotations

import torch

from . import _lib as L
from .dp import allreduce_load, global_tokens_times_k
from .layer import pack_gate_up, to_device_bf16


class EPRank:
    """Rank `rank` of `world`: its routed experts [rank * E / world, (rank + 1) * E / world)."""

    def __init__(self, spec, host: dict, t_local: int, rank: int, world: int, device="cuda"):
        if spec.E % world:
            raise ValueError("E must be a multiple of the number of ranks")
        if spec.w_format != "bf16" or spec.x_dtype != "bf16":
            raise ValueError("expert parallelism runs the bf16 layer with bf16 tokens")
        dev = torch.device(device)
        self.spec, self.rank, self.world, self.device = spec, rank, world, dev
        self.el = spec.E // world
        self.t = t_local
        e0 = rank * self.el
        self.shape = L.make_shape(t_local, spec.d, spec.E, spec.f, spec.F, spec.k, renorm=spec.renorm)
        self.w_router = torch.from_numpy(host["w_router"]).to(dev)
        self.bias = torch.from_numpy(host["bias"].copy()).to(dev)
        lo = host.get("logit_offset")
        self.logit_offset = None if lo is None else torch.from_numpy(lo).to(dev)
        self.gamma = float(host["gamma"])
        wg = to_device_bf16(host["w_gate"][e0:e0 + self.el], dev)
        wu = to_device_bf16(host["w_up"][e0:e0 + self.el], dev)
        self.w_gate_up = pack_gate_up(wg, wu)
        self.w_down = to_device_bf16(host["w_down"][e0:e0 + self.el], dev)
        self.local_weights = L.make_weights(self.w_gate_up, self.w_down)
        self.shared_weights = None
        if spec.F:
            sg = to_device_bf16(host["s_gate"], dev)[None]
            su = to_device_bf16(host["s_up"], dev)[None]
            self.s_gate_up = pack_gate_up(sg, su)
            self.s_down = to_device_bf16(host["s_down"], dev)[None]
            self.shared_weights = L.make_weights(self.s_gate_up, self.s_down)
            # The shared expert as one routed group over all of the rank's tokens.
            self.shared_shape = L.make_shape(t_local, spec.d, 1, spec.F, 0, 1, renorm=False)
            self.shared_offsets = torch.tensor([0, t_local], dtype=torch.int32, device=dev)
            self.shared_perm = torch.arange(t_local, dtype=torch.int32, device=dev)
            self.shared_ws = torch.empty(L.moe_expert_ffn_workspace_size(self.shared_shape), dtype=torch.uint8,
                                         device=dev)
        self.route_ws = torch.empty(max(1, L.moe_route_workspace_size(self.shape)), dtype=torch.uint8, device=dev)
        self.perm_ws = torch.empty(L.moe_permute_workspace_size(self.shape), dtype=torch.uint8, device=dev)

    # 1. route, permute, gather
    def dispatch(self, x: torch.Tensor, stream=None) -> dict:
        s, dev, tk = self.spec, self.device, self.t * self.spec.k
        idx = torch.empty(self.t, s.k, dtype=torch.int32, device=dev)
        gate = torch.empty(self.t, s.k, dtype=torch.float32, device=dev)
        load = torch.empty(s.E, dtype=torch.int32, device=dev)
        L.moe_route(self.shape, x, self.w_router, self.logit_offset, self.bias, None, idx, gate, load,
                    self.route_ws, stream=stream)
        offsets = torch.empty(s.E + 1, dtype=torch.int32, device=dev)
        perm_tok = torch.empty(tk, dtype=torch.int32, device=dev)
        inv_pos = torch.empty(self.t, s.k, dtype=torch.int32, device=dev)
        L.moe_permute(self.shape, idx, offsets, perm_tok, inv_pos, self.perm_ws, stream=stream)
        xp = torch.empty(tk, s.d, dtype=torch.bfloat16, device=dev)
        L.moe_gather_rows(tk, s.d, x, perm_tok, xp, stream=stream)
        # counts[q][e]: rows for owner q's local expert e (the loads, viewed per owner)
        return dict(idx=idx, gate=gate, load=load, inv_pos=inv_pos, xp=xp,
                    counts=load.view(self.world, self.el))

    # 3. the owner's experts over the rows it received
    def experts(self, recv_x: torch.Tensor, recv_counts: torch.Tensor, stream=None) -> torch.Tensor:
        s, dev = self.spec, self.device
        rows = recv_x.shape[0]
        y = torch.empty(rows, s.d, dtype=torch.bfloat16, device=dev)
        if rows == 0:
            return y
        perm = torch.empty(rows, dtype=torch.int32, device=dev)
        inv = torch.empty(rows, dtype=torch.int32, device=dev)
        offsets = torch.empty(self.el + 1, dtype=torch.int32, device=dev)
        L.moe_ep_regroup(self.world, self.el, recv_counts.contiguous(), perm, inv, offsets, stream=stream)
        shape = L.make_shape(rows, s.d, self.el, s.f, 0, 1, renorm=False)
        ws = torch.empty(L.moe_expert_ffn_workspace_size(shape), dtype=torch.uint8, device=dev)
        y_grouped = torch.empty(rows, s.d, dtype=torch.bfloat16, device=dev)
        L.moe_expert_ffn(shape, recv_x, offsets, perm, self.local_weights, y_grouped, None, ws, stream=stream)
        L.moe_gather_rows(rows, s.d, y_grouped, inv, y, stream=stream)
        return y

    # 5. shared expert and combine
    def combine(self, state: dict, x: torch.Tensor, y_back: torch.Tensor, out: torch.Tensor,
                residual: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        s_out = None
        if self.shared_weights is not None:
            s_out = torch.empty(self.t, self.spec.d, dtype=torch.bfloat16, device=self.device)
            L.moe_expert_ffn(self.shared_shape, x, self.shared_offsets, self.shared_perm, self.shared_weights,
                             s_out, None, self.shared_ws, stream=stream)
        L.moe_combine(self.shape, y_back, s_out, state["inv_pos"], state["gate"], residual, out, stream=stream)
        return out

    # 6. the bias update from the summed loads; tokens_times_k is the global T*k (the sum
    # of the summed loads), or MOE_TK_FROM_LOAD to have the kernel take that sum itself
    def bias_update(self, global_load: torch.Tensor, tokens_times_k: int, stream=None):
        L.moe_bias_update(self.spec.E, tokens_times_k, global_load, self.gamma, self.bias, stream=stream)


def rows_per_owner(counts: torch.Tensor) -> list[int]:
    """Row counts per owner rank from a [world][E_local] count table (host integers)."""
    return [int(v) for v in counts.sum(dim=1).tolist()]


def ep_forward(rank: EPRank, x: torch.Tensor, out: torch.Tensor, update_bias: bool = True,
               residual: torch.Tensor | None = None, group=None) -> torch.Tensor:
    """One expert-parallel forward of this process's rank over torch.distributed."""
    import torch.distributed as dist

    st = rank.dispatch(x)
    send_counts = st["counts"].contiguous()
    recv_counts = torch.empty_like(send_counts)
    dist.all_to_all_single(recv_counts, send_counts, group=group)
    send_rows, recv_rows = rows_per_owner(send_counts), rows_per_owner(recv_counts)
    xp = st["xp"]
    recv_x = torch.empty(sum(recv_rows), xp.shape[1], dtype=xp.dtype, device=xp.device)
    dist.all_to_all_single(recv_x, xp, recv_rows, send_rows, group=group)
    y_recv = rank.experts(recv_x, recv_counts)
    y_back = torch.empty_like(xp)
    dist.all_to_all_single(y_back, y_recv, send_rows, recv_rows, group=group)
    rank.combine(st, x, y_back, out, residual)
    if update_bias:
        load = st["load"].clone()
        allreduce_load(load, group)
        # The global T*k from the summed loads: right for shards of any sizes.
        rank.bias_update(load, global_tokens_times_k(load))
    return out


def ep_forward_emulated(ranks: list[EPRank], xs: list[torch.Tensor], outs: list[torch.Tensor],
                        update_bias: bool = True, residuals=None) -> list[torch.Tensor]:
    """All ranks in one process (one GPU): the exchanges become copies between the ranks'
    buffers, in the order the all-to-alls would deliver them."""
    world = len(ranks)
    st = [r.dispatch(x) for r, x in zip(ranks, xs)]
    send_rows = [rows_per_owner(s["counts"]) for s in st]
    starts = [[sum(rows[:q]) for q in range(world)] for rows in send_rows]
    y_recv = []
    for q, r in enumerate(ranks):
        recv_counts = torch.stack([st[src]["counts"][q] for src in range(world)])
        recv_x = torch.cat([st[src]["xp"][starts[src][q]:starts[src][q] + send_rows[src][q]]
                            for src in range(world)])
        y_recv.append(r.experts(recv_x, recv_counts))
    for src, r in enumerate(ranks):
        pieces = []
        for q in range(world):
            first = sum(send_rows[s][q] for s in range(src))  # src's rows in q's received order
            pieces.append(y_recv[q][first:first + send_rows[src][q]])
        y_back = torch.cat(pieces)
        r.combine(st[src], xs[src], y_back, outs[src], None if residuals is None else residuals[src])
    if update_bias:
        load = torch.stack([s["load"] for s in st]).sum(dim=0, dtype=torch.int32)
        for r in ranks:
            r.bias_update(load, L.MOE_TK_FROM_LOAD)  # global T*k = sum of the summed loads
    return outs

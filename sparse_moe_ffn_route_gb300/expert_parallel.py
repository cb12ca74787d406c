"""Expert parallelism for the sparse MoE FFN layer: dispatch and combine of
(token, slot) rows across ranks.

"Phase 19: MoE - gpt-oss-20b", section 6 leaves expert parallelism (experts spread
over several GPUs) for later work; this module is that step's bookkeeping.  G ranks
each hold tokens of their own (data-parallel over tokens) and the routed experts
[r E/G, (r+1) E/G) of rank r.  One layer then runs as:

  1. route locally: topk_ids [T, k], topk_w [T, k] on every rank (the router and
     the shared expert are data-parallel and stay local);
  2. plan: the owner rank of slot s = t k + j is topk_ids[t, j] // (E/G); the slots
     are sent grouped by owner, in slot order within an owner (a stable sort), and
     the per-destination counts are exchanged (one all-to-all of G integers);
  3. dispatch: the token row x[t] of every slot, and its expert's local index, go
     to the owner (one all-to-all of rows of d values, one of ids);
  4. the owner evaluates its experts on the received rows, one expert per row, with
     routing weight 1 (moe_ffn_forward_routed with top_k = 1 and fp32 output on a
     GPU): the unweighted expert outputs Y;
  5. return: the Y rows travel back by the reverse all-to-all and land in slot
     order;
  6. combine: y[t] = sum_j topk_w[t, j] Y[t k + j], j = 0..k-1 in that fixed order
     (the caller adds the shared expert's sgate * shexp and the residual).

Rows leave a rank once per (token, slot) whose expert lives elsewhere (a real
deployment would keep the local slots out of the exchange; here every slot takes
the same path, which the tests need to see).  Y comes back at the precision the
owner computed it in (fp32 from the library), so the combine adds the same terms
the single-GPU layer adds.  The plan is integer work on the routing ids; the
exchange is torch.distributed (gloo on CPU ranks, NCCL on GPUs).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional

import torch
import torch.distributed as dist


@dataclasses.dataclass
class DispatchPlan:
    """Where every (token, slot) row of one rank goes, and what it receives."""
    world: int
    experts_per_rank: int
    top_k: int
    tokens: int
    send_order: torch.Tensor      # int64 [T k]: slot index of each sent row, grouped by owner
    send_counts: List[int]        # rows sent to each rank
    recv_counts: List[int]        # rows received from each rank
    recv_local_ids: torch.Tensor  # int32 [R]: local expert index (0..E/G-1) of each received row

    @property
    def rows_received(self) -> int:
        return int(sum(self.recv_counts))


def owner_of(topk_ids: torch.Tensor, n_experts: int, world: int) -> torch.Tensor:
    """Rank that holds each selected expert: contiguous blocks of E/G experts."""
    if n_experts % world:
        raise ValueError(f"{n_experts} experts do not split evenly over {world} ranks")
    return torch.div(topk_ids.to(torch.int64), n_experts // world, rounding_mode="floor")


def _a2a(out: torch.Tensor, inp: torch.Tensor, out_splits, in_splits, group) -> torch.Tensor:
    dist.all_to_all_single(out, inp.contiguous(), list(out_splits), list(in_splits), group=group)
    return out


def dispatch_plan(topk_ids: torch.Tensor, n_experts: int, group=None) -> DispatchPlan:
    """Step 2: owners, send order and counts, and the exchange of counts and local ids."""
    world = dist.get_world_size(group)
    T, k = topk_ids.shape
    epr = n_experts // world
    owner = owner_of(topk_ids, n_experts, world).reshape(-1)
    if owner.numel() and (int(owner.min()) < 0 or int(owner.max()) >= world):
        raise ValueError("a routing id lies outside [0, n_experts)")
    send_order = torch.sort(owner, stable=True).indices
    send_counts_t = torch.bincount(owner, minlength=world).to(torch.int64)
    recv_counts_t = torch.empty(world, dtype=torch.int64, device=send_counts_t.device)
    _a2a(recv_counts_t, send_counts_t, [1] * world, [1] * world, group)
    send_counts = [int(c) for c in send_counts_t.tolist()]
    recv_counts = [int(c) for c in recv_counts_t.tolist()]
    local = (topk_ids.reshape(-1).to(torch.int64) - owner * epr)[send_order].to(torch.int32)
    recv_ids = torch.empty(sum(recv_counts), dtype=torch.int32, device=topk_ids.device)
    _a2a(recv_ids, local, recv_counts, send_counts, group)
    return DispatchPlan(world, epr, k, T, send_order, send_counts, recv_counts, recv_ids)


def dispatch(x: torch.Tensor, plan: DispatchPlan, group=None) -> torch.Tensor:
    """Step 3: the token row of every sent slot, delivered to the owner of its expert.
    x [T, d] -> rows [R, d] on the receiving side, grouped by source rank."""
    rows = x.index_select(0, torch.div(plan.send_order, plan.top_k, rounding_mode="floor"))
    out = torch.empty((plan.rows_received, x.shape[1]), dtype=x.dtype, device=x.device)
    return _a2a(out, rows, plan.recv_counts, plan.send_counts, group)


def gather_back(Y_recv: torch.Tensor, plan: DispatchPlan, group=None) -> torch.Tensor:
    """Step 5: expert outputs of the received rows back to their sources, in slot
    order: [R, d] -> [T k, d]."""
    back = torch.empty((plan.tokens * plan.top_k, Y_recv.shape[1]), dtype=Y_recv.dtype,
                       device=Y_recv.device)
    _a2a(back, Y_recv, plan.send_counts, plan.recv_counts, group)
    Y_slots = torch.empty_like(back)
    Y_slots.index_copy_(0, plan.send_order, back)
    return Y_slots


def combine(Y_slots: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
    """Step 6: y[t] = sum_j topk_w[t, j] * Y[t k + j], added in slot order j = 0..k-1
    in Y's precision."""
    T, k = topk_w.shape
    Y = Y_slots.view(T, k, Y_slots.shape[1])
    w = topk_w.to(Y.dtype)
    y = torch.zeros((T, Y.shape[2]), dtype=Y.dtype, device=Y.device)
    for j in range(k):
        y = y + w[:, j:j + 1] * Y[:, j]
    return y


def forward(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, n_experts: int,
            local_experts: Callable[[torch.Tensor, torch.Tensor], torch.Tensor],
            group=None) -> torch.Tensor:
    """Steps 2-6 for one rank: the routed part of the layer for this rank's tokens.

    local_experts(rows [R, d], local_ids int32 [R]) -> Y [R, d] evaluates this rank's
    experts, one per row, unweighted (e.g. library_local_experts below)."""
    plan = dispatch_plan(topk_ids, n_experts, group)
    rows = dispatch(x, plan, group)
    Y = local_experts(rows, plan.recv_local_ids)
    if Y.shape[0] != plan.rows_received:
        raise ValueError("local_experts returned a different number of rows")
    return combine(gather_back(Y, plan, group), topk_w)


def library_local_experts(cfg, experts, rank: int, world: int, stream=None):
    """local_experts for a GPU rank: this rank's slice of the expert weights run by
    moe_ffn_forward_routed, one expert per row with weight 1, fp32 output.

    cfg is the whole layer's moe_cfg_t; `experts` holds all E experts' tensors (the
    slice [r E/G, (r+1) E/G) is taken here, as views)."""
    from . import Experts, moe_ffn_forward_routed
    E = cfg.n_experts
    if E % world:
        raise ValueError(f"{E} experts do not split evenly over {world} ranks")
    epr = E // world
    lo, hi = rank * epr, (rank + 1) * epr
    local = Experts(**{f.name: (None if getattr(experts, f.name) is None
                                else getattr(experts, f.name)[lo:hi])
                       for f in dataclasses.fields(Experts)})
    lcfg = cfg.replace(n_experts=epr, top_k=1, shared_ff=0, y_fp32=1, residual=0, rms_norm=0)

    def run(rows: torch.Tensor, local_ids: torch.Tensor) -> torch.Tensor:
        R = rows.shape[0]
        if R == 0:
            return torch.empty((0, rows.shape[1]), dtype=torch.float32, device=rows.device)
        ids = local_ids.view(R, 1).contiguous()
        w = torch.ones((R, 1), dtype=torch.float32, device=rows.device)
        return moe_ffn_forward_routed(lcfg, rows.contiguous(), ids, w, local, stream=stream)

    return run

"""Expert-parallel MoE layer: G ranks (one GPU each), rank r owning the
E_local = E / G consecutive experts [r * E_local, (r + 1) * E_local).

Megatron-LM ``fused_indices_converter.py`` (``_indices_to_multihot_kernel``)
restricts a rank's routing map to its local experts; every owner runs the
grouped FFN of project_6 ``moe_expert_gemm.cpp`` (``moe_prefill_experts``) on the
rows routed to its experts, and each token's k weighted results are summed as
in mlc-llm ``moe_misc.py`` (``scatter_output``, ``moe_sum``).

One step, on every rank for its own T tokens:

1. gating and align over all E experts (``moe_gating_softmax_topk``,
   ``moe_align_by_expert``), then the expert-sorted rows
   (``moe_gather_rows``). The align order is expert-major, so the rows for
   owner r are one contiguous range of x_sorted.
2. exchange 1: the [G, E_local] table of counts (row r = the counts of owner
   r's experts), then the rows themselves (all-to-all, rank order). This rank
   receives its experts' rows source-major.
3. ``moe_ep_receive_index`` turns the received counts table into local
   counts / offsets and the permutation from expert-major position to
   received row; ``moe_grouped_ffn`` runs with k = 1, gathering through it and
   writing every result back to the received row it came from.
4. exchange 2: the results go back along the same splits, reversed, and
   arrive in the sender's x_sorted order; ``moe_ep_combine`` forms
   out[t] = sum_j w[t, j] * y[pos(t, j)].

The split sizes of the row exchanges are host integers, so each step reads
the E expert counts back to the host once (after align). The planning below
is O(G * E) host arithmetic; all O(T) work runs in the library's kernels.
The compute steps are a parameter of the layer: ``GpuCompute`` (the
library's kernels) is the product path; tests on CPU ranks pass their own.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


def expert_range(E: int, G: int, r: int) -> tuple[int, int]:
    """[lo, hi) of the experts rank r owns (E divisible by G)."""
    if E % G:
        raise ValueError(f"E={E} must be divisible by the {G} ranks")
    El = E // G
    return r * El, (r + 1) * El


def owner_of(e: int, E: int, G: int) -> int:
    """Rank that owns expert e."""
    return e // (E // G)


@dataclass
class ExchangePlan:
    """Sizes of one step's two row exchanges, from this rank's point of view."""
    send_table: torch.Tensor   # [G, E_local] int32: counts of each owner's experts among this rank's slots
    recv_table: torch.Tensor   # [G, E_local] int32: counts of this rank's experts among each source's slots
    send_rows: list            # rows to each owner (exchange 1), received back from it (exchange 2)
    recv_rows: list            # rows from each source (exchange 1), returned to it (exchange 2)

    @property
    def sent(self) -> int:
        return sum(self.send_rows)

    @property
    def received(self) -> int:
        return sum(self.recv_rows)


def send_table(counts: torch.Tensor, G: int) -> torch.Tensor:
    """[E] expert counts -> [G, E_local]: row r = the counts of owner r's experts."""
    E = counts.numel()
    if E % G:
        raise ValueError(f"E={E} must be divisible by the {G} ranks")
    return counts.reshape(G, E // G).to(torch.int32).contiguous()


def plan_from_tables(send_tab: torch.Tensor, recv_tab: torch.Tensor) -> ExchangePlan:
    return ExchangePlan(send_tab, recv_tab, [int(x) for x in send_tab.sum(1).tolist()],
                        [int(x) for x in recv_tab.sum(1).tolist()])


def exchange_counts(send_tab: torch.Tensor, group=None) -> torch.Tensor:
    """All-to-all of the [G, E_local] counts tables: row g of the result comes from rank g."""
    recv = torch.empty_like(send_tab)
    dist.all_to_all_single(recv, send_tab, group=group)
    return recv


def exchange_rows(rows: torch.Tensor, send_rows: list, recv_rows: list, group=None) -> torch.Tensor:
    """All-to-all of row blocks: rows[0:send_rows[0]] to rank 0, the next send_rows[1] to rank 1,
    ...; returns the received blocks concatenated in source-rank order."""
    out = rows.new_empty((sum(recv_rows),) + tuple(rows.shape[1:]))
    dist.all_to_all_single(out, rows[:sum(send_rows)].contiguous(), recv_rows, send_rows, group=group)
    return out


class GpuCompute:
    """The layer's compute steps on the library's kernels (this rank's GPU)."""

    def __init__(self):
        from . import _binding as b
        self.b = b
        b.lib()   # fails loudly when the library is missing

    def route(self, logits, k, norm):
        w, idx = self.b.moe_gating_softmax_topk(logits, k, norm)
        al = self.b.moe_align_by_expert(idx, w, logits.shape[1])
        return w, idx, al

    def gather_rows(self, hidden, al, k):
        return self.b.moe_gather_rows(hidden, al["sorted_token_ids"], al["offsets"], k)

    def receive_index(self, recv_tab, R):
        return self.b.moe_ep_receive_index(recv_tab.to(torch.int32).contiguous(), R)

    def expert_ffn(self, rows, w13_local, w2_local, counts, offsets, perm):
        R = rows.shape[0]
        ones = torch.ones(R, dtype=torch.float32, device=rows.device)
        return self.b.moe_grouped_ffn(rows, w13_local, w2_local, 1, counts, offsets, perm, ones, perm)

    def combine(self, y_sorted, w, al):
        return self.b.moe_ep_combine(y_sorted, w, al["reverse_indices"], al["offsets"])


class ExpertParallelLayer:
    """The MoE layer forward with the experts split over the ranks of `group`.

    w13_local [E_local, 2I, H] and w2_local [E_local, H, I] are this rank's
    experts. forward(hidden [T, H], logits [T, E]) -> out [T, H] for this
    rank's own tokens (every rank calls it in the same step).
    """

    def __init__(self, w13_local, w2_local, E: int, k: int, norm_topk_prob: bool = True, group=None,
                 compute=None):
        self.group = group
        self.G = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.G or w13_local.shape[0] != E // self.G or w2_local.shape[0] != E // self.G:
            raise ValueError("each rank holds E / G experts")
        self.w13, self.w2 = w13_local, w2_local
        self.E, self.k, self.norm = E, k, bool(norm_topk_prob)
        self.compute = compute if compute is not None else GpuCompute()

    def forward(self, hidden, logits):
        c = self.compute
        w, idx, al = c.route(logits, self.k, self.norm)
        xs = c.gather_rows(hidden, al, self.k)
        send_tab = send_table(al["counts"], self.G)
        plan = plan_from_tables(send_tab.cpu(), exchange_counts(send_tab, self.group).cpu())
        recv_x = exchange_rows(xs, plan.send_rows, plan.recv_rows, self.group)
        counts, offsets, perm = c.receive_index(plan.recv_table.to(recv_x.device), plan.received)
        y_recv = c.expert_ffn(recv_x, self.w13, self.w2, counts, offsets, perm)
        y_back = exchange_rows(y_recv, plan.recv_rows, plan.send_rows, self.group)
        if y_back.shape[0] < xs.shape[0]:   # slots beyond offsets[E] (none for the layer's own gating)
            pad = y_back.new_zeros((xs.shape[0] - y_back.shape[0],) + tuple(y_back.shape[1:]))
            y_back = torch.cat([y_back, pad])
        return c.combine(y_back, w, al)

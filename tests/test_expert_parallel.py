"""Expert-parallel layer on CPU ranks (gloo): the host planning and the two
all-to-all exchanges of mixture_experts_routing_token_gb300.expert_parallel,
with the compute steps done by the oracle on the CPU, against the
single-process oracle layer on each rank's tokens.

The device kernels of the same steps (row gather, receive index, combine) are
checked on the GPU in test_gpu_expert_parallel.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from moe_inputs import make_layer_inputs
from oracle import align, ffn, gating


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def receive_index_reference(recv_tab):
    """Local counts, exclusive offsets and perm (expert-major position -> received row)
    written out from their definition: rows arrive source-major, each source's rows
    expert-major; the expert-major order keeps the sources in rank order."""
    tab = np.asarray(recv_tab, dtype=np.int64)
    G, El = tab.shape
    src_start = np.zeros((G, El), np.int64)
    run = 0
    for g in range(G):
        for e in range(El):
            src_start[g, e] = run
            run += tab[g, e]
    counts = tab.sum(0)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm = []
    for e in range(El):
        for g in range(G):
            perm.extend(range(src_start[g, e], src_start[g, e] + tab[g, e]))
    return counts.astype(np.int32), offsets.astype(np.int32), np.asarray(perm, np.int32)


class OracleCompute:
    """The layer's compute steps on the CPU: the oracle (float64) for gating, align and
    the expert FFN; gather, receive index and combine from their definitions."""

    def __init__(self, dtype):
        self.dtype = dtype

    def route(self, logits, k, norm):
        w, idx = gating.softmax_topk(logits.numpy(), k, norm)
        al = align.align_by_expert(idx, w, logits.shape[1])
        al = {n: torch.from_numpy(np.ascontiguousarray(al[n])) for n in
              ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")}
        return torch.from_numpy(w), torch.from_numpy(idx), al

    def gather_rows(self, hidden, al, k):
        n = int(al["offsets"][-1])
        xs = torch.zeros((hidden.shape[0] * k, hidden.shape[1]), dtype=hidden.dtype)
        xs[:n] = hidden[al["sorted_token_ids"][:n].long()]
        return xs

    def receive_index(self, recv_tab, R):
        self.recv_tab = recv_tab.clone()
        c, o, p = receive_index_reference(recv_tab.numpy())
        assert p.size == R
        return torch.from_numpy(c), torch.from_numpy(o), torch.from_numpy(p)

    def expert_ffn(self, rows, w13_local, w2_local, counts, offsets, perm):
        y = torch.zeros_like(rows)
        for e in range(len(counts)):
            sel = perm[int(offsets[e]):int(offsets[e + 1])].long()
            if sel.numel():
                y[sel] = torch.from_numpy(ffn.expert_ffn(rows[sel].numpy(), ffn.to_f64(w13_local[e], self.dtype),
                                                         ffn.to_f64(w2_local[e], self.dtype), self.dtype))
        return y

    def combine(self, y_sorted, w, al):
        T, k = w.shape
        pos = np.full(T * k, -1, np.int64)
        n = int(al["offsets"][-1])
        pos[al["reverse_indices"][:n].numpy()] = np.arange(n)
        out = np.zeros((T, y_sorted.shape[1]))
        for j in range(k):
            p = pos.reshape(T, k)[:, j]
            ok = p >= 0
            out[ok] += w.numpy()[ok, j:j + 1].astype(np.float64) * y_sorted.numpy()[p[ok]]
        return torch.from_numpy(ffn.bf16_round(out) if self.dtype == "bf16"
                                else out.astype(np.float32).astype(np.float64))


def _worker(rank, world, port, cfg, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixture_experts_routing_token_gb300 import expert_parallel as ep
        T, H, I, E, k, dtype, bias = cfg
        d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype=dtype, logits="distinct", seed=7)   # weights: shared
        tok = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype=dtype, logits="distinct", seed=100 + rank,
                                with_weights=False)                                              # tokens: per rank
        d["hidden"] = tok["hidden"]
        logits = tok["logits"] + np.asarray(bias, np.float32)[None, :]
        lo, hi = ep.expert_range(E, world, rank)
        compute = OracleCompute(dtype)
        layer = ep.ExpertParallelLayer(d["w13"][lo:hi], d["w2"][lo:hi], E, k, True, compute=compute)
        got = layer.forward(torch.from_numpy(ffn.to_f64(d["hidden"], dtype)), torch.from_numpy(logits)).numpy()
        ref = ffn.layer_forward(logits, d["hidden"], d["w13"], d["w2"], k, True, dtype)
        err = float(np.abs(got - ref["out"]).max())
        scale = float(np.abs(ref["out"]).max())
        # what this rank received: row g = the slots of rank g's tokens routed to this
        # rank's experts, counted here from every rank's own gating result
        mine = torch.tensor(np.bincount(ref["topk_indices"].ravel(), minlength=E), dtype=torch.int64)
        every = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(every, mine)
        want = torch.stack([x[lo:hi] for x in every]).tolist()
        out[rank] = (err, scale, compute.recv_tab.tolist() == want)
    finally:
        dist.destroy_process_group()


CONFIGS = [
    # T, H, I, E, k, dtype, logit bias per expert
    (40, 16, 24, 8, 2, "bf16", [0.0] * 8),
    (33, 8, 12, 16, 4, "f32", [0.0] * 16),
    (25, 16, 8, 8, 2, "bf16", [6.0] * 4 + [0.0] * 4),        # every slot goes to rank 0's experts
]


@pytest.mark.parametrize("cfg", CONFIGS)
def test_two_gloo_ranks_match_the_single_process_oracle(cfg):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(2, _free_port(), cfg, out), nprocs=2, start_method="spawn", join=True)
    tol = 2e-2 if cfg[5] == "bf16" else 1e-4
    for rank in range(2):
        err, scale, table_ok = out[rank]
        assert scale > 0 and err <= tol * scale, (rank, err, scale)
        assert table_ok, rank                   # received counts table, bit for bit


def test_plan_helpers():
    from mixture_experts_routing_token_gb300 import expert_parallel as ep
    assert ep.expert_range(8, 2, 1) == (4, 8) and ep.owner_of(5, 8, 2) == 1 and ep.owner_of(3, 8, 4) == 1
    with pytest.raises(ValueError):
        ep.expert_range(6, 4, 0)
    counts = torch.tensor([3, 0, 2, 5, 1, 1], dtype=torch.int32)
    tab = ep.send_table(counts, 3)
    assert tab.tolist() == [[3, 0], [2, 5], [1, 1]]
    plan = ep.plan_from_tables(tab, torch.tensor([[1, 2], [0, 0], [4, 1]], dtype=torch.int32))
    assert plan.send_rows == [3, 7, 2] and plan.recv_rows == [3, 0, 5]
    assert plan.sent == 12 and plan.received == 8


def test_receive_index_reference_by_hand():
    # sources 0..2, two local experts; received rows (source-major, expert-major within):
    #   src0: e0 x2 (rows 0,1), e1 x1 (row 2); src1: e1 x2 (rows 3,4); src2: e0 x1 (row 5)
    c, o, p = receive_index_reference([[2, 1], [0, 2], [1, 0]])
    assert c.tolist() == [3, 3] and o.tolist() == [0, 3, 6]
    assert p.tolist() == [0, 1, 5, 2, 3, 4]

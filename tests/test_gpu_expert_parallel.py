"""Expert-parallel entry points on the GPU, through the C ABI: the row gather, the
owner-side receive index and the sender-side combine against references written
from their definitions, and a two-rank layer emulated on one GPU (the ranks' steps
run one after the other; the exchanges are slices of device tensors) against the
oracle."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_close_rel_max, layer_tolerance, need_gpu, to_dev, to_np64
from moe_inputs import make_layer_inputs
from oracle import align, ffn, gating
from test_expert_parallel import receive_index_reference

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed, drop=0.0):
    d = make_layer_inputs(T=T, H=8, I=8, E=E, k=k, dtype="f32", logits="distinct", seed=seed, with_weights=False)
    w, idx = gating.softmax_topk(d["logits"], k, True)
    if drop:
        rng = np.random.default_rng(seed)
        idx = idx.copy()
        idx[rng.random(idx.shape) < drop] = -1
    return w, idx, align.align_by_expert(idx, w, E)


@pytest.mark.parametrize("dtype,H", [("bf16", 64), ("bf16", 4096), ("f32", 12), ("bf16", 8200)])
@pytest.mark.parametrize("drop", [0.0, 0.1])
def test_gather_rows_matches_indexing(dtype, H, drop):
    moe = need_gpu()
    T, E, k = 300, 16, 4
    w, idx, al = _routing(T, E, k, seed=H, drop=drop)
    hidden = torch.randn((T, H), device=DEV).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    ids = torch.from_numpy(al["sorted_token_ids"]).to(DEV)
    offs = torch.from_numpy(al["offsets"]).to(DEV)
    out = torch.full((T * k, H), 7.0, device=DEV, dtype=hidden.dtype)
    moe.moe_gather_rows(hidden, ids, offs, k, out=out)
    torch.cuda.synchronize()
    n = int(al["offsets"][-1])
    assert torch.equal(out[:n], hidden[ids[:n].long()])
    assert bool((out[n:] == 7.0).all())          # rows past offsets[E] untouched


@pytest.mark.parametrize("G,El", [(1, 1), (2, 4), (8, 16), (3, 5), (64, 128), (16, 1024)])
def test_receive_index_matches_reference(G, El):
    moe = need_gpu()
    rng = np.random.default_rng(G * 1000 + El)
    tab = rng.integers(0, 40, size=(G, El)).astype(np.int32)
    tab[rng.random((G, El)) < 0.3] = 0
    if G > 1:
        tab[G // 2] = 0                                  # a source that sends nothing
    R = int(tab.sum())
    c, o, p = moe.moe_ep_receive_index(torch.from_numpy(tab).to(DEV), R)
    torch.cuda.synchronize()
    rc, ro, rp = receive_index_reference(tab)
    assert c.cpu().numpy().tolist() == rc.tolist()
    assert o.cpu().numpy().tolist() == ro.tolist()
    assert p.cpu().numpy().tolist() == rp.tolist()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("drop", [0.0, 0.15])
def test_ep_combine_matches_reference(dtype, drop):
    moe = need_gpu()
    T, E, k, H = 257, 8, 3, 136
    w, idx, al = _routing(T, E, k, seed=5, drop=drop)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    y = torch.randn((T * k, H), device=DEV).to(tdt)
    out = moe.moe_ep_combine(y, torch.from_numpy(w).to(DEV), torch.from_numpy(al["reverse_indices"]).to(DEV),
                             torch.from_numpy(al["offsets"]).to(DEV))
    torch.cuda.synchronize()
    # out[t] = sum_j w[t, j] * y[pos(t, j)], pos inverting reverse_indices
    n = int(al["offsets"][-1])
    pos = np.full(T * k, -1)
    pos[al["reverse_indices"][:n]] = np.arange(n)
    yv = to_np64(y)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            if pos[t * k + j] >= 0:
                ref[t] += float(w[t, j]) * yv[pos[t * k + j]]
    ref = ffn.bf16_round(ref) if dtype == "bf16" else ref
    tol = 2 ** -8 if dtype == "bf16" else 1e-6
    assert_close_rel_max(to_np64(out), ref, tol, "ep combine")


@pytest.mark.parametrize("G,T,H,I,E,k", [(2, 300, 256, 384, 8, 2), (4, 160, 128, 256, 16, 4)])
def test_ranks_emulated_on_one_gpu_match_the_oracle(G, T, H, I, E, k):
    """Each virtual rank r: gating, align, gather on its own tokens; exchange 1 as slices
    of the senders' x_sorted; receive index + grouped FFN (k = 1) on the owner; exchange 2
    as slices of the owners' results; combine. Output vs the oracle per rank."""
    from mixture_experts_routing_token_gb300 import expert_parallel as ep
    moe = need_gpu()
    c = ep.GpuCompute()
    wts = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=3)
    ranks = []
    for r in range(G):
        tok = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=50 + r,
                                with_weights=False)
        hidden = to_dev(tok["hidden"], "bf16")
        logits = torch.from_numpy(tok["logits"]).to(DEV)
        w, idx, al = c.route(logits, k, True)
        xs = c.gather_rows(hidden, al, k)
        ranks.append(dict(tok=tok, w=w, idx=idx, al=al, xs=xs, send=ep.send_table(al["counts"], G).cpu()))
    El = E // G
    y_recv = []
    for o in range(G):                                  # owner o
        lo, hi = ep.expert_range(E, G, o)
        recv_tab = torch.stack([ranks[g]["send"][o] for g in range(G)])
        blocks = []
        for g in range(G):                              # rows of source g for owner o: its x_sorted range
            a = int(ranks[g]["al"]["offsets"][lo])
            blocks.append(ranks[g]["xs"][a:a + int(ranks[g]["send"][o].sum())])
        rows = torch.cat(blocks)
        cnt, off, perm = c.receive_index(recv_tab.to(DEV), rows.shape[0])
        y_recv.append(c.expert_ffn(rows, to_dev(wts["w13"][lo:hi], "bf16"), to_dev(wts["w2"][lo:hi], "bf16"),
                                   cnt, off, perm))
        assert cnt.cpu().tolist() == recv_tab.sum(0).tolist()
    tol = layer_tolerance("bf16")
    for g in range(G):                                  # sender g gets its rows back in x_sorted order
        back = []
        for o in range(G):
            start = sum(int(ranks[s]["send"][o].sum()) for s in range(g))
            back.append(y_recv[o][start:start + int(ranks[g]["send"][o].sum())])
        out = c.combine(torch.cat(back), ranks[g]["w"], ranks[g]["al"])
        torch.cuda.synchronize()
        tok = ranks[g]["tok"]
        ref = ffn.layer_forward(tok["logits"], tok["hidden"], wts["w13"], wts["w2"], k, True, "bf16")
        assert np.array_equal(ranks[g]["idx"].cpu().numpy(), ref["topk_indices"])
        assert_close_rel_max(to_np64(out), ref["out"], tol, f"rank {g}")

"""Pins for the FFN backward oracle (CPU only): torch autograd in float64 over the same forward.

torch differentiates its own forward (gather, matmuls, silu, weighted k-sum), so a
dropped term, a wrong sign or a transposed operand in the written-out derivative
fails here. The bf16 case checks the stated reading (the activation's rounding is
differentiated as the identity) with a straight-through rounding in the torch graph.
"""
import numpy as np
import pytest
import torch

from moe_inputs import make_layer_inputs
from oracle import align, ffn, gating
from oracle.ffn_backward import grouped_ffn_backward


def _torch_grads(d, w, idx, dO):
    """float64 autograd of out[t] = sum_j w[t,j] * W2[e] (silu(W1[e] x) * W3[e] x)."""
    dt = d["dtype"]
    x = torch.tensor(ffn.to_f64(d["hidden"], dt), requires_grad=True)
    W13 = torch.tensor(ffn.to_f64(d["w13"], dt), requires_grad=True)
    W2 = torch.tensor(ffn.to_f64(d["w2"], dt), requires_grad=True)
    wt = torch.tensor(w.astype(np.float64), requires_grad=True)
    I = d["I"]
    ii = torch.tensor(idx, dtype=torch.int64)
    T, k = idx.shape
    out = torch.zeros((T, d["H"]), dtype=torch.float64)
    for j in range(k):
        e = ii[:, j]
        g = torch.einsum("th,tih->ti", x, W13[e, :I])
        u = torch.einsum("th,tih->ti", x, W13[e, I:])
        a = torch.nn.functional.silu(g) * u
        if dt == "bf16":   # straight-through: the forward value is rounded, the derivative is the identity
            a = a + (a.to(torch.bfloat16).to(torch.float64) - a).detach()
        y = torch.einsum("ti,thi->th", a, W2[e])
        out = out + wt[:, j:j + 1] * y
    (out * torch.tensor(dO)).sum().backward()
    return dict(d_hidden=x.grad.numpy(), d_w13=W13.grad.numpy(), d_w2=W2.grad.numpy(), d_weights=wt.grad.numpy())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,H,I,E,k,norm", [(13, 8, 6, 4, 2, True), (40, 16, 12, 7, 3, False), (5, 4, 4, 3, 3, True)])
def test_backward_matches_torch_autograd(dtype, T, H, I, E, k, norm):
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=norm, dtype=dtype, logits="distinct",
                          seed=T * H + k)
    w, idx = gating.softmax_topk(d["logits"], k, norm)
    al = align.align_by_expert(idx, w, E)
    dO = np.random.default_rng(T).standard_normal((T, H))
    dO = ffn.bf16_round(dO) if dtype == "bf16" else dO.astype(np.float32).astype(np.float64)
    got = grouped_ffn_backward(d["hidden"], d["w13"], d["w2"], dtype, k, al["counts"], al["offsets"],
                               al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"],
                               dO.astype(np.float32) if dtype == "f32" else
                               (dO.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    ref = _torch_grads(d, w, idx, dO)
    for name in ("d_hidden", "d_w13", "d_w2", "d_weights"):
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-12, err_msg=name)


def test_backward_of_unused_experts_is_zero():
    d = make_layer_inputs(T=6, H=8, I=4, E=5, k=1, dtype="f32", logits="distinct", seed=3)
    idx = np.array([[0], [2], [2], [0], [0], [2]], np.int32)
    w = np.full((6, 1), 0.5, np.float32)
    al = align.align_by_expert(idx, w, 5)
    got = grouped_ffn_backward(d["hidden"], d["w13"], d["w2"], "f32", 1, al["counts"], al["offsets"],
                               al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"],
                               np.ones((6, 8), np.float32))
    for e in (1, 3, 4):
        assert not got["d_w13"][e].any() and not got["d_w2"][e].any()
    assert got["d_w13"][0].any() and got["d_w2"][2].any()

"""GPU parity of the grouped FFN backward against the oracle, through the C ABI.

Tolerance: max|err| <= 2e-2 * max|ref| per output (bf16 operands: the gathered
rows, the scaled upstream gradient, the activation and its gradient are bf16;
accumulation is float32), the same bar as the bf16 forward.
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_close_rel_max, need_gpu, to_dev, to_np64
from moe_inputs import gen_normal, make_layer_inputs
from oracle import align, gating
from oracle.ffn_backward import grouped_ffn_backward

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _routing_tensors(al):
    return {k_: torch.from_numpy(np.ascontiguousarray(al[k_])).to(DEV)
            for k_ in ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")}


def _check(moe, d, al, k, seed, workspace=None):
    T, H = d["T"], d["H"]
    dO = gen_normal(np.random.SeedSequence(seed), (T, H), 1.0, "bf16")
    t = _routing_tensors(al)
    dh, dw13, dw2, dwt = moe.moe_grouped_ffn_backward(
        to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16"), k, t["counts"],
        t["offsets"], t["sorted_token_ids"], t["sorted_weights"], t["reverse_indices"], to_dev(dO, "bf16"),
        workspace=workspace)
    torch.cuda.synchronize()
    ref = grouped_ffn_backward(d["hidden"], d["w13"], d["w2"], "bf16", k, al["counts"], al["offsets"],
                               al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"], dO)
    assert_close_rel_max(to_np64(dh), ref["d_hidden"], TOL, "d_hidden")
    assert_close_rel_max(to_np64(dw13), ref["d_w13"], TOL, "d_w13")
    assert_close_rel_max(to_np64(dw2), ref["d_w2"], TOL, "d_w2")
    assert_close_rel_max(dwt.cpu().numpy().astype(np.float64), ref["d_weights"], TOL, "d_weights")
    return dh, dw13, dw2, dwt


@pytest.mark.parametrize("T,H,I,E,k", [
    (300, 256, 256, 8, 2),       # ragged 256-row tiles
    (700, 512, 384, 8, 2),       # I % 256 == 128: half-empty N tiles, 768-row dW13
    (1000, 256, 128, 16, 4),     # I < 256
    (513, 320, 640, 5, 3),       # H % 256 == 64: partial dx / dW tiles
    (40, 128, 128, 256, 2),      # 80 slots over 256 experts: most experts have no rows
    (5, 128, 192, 8, 2),         # a few tokens
    # H above 3072: FC1 recompute and dA as two kernels (f32 gate/up buffer) instead of one
    (300, 4096, 256, 8, 2),
    (200, 3200, 384, 4, 3),      # H % 256 == 128
])
def test_backward_shapes(T, H, I, E, k):
    moe = need_gpu()
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=T + H + I)
    w, idx = gating.softmax_topk(d["logits"], k, True)
    al = align.align_by_expert(idx, w, E)
    _check(moe, d, al, k, seed=T * 3)


@pytest.mark.parametrize("T,H,I,E,k", [
    (50, 64, 64, 1, 1),          # one expert, the smallest tensor-core shape
    (33, 128, 128, 4, 4),        # k = E: every token on every expert
    (70, 192, 320, 3, 1),        # odd expert count, I % 256 == 64
])
def test_backward_edge_shapes(T, H, I, E, k):
    moe = need_gpu()
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=T + E)
    w, idx = gating.softmax_topk(d["logits"], k, True)
    _check(moe, d, align.align_by_expert(idx, w, E), k, seed=E)


def test_backward_all_rows_on_one_expert():
    moe = need_gpu()
    T, H, I, E, k = 300, 128, 192, 8, 1
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=4)
    idx = np.full((T, 1), 5, np.int32)
    w = np.random.default_rng(1).uniform(0.1, 1.0, (T, 1)).astype(np.float32)
    _, dw13, dw2, _ = _check(moe, d, align.align_by_expert(idx, w, E), k, seed=3)
    assert not dw13[torch.arange(E, device=DEV) != 5].any() and not dw2[torch.arange(E, device=DEV) != 5].any()


def test_backward_zero_tokens():
    moe = need_gpu()
    z = torch.zeros(0, dtype=torch.int32, device=DEV)
    h = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    w13 = torch.zeros((2, 128, 64), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device=DEV)
    counts = torch.zeros(2, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(3, dtype=torch.int32, device=DEV)
    dw13_out = torch.full_like(w13, 3.0)   # must be overwritten with zeros
    dw2_out = torch.full_like(w2, 3.0)
    dh, dw13, dw2, dwt = moe.moe_grouped_ffn_backward(h, w13, w2, 1, counts, offsets, z, z.float(), z, h,
                                                     d_w13=dw13_out, d_w2=dw2_out)
    torch.cuda.synchronize()
    assert dh.shape == (0, 64) and dwt.shape == (0, 1)
    assert not dw13.any() and not dw2.any()   # no rows: zero weight gradients


def test_backward_dropped_slots_and_stale_workspace():
    """Dropped slots get d_weights 0 and contribute nothing, whatever the workspace held."""
    moe = need_gpu()
    T, H, I, E, k = 400, 256, 256, 12, 3
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=11)
    w, idx = gating.softmax_topk(d["logits"], k, True)
    idx = idx.copy()
    rng = np.random.default_rng(5)
    idx[rng.random(idx.shape) < 0.15] = -1
    al = align.align_by_expert(idx, w, E)
    ws = torch.full((moe.moe_grouped_ffn_backward_workspace_size(moe.MOE_BF16, T, H, I, E, k),), 0xFF,
                    dtype=torch.uint8, device=DEV)
    _, _, _, dwt = _check(moe, d, al, k, seed=2, workspace=ws)
    assert (dwt.cpu().numpy()[idx < 0] == 0).all()


def test_backward_weight_gradients_16_byte_aligned_only():
    """d_w13 / d_w2 on a 16- but not 32-byte boundary take 16-byte stores; same results.
    Tokens go to experts 0..3 only, so the zeroing of experts without rows is covered too."""
    moe = need_gpu()
    T, H, I, E, k = 300, 256, 256, 8, 2
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=21)
    w, idx = gating.softmax_topk(d["logits"][:, :4], k, True)
    al = align.align_by_expert(idx, w, E)
    t = _routing_tensors(al)
    dO = to_dev(gen_normal(np.random.SeedSequence(4), (T, H), 1.0, "bf16"), "bf16")
    args = (to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16"), k, t["counts"],
            t["offsets"], t["sorted_token_ids"], t["sorted_weights"], t["reverse_indices"], dO)
    n13, n2 = E * 2 * I * H, E * H * I
    b13 = torch.full((n13 + 16,), 7.0, dtype=torch.bfloat16, device=DEV)
    b2 = torch.full((n2 + 16,), 7.0, dtype=torch.bfloat16, device=DEV)
    dw13 = b13[8:8 + n13].view(E, 2 * I, H)
    dw2 = b2[8:8 + n2].view(E, H, I)
    assert dw13.data_ptr() % 32 == 16 and dw2.data_ptr() % 32 == 16
    moe.moe_grouped_ffn_backward(*args, d_w13=dw13, d_w2=dw2)
    ref = moe.moe_grouped_ffn_backward(*args)
    torch.cuda.synchronize()
    assert torch.equal(dw13, ref[1]) and torch.equal(dw2, ref[2])
    assert not dw13[4:].any() and not dw2[4:].any() and dw13[:4].any()
    for b, n in ((b13, n13), (b2, n2)):   # nothing written outside the views
        assert (b[:8] == 7).all() and (b[8 + n:] == 7).all()


def test_backward_repeated_calls_are_identical():
    moe = need_gpu()
    T, H, I, E, k = 600, 256, 256, 8, 2
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=9)
    w, idx = gating.softmax_topk(d["logits"], k, True)
    t = _routing_tensors(align.align_by_expert(idx, w, E))
    dO = to_dev(gen_normal(np.random.SeedSequence(1), (T, H), 1.0, "bf16"), "bf16")
    args = (to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16"), k, t["counts"],
            t["offsets"], t["sorted_token_ids"], t["sorted_weights"], t["reverse_indices"], dO)
    a = moe.moe_grouped_ffn_backward(*args)
    b = moe.moe_grouped_ffn_backward(*args)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_rejects_float32():
    moe = need_gpu()
    x = torch.zeros((4, 64), device=DEV)
    w13 = torch.zeros((2, 128, 64), device=DEV)
    w2 = torch.zeros((2, 64, 64), device=DEV)
    z = torch.zeros(8, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoeError):
        moe.moe_grouped_ffn_backward(x, w13, w2, 2, z[:2], z[:3], z, torch.zeros(8, device=DEV), z, x,
                                     workspace=torch.empty(256, dtype=torch.uint8, device=DEV))

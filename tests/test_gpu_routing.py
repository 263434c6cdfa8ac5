"""GPU parity of the routing steps against the oracle, through the C ABI.

Bit-exact: indices, multihot, position maps, counts, offsets, sorted ids,
reverse ids, sorted weights (a copy of routing weights). Routing weights:
within 1e-6 relative of the oracle's float64 value rounded to float32.
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, need_gpu
from moe_inputs import WORKLOADS, gen_logits
from oracle import align, gating, multihot

pytestmark = pytest.mark.gpu

W_RTOL = 1e-6


def _gating_case(moe, x, k, norm):
    w_ref, i_ref = gating.softmax_topk(x, k, norm)
    w, i = moe.moe_gating_softmax_topk(torch.from_numpy(x).to(DEV), k, norm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(i.cpu().numpy(), i_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=W_RTOL, atol=0)
    return w, i, w_ref, i_ref


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_gating_on_workload_logits(name):
    moe = need_gpu()
    wl = WORKLOADS[name]
    x = gen_logits(np.random.SeedSequence(wl.seed).spawn(5)[0], wl.T, wl.E, wl.logits,
                   np.random.SeedSequence(wl.seed).spawn(5)[4])
    _gating_case(moe, x, wl.k, wl.norm_topk_prob)
    _gating_case(moe, x, wl.k, not wl.norm_topk_prob)


@pytest.mark.parametrize("E,k", [(1, 1), (2, 1), (3, 2), (4, 4), (5, 5), (7, 3), (7, 7), (8, 4), (8, 6), (8, 8),
                                 (16, 4), (31, 1),
                                 (32, 32), (33, 8), (64, 4), (96, 8), (100, 6), (128, 1), (128, 8), (200, 16),
                                 (256, 8), (1000, 32), (1024, 2)])
@pytest.mark.parametrize("norm", [True, False])
def test_gating_shapes(E, k, norm):
    moe = need_gpu()
    x = gen_logits(np.random.SeedSequence(E * 1000 + k), 257, E, "distinct")
    _gating_case(moe, x, k, norm)


@pytest.mark.parametrize("E,k", [(8, 2), (64, 8), (6, 6), (40, 5)])
def test_gating_ties_go_to_lower_index(E, k):
    moe = need_gpu()
    rng = np.random.default_rng(E)
    x = (rng.integers(-2, 3, size=(300, E)) * 0.5).astype(np.float32)
    x[0] = 1.0  # a row of all-equal values
    _gating_case(moe, x, k, True)
    _gating_case(moe, x, k, False)


# bf16 logits: same indices and bit-identical weights as the float32 entry on the widened
# rows; both within 1e-6 of the oracle. Shapes cover every kernel of the dispatch, vector and
# scalar row loads (E % 8), and heavy ties (8-bit mantissas).
@pytest.mark.parametrize("E,k", [(8, 2), (6, 3), (16, 4), (36, 5), (64, 4), (64, 8), (96, 8), (100, 6),
                                 (128, 8), (256, 8), (520, 16), (1024, 32)])
@pytest.mark.parametrize("norm", [True, False])
def test_gating_bf16_logits(E, k, norm):
    moe = need_gpu()
    x = gen_logits(np.random.SeedSequence(E * 77 + k), 300, E, "plain")
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    w_ref, i_ref = gating.softmax_topk_bf16(bits, k, norm)
    w, i = moe.moe_gating_softmax_topk_bf16(xb, k, norm)
    w32, i32 = moe.moe_gating_softmax_topk(xb.float(), k, norm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(i.cpu().numpy(), i_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=W_RTOL, atol=0)
    assert torch.equal(i, i32) and torch.equal(w.view(torch.int32), w32.view(torch.int32))


# rows of at most 8 experts on enough tokens that the grid-stride kernel loops (more
# rows than 6 blocks of 256 threads per SM) with a ragged last pass; float32 and bf16
# (bit-identical to the float32 entry on the widened rows), full (E = 8) and partial rows
@pytest.mark.parametrize("E,k,norm", [(8, 2, True), (8, 3, False), (6, 2, True), (8, 8, True)])
def test_gating_small_rows_over_many_tokens(E, k, norm):
    moe = need_gpu()
    T = 400_003
    x = gen_logits(np.random.SeedSequence(E * 131 + k), T, E, "plain")
    _gating_case(moe, x, k, norm)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    w_ref, i_ref = gating.softmax_topk_bf16(bits, k, norm)
    w, i = moe.moe_gating_softmax_topk_bf16(xb, k, norm)
    w32, i32 = moe.moe_gating_softmax_topk(xb.float(), k, norm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(i.cpu().numpy(), i_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=W_RTOL, atol=0)
    assert torch.equal(i, i32) and torch.equal(w.view(torch.int32), w32.view(torch.int32))


@pytest.mark.parametrize("E,gap", [(64, 1.0), (64, 2.3), (128, 2.3), (128, 4.0)])
def test_gating_full_softmax_near_flat_rows(E, gap):
    """norm_topk_prob = False sums all E exponentials; rows whose other logits sit
    just below the maximum at a distance `gap` weigh the terms whose rounding
    grows with the distance (the worst case of the denominator's error bound)."""
    moe = need_gpu()
    rng = np.random.default_rng(E + int(gap * 10))
    x = (-gap + 0.05 * rng.standard_normal((513, E))).astype(np.float32)
    x[np.arange(513), rng.integers(0, E, 513)] = 0.0
    _gating_case(moe, x, 8, False)


def test_gating_empty_and_single():
    moe = need_gpu()
    w, i = moe.moe_gating_softmax_topk(torch.zeros((0, 8), device=DEV), 2)
    assert w.shape == (0, 2)
    _gating_case(moe, np.array([[0.5, -1.0, 3.0]], np.float32), 2, True)


@pytest.mark.parametrize("T,E,k", [(16384, 64, 8), (37, 5, 2), (37, 12, 3), (3, 1024, 32), (1000, 128, 8),
                                   (1, 4, 4), (5000, 8, 2), (333, 320, 6)])
def test_multihot_round_trip(T, E, k):
    moe = need_gpu()
    x = gen_logits(np.random.SeedSequence(T + E), T, E, "distinct")
    w_ref, i_ref = gating.softmax_topk(x, k, True)
    mh_r, pm_r, pos_r = multihot.indices_to_multihot(i_ref, w_ref, E)
    mh, pm, pos = moe.moe_indices_to_multihot(torch.from_numpy(i_ref).to(DEV),
                                              torch.from_numpy(w_ref).to(DEV), E)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(mh.cpu().numpy(), mh_r)
    np.testing.assert_array_equal(pm.cpu().numpy(), pm_r)
    np.testing.assert_array_equal(pos.cpu().numpy(), pos_r)
    p2, i2 = moe.moe_multihot_to_indices(pm, pos, k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(p2.cpu().numpy(), w_ref)
    np.testing.assert_array_equal(i2.cpu().numpy(), i_ref)


def test_multihot_page_examples(gold):
    moe = need_gpu()
    g = gold("indices_to_multihot")
    mh, pm, pos = moe.moe_indices_to_multihot(torch.tensor(g["indices"], dtype=torch.int32, device=DEV),
                                              torch.tensor(g["probs"], dtype=torch.float32, device=DEV), g["E"])
    assert mh.cpu().tolist() == g["multihot"]
    assert pos.cpu().tolist() == g["position_map"]
    np.testing.assert_array_equal(pm.cpu().numpy(), np.array(g["probs_in_multihot"], np.float32))
    g = gold("multihot_to_indices")
    p, _ = moe.moe_multihot_to_indices(torch.tensor(g["probs_in_multihot"], dtype=torch.float32, device=DEV),
                                       torch.tensor(g["position_map"], dtype=torch.int32, device=DEV), g["k"])
    np.testing.assert_array_equal(p.cpu().numpy(), np.array(g["probs"], np.float32))


def test_multihot_invalid_and_duplicate_indices():
    moe = need_gpu()
    idx = np.array([[-1, 2], [5, -7], [1, 1], [3, 0], [9, 6]], np.int32)
    pr = np.array([[0.5, 0.25], [0.1, 0.2], [0.3, 0.4], [0.6, 0.7], [0.8, 0.9]], np.float32)
    for E in (4, 5, 8, 16):   # four-wide vector, scalar and eight-wide store paths
        ref = multihot.indices_to_multihot(idx, pr, E)
        got = moe.moe_indices_to_multihot(torch.from_numpy(idx).to(DEV), torch.from_numpy(pr).to(DEV), E)
        for r, g_ in zip(ref, got):
            np.testing.assert_array_equal(g_.cpu().numpy(), r)
        rp, ri = multihot.multihot_to_indices(ref[1], ref[2], 2)
        gp, gi = moe.moe_multihot_to_indices(got[1], got[2], 2)
        np.testing.assert_array_equal(gp.cpu().numpy(), rp)
        np.testing.assert_array_equal(gi.cpu().numpy(), ri)


@pytest.mark.parametrize("E,k", [(64, 8), (320, 6)])
def test_multihot_outputs_16_byte_aligned_only(E, k):
    """Outputs on a 16- but not 32-byte boundary take the 128-bit store form."""
    moe = need_gpu()
    T = 777
    x = gen_logits(np.random.SeedSequence(E), T, E, "distinct")
    w_ref, i_ref = gating.softmax_topk(x, k, True)
    ref = multihot.indices_to_multihot(i_ref, w_ref, E)
    bufs = [torch.full((T * E + 16,), 7, dtype=dt, device=DEV) for dt in (torch.uint8, torch.float32, torch.int32)]
    n = T * E
    mh, pm, pos = (bufs[0][16:16 + n].view(T, E), bufs[1][4:4 + n].view(T, E), bufs[2][4:4 + n].view(T, E))
    assert pm.data_ptr() % 32 == 16 and pos.data_ptr() % 32 == 16
    moe.moe_indices_to_multihot(torch.from_numpy(i_ref).to(DEV), torch.from_numpy(w_ref).to(DEV), E,
                                multihot=mh, probs_in_multihot=pm, position_map=pos)
    torch.cuda.synchronize()
    for r, g_ in zip(ref, (mh, pm, pos)):
        np.testing.assert_array_equal(g_.cpu().numpy(), r)
    for b, lo in zip(bufs, (16, 4, 4)):   # nothing written outside the views
        assert (b[:lo] == 7).all() and (b[lo + n:] == 7).all()


def _align_case(moe, i_np, w_np, E):
    ref = align.align_by_expert(i_np, w_np, E)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = moe.moe_align_by_expert(torch.from_numpy(i_np).to(DEV), torch.from_numpy(w_np).to(DEV), E,
                                  status=status)
    torch.cuda.synchronize()
    n = ref["valid_slots"]
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(got["offsets"].cpu().numpy(), ref["offsets"])
    for key in ("sorted_token_ids", "sorted_weights", "reverse_indices"):
        np.testing.assert_array_equal(got[key].cpu().numpy()[:n], ref[key][:n], err_msg=key)
    return int(status.item())


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_align_on_workload_routing(name):
    moe = need_gpu()
    wl = WORKLOADS[name]
    ss = np.random.SeedSequence(wl.seed).spawn(5)
    x = gen_logits(ss[0], wl.T, wl.E, wl.logits, ss[4])
    w, i = gating.softmax_topk(x, wl.k, wl.norm_topk_prob)
    assert _align_case(moe, i, w, wl.E) == 0
    if name == "skew":
        assert (np.bincount(i.reshape(-1), minlength=wl.E) == 0).any()   # empty experts exercised


@pytest.mark.parametrize("T,E,k", [(0, 8, 2), (1, 8, 8), (4095, 3, 1), (4096, 7, 2), (4097, 64, 8),
                                   (9000, 1024, 4), (50000, 16, 2), (3, 1, 1)])
def test_align_shapes(T, E, k):
    moe = need_gpu()
    x = gen_logits(np.random.SeedSequence(T * 3 + E), T, E, "distinct")
    w, i = gating.softmax_topk(x, k, True) if T else (np.zeros((0, k), np.float32), np.zeros((0, k), np.int32))
    assert _align_case(moe, i, w, E) == 0


def test_align_all_to_one_expert_and_page_example(gold):
    moe = need_gpu()
    T, E = 10000, 16
    i = np.zeros((T, 1), np.int32) + 11
    w = np.random.default_rng(0).random((T, 1)).astype(np.float32)
    assert _align_case(moe, i, w, E) == 0
    g = gold("moe_cumsum")
    i = np.array(g["indices"], np.int32)
    assert _align_case(moe, i, np.ones(i.shape, np.float32), g["E"]) == 0


def test_align_repeated_expert_in_a_row_k8():
    """Rows naming an expert twice are outside what top-k routing produces (the
    oracle's reading); the k = 8 ranking detects them and falls back to the
    general ranking, so the result is still the stable sort of the slots by
    expert: checked against numpy's stable argsort on chunks with and without
    repeats."""
    moe = need_gpu()
    T, E, k = 3000, 64, 8
    rng = np.random.default_rng(5)
    i = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    i[700, 3] = i[700, 1]          # a repeat in chunk 1 (tokens 512..1023)
    i[10, 7] = i[10, 0]            # and one in chunk 0; chunks 2.. have none
    w = rng.random((T, k)).astype(np.float32)
    got = moe.moe_align_by_expert(torch.from_numpy(i).to(DEV), torch.from_numpy(w).to(DEV), E)
    torch.cuda.synchronize()
    flat = i.reshape(-1)
    order = np.argsort(flat, kind="stable")
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(got["reverse_indices"].cpu().numpy(), order)
    np.testing.assert_array_equal(got["sorted_token_ids"].cpu().numpy(), order // k)
    np.testing.assert_array_equal(got["sorted_weights"].cpu().numpy(), w.reshape(-1)[order])


def test_align_invalid_index_sets_status_and_drops_slot():
    moe = need_gpu()
    for T in (3, 6000):    # single-chunk and multi-chunk launches
        i = np.tile(np.array([[0, 9], [-1, 1], [1, 0]], np.int32), (T // 3, 1))
        w = np.ones(i.shape, np.float32)
        st = _align_case(moe, i, w, 3)
        assert st & moe.MOE_STATUS_BAD_INDEX


# ---- group-limited top-k ------------------------------------------------------------

def _group_case(moe, x, bias, k, n_group, topk_group, method):
    w_ref, i_ref = gating.group_limited_topk(x, k, n_group, topk_group, method, bias)
    b = torch.from_numpy(bias).to(DEV) if bias is not None else None
    w, i = moe.moe_group_limited_topk(torch.from_numpy(x).to(DEV), k, n_group, topk_group, method, bias=b)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(i.cpu().numpy(), i_ref)
    np.testing.assert_array_equal(w.cpu().numpy(), w_ref)     # weights are copies of input scores


def _sigmoid_scores(T, E, seed):
    x = gen_logits(np.random.SeedSequence(seed), T, E, "distinct").astype(np.float64)
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


@pytest.mark.parametrize("T,E,k,n_group,topk_group", [
    (4096, 256, 8, 8, 4),      # DeepSeek-V3-shaped routing
    (40000, 256, 8, 8, 4),     # more token groups than resident blocks: the persistent loop
    (3000, 160, 6, 8, 3),      # DeepSeek-V2-shaped routing
    (777, 64, 6, 8, 3), (100, 8, 2, 4, 2), (50, 1024, 32, 32, 7), (1, 256, 8, 8, 4), (0, 256, 8, 8, 4),
    (64, 96, 4, 3, 1), (64, 32, 3, 16, 2),
    (300, 512, 8, 4, 2),       # groups of 128 experts: warp-per-token form
    (200, 320, 6, 10, 4),      # E > 256 with groups of 32: lane-per-group form
    (70, 64, 4, 2, 1), (90, 128, 8, 4, 3), (33, 512, 16, 16, 5),   # more groups of 32
])
@pytest.mark.parametrize("method", ["group_limited_greedy", "noaux_tc"])
def test_group_limited_topk(T, E, k, n_group, topk_group, method):
    moe = need_gpu()
    x = _sigmoid_scores(T, E, T + E)
    bias = (gen_logits(np.random.SeedSequence(E), 1, E, "distinct")[0] * np.float32(0.05)).astype(np.float32)
    _group_case(moe, x, bias if method == "noaux_tc" else None, k, n_group, topk_group, method)


@pytest.mark.parametrize("method", ["group_limited_greedy", "noaux_tc"])
def test_group_limited_topk_ties_and_golden(method, gold):
    moe = need_gpu()
    rng = np.random.default_rng(4)
    x = (rng.integers(0, 4, size=(500, 48)) * 0.25).astype(np.float32)
    bias = (rng.integers(-1, 2, size=48) * 0.25).astype(np.float32)
    _group_case(moe, x, bias, 5, 6, 3, method)
    # groups of 32 with ties inside groups, between group scores and between experts
    x = (rng.integers(0, 4, size=(700, 256)) * 0.25).astype(np.float32)
    bias = (rng.integers(-1, 2, size=256) * 0.25).astype(np.float32)
    _group_case(moe, x, bias, 8, 8, 4, method)
    g = gold("group_limited_topk")
    x = np.array(g["scores"], np.float32)
    _group_case(moe, x, np.array(g["bias"], np.float32), g["k"], g["n_group"], g["topk_group"], method)


def test_group_limited_topk_rejects_bad_arguments():
    moe = need_gpu()
    x = torch.rand((4, 256), device=DEV)
    with pytest.raises(moe.MoeError):
        moe.moe_group_limited_topk(x, 8, 7, 3)                      # 7 does not divide 256
    with pytest.raises(moe.MoeError):
        moe.moe_group_limited_topk(x, 8, 8, 4, "noaux_tc")          # no bias
    with pytest.raises(moe.MoeError):
        moe.moe_group_limited_topk(x, 100, 8, 1)                    # k > topk_group * group size


def test_converter_backward_on_dense_gradient():
    """The converter's backward is the inverse kernel applied to the upstream gradient
    (Megatron-LM IndicesToMultihot.backward); checked with a dense gradient."""
    moe = need_gpu()
    T, E, k = 3000, 64, 8
    x = gen_logits(np.random.SeedSequence(77), T, E, "distinct")
    w, i = gating.softmax_topk(x, k, True)
    _, _, pos = multihot.indices_to_multihot(i, w, E)
    grad = np.random.default_rng(6).standard_normal((T, E)).astype(np.float32)
    ref, _ = multihot.multihot_to_indices(grad, pos, k)
    got, _ = moe.moe_multihot_to_indices(torch.from_numpy(grad).to(DEV), torch.from_numpy(pos).to(DEV), k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), ref)

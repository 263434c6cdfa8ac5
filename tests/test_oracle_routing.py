"""Pins for the multihot and align oracles (CPU only)."""
import numpy as np
import pytest

from oracle import align, gating, multihot
from moe_inputs import gen_logits


def test_indices_to_multihot_golden(gold):
    g = gold("indices_to_multihot")
    mh, pm, pos = multihot.indices_to_multihot(np.array(g["indices"]), np.array(g["probs"], np.float32), g["E"])
    assert mh.tolist() == g["multihot"]
    np.testing.assert_array_equal(pm, np.array(g["probs_in_multihot"], np.float32))
    assert pos.tolist() == g["position_map"]


def test_multihot_to_indices_golden(gold):
    g = gold("multihot_to_indices")
    p, i = multihot.multihot_to_indices(np.array(g["probs_in_multihot"], np.float32),
                                        np.array(g["position_map"]), g["k"])
    np.testing.assert_array_equal(p, np.array(g["probs"], np.float32))
    assert i.tolist() == [[0, 1], [1, 2]]


@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (64, 8), (128, 8), (7, 7), (9, 1)])
def test_multihot_round_trip(E, k):
    x = gen_logits(np.random.SeedSequence(E * 100 + k), 300, E, "distinct")
    w, i = gating.softmax_topk(x, k, True)
    mh, pm, pos = multihot.indices_to_multihot(i, w, E)
    assert (mh.sum(1) == k).all()
    assert ((pos >= 0) == (mh == 1)).all()
    np.testing.assert_array_equal(pm.sum(1, dtype=np.float64), w.sum(1, dtype=np.float64))
    p2, i2 = multihot.multihot_to_indices(pm, pos, k)
    np.testing.assert_array_equal(p2, w)
    np.testing.assert_array_equal(i2, i)


def test_multihot_invalid_and_duplicate_indices():
    idx = np.array([[-1, 2], [5, -7], [1, 1]])
    pr = np.array([[0.5, 0.25], [0.1, 0.2], [0.3, 0.4]], np.float32)
    mh, pm, pos = multihot.indices_to_multihot(idx, pr, 4)
    assert mh.tolist() == [[0, 0, 1, 0], [0, 0, 0, 0], [0, 1, 0, 0]]
    assert pos.tolist() == [[-1, -1, 1, -1], [-1, -1, -1, -1], [-1, 0, -1, -1]]
    assert pm[2].tolist() == [0.0, np.float32(0.3), 0.0, 0.0]
    p2, i2 = multihot.multihot_to_indices(pm, pos, 2)
    assert i2.tolist() == [[-1, 2], [-1, -1], [1, -1]]
    assert p2.tolist() == [[0.0, 0.25], [0.0, 0.0], [np.float32(0.3), 0.0]]


def test_moe_cumsum_golden(gold):
    g = gold("moe_cumsum")
    idx = np.array(g["indices"])
    E = g["E"]
    cs = align.moe_cumsum(idx, E)
    assert cs.reshape(E, -1).tolist() == g["cumsum_2d"]
    assert align.get_indptr(cs, E, idx.shape[0]).tolist() == g["indptr_exclusive"]
    rev, tok, _ = align.get_indices(cs, idx, E)
    assert rev.tolist() == g["reverse_indices"]
    assert tok.tolist() == g["token_indices"]
    al = align.align_by_expert(idx, np.arange(8, dtype=np.float32).reshape(4, 2), E)
    assert al["counts"].tolist() == g["counts"]
    # the weight of slot (b, j) travels with it: weight value == b*k + j == reverse index
    assert al["sorted_weights"].tolist() == [float(r) for r in g["reverse_indices"]]


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (13, 8, 2), (200, 64, 8), (64, 128, 8), (33, 5, 5)])
def test_align_matches_stable_sort_and_invariants(T, E, k):
    x = gen_logits(np.random.SeedSequence(T + 7 * E + k), T, E, "distinct")
    w, i = gating.softmax_topk(x, k, True)
    al = align.align_by_expert(i, w, E)
    S = T * k
    # brute force: a stable sort of the flattened slots by expert id gives the same order
    order = np.argsort(i.reshape(-1), kind="stable")
    np.testing.assert_array_equal(al["reverse_indices"], order)
    np.testing.assert_array_equal(al["sorted_token_ids"], order // k)
    np.testing.assert_array_equal(al["sorted_weights"], w.reshape(-1)[order])
    assert al["counts"].sum() == S and al["valid_slots"] == S
    assert al["offsets"][0] == 0 and (np.diff(al["offsets"]) == al["counts"]).all()
    assert np.array_equal(np.sort(al["reverse_indices"]), np.arange(S))
    np.testing.assert_array_equal(al["counts"], np.bincount(i.reshape(-1), minlength=E))
    for e in range(E):
        seg = al["sorted_token_ids"][al["offsets"][e]:al["offsets"][e + 1]]
        assert (np.diff(seg) > 0).all()


def test_align_drops_invalid_slots():
    idx = np.array([[0, 9], [-1, 1], [1, 0]])
    al = align.align_by_expert(idx, np.ones((3, 2), np.float32), 3)
    assert al["counts"].tolist() == [2, 2, 0]
    assert al["valid_slots"] == 4
    assert al["reverse_indices"][:4].tolist() == [0, 5, 3, 4]
    assert al["sorted_token_ids"][:4].tolist() == [0, 2, 1, 2]


def test_align_empty():
    al = align.align_by_expert(np.zeros((0, 2), np.int32), np.zeros((0, 2), np.float32), 4)
    assert al["counts"].tolist() == [0, 0, 0, 0] and al["offsets"].tolist() == [0] * 5


def test_converter_backward_is_the_inverse_map_on_the_gradient():
    """Megatron-LM IndicesToMultihot.backward: grad of probs_in_multihot -> grad of the
    [T, k] probs through the saved position map. Pinned against torch autograd of the
    forward scatter (a library differentiation, independent of the oracle)."""
    import torch
    x = gen_logits(np.random.SeedSequence(41), 50, 12, "distinct")
    w, i = gating.softmax_topk(x, 3, True)
    _, _, pos = multihot.indices_to_multihot(i, w, 12)
    grad = np.random.default_rng(5).standard_normal((50, 12)).astype(np.float32)   # dense upstream grad
    probs = torch.tensor(w, requires_grad=True)
    pm = torch.zeros((50, 12)).scatter(1, torch.tensor(i, dtype=torch.int64), probs)
    pm.backward(torch.tensor(grad))
    got, _ = multihot.multihot_to_indices(grad, pos, 3)
    np.testing.assert_array_equal(got, probs.grad.numpy())

"""Pins for the gating oracle (CPU only).

The oracle writes top-k as a stable sort; these tests hold it to the page's
own insertion procedure, hand-computed closed forms, a library softmax and
invariants.
"""
import itertools

import numpy as np
import pytest
import scipy.special

from oracle import gating
from moe_inputs import gen_logits

FLT_MIN_VALUE = -3.4028234663852886e38   # lowest finite float32, the page's initial slot value


def insertion_topk(row, k):
    """The page's procedure for one row: k slots start at the lowest float32 value; each
    candidate, scanned in expert order, goes into the first slot it strictly exceeds and
    pushes the later slots down one place."""
    vals = [FLT_MIN_VALUE] * k
    idx = list(range(k))
    for e, x in enumerate(row):
        for i in range(k):
            if x > vals[i]:
                vals[i + 1:] = vals[i:k - 1]
                idx[i + 1:] = idx[i:k - 1]
                vals[i] = x
                idx[i] = e
                break
    return vals, idx


def brute_topk(row, k):
    """Exhaustive: the ordered k-tuple of distinct experts that is lexicographically best
    under (value descending, index ascending) at every position."""
    best = None
    for combo in itertools.permutations(range(len(row)), k):
        key = [(-row[e], e) for e in combo]
        if best is None or key < best[0]:
            best = (key, combo)
    return list(best[1])


def test_ties_golden(gold):
    g = gold("topk_ties")
    v, i = gating.topk(np.array(g["scores"], dtype=np.float32), 3)
    assert i.tolist() == g["k3_indices"]
    assert v.tolist() == g["k3_values"]


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_insertion_procedure(seed):
    rng = np.random.default_rng(seed)
    for E in (1, 2, 3, 5, 8, 13, 16):
        for k in sorted({1, 2, min(E, 3), E}):
            if k > E:
                continue
            # coarse values force many ties
            x = rng.integers(-3, 4, size=(20, E)).astype(np.float32) * np.float32(0.5)
            v, i = gating.topk(x, k)
            for r in range(x.shape[0]):
                pv, pi = insertion_topk(x[r].tolist(), k)
                assert i[r].tolist() == pi
                assert v[r].tolist() == pv


def test_topk_matches_brute_force():
    rng = np.random.default_rng(7)
    for E, k in [(4, 2), (5, 3), (6, 2), (6, 6)]:
        x = rng.integers(-2, 3, size=(30, E)).astype(np.float32)
        _, i = gating.topk(x, k)
        for r in range(x.shape[0]):
            assert i[r].tolist() == brute_topk(x[r].tolist(), k)


def test_softmax_topk_closed_forms(gold):
    g = gold("softmax_topk_closed_form")
    x = np.array(g["logits"], dtype=np.float32)
    w, i = gating.softmax_topk(x, g["k"], True)
    assert i.tolist() == g["indices"]
    np.testing.assert_allclose(w, np.array(g["weights_norm_true"], np.float32), rtol=1e-7)
    w, i = gating.softmax_topk(x, g["k"], False)
    assert i.tolist() == g["indices"]
    np.testing.assert_allclose(w, np.array(g["weights_norm_false"], np.float32), rtol=1e-7)


@pytest.mark.parametrize("E,k", [(8, 2), (64, 8), (128, 8), (5, 5)])
def test_softmax_topk_against_library_softmax(E, k):
    x = gen_logits(np.random.SeedSequence(11), 200, E, "distinct")
    ref = scipy.special.softmax(x.astype(np.float64), axis=1)
    w, i = gating.softmax_topk(x, k, False)
    np.testing.assert_allclose(w, np.take_along_axis(ref, i, 1).astype(np.float32), rtol=1e-7)
    # norm=True with k=E: the full softmax listed in descending order
    wf, iF = gating.softmax_topk(x, E, True)
    np.testing.assert_allclose(wf, np.take_along_axis(ref, iF, 1).astype(np.float32), rtol=1e-6)
    assert (np.diff(np.take_along_axis(x, iF, 1), axis=1) < 0).all()


@pytest.mark.parametrize("norm", [True, False])
def test_softmax_topk_invariants(norm):
    x = gen_logits(np.random.SeedSequence(3), 500, 64, "distinct")
    w, i = gating.softmax_topk(x, 8, norm)
    assert i.dtype == np.int32 and w.dtype == np.float32
    assert ((i >= 0) & (i < 64)).all()
    assert all(len(set(r)) == 8 for r in i.tolist())
    assert (np.diff(w.astype(np.float64), axis=1) <= 0).all()      # descending weights
    s = w.astype(np.float64).sum(1)
    if norm:
        np.testing.assert_allclose(s, 1.0, atol=1e-6)
    else:
        assert (s < 1.0 + 1e-6).all()
    # chosen experts beat every unchosen one
    vals = np.take_along_axis(x, i, 1)
    mask = np.ones_like(x, bool)
    np.put_along_axis(mask, i.astype(np.int64), False, 1)
    rest = np.where(mask, x, -np.inf).max(1)
    assert (vals[:, -1] > rest).all()


def test_softmax_topk_shift_invariance():
    x = gen_logits(np.random.SeedSequence(5), 64, 16, "distinct").astype(np.float64)
    w0, i0 = gating.softmax_topk(x.astype(np.float32), 4, True)
    w1, i1 = gating.softmax_topk((x + 8.0).astype(np.float32), 4, True)
    assert (i0 == i1).all()
    np.testing.assert_allclose(w0, w1, rtol=5e-6)


def test_rejects_non_finite_and_bad_k():
    with pytest.raises(ValueError):
        gating.softmax_topk(np.array([[0.0, np.inf]], np.float32), 1)
    with pytest.raises(ValueError):
        gating.topk(np.zeros((2, 3), np.float32), 4)


# ---- group-limited greedy / noaux_tc top-k ------------------------------------------

def _page_group_limited(row, k, n_group, topk_group, method, bias):
    """The page's steps for one row, written with the insertion top-k above."""
    row = [np.float32(v) for v in row]
    choice = row if method != "noaux_tc" else [np.float32(a + np.float32(b)) for a, b in zip(row, bias)]
    gs = len(row) // n_group
    gscore = []
    for g in range(n_group):
        grp = choice[g * gs:(g + 1) * gs]
        if method == "noaux_tc":
            v, _ = insertion_topk(grp, 2)
            gscore.append(np.float32(v[0] + v[1]))
        else:
            gscore.append(max(grp))
    _, gsel = insertion_topk(gscore, topk_group)
    masked = [FLT_MIN_VALUE] * len(row)
    for g in gsel:
        for c in range(gs):
            masked[g * gs + c] = choice[g * gs + c]
    v, i = insertion_topk(masked, k)
    if method == "noaux_tc":
        v = [row[e] for e in i]
    return [float(x) for x in v], i


def test_group_limited_golden(gold):
    g = gold("group_limited_topk")
    x = np.array(g["scores"], np.float32)
    w, i = gating.group_limited_topk(x, g["k"], g["n_group"], g["topk_group"], "group_limited_greedy")
    assert i.tolist() == g["greedy_indices"]
    np.testing.assert_array_equal(w, np.array(g["greedy_weights"], np.float32))
    w, i = gating.group_limited_topk(x, g["k"], g["n_group"], g["topk_group"], "noaux_tc", np.zeros(8, np.float32))
    assert i.tolist() == g["noaux_zero_bias_indices"]
    np.testing.assert_array_equal(w, np.array(g["noaux_zero_bias_weights"], np.float32))
    w, i = gating.group_limited_topk(x, g["k"], g["n_group"], g["topk_group"], "noaux_tc",
                                     np.array(g["bias"], np.float32))
    assert i.tolist() == g["noaux_bias_indices"]
    np.testing.assert_array_equal(w, np.array(g["noaux_bias_weights"], np.float32))


@pytest.mark.parametrize("method", ["group_limited_greedy", "noaux_tc"])
@pytest.mark.parametrize("E,n_group,topk_group,k", [(8, 4, 2, 2), (12, 3, 2, 5), (16, 8, 3, 4), (12, 6, 6, 3)])
def test_group_limited_matches_page_steps(method, E, n_group, topk_group, k):
    rng = np.random.default_rng(E * 31 + k)
    x = (rng.integers(0, 5, size=(40, E)) * 0.25).astype(np.float32)   # coarse: many ties
    bias = (rng.integers(-2, 3, size=E) * 0.125).astype(np.float32)
    w, i = gating.group_limited_topk(x, k, n_group, topk_group, method, bias)
    for r in range(x.shape[0]):
        pw, pi = _page_group_limited(x[r].tolist(), k, n_group, topk_group, method, bias.tolist())
        assert i[r].tolist() == pi
        assert w[r].tolist() == [float(np.float32(v)) for v in pw]


@pytest.mark.parametrize("method", ["group_limited_greedy", "noaux_tc"])
def test_group_limited_reduces_to_plain_topk(method):
    x = gen_logits(np.random.SeedSequence(9), 100, 32, "distinct")
    z = np.zeros(32, np.float32)
    for n_group, topk_group in [(1, 1), (4, 4), (16, 16)]:
        w, i = gating.group_limited_topk(x, 6, n_group, topk_group, method, z)
        v, j = gating.topk(x, 6)
        np.testing.assert_array_equal(i, j)
        np.testing.assert_array_equal(w, v)


def test_group_limited_choice_stays_in_kept_groups():
    x = gen_logits(np.random.SeedSequence(2), 300, 256, "distinct")
    bias = gen_logits(np.random.SeedSequence(3), 1, 256, "distinct")[0] * np.float32(0.1)
    w, i = gating.group_limited_topk(x, 8, 8, 4, "noaux_tc", bias)
    groups = i // 32
    assert all(len(set(r)) <= 4 for r in groups.tolist())
    np.testing.assert_array_equal(w, np.take_along_axis(x, i.astype(np.int64), 1))
    with pytest.raises(ValueError):
        gating.group_limited_topk(x, 200, 8, 4, "noaux_tc", bias)
    with pytest.raises(ValueError):
        gating.group_limited_topk(x, 4, 256, 4, "noaux_tc", bias)      # one expert per group


# ---- bf16 logits ------------------------------------------------------------------------

def test_bf16_widening_matches_known_bit_patterns():
    """bf16 bit patterns with textbook values: 1.0, -2.0, 0.5, the largest finite bf16,
    the smallest normal, and a value whose float32 tail is zero by definition."""
    bits = np.array([0x3F80, 0xC000, 0x3F00, 0x7F7F, 0x0080, 0x4049], np.uint16)
    want = [1.0, -2.0, 0.5, 3.3895313892515355e38, 2.0 ** -126, 3.140625]
    assert gating.bf16_bits_as_float32(bits).astype(np.float64).tolist() == want


def test_bf16_topk_ties_follow_the_insertion_procedure():
    """Coarse bf16 values tie often; the order must be the page's insertion procedure."""
    rng = np.random.default_rng(4)
    for E, k in [(8, 2), (16, 4), (12, 12)]:
        x = (rng.integers(-4, 5, size=(30, E)) * 0.25).astype(np.float32)
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)          # exact: x has short mantissas
        w, i = gating.softmax_topk_bf16(bits, k, True)
        for r in range(x.shape[0]):
            _, pi = insertion_topk(x[r].tolist(), k)
            assert i[r].tolist() == pi
        np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)

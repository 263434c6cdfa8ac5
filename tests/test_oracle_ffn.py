"""Pins for the FFN oracle (CPU only).

The pages print no numeric FFN example, so the oracle is pinned by: a
hand-evaluated scalar closed form (which also fixes which half of ``w13`` is
gated), agreement between the page's decode form (loop over one token's k
experts) and its prefill form (loop over experts, scatter, sum over k),
linearity and permutation properties, and the bf16 rounding against two
independent implementations.
"""
import math

import numpy as np
import pytest
import torch

from oracle import align, ffn, gating
from moe_inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_layer_inputs


def test_scalar_closed_form(gold):
    g = gold("ffn_scalar_closed_form")
    x = np.array([[g["x"]]], np.float32)
    w13 = np.array([g["w13"]], np.float32)
    w2 = np.array([g["w2"]], np.float32)
    res = ffn.layer_forward(np.array([[0.0]], np.float32), x, w13, w2, 1, True, "f32")
    assert res["topk_weights"].tolist() == [[1.0]]
    assert res["out"][0, 0] == pytest.approx(g["out"], rel=1e-7)
    assert abs(res["out"][0, 0] - g["out_if_halves_swapped"]) > 0.5


def test_silu_values():
    z = np.array([0.0, 1.0, -1.0, 3.0, -40.0, 800.0, -800.0])
    s = ffn.silu(z)
    assert s[0] == 0.0
    assert s[1] == pytest.approx(0.7310585786300049, rel=1e-15)
    assert s[1] - s[2] == pytest.approx(1.0, rel=1e-15)   # silu(z) - silu(-z) = z
    assert s[5] == 800.0 and s[6] == 0.0
    assert s[4] == pytest.approx(-40.0 * math.exp(-40.0), rel=1e-12)


def test_bf16_round_against_bit_definition_and_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, 3.3895e38, 3.4e38], np.float32),
    ])
    ours = ffn.bf16_round(x.astype(np.float64))
    bits = bf16_bits_to_f32(f32_to_bf16_bits(x)).astype(np.float64)
    np.testing.assert_array_equal(ours, bits)
    tch = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, tch)
    assert ours[-6] == 1.0 and ours[-5] == 1 + 2 ** -6


def _small(dtype, T=24, H=16, I=12, E=5, k=2, seed=1, norm=True):
    return make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=norm, dtype=dtype,
                             logits="distinct", seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k,norm", [(1, True), (2, True), (3, False), (5, True)])
def test_decode_form_equals_prefill_form(dtype, k, norm):
    d = _small(dtype, k=k, norm=norm)
    res = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], k, norm, dtype)
    for t in range(d["T"]):
        ref = ffn.decode_form(d["hidden"][t], d["w13"], d["w2"], dtype,
                              res["topk_indices"][t], res["topk_weights"][t])
        np.testing.assert_allclose(res["out"][t], ref, rtol=1e-12, atol=1e-12)


def test_output_is_linear_in_w2_and_token_permutation_equivariant():
    d = _small("f32", T=30, k=3)
    res = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], 3, True, "f32")
    res2 = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"] * np.float32(2.0), 3, True, "f32")
    np.testing.assert_allclose(res2["out"], 2.0 * res["out"], rtol=1e-6)
    perm = np.random.default_rng(3).permutation(30)
    res3 = ffn.layer_forward(d["logits"][perm], d["hidden"][perm], d["w13"], d["w2"], 3, True, "f32")
    np.testing.assert_allclose(res3["out"], res["out"][perm], rtol=1e-12)


def test_up_half_zero_gives_zero_and_gate_half_matters():
    d = _small("f32", T=8, k=2)
    w13 = d["w13"].copy()
    I = w13.shape[1] // 2
    w13[:, I:, :] = 0
    res = ffn.layer_forward(d["logits"], d["hidden"], w13, d["w2"], 2, True, "f32")
    assert np.all(res["out"] == 0)
    # a very negative gate drives silu to 0 whatever the up half is
    w13 = d["w13"].copy()
    w13[:, :I, :] = 0
    x = d["hidden"].copy()
    res = ffn.layer_forward(d["logits"], x, w13, d["w2"], 2, True, "f32")
    assert np.all(res["out"] == 0)


def test_layer_rows_equals_full_layer():
    d = _small("bf16", T=40, E=6, k=2)
    res = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], 2, True, "bf16")
    tok = np.array([39, 0, 17, 5])
    rows = ffn.layer_rows(d["hidden"], d["w13"], d["w2"], "bf16", res["topk_weights"],
                          res["topk_indices"], tok)
    np.testing.assert_array_equal(rows, res["out"][tok])


def test_bf16_outputs_are_bf16_values():
    d = _small("bf16")
    res = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], 2, True, "bf16")
    o = res["out"]
    np.testing.assert_array_equal(ffn.bf16_round(o), o)


def test_empty_experts_and_zero_tokens():
    d = _small("f32", T=3, E=16, k=1)
    res = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], 1, True, "f32")
    assert (res["counts"] == 0).sum() >= 13
    z = ffn.layer_forward(np.zeros((0, 4), np.float32), np.zeros((0, 8), np.float32),
                          np.zeros((4, 6, 8), np.float32), np.zeros((4, 8, 3), np.float32), 2, True, "f32")
    assert z["out"].shape == (0, 8)


def _torch_token_major_forward(d, w, idx):
    """An independent float64 forward, token-major: for every token and each of its k
    slots, gather the slot's expert weights and evaluate silu(W1 x) * (W3 x), W2, the
    routing weight and the running sum with torch einsums. No align step, no expert
    loop, no scatter: it shares with the oracle only the input decoding (to_f64) and
    the bf16 rounding (pinned on its own above)."""
    dt = d["dtype"]
    x = torch.tensor(ffn.to_f64(d["hidden"], dt))
    W13 = torch.tensor(ffn.to_f64(d["w13"], dt))
    W2 = torch.tensor(ffn.to_f64(d["w2"], dt))
    I = d["I"]
    ii = torch.tensor(idx, dtype=torch.int64)
    wt = torch.tensor(np.asarray(w, np.float32).astype(np.float64))
    out = torch.zeros((x.shape[0], x.shape[1]), dtype=torch.float64)
    for j in range(idx.shape[1]):
        e = ii[:, j]
        g = torch.einsum("th,tih->ti", x, W13[e, :I])
        u = torch.einsum("th,tih->ti", x, W13[e, I:])
        a = (torch.nn.functional.silu(g) * u).numpy()
        if dt == "bf16":
            a = ffn.bf16_round(a)
        out = out + wt[:, j:j + 1] * torch.einsum("ti,thi->th", torch.tensor(a), W2[e])
    out = out.numpy()
    return ffn.bf16_round(out) if dt == "bf16" else out.astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,H,I,E,k,norm", [(37, 24, 40, 6, 3, False), (64, 128, 96, 8, 2, True),
                                            (19, 16, 8, 16, 4, True)])
def test_layer_forward_matches_an_independent_token_major_forward(dtype, T, H, I, E, k, norm):
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=norm, dtype=dtype, logits="distinct",
                          seed=T + H + I)
    res = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], k, norm, dtype)
    ref = _torch_token_major_forward(d, res["topk_weights"], res["topk_indices"])
    assert np.abs(ref).max() > 0
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-300)

"""Oracle: gating top-k and softmax (test infrastructure only).

Source: mlc-llm ``moe_misc.py`` — ``gating_topk`` with its helpers
``_gating_topk_init_local_top_k`` / ``_gating_topk_process_value``, and
``gating_softmax_topk`` (both the ``norm_topk_prob`` branch and the
full-softmax branch).

What the page computes, restated:

* top-k keeps, per row, the ``k`` largest values in descending order. A
  candidate displaces a kept value only when it is strictly greater, so of two
  equal values the one with the lower expert index ranks first. That is the
  same as a stable sort of the row by descending value; the oracle writes it
  that way (a library stable sort is the step);
* ``norm_topk_prob=True``: softmax over the ``k`` selected values only,
  ``w_j = exp(l_j - m) / sum_i exp(l_i - m)`` with ``m`` the largest selected;
* ``norm_topk_prob=False``: softmax over the whole row, then top-k of the
  probabilities. Softmax is strictly increasing in the logit, so the selected
  experts and their order are those of the logits; the weights are the full
  softmax probabilities at the selected experts.

Arithmetic is float64, rounded once to float32 (the logits' dtype, the page
casts back to it). Logits must be finite.

``gating_softmax_topk`` is written for any logits dtype. For bf16 logits
(``softmax_topk_bf16``) the reading is: each bf16 value is exactly a float32
value (its 16 bits followed by 16 zero bits), and the result is the float32
computation on those values, with the weights kept in float32 (the dtype the
align and FFN steps take) rather than cast back to bf16.
"""
from __future__ import annotations

import numpy as np

__all__ = ["topk", "softmax_topk", "softmax_topk_bf16", "bf16_bits_as_float32", "group_limited_topk",
           "FLOAT32_LOWEST"]

FLOAT32_LOWEST = np.float32(np.finfo(np.float32).min)


def topk(scores: np.ndarray, k: int):
    """``gating_topk``: (values [T,k], indices [T,k] int32), descending, ties to lower index."""
    scores = np.asarray(scores)
    T, E = scores.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # stable ascending sort of the negated row == descending with lower index first on ties
    order = np.argsort(-scores, axis=1, kind="stable")[:, :k].astype(np.int32)
    return np.take_along_axis(scores, order, axis=1), order


def softmax_topk(logits: np.ndarray, k: int, norm_topk_prob: bool = True):
    """``gating_softmax_topk``: (weights [T,k] float32, indices [T,k] int32)."""
    x = np.asarray(logits, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("logits must be finite")
    vals, idx = topk(x, k)
    v = vals.astype(np.float64)
    if norm_topk_prob:
        m = v.max(axis=1, keepdims=True)
        ex = np.exp(v - m)
        w = ex / ex.sum(axis=1, keepdims=True)
    else:
        full = x.astype(np.float64)
        m = full.max(axis=1, keepdims=True)
        ex = np.exp(full - m)
        prob = ex / ex.sum(axis=1, keepdims=True)
        w = np.take_along_axis(prob, idx, axis=1)
    return w.astype(np.float32), idx


def bf16_bits_as_float32(bits: np.ndarray) -> np.ndarray:
    """bf16 values given as uint16 bit patterns -> the equal float32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def softmax_topk_bf16(logit_bits: np.ndarray, k: int, norm_topk_prob: bool = True):
    """``gating_softmax_topk`` on bf16 logits (uint16 bits): float32 weights, int32 indices."""
    return softmax_topk(bf16_bits_as_float32(logit_bits), k, norm_topk_prob)


def group_limited_topk(scores: np.ndarray, k: int, n_group: int, topk_group: int,
                       method: str = "group_limited_greedy", bias: np.ndarray | None = None):
    """``group_limited_greedy_topk`` (mlc-llm ``moe_misc.py``): (weights [T,k] f32, indices [T,k] i32).

    Steps, as the page takes them (all on float32 tensors, the page asserts
    float32 scores):

    1. scores for choice: the scores, plus ``bias`` for ``noaux_tc``;
    2. experts are cut into ``n_group`` groups of ``E / n_group`` consecutive
       experts; a group's score is its largest choice score
       (``group_limited_greedy``) or the sum of its two largest (``noaux_tc``);
    3. the ``topk_group`` best groups are kept (top-k rule: descending, ties to
       the lower group index);
    4. choice scores outside the kept groups become the lowest float32 value;
    5. top-k of the result; the weights are those values (``group_limited_greedy``)
       or the un-biased scores of the chosen experts (``noaux_tc``).

    Needs ``k <= topk_group * E / n_group`` so that only kept experts are chosen,
    and, for ``noaux_tc``, at least two experts per group (the page takes a
    top-2 inside each group).
    """
    s32 = np.asarray(scores, dtype=np.float32)
    T, E = s32.shape
    if E % n_group or not 1 <= topk_group <= n_group or not 1 <= k <= topk_group * (E // n_group):
        raise ValueError("need E % n_group == 0, 1 <= topk_group <= n_group, 1 <= k <= topk_group*E/n_group")
    if method not in ("group_limited_greedy", "noaux_tc"):
        raise ValueError(f"unknown method {method!r}")
    choice = s32
    if method == "noaux_tc":
        if bias is None:
            raise ValueError("noaux_tc needs a bias")
        choice = (s32 + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    gs = E // n_group
    if method == "noaux_tc" and gs < 2:
        raise ValueError("noaux_tc needs at least two experts per group")
    grouped = choice.reshape(T * n_group, gs)
    if method == "noaux_tc":
        top2 = topk(grouped, 2)[0].astype(np.float32)
        gscore = top2[:, 0] + top2[:, 1]                                    # float32 sum of the two
    else:
        gscore = grouped.max(axis=1)
    gscore = np.asarray(gscore, dtype=np.float32).reshape(T, n_group)
    gidx = topk(gscore, topk_group)[1]
    masked = np.full((T, E), FLOAT32_LOWEST, dtype=np.float32)
    for j in range(topk_group):
        for c in range(gs):
            col = gidx[:, j].astype(np.int64) * gs + c
            masked[np.arange(T), col] = choice[np.arange(T), col]
    vals, idx = topk(masked, k)
    if method == "noaux_tc":
        vals = np.take_along_axis(s32, idx.astype(np.int64), axis=1)
    return vals.astype(np.float32), idx

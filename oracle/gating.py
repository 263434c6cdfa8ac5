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
"""
from __future__ import annotations

import numpy as np

__all__ = ["topk", "softmax_topk"]


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

"""Oracle: expert FFN, weighting and the sum over k (test infrastructure only).

Sources:

* project_6 ``moe_expert_gemm.cpp`` — ``moe_prefill_experts`` (per expert with
  a non-zero count: gather its tokens, FC1 with ``w13[e]`` used as
  ``x @ W^T``, ``silu_and_mul``, FC2 with ``w2[e]``, scale by the slot's
  routing weight, accumulate into the token's output row) and
  ``moe_decode_experts`` (the same steps for one token, looping over its k
  experts);
* mlc-llm ``moe_misc.py`` — ``scatter_output`` (row ``p`` of the expert
  outputs goes back to slot ``reverse_indices[p]``) and ``moe_sum`` (sum of
  the ``[T, k, H]`` slot outputs over ``k``).

Readings (the pages leave them open):

* ``silu_and_mul`` on a ``[.., 2I]`` row gates the first half:
  ``act = silu(g) * u`` with ``g`` from rows ``0..I-1`` of ``w13[e]`` and ``u``
  from rows ``I..2I-1`` (the name ``w13`` = w1 stacked over w3);
* both GEMMs accumulate at full precision (float64 here); silu acts on the
  unrounded FC1 result; for bf16 the activation is rounded once to bf16
  (it is the FC2 operand); weighting and the k-sum are full precision; the
  layer output is rounded once to the output dtype (bf16: round to nearest,
  ties to even, written here from the definition of the format);
* the k-sum runs ``j = 0 .. k-1``;
* the layer output is in the original token order.
"""
from __future__ import annotations

import numpy as np

from . import align as _align
from . import gating as _gating

__all__ = [
    "bf16_round", "to_f64", "silu", "expert_ffn", "grouped_ffn", "decode_form",
    "layer_forward", "layer_rows",
]


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (8 significant bits), ties to even.

    bfloat16 keeps float32's exponent range (normal down to 2**-126, subnormal
    quantum 2**-133) and a significand of 8 bits including the implicit one.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2**e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)               # below 2**-126 the quantum is fixed at 2**-133
    q = np.ldexp(1.0, e - 8)              # spacing of 8-bit significands at this exponent
    r = np.rint(x / q) * q                # np.rint rounds half to even
    r = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, x), r)
    return r


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Input tensor as float64: float32 as is, bf16 given as uint16 bit patterns."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return bits.view(np.float32).astype(np.float64)


def silu(z: np.ndarray) -> np.ndarray:
    """``z * sigmoid(z) = z / (1 + exp(-z))``."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn(x: np.ndarray, w13_e: np.ndarray, w2_e: np.ndarray, dtype: str) -> np.ndarray:
    """One expert on float64 rows ``x [n, H]``: FC1 -> silu_and_mul -> FC2, float64 ``[n, H]``."""
    I = w13_e.shape[0] // 2
    gate_up = x @ w13_e.T                  # [n, 2I]
    act = silu(gate_up[:, :I]) * gate_up[:, I:]
    if dtype == "bf16":
        act = bf16_round(act)
    return act @ w2_e.T


def _round_out(y: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_round(y) if dtype == "bf16" else y.astype(np.float32).astype(np.float64)


def grouped_ffn(hidden, w13, w2, dtype: str, k: int, counts, offsets, sorted_token_ids,
                sorted_weights, reverse_indices, T: int | None = None, return_staging=False):
    """Prefill form: loop over experts with tokens, scatter to slots, sum over k.

    Returns the layer output as float64 holding values of the output dtype
    (and the float64 ``[T*k, H]`` weighted slot outputs when asked).
    """
    x = to_f64(hidden, dtype)
    T = x.shape[0] if T is None else T
    H = x.shape[1]
    E = len(counts)
    staging = np.zeros((T * k, H), dtype=np.float64)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        lo = int(offsets[e])
        tok = np.asarray(sorted_token_ids[lo:lo + c], dtype=np.int64)
        y = expert_ffn(x[tok], to_f64(w13[e], dtype), to_f64(w2[e], dtype), dtype)
        wt = np.asarray(sorted_weights[lo:lo + c], dtype=np.float32).astype(np.float64)
        staging[np.asarray(reverse_indices[lo:lo + c], dtype=np.int64)] = y * wt[:, None]
    out = np.zeros((T, H), dtype=np.float64)
    st = staging.reshape(T, k, H)
    for j in range(k):                     # moe_sum over the k axis, j ascending
        out += st[:, j, :]
    out = _round_out(out, dtype)
    return (out, staging) if return_staging else out


def decode_form(hidden_row, w13, w2, dtype: str, expert_ids, expert_weights) -> np.ndarray:
    """Decode form for one token: loop over its k experts and accumulate (float64 ``[H]``)."""
    x = to_f64(np.asarray(hidden_row)[None, :], dtype)
    out = np.zeros(x.shape[1], dtype=np.float64)
    for e, w in zip(expert_ids, expert_weights):
        y = expert_ffn(x, to_f64(w13[int(e)], dtype), to_f64(w2[int(e)], dtype), dtype)
        out += float(np.float32(w)) * y[0]
    return _round_out(out, dtype)


def layer_forward(logits, hidden, w13, w2, k: int, norm_topk_prob: bool, dtype: str) -> dict:
    """Whole path: gating -> align -> grouped FFN -> sum over k."""
    w, idx = _gating.softmax_topk(logits, k, norm_topk_prob)
    E = np.asarray(logits).shape[1]
    al = _align.align_by_expert(idx, w, E)
    out = grouped_ffn(hidden, w13, w2, dtype, k, al["counts"], al["offsets"],
                      al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"])
    return dict(out=out, topk_weights=w, topk_indices=idx, **al)


def layer_rows(hidden, w13, w2, dtype: str, topk_weights, topk_indices, tokens) -> np.ndarray:
    """Layer output rows for a subset of tokens, given their routing.

    Each output row depends only on its own token, its k experts and weights,
    so the grouped form restricted to ``tokens`` gives those rows exactly.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    idx = np.asarray(topk_indices)[tokens]
    wts = np.asarray(topk_weights)[tokens]
    E = len(w13)          # w13 / w2 may be any per-expert indexable (array or mapping)
    al = _align.align_by_expert(idx, wts, E)
    k = idx.shape[1]
    return grouped_ffn(np.asarray(hidden)[tokens], w13, w2, dtype, k, al["counts"],
                       al["offsets"], al["sorted_token_ids"], al["sorted_weights"],
                       al["reverse_indices"])

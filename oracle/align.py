"""Oracle: group routed slots by expert (test infrastructure only).

Source: mlc-llm ``moe_misc.py`` — ``moe_cumsum`` (expert mask, transposed,
flattened, inclusive cumsum), ``get_indptr`` (exclusive form, ``E + 1``
entries) and ``get_indices`` (shuffle and reverse indices); project_6
``moe_expert_gemm.cpp``, ``moe_prefill_experts`` (per-expert counts and the
routing weight that travels with each sorted slot).

The functions follow the page's steps literally: the full ``E * T`` mask
cumsum is materialised. For slot ``(b, j)`` routed to expert ``e`` its
sorted position is ``cumsum[e * T + b] - 1``: expert-major, then ascending
token.

Readings:

* ``get_indptr``'s docstring gives the inclusive form ``E + 1`` entries but its
  code gives the exclusive form ``E + 1`` and the inclusive form ``E``; the
  code is followed and the exclusive form is what the path exports;
* indices are int32 (page 3 carries int64);
* the rows name ``k`` distinct experts (what gating produces); a slot whose
  expert lies outside ``[0, E)`` is not routed: it is left out of the counts
  and the sorted arrays, and ``valid_slots`` reports how many were kept.
"""
from __future__ import annotations

import numpy as np

__all__ = ["moe_cumsum", "get_indptr", "get_indices", "align_by_expert"]


def moe_cumsum(indices: np.ndarray, E: int) -> np.ndarray:
    """Inclusive cumsum over the transposed-then-flattened expert mask, length ``E*T``."""
    idx = np.asarray(indices, dtype=np.int64)
    T, k = idx.shape
    mask = np.zeros((T, E), dtype=np.int64)
    for j in range(k):
        e = idx[:, j]
        ok = (e >= 0) & (e < E)
        mask[np.nonzero(ok)[0], e[ok]] = 1
    return np.cumsum(mask.T.reshape(E * T))


def get_indptr(cumsum: np.ndarray, E: int, T: int) -> np.ndarray:
    """Exclusive indptr: ``indptr[0] = 0``, ``indptr[i] = cumsum[i*T - 1]`` (``E + 1`` entries)."""
    indptr = np.zeros(E + 1, dtype=np.int64)
    for i in range(1, E + 1):
        indptr[i] = cumsum[i * T - 1] if T > 0 else 0
    return indptr


def get_indices(cumsum: np.ndarray, indices: np.ndarray, E: int):
    """(reverse_indices, token_indices, slot_position) following ``get_indices``.

    ``slot_position[b, j]`` is the sorted position of slot ``(b, j)`` (``-1``
    when not routed); ``reverse_indices[p] = b*k + j`` and
    ``token_indices[p] = b``.
    """
    idx = np.asarray(indices, dtype=np.int64)
    T, k = idx.shape
    rev = np.full(T * k, -1, dtype=np.int64)
    tok = np.full(T * k, -1, dtype=np.int64)
    posn = np.full((T, k), -1, dtype=np.int64)
    b = np.repeat(np.arange(T), k).reshape(T, k)
    j = np.tile(np.arange(k), T).reshape(T, k)
    ok = (idx >= 0) & (idx < E)
    p = cumsum[(idx[ok] * T + b[ok])] - 1
    rev[p] = b[ok] * k + j[ok]
    tok[p] = b[ok]
    posn[ok] = p
    return rev, tok, posn


def align_by_expert(indices: np.ndarray, weights: np.ndarray, E: int) -> dict:
    """All align outputs: counts [E], offsets [E+1], sorted_token_ids, sorted_weights,
    reverse_indices (each ``[T*k]``, valid up to ``offsets[E]``), plus ``valid_slots``."""
    idx = np.asarray(indices, dtype=np.int64)
    w = np.asarray(weights, dtype=np.float32)
    T, k = idx.shape
    cs = moe_cumsum(idx, E)
    indptr = get_indptr(cs, E, T)
    rev, tok, posn = get_indices(cs, idx, E)
    sw = np.zeros(T * k, dtype=np.float32)
    ok = posn >= 0
    sw[posn[ok]] = w[ok]
    n = int(indptr[E])
    return dict(
        counts=np.diff(indptr).astype(np.int32),
        offsets=indptr.astype(np.int32),
        sorted_token_ids=tok.astype(np.int32),
        sorted_weights=sw,
        reverse_indices=rev.astype(np.int32),
        valid_slots=n,
        slot_position=posn.astype(np.int32),
    )

"""Oracle: indices <-> multihot routing map (test infrastructure only).

Source: Megatron-LM ``fused_indices_converter.py`` —
``_indices_to_multihot_kernel`` (forward) and ``_multihot_to_indices_kernel``
(the inverse that the autograd backward runs), with the docstring examples
for ``topk = 2``, four local experts, two tokens.

Readings taken where the page is silent or garbled:

* the multihot output is 0/1 (the kernel stores 0, then 1, into a bool
  buffer; the docstring's ``-1`` entries are not what it stores);
* an index is routed only when ``0 <= idx < E``; the page masks ``-1`` and
  ``idx >= E`` and this reading also skips every other negative value;
* a row that names the same expert twice keeps the lowest slot ``j``;
* the inverse leaves an unfilled slot at 0.0 (the page's initial store) and,
  for the optional index output, at ``-1``; a position outside ``[0, k)``
  is skipped.
"""
from __future__ import annotations

import numpy as np

__all__ = ["indices_to_multihot", "multihot_to_indices"]


def indices_to_multihot(indices: np.ndarray, probs: np.ndarray, E: int):
    """Returns (multihot [T,E] uint8, probs_in_multihot [T,E] float32, position_map [T,E] int32)."""
    indices = np.asarray(indices, dtype=np.int64)
    probs = np.asarray(probs, dtype=np.float32)
    T, k = indices.shape
    multihot = np.zeros((T, E), dtype=np.uint8)
    probs_mh = np.zeros((T, E), dtype=np.float32)
    pos = np.full((T, E), -1, dtype=np.int32)
    for j in range(k - 1, -1, -1):          # lower j written last, so it wins a duplicate
        e = indices[:, j]
        ok = (e >= 0) & (e < E)
        t = np.nonzero(ok)[0]
        multihot[t, e[ok]] = 1
        probs_mh[t, e[ok]] = probs[t, j]
        pos[t, e[ok]] = j
    return multihot, probs_mh, pos


def multihot_to_indices(probs_in_multihot: np.ndarray, position_map: np.ndarray, k: int):
    """Returns (probs [T,k] float32, indices [T,k] int32) restored to slot order."""
    pm = np.asarray(probs_in_multihot, dtype=np.float32)
    pos = np.asarray(position_map, dtype=np.int64)
    T, E = pm.shape
    out = np.zeros((T, k), dtype=np.float32)
    idx = np.full((T, k), -1, dtype=np.int32)
    for e in range(E):
        p = pos[:, e]
        ok = (p >= 0) & (p < k)
        t = np.nonzero(ok)[0]
        out[t, p[ok]] = pm[t, e]
        idx[t, p[ok]] = e
    return out, idx

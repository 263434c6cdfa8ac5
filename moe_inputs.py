"""Seeded synthetic inputs for the MoE layer forward path.

This module only draws random numbers and packs them into the dtypes the
path consumes. It holds none of the method's arithmetic (no top-k, no
softmax, no routing, no FFN), so both the CPU oracle and the CUDA path can be
fed from it without sharing any computation.

Recipes (one per named workload):

* every tensor gets its own substream: ``SeedSequence(seed).spawn`` in a
  fixed order (logits, hidden, w13, w2, expert permutation); large tensors
  spawn one further substream per block of leading-axis slices (block size a
  function of the shape alone) so that blocks can be drawn in parallel
  threads and still be reproducible;
* normal draws are made in float32 with numpy's ``Generator(PCG64)``;
  bf16 tensors are the round-to-nearest-even narrowing of those float32
  draws, stored as raw ``uint16`` bit patterns;
* ``N(0, 1/sqrt(fan_in))`` is read as standard deviation ``1/sqrt(fan_in)``
  with fan_in = H for ``w13`` and I for ``w2``;
* router logits are float32 ``N(0,1)``; rows holding two equal values are
  redrawn until every row is duplicate-free ("distinct values");
* ``tiny`` adds ``1e-3 * e`` to logit column ``e``;
* ``skew`` adds ``bias_e = 2 * ln(p_r)`` where ``p_r`` is the Zipf(s=1.2)
  mass of rank ``r`` over ``E`` ranks and ranks are dealt to experts by a
  seeded permutation, which leaves some experts empty.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "gen_logits", "gen_normal", "make_layer_inputs",
]


@dataclass(frozen=True)
class Workload:
    """Shape and recipe of one synthetic MoE layer workload."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    norm_topk_prob: bool
    dtype: str           # "f32" or "bf16": hidden, weights, act and output
    logits: str          # "jitter" | "distinct" | "zipf"
    seed: int = 0

    @property
    def S(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "tiny": Workload("tiny", 64, 128, 256, 8, 2, True, "f32", "jitter"),
    "mixtral": Workload("mixtral", 4096, 4096, 14336, 8, 2, True, "bf16", "distinct"),
    "decode1": Workload("decode1", 1, 2048, 1408, 64, 8, True, "bf16", "distinct"),
    "decode8": Workload("decode8", 8, 2048, 1408, 64, 8, True, "bf16", "distinct"),
    "decode64": Workload("decode64", 64, 2048, 1408, 64, 8, True, "bf16", "distinct"),
    "fine": Workload("fine", 16384, 2048, 1408, 64, 8, False, "bf16", "distinct"),
    "skew": Workload("skew", 32768, 4096, 1536, 128, 8, True, "bf16", "zipf"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def f32_to_bf16_bits(a: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Narrow float32 to bfloat16 with round-to-nearest-even; returns uint16 bits.

    Input packing only (NaN never occurs in these recipes). ``a`` is used as
    scratch when it is a writable contiguous float32 array and ``out`` is given.
    """
    if out is None:
        a = np.array(a, dtype=np.float32, copy=True)
        out = np.empty(a.shape, dtype=np.uint16)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += lsb
    u += np.uint32(0x7FFF)
    u >>= np.uint32(16)
    np.copyto(out, u, casting="unsafe")
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def gen_normal(ss: np.random.SeedSequence, shape, std: float, dtype: str) -> np.ndarray:
    """``N(0, std)`` of ``shape``.

    The leading axis is cut into blocks of ``ceil(2**22 / row_size)`` slices
    (a function of the shape only); each block draws from its own substream of
    ``ss``, so blocks can be filled by parallel threads reproducibly.
    Returns float32 for ``dtype == "f32"`` and uint16 bf16 bits for ``"bf16"``.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.float32 if dtype == "f32" else np.uint16)
    if out.size == 0:
        return out
    lead = shape[0]
    row = max(1, out.size // lead)
    per = max(1, -(-(1 << 22) // row))
    nblk = -(-lead // per)
    subs = ss.spawn(nblk)

    def one(b):
        lo, hi = b * per, min(lead, (b + 1) * per)
        g = np.random.Generator(np.random.PCG64(subs[b]))
        x = g.standard_normal((hi - lo,) + shape[1:], dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if dtype == "f32":
            out[lo:hi] = x
        else:
            f32_to_bf16_bits(x, out[lo:hi])

    if nblk > 1:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(nblk)))
    else:
        one(0)
    return out


def _zipf_bias(E: int, perm_ss: np.random.SeedSequence, s: float = 1.2) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    bias_by_rank = 2.0 * np.log(p)
    perm = np.random.Generator(np.random.PCG64(perm_ss)).permutation(E)
    bias = np.empty(E, dtype=np.float64)
    bias[perm] = bias_by_rank          # expert perm[r] receives rank r's bias
    return bias.astype(np.float32)


def gen_logits(ss: np.random.SeedSequence, T: int, E: int, kind: str,
               perm_ss: np.random.SeedSequence | None = None) -> np.ndarray:
    """Router logits ``[T, E]`` float32 following the named recipe.

    ``plain`` draws ``N(0,1)`` and nothing more (ties allowed); the other
    recipes redraw any row that holds a repeated value.
    """
    if kind not in ("plain", "distinct", "jitter", "zipf"):
        raise ValueError(f"unknown logits recipe {kind!r}")
    g = np.random.Generator(np.random.PCG64(ss))
    bias = np.zeros(E, dtype=np.float32)
    if kind == "jitter":
        bias = np.float32(1e-3) * np.arange(E, dtype=np.float32)
    elif kind == "zipf":
        bias = _zipf_bias(E, perm_ss if perm_ss is not None else ss.spawn(1)[0])
    x = g.standard_normal((T, E), dtype=np.float32) + bias[None, :]
    if kind == "plain" or T == 0 or E < 2:
        return x
    for _ in range(100):
        srt = np.sort(x, axis=1)
        bad = np.nonzero((srt[:, 1:] == srt[:, :-1]).any(axis=1))[0]
        if bad.size == 0:
            break
        x[bad] = g.standard_normal((bad.size, E), dtype=np.float32) + bias[None, :]
    return x


def make_layer_inputs(w: Workload | str | None = None, *, T=None, H=None, I=None, E=None,
                      k=None, norm_topk_prob=None, dtype=None, logits=None, seed=None,
                      with_weights: bool = True) -> dict:
    """Draw one full set of layer inputs.

    Returns a dict with ``logits`` (float32 ``[T,E]``), ``hidden`` (``[T,H]``),
    ``w13`` (``[E,2I,H]``), ``w2`` (``[E,H,I]``) and the shape parameters.
    Float tensors are float32 for ``dtype == "f32"`` and uint16 bf16 bit patterns
    for ``"bf16"``. Keyword arguments override the named workload's fields.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    base = w or Workload("custom", 0, 0, 0, 0, 0, True, "bf16", "distinct")
    T = base.T if T is None else T
    H = base.H if H is None else H
    I = base.I if I is None else I
    E = base.E if E is None else E
    k = base.k if k is None else k
    norm = base.norm_topk_prob if norm_topk_prob is None else norm_topk_prob
    dtype = base.dtype if dtype is None else dtype
    kind = base.logits if logits is None else logits
    seed = base.seed if seed is None else seed
    ss_logits, ss_hidden, ss_w13, ss_w2, ss_perm = np.random.SeedSequence(seed).spawn(5)
    out = dict(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=bool(norm), dtype=dtype, seed=seed)
    out["logits"] = gen_logits(ss_logits, T, E, kind, ss_perm)
    out["hidden"] = gen_normal(ss_hidden, (T, H), 1.0, dtype) if T > 0 else \
        np.empty((0, H), dtype=np.float32 if dtype == "f32" else np.uint16)
    if with_weights:
        out["w13"] = gen_normal(ss_w13, (E, 2 * I, H), 1.0 / np.sqrt(H), dtype)
        out["w2"] = gen_normal(ss_w2, (E, H, I), 1.0 / np.sqrt(I), dtype)
    return out

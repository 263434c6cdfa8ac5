"""CPU oracle for the MoE layer forward path — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the three source pages
compute, in numpy with float64 arithmetic:

* mlc-llm, ``python/mlc_llm/op/moe_misc.py`` ("Mixture of Experts operators"):
  ``gating_topk``, ``gating_softmax_topk``, ``moe_cumsum``, ``get_indices``,
  ``get_indptr``, ``scatter_output``, ``moe_sum``;
* Megatron-LM, ``megatron/core/fusions/fused_indices_converter.py``:
  ``_indices_to_multihot_kernel``, ``_multihot_to_indices_kernel``;
* project_6, ``ex_engine/csrc/moe_expert_gemm.cpp``: ``moe_decode_experts``,
  ``moe_prefill_experts``.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package. The CUDA library never calls it, shares no code
with it, and must fail loudly rather than fall back to it.

Modules:

* :mod:`oracle.gating` — top-k selection and the two softmax variants;
* :mod:`oracle.multihot` — indices <-> multihot / position map;
* :mod:`oracle.align` — mask cumsum, indptr, shuffle and reverse indices;
* :mod:`oracle.ffn` — per-expert FC1 / silu_and_mul / FC2, weighting and the
  sum over k.

Every function is pinned by a ``-m "not gpu"`` test against the pages' worked
examples, closed forms, brute force on tiny inputs or invariants, except the
FFN, whose pins are closed forms on special cases and agreement between the
page's two loop forms (decode form vs. prefill form); the pages print no
numeric FFN example ("parity pinned by special cases only").
"""
from . import align, ffn, gating, multihot  # noqa: F401

"""Oracle: gradients of the grouped expert FFN and the weighted k-sum (test infrastructure only).

The forward is the one in ``ffn.py`` (project_6 ``moe_expert_gemm.cpp``,
``moe_prefill_experts``; mlc-llm ``moe_misc.py``, ``scatter_output`` and
``moe_sum``). Its backward is not printed on the pages; the training side
they name (Megatron-LM's multihot converter carries a backward) needs it, and
it is the derivative of that forward, written out here.

Per routed slot ``p`` of expert ``e`` with token ``t`` and routing weight
``w_p`` (``x = hidden[t]``, ``W1 = w13[e][:I]``, ``W3 = w13[e][I:]``):

    g = W1 x,  u = W3 x,  s = sigmoid(g),  a = g s u,  y = W2 a,
    out[t] = sum over the token's k slots of w_p y_p.

Given ``dO = d loss / d out``:

    d w_p   = <dO[t], y_p>
    dy_p    = w_p dO[t]
    dW2[e]  = sum_p dy_p a_p^T
    da_p    = W2^T dy_p
    dg_p    = da_p * u_p * s_p * (1 + g_p (1 - s_p))      (silu'(g) = s (1 + g (1 - s)))
    du_p    = da_p * g_p * s_p                            (silu(g) = g s)
    dW1[e]  = sum_p dg_p x_t^T,   dW3[e] = sum_p du_p x_t^T
    dx_t    = sum over the token's slots of W1^T dg_p + W3^T du_p

Reading (the pages leave it open): for bf16 the forward rounds ``a`` to bf16
(the FC2 operand). That rounding is differentiated as the identity: ``y``,
``dW2`` and ``d w_p`` use the rounded ``a`` the forward used, while ``dg`` and
``du`` use the unrounded ``g`` and ``u``. (The literal derivative of a
rounding is zero almost everywhere and would zero every gradient before FC2.)

Arithmetic is float64; results are float64.
"""
from __future__ import annotations

import numpy as np

from .ffn import bf16_round, to_f64

__all__ = ["grouped_ffn_backward"]


def grouped_ffn_backward(hidden, w13, w2, dtype: str, k: int, counts, offsets, sorted_token_ids,
                         sorted_weights, reverse_indices, d_out) -> dict:
    """Gradients of the layer output w.r.t. hidden, w13, w2 and the routing weights.

    Returns float64 ``d_hidden [T, H]``, ``d_w13 [E, 2I, H]``, ``d_w2 [E, H, I]`` and
    ``d_weights [T, k]`` (slot ``t*k + j``, the layout of the top-k weights).
    """
    x = to_f64(hidden, dtype)
    dO = to_f64(d_out, dtype)
    T, H = x.shape
    E = len(counts)
    I = np.asarray(w2[0]).shape[1]
    d_hidden = np.zeros((T, H))
    d_w13 = np.zeros((E, 2 * I, H))
    d_w2 = np.zeros((E, H, I))
    d_w = np.zeros(T * k)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        lo = int(offsets[e])
        tok = np.asarray(sorted_token_ids[lo:lo + c], dtype=np.int64)
        slot = np.asarray(reverse_indices[lo:lo + c], dtype=np.int64)
        wp = np.asarray(sorted_weights[lo:lo + c], dtype=np.float32).astype(np.float64)
        W13 = to_f64(w13[e], dtype)
        W1, W3 = W13[:I], W13[I:]
        W2 = to_f64(w2[e], dtype)
        X = x[tok]
        G = X @ W1.T
        U = X @ W3.T
        S = 1.0 / (1.0 + np.exp(-G))
        A = G * S * U
        if dtype == "bf16":
            A = bf16_round(A)
        Y = A @ W2.T
        dO_t = dO[tok]
        d_w[slot] = np.sum(dO_t * Y, axis=1)
        dY = wp[:, None] * dO_t
        d_w2[e] = dY.T @ A
        dA = dY @ W2
        dG = dA * U * S * (1.0 + G * (1.0 - S))
        dU = dA * G * S
        d_w13[e, :I] = dG.T @ X
        d_w13[e, I:] = dU.T @ X
        np.add.at(d_hidden, tok, dG @ W1 + dU @ W3)
    return dict(d_hidden=d_hidden, d_w13=d_w13, d_w2=d_w2, d_weights=d_w.reshape(T, k))

"""ctypes binding of ``libmoe_gb300.so`` (the C ABI declared in ``include/moe.h``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch supplies device memory (output and workspace tensors when
the caller gives none) and the current CUDA stream. There is no CPU or
PyTorch fallback: if the library is missing or a call fails, an exception is
raised.
"""
from __future__ import annotations

import ctypes
import json
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE = 0, 1, 2, 3, 4
MOE_F32, MOE_BF16 = 0, 1
MOE_STATUS_BAD_INDEX, MOE_STATUS_TIMEOUT = 1, 2
MOE_GROUP_TOPK_GREEDY, MOE_GROUP_TOPK_NOAUX_TC = 0, 1
MOE_MAX_TOPK, MOE_MAX_EXPERTS = 32, 1024
MOE_ALIGN_NOALLOC_SCRATCH_INTS = 65536

_p, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_gating_softmax_topk": (_i, [_p, _i, _i, _i, _i, _p, _p, _p]),
    "moe_gating_softmax_topk_bf16": (_i, [_p, _i, _i, _i, _i, _p, _p, _p]),
    "moe_group_limited_topk": (_i, [_p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p]),
    "moe_indices_to_multihot": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _p]),
    "moe_multihot_to_indices": (_i, [_p, _p, _i, _i, _i, _p, _p, _p]),
    "moe_align_workspace_size": (_sz, [_i, _i, _i]),
    "moe_align_by_expert": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _sz, _p, _p]),
    "moe_align_by_expert_noalloc": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p]),
    "moe_grouped_ffn_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_grouped_ffn": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _sz, _p, _p]),
    "moe_grouped_ffn_backward_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_grouped_ffn_backward": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                      _p, _p, _sz, _p, _p]),
    "moe_layer_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_layer_forward": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _sz, _p, _p]),
    "moe_gather_rows": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p]),
    "moe_ep_receive_workspace_size": (_sz, [_i, _i]),
    "moe_ep_receive_index": (_i, [_p, _i, _i, _i, _p, _p, _p, _p, _sz, _p]),
    "moe_ep_combine_workspace_size": (_sz, [_i, _i]),
    "moe_ep_combine": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _sz, _p]),
    "moe_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "moe_profiler_enable": (_i, [_i]),
    "moe_profiler_report": (_i, [ctypes.c_char_p, _sz]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_version": (ctypes.c_char_p, []),
}


class MoeError(RuntimeError):
    """A library call returned a non-zero status."""

    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with code {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device):
    if stream is None:
        if _raw_stream is not None:      # the current stream's handle without a Stream object
            return ctypes.c_void_p(_raw_stream(device.index if device.index is not None else
                                               torch.cuda.current_device()))
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc, lib().moe_last_error().decode())


def _dev(t, name, dtype=None):
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    return t


def _dtype_code(t):
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _out(t, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _dev(t, name, dtype)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}")
    return t


def version() -> str:
    return lib().moe_version().decode()


def moe_gating_softmax_topk(logits, k, norm_topk_prob=True, weights=None, indices=None, stream=None):
    """Top-k experts per row of ``logits [T,E]`` (float32) -> (weights [T,k] f32, indices [T,k] i32)."""
    _dev(logits, "logits", torch.float32)
    T, E = logits.shape
    weights = _out(weights, (T, k), torch.float32, logits.device, "weights")
    indices = _out(indices, (T, k), torch.int32, logits.device, "indices")
    _check("moe_gating_softmax_topk", lib().moe_gating_softmax_topk(
        _ptr(logits), T, E, k, int(bool(norm_topk_prob)), _ptr(weights), _ptr(indices),
        _stream(stream, logits.device)))
    return weights, indices


def moe_gating_softmax_topk_bf16(logits, k, norm_topk_prob=True, weights=None, indices=None, stream=None):
    """Top-k experts per row of bf16 ``logits [T,E]`` -> (weights [T,k] f32, indices [T,k] i32)."""
    _dev(logits, "logits", torch.bfloat16)
    T, E = logits.shape
    weights = _out(weights, (T, k), torch.float32, logits.device, "weights")
    indices = _out(indices, (T, k), torch.int32, logits.device, "indices")
    _check("moe_gating_softmax_topk_bf16", lib().moe_gating_softmax_topk_bf16(
        _ptr(logits), T, E, k, int(bool(norm_topk_prob)), _ptr(weights), _ptr(indices),
        _stream(stream, logits.device)))
    return weights, indices


def moe_group_limited_topk(scores, k, n_group, topk_group, method="group_limited_greedy", bias=None,
                           weights=None, indices=None, stream=None):
    """Group-limited top-k of ``scores [T,E]`` f32 -> (weights [T,k] f32, indices [T,k] i32).

    ``method`` is "group_limited_greedy" or "noaux_tc" (needs ``bias [E]`` f32)."""
    _dev(scores, "scores", torch.float32)
    T, E = scores.shape
    code = {"group_limited_greedy": MOE_GROUP_TOPK_GREEDY, "noaux_tc": MOE_GROUP_TOPK_NOAUX_TC}[method]
    if bias is not None:
        _dev(bias, "bias", torch.float32)
    weights = _out(weights, (T, k), torch.float32, scores.device, "weights")
    indices = _out(indices, (T, k), torch.int32, scores.device, "indices")
    _check("moe_group_limited_topk", lib().moe_group_limited_topk(
        _ptr(scores), _ptr(bias), T, E, k, n_group, topk_group, code, _ptr(weights), _ptr(indices),
        _stream(stream, scores.device)))
    return weights, indices


def moe_indices_to_multihot(indices, probs, num_experts, multihot=None, probs_in_multihot=None,
                            position_map=None, stream=None):
    """-> (multihot [T,E] uint8, probs_in_multihot [T,E] f32, position_map [T,E] i32)."""
    _dev(indices, "indices", torch.int32)
    _dev(probs, "probs", torch.float32)
    T, k = indices.shape
    E = int(num_experts)
    d = indices.device
    multihot = _out(multihot, (T, E), torch.uint8, d, "multihot")
    probs_in_multihot = _out(probs_in_multihot, (T, E), torch.float32, d, "probs_in_multihot")
    position_map = _out(position_map, (T, E), torch.int32, d, "position_map")
    _check("moe_indices_to_multihot", lib().moe_indices_to_multihot(
        _ptr(indices), _ptr(probs), T, k, E, _ptr(multihot), _ptr(probs_in_multihot),
        _ptr(position_map), _stream(stream, d)))
    return multihot, probs_in_multihot, position_map


def moe_multihot_to_indices(probs_in_multihot, position_map, k, probs=None, indices=None,
                            with_indices=True, stream=None):
    """-> (probs [T,k] f32, indices [T,k] i32 or None)."""
    _dev(probs_in_multihot, "probs_in_multihot", torch.float32)
    _dev(position_map, "position_map", torch.int32)
    T, E = probs_in_multihot.shape
    d = probs_in_multihot.device
    probs = _out(probs, (T, k), torch.float32, d, "probs")
    if with_indices or indices is not None:
        indices = _out(indices, (T, k), torch.int32, d, "indices")
    _check("moe_multihot_to_indices", lib().moe_multihot_to_indices(
        _ptr(probs_in_multihot), _ptr(position_map), T, E, k, _ptr(probs), _ptr(indices),
        _stream(stream, d)))
    return probs, indices


def moe_align_workspace_size(T, k, E) -> int:
    return int(lib().moe_align_workspace_size(T, k, E))


def moe_align_by_expert(indices, weights, num_experts, out=None, workspace=None, status=None,
                        stream=None):
    """-> dict(counts [E], offsets [E+1], sorted_token_ids, sorted_weights, reverse_indices [T*k])."""
    _dev(indices, "indices", torch.int32)
    _dev(weights, "weights", torch.float32)
    T, k = indices.shape
    E = int(num_experts)
    S = T * k
    d = indices.device
    out = dict(out or {})
    counts = _out(out.get("counts"), (E,), torch.int32, d, "counts")
    offsets = _out(out.get("offsets"), (E + 1,), torch.int32, d, "offsets")
    ids = _out(out.get("sorted_token_ids"), (S,), torch.int32, d, "sorted_token_ids")
    sw = _out(out.get("sorted_weights"), (S,), torch.float32, d, "sorted_weights")
    rev = _out(out.get("reverse_indices"), (S,), torch.int32, d, "reverse_indices")
    need = moe_align_workspace_size(T, k, E)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=d)
    _check("moe_align_by_expert", lib().moe_align_by_expert(
        _ptr(indices), _ptr(weights), T, k, E, _ptr(counts), _ptr(offsets), _ptr(ids), _ptr(sw),
        _ptr(rev), _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream, d)))
    return dict(counts=counts, offsets=offsets, sorted_token_ids=ids, sorted_weights=sw,
                reverse_indices=rev)


def moe_align_by_expert_noalloc(indices, weights, num_experts, out=None, status=None, stream=None):
    """Align by expert for callers that cannot allocate device memory at call time.

    Same results as :func:`moe_align_by_expert`; the library keeps the scratch in
    a fixed device array of its own (limit: ceil(T*k / 4096) * E <=
    MOE_ALIGN_NOALLOC_SCRATCH_INTS), so no workspace is passed. Calls that
    overlap on the GPU share that array and race. Output tensors are created
    here only when ``out`` does not supply them.
    """
    _dev(indices, "indices", torch.int32)
    _dev(weights, "weights", torch.float32)
    T, k = indices.shape
    E = int(num_experts)
    S = T * k
    d = indices.device
    out = dict(out or {})
    counts = _out(out.get("counts"), (E,), torch.int32, d, "counts")
    offsets = _out(out.get("offsets"), (E + 1,), torch.int32, d, "offsets")
    ids = _out(out.get("sorted_token_ids"), (S,), torch.int32, d, "sorted_token_ids")
    sw = _out(out.get("sorted_weights"), (S,), torch.float32, d, "sorted_weights")
    rev = _out(out.get("reverse_indices"), (S,), torch.int32, d, "reverse_indices")
    _check("moe_align_by_expert_noalloc", lib().moe_align_by_expert_noalloc(
        _ptr(indices), _ptr(weights), T, k, E, _ptr(counts), _ptr(offsets), _ptr(ids), _ptr(sw),
        _ptr(rev), _ptr(status), _stream(stream, d)))
    return dict(counts=counts, offsets=offsets, sorted_token_ids=ids, sorted_weights=sw,
                reverse_indices=rev)


def moe_grouped_ffn_workspace_size(dtype_code, T, H, I, E, k) -> int:
    return int(lib().moe_grouped_ffn_workspace_size(dtype_code, T, H, I, E, k))


def moe_grouped_ffn(hidden, w13, w2, k, counts, offsets, sorted_token_ids, sorted_weights,
                    reverse_indices, out=None, workspace=None, status=None, stream=None):
    """Expert FFN + weighted combine -> out [T,H] (hidden's dtype)."""
    _dev(hidden, "hidden")
    dt = _dtype_code(hidden)
    T, H = hidden.shape
    E, I2, H2 = w13.shape
    I = I2 // 2
    _dev(w13, "w13", hidden.dtype)
    _dev(w2, "w2", hidden.dtype)
    if H2 != H or tuple(w2.shape) != (E, H, I):
        raise ValueError("w13 must be [E, 2I, H] and w2 [E, H, I]")
    d = hidden.device
    out = _out(out, (T, H), hidden.dtype, d, "out")
    need = moe_grouped_ffn_workspace_size(dt, T, H, I, E, k)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d)
    _check("moe_grouped_ffn", lib().moe_grouped_ffn(
        _ptr(hidden), _ptr(w13), _ptr(w2), dt, T, H, I, E, k, _ptr(counts), _ptr(offsets),
        _ptr(sorted_token_ids), _ptr(sorted_weights), _ptr(reverse_indices), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream, d)))
    return out


def moe_grouped_ffn_backward_workspace_size(dtype_code, T, H, I, E, k) -> int:
    return int(lib().moe_grouped_ffn_backward_workspace_size(dtype_code, T, H, I, E, k))


def moe_grouped_ffn_backward(hidden, w13, w2, k, counts, offsets, sorted_token_ids, sorted_weights,
                             reverse_indices, d_out, d_hidden=None, d_w13=None, d_w2=None, d_weights=None,
                             workspace=None, status=None, stream=None, want_d_weights=True):
    """Backward of moe_grouped_ffn (bf16) -> (d_hidden [T,H], d_w13 [E,2I,H], d_w2 [E,H,I], d_weights [T,k] f32)."""
    _dev(hidden, "hidden")
    dt = _dtype_code(hidden)
    T, H = hidden.shape
    E, I2, H2 = w13.shape
    I = I2 // 2
    _dev(w13, "w13", hidden.dtype)
    _dev(w2, "w2", hidden.dtype)
    _dev(d_out, "d_out", hidden.dtype)
    if H2 != H or tuple(w2.shape) != (E, H, I) or tuple(d_out.shape) != (T, H):
        raise ValueError("shape mismatch")
    d = hidden.device
    d_hidden = _out(d_hidden, (T, H), hidden.dtype, d, "d_hidden")
    d_w13 = _out(d_w13, (E, 2 * I, H), hidden.dtype, d, "d_w13")
    d_w2 = _out(d_w2, (E, H, I), hidden.dtype, d, "d_w2")
    if want_d_weights:
        d_weights = _out(d_weights, (T, k), torch.float32, d, "d_weights")
    need = moe_grouped_ffn_backward_workspace_size(dt, T, H, I, E, k)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d)
    _check("moe_grouped_ffn_backward", lib().moe_grouped_ffn_backward(
        _ptr(hidden), _ptr(w13), _ptr(w2), dt, T, H, I, E, k, _ptr(counts), _ptr(offsets),
        _ptr(sorted_token_ids), _ptr(sorted_weights), _ptr(reverse_indices), _ptr(d_out), _ptr(d_hidden),
        _ptr(d_w13), _ptr(d_w2), _ptr(d_weights) if want_d_weights else None, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream, d)))
    return d_hidden, d_w13, d_w2, (d_weights if want_d_weights else None)


def moe_layer_workspace_size(dtype_code, T, H, I, E, k) -> int:
    return int(lib().moe_layer_workspace_size(dtype_code, T, H, I, E, k))


def moe_layer_forward(hidden, router_logits, w13, w2, k, norm_topk_prob=True, out=None,
                      topk_weights=None, topk_indices=None, workspace=None, status=None,
                      stream=None):
    """Whole MoE layer forward -> out [T,H] (hidden's dtype)."""
    _dev(hidden, "hidden")
    _dev(router_logits, "router_logits", torch.float32)
    dt = _dtype_code(hidden)
    T, H = hidden.shape
    E, I2, H2 = w13.shape
    I = I2 // 2
    _dev(w13, "w13", hidden.dtype)
    _dev(w2, "w2", hidden.dtype)
    if H2 != H or tuple(w2.shape) != (E, H, I) or tuple(router_logits.shape) != (T, E):
        raise ValueError("shapes must be hidden [T,H], router_logits [T,E], w13 [E,2I,H], w2 [E,H,I]")
    d = hidden.device
    out = _out(out, (T, H), hidden.dtype, d, "out")
    if topk_weights is not None:
        _out(topk_weights, (T, k), torch.float32, d, "topk_weights")
    if topk_indices is not None:
        _out(topk_indices, (T, k), torch.int32, d, "topk_indices")
    if workspace is None:
        need = moe_layer_workspace_size(dt, T, H, I, E, k)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d)
    _check("moe_layer_forward", lib().moe_layer_forward(
        _ptr(hidden), _ptr(router_logits), _ptr(w13), _ptr(w2), dt, T, H, I, E, k,
        int(bool(norm_topk_prob)), _ptr(out), _ptr(topk_weights), _ptr(topk_indices),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream, d)))
    return out


def moe_gather_rows(hidden, sorted_token_ids, offsets, k, out=None, stream=None):
    """Expert-sorted copy of the routed token rows -> x_sorted [T*k, H] (rows p < offsets[E])."""
    _dev(hidden, "hidden")
    dt = _dtype_code(hidden)
    T, H = hidden.shape
    E = offsets.numel() - 1
    d = hidden.device
    out = _out(out, (T * k, H), hidden.dtype, d, "out")
    _check("moe_gather_rows", lib().moe_gather_rows(
        _ptr(hidden), _ptr(sorted_token_ids), _ptr(offsets), dt, T, H, E, k, _ptr(out), _stream(stream, d)))
    return out


def moe_ep_receive_index(recv_counts, R, local_counts=None, local_offsets=None, perm=None, workspace=None,
                         stream=None):
    """Owner side of the expert-parallel exchange: recv_counts [G, E_local] int32 (device) ->
    (local_counts [E_local], local_offsets [E_local+1], perm [R]) int32."""
    _dev(recv_counts, "recv_counts", torch.int32)
    G, El = recv_counts.shape
    d = recv_counts.device
    local_counts = _out(local_counts, (El,), torch.int32, d, "local_counts")
    local_offsets = _out(local_offsets, (El + 1,), torch.int32, d, "local_offsets")
    perm = _out(perm, (R,), torch.int32, d, "perm")
    need = int(lib().moe_ep_receive_workspace_size(G, El))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d)
    _check("moe_ep_receive_index", lib().moe_ep_receive_index(
        _ptr(recv_counts), G, El, int(R), _ptr(local_counts), _ptr(local_offsets), _ptr(perm), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream, d)))
    return local_counts, local_offsets, perm


def moe_ep_combine(y_sorted, topk_weights, reverse_indices, offsets, out=None, workspace=None, stream=None):
    """Sender side after the return exchange: out[t] = sum_j w[t,j] * y_sorted[pos(t, j)] -> [T, H]."""
    _dev(y_sorted, "y_sorted")
    dt = _dtype_code(y_sorted)
    T, k = topk_weights.shape
    H = y_sorted.shape[1]
    E = offsets.numel() - 1
    d = y_sorted.device
    out = _out(out, (T, H), y_sorted.dtype, d, "out")
    need = int(lib().moe_ep_combine_workspace_size(T, k))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d)
    _check("moe_ep_combine", lib().moe_ep_combine(
        _ptr(y_sorted), _ptr(topk_weights), _ptr(reverse_indices), _ptr(offsets), dt, T, k, H, E, _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, d)))
    return out


def set_wait_limit_ns(ns: int) -> int:
    """Limit of the tensor-core FFN kernels' waits on their other roles (0: the default, 2 s);
    returns the previous limit."""
    return int(lib().moe_set_wait_limit_ns(int(ns)))


def profiler_enable(on: bool = True) -> None:
    lib().moe_profiler_enable(int(bool(on)))


def profiler_report() -> dict:
    """Per-kernel {"launches": n, "total_ms": t} since the last report (synchronises)."""
    buf = ctypes.create_string_buffer(1 << 20)
    n = lib().moe_profiler_report(buf, len(buf))
    if n >= len(buf):
        raise RuntimeError("profiler report truncated")
    return json.loads(buf.value.decode())

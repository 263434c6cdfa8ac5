"""Helpers for the GPU parity tests: move seeded numpy inputs to the device and back."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_routing_token_gb300 as moe
    from mixture_experts_routing_token_gb300.build import build
    build()
    moe.lib()
    return moe


DEV = "cuda:0"


def to_dev(a, dtype):
    """numpy float32 (dtype "f32") or uint16 bf16 bits ("bf16") -> device tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(DEV)


def to_np64(t):
    return t.float().cpu().numpy().astype(np.float64)


def layer_tolerance(dtype):
    """max|err| <= tol * max|ref|: 2e-2 for bf16 inputs with fp32 accumulation, 1e-4 for fp32."""
    return 2e-2 if dtype == "bf16" else 1e-4


def assert_close_rel_max(got, ref, tol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return
    err = float(np.abs(got - ref).max())
    scale = float(np.abs(ref).max())
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err <= tol * scale, f"{what}: max|err| {err:.4e} > {tol} * max|ref| {scale:.4e}"

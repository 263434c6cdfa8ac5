"""moe_align_by_expert_noalloc: align by expert for callers that cannot allocate.

Some callers cannot allocate device memory when they call the library (host
code that is handed tensors by a framework whose allocator it cannot reach, or
a runtime whose device memory is fixed at start-up), so they cannot pass the
workspace that moe_align_by_expert needs. The no-allocation entry point keeps
that scratch in a fixed array inside the library instead. These tests call it
through the C ABI and check it against moe_align_by_expert, bit for bit (the
outputs are integers and copied floats), on two calls in a row, since every
call reuses the same array.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, need_gpu
from moe_inputs import gen_logits
from oracle import gating

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")


def _routing(T, E, k, seed, kind="distinct"):
    x = gen_logits(np.random.SeedSequence(seed), T, E, kind)
    w, i = gating.softmax_topk(x, k, True)
    return torch.from_numpy(i).to(DEV), torch.from_numpy(w).to(DEV)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (4096, 8, 2), (16384, 64, 8), (32768, 128, 8), (5000, 1000, 3)])
def test_noalloc_matches_workspace_entry_point_twice(T, E, k):
    moe = need_gpu()
    for call in range(2):   # second call runs over the array the first one left behind
        idx, w = _routing(T, E, k, seed=T + E + call, kind="zipf" if E >= 64 else "distinct")
        st_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        ref = moe.moe_align_by_expert(idx, w, E, status=st_ref)
        got = moe.moe_align_by_expert_noalloc(idx, w, E, status=st)
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(got[key], ref[key]), (call, key)
        assert int(st.item()) == int(st_ref.item()) == 0


def test_noalloc_into_caller_outputs_and_bad_index_status():
    moe = need_gpu()
    T, E, k = 9000, 16, 2
    idx, w = _routing(T, E, k, seed=3)
    idx[5, 1] = 99                     # one slot with an expert outside [0, E)
    S = T * k
    out = {"counts": torch.full((E,), -7, dtype=torch.int32, device=DEV),
           "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
           "sorted_token_ids": torch.full((S,), -7, dtype=torch.int32, device=DEV),
           "sorted_weights": torch.full((S,), -7.0, dtype=torch.float32, device=DEV),
           "reverse_indices": torch.full((S,), -7, dtype=torch.int32, device=DEV)}
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = moe.moe_align_by_expert_noalloc(idx, w, E, out=out, status=st)
    st_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref = moe.moe_align_by_expert(idx, w, E, status=st_ref)
    torch.cuda.synchronize()
    n = int(ref["offsets"][E].item())
    assert n == S - 1
    for key in KEYS:
        a, b = got[key], ref[key]
        if a.numel() == S:
            a, b = a[:n], b[:n]
        assert torch.equal(a, b), key
    assert got["counts"].data_ptr() == out["counts"].data_ptr()
    assert int(st.item()) & moe.MOE_STATUS_BAD_INDEX
    assert int(st.item()) == int(st_ref.item())


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    moe = need_gpu()
    E, k = 1024, 4
    T = (moe.MOE_ALIGN_NOALLOC_SCRATCH_INTS // E + 1) * 4096 // k   # one chunk too many
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    w = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    with pytest.raises(moe.MoeError) as ex:
        moe.moe_align_by_expert_noalloc(idx, w, E)
    assert ex.value.code == 2 and "without workspace" in str(ex.value)
    T_ok = (moe.MOE_ALIGN_NOALLOC_SCRATCH_INTS // E) * 4096 // k     # exactly at the limit
    idx, w = _routing(T_ok, E, k, seed=1)
    ref = moe.moe_align_by_expert(idx, w, E)
    got = moe.moe_align_by_expert_noalloc(idx, w, E)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(got[key], ref[key]), key


def test_noalloc_under_a_second_context_of_the_same_device():
    """A caller with a driver context of its own (beside the runtime's primary
    context, which torch uses) gets that context's copy of the fixed array: the
    entry point must not reuse the address it looked up in the primary context."""
    import ctypes
    moe = need_gpu()
    cu = ctypes.CDLL("libcuda.so.1")

    def ok(rc, what):
        assert rc == 0, f"{what} returned CUresult {rc}"

    T, E, k = 16384, 64, 8            # 32 chunks: the scratch array (and the scan launch) is used
    S = T * k
    idx, w = _routing(T, E, k, seed=11, kind="zipf")
    ref = moe.moe_align_by_expert(idx, w, E)
    moe.moe_align_by_expert_noalloc(idx, w, E)   # caches the primary context's address first
    torch.cuda.synchronize()
    want = {key: ref[key].cpu().numpy() for key in KEYS}
    host_in = {"indices": np.ascontiguousarray(idx.cpu().numpy()), "weights": np.ascontiguousarray(w.cpu().numpy())}
    out_shapes = {"counts": (E, np.int32), "offsets": (E + 1, np.int32), "sorted_token_ids": (S, np.int32),
                  "sorted_weights": (S, np.float32), "reverse_indices": (S, np.int32)}

    dev = ctypes.c_int()
    ok(cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()), "cuDeviceGet")
    ctx = ctypes.c_void_p()
    ok(cu.cuCtxCreate_v4(ctypes.byref(ctx), None, 0, dev), "cuCtxCreate")   # current on this thread now
    ptrs = {}
    try:
        def alloc(name, nbytes):
            p = ctypes.c_uint64()
            ok(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
            ptrs[name] = p.value
        for name, a in host_in.items():
            alloc(name, a.nbytes)
            ok(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(ptrs[name]), a.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(a.nbytes)), "cuMemcpyHtoD")
        for name, (n, dt) in out_shapes.items():
            alloc(name, n * np.dtype(dt).itemsize)
        alloc("status", 4)
        zero = np.zeros(1, np.int32)
        ok(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(ptrs["status"]), zero.ctypes.data_as(ctypes.c_void_p),
                              ctypes.c_size_t(4)), "cuMemcpyHtoD")
        for call in range(2):
            rc = moe.lib().moe_align_by_expert_noalloc(
                ptrs["indices"], ptrs["weights"], T, k, E, ptrs["counts"], ptrs["offsets"],
                ptrs["sorted_token_ids"], ptrs["sorted_weights"], ptrs["reverse_indices"], ptrs["status"], None)
            assert rc == 0, moe.lib().moe_last_error().decode()
            ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
            for name, (n, dt) in out_shapes.items():
                got = np.empty(n, dt)
                ok(cu.cuMemcpyDtoH_v2(got.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(ptrs[name]),
                                      ctypes.c_size_t(got.nbytes)), "cuMemcpyDtoH")
                assert np.array_equal(got.view(np.int32), want[name].reshape(-1).view(np.int32)), (call, name)
            st = np.empty(1, np.int32)
            ok(cu.cuMemcpyDtoH_v2(st.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(ptrs["status"]),
                                  ctypes.c_size_t(4)), "cuMemcpyDtoH")
            assert st[0] == 0
    finally:
        for p in ptrs.values():
            cu.cuMemFree_v2(ctypes.c_uint64(p))
        cu.cuCtxDestroy_v2(ctx)
    # back in the primary context, the cached address still serves
    got = moe.moe_align_by_expert_noalloc(idx, w, E)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(got[key], ref[key]), key

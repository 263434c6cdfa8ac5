"""GPU parity of the grouped FFN and of the whole layer against the oracle, through the C ABI.

Tolerance: max|err| <= 2e-2 * max|ref| for bf16 inputs with fp32
accumulation, 1e-4 for float32. Full-size workloads are compared on a
seeded sample of tokens (plus every token of the least-loaded experts), each
row computed independently by the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_close_rel_max, layer_tolerance, need_gpu, to_dev, to_np64
from moe_inputs import WORKLOADS, make_layer_inputs
from oracle import align, ffn, gating

pytestmark = pytest.mark.gpu


def _layer(moe, d, status=None):
    dt = d["dtype"]
    tw = torch.empty((d["T"], d["k"]), dtype=torch.float32, device=DEV)
    ti = torch.empty((d["T"], d["k"]), dtype=torch.int32, device=DEV)
    out = moe.moe_layer_forward(to_dev(d["hidden"], dt), torch.from_numpy(d["logits"]).to(DEV),
                                to_dev(d["w13"], dt), to_dev(d["w2"], dt), d["k"], d["norm_topk_prob"],
                                topk_weights=tw, topk_indices=ti, status=status)
    torch.cuda.synchronize()
    return out, tw, ti


def _full_check(moe, d):
    out, tw, ti = _layer(moe, d)
    ref = ffn.layer_forward(d["logits"], d["hidden"], d["w13"], d["w2"], d["k"], d["norm_topk_prob"],
                            d["dtype"])
    np.testing.assert_array_equal(ti.cpu().numpy(), ref["topk_indices"])
    np.testing.assert_allclose(tw.cpu().numpy(), ref["topk_weights"], rtol=1e-6, atol=0)
    assert_close_rel_max(to_np64(out), ref["out"], layer_tolerance(d["dtype"]), "layer out")


def test_tiny_f32_workload_full():
    moe = need_gpu()
    _full_check(moe, make_layer_inputs("tiny"))


@pytest.mark.parametrize("name", ["decode1", "decode8", "decode64"])
def test_decode_workloads_full(name):
    moe = need_gpu()
    _full_check(moe, make_layer_inputs(name))


# tensor-core path: H, I multiples of 64; ragged expert counts, several tiles, a tail
@pytest.mark.parametrize("T,H,I,E,k,norm", [
    (1, 64, 64, 4, 1, True),
    (5, 128, 192, 8, 2, True),          # I % 128 == 64: half-empty last gate/up tile
    (300, 256, 256, 8, 2, True),        # counts ~75 per expert, one ragged M tile each
    (700, 512, 384, 8, 2, False),
    (1000, 256, 128, 16, 4, True),      # several M tiles per expert + tail
    (513, 320, 640, 5, 3, True),        # H % 256 == 64: partial FC2 N tile
    (2048, 1024, 512, 64, 8, False),
    (257, 128, 128, 128, 8, True),      # many empty experts
    (128, 128, 256, 128, 8, True),      # largest batch of the one-launch routing, E = 128
    (100, 128, 128, 256, 8, False),     # one-launch routing with a warp per token (E > 128)
    (129, 256, 128, 64, 8, True),       # first batch size past the one-launch routing
    (90, 192, 192, 12, 3, False),       # E % 4 != 0: scalar row staging
    (150, 8256, 128, 4, 2, True),       # rows over 16 KB: the vector-copy gather instead of bulk copies
])
def test_layer_tensor_core_shapes(T, H, I, E, k, norm):
    moe = need_gpu()
    _full_check(moe, make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=norm, dtype="bf16",
                                       logits="distinct", seed=T + H))


# decode (weight-streaming, T <= 64) kernels at every token-chunk width and around the threshold;
# in the layer call FC1 routes its tokens itself when E <= 64 and T <= 16 (else it waits
# for the routing kernel): E % 4 != 0, k > 8, norm=False and both fallbacks are covered
@pytest.mark.parametrize("T,H,I,E,k,norm", [
    (1, 256, 128, 8, 2, True), (3, 128, 192, 16, 4, True), (16, 256, 256, 64, 8, True),
    (17, 128, 384, 32, 8, True), (33, 192, 320, 64, 8, True), (64, 256, 128, 8, 2, True),
    (64, 128, 256, 64, 8, True), (65, 128, 256, 64, 8, True),
    (2, 128, 128, 5, 3, False), (12, 128, 128, 64, 10, True), (8, 128, 128, 100, 8, True),
    (60, 128, 128, 64, 9, False),
])
def test_layer_decode_shapes(T, H, I, E, k, norm):
    moe = need_gpu()
    _full_check(moe, make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=norm, dtype="bf16",
                                       logits="distinct", seed=T * 7))


# matrix-vector path (bf16, T <= 2): rows longer than one round of a warp's pieces (H > 2048),
# piece counts that are not a multiple of 32 (I = 1408, 448), rows of only 8 pieces
# (H = I = 64), experts shared by both tokens, routing inside each CTA (E <= 64) and from
# the routing kernel (E > 64), 64 slots (k = 32); in the one-kernel form, output columns
# enough for many rounds of FC2 buffers per CTA (H = 8192 / 4096) and an odd H / 64
@pytest.mark.parametrize("T,H,I,E,k,norm", [
    (1, 2112, 1408, 4, 4, True), (2, 2112, 448, 4, 3, False), (1, 64, 64, 8, 8, True),
    (2, 64, 192, 3, 3, True), (2, 256, 128, 100, 8, True), (2, 128, 128, 64, 32, False),
    (1, 128, 320, 200, 32, True), (1, 8192, 64, 4, 2, True), (2, 4096, 128, 8, 5, False),
    (1, 4160, 192, 16, 9, True),
])
def test_layer_matrix_vector_shapes(T, H, I, E, k, norm):
    moe = need_gpu()
    _full_check(moe, make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=norm, dtype="bf16",
                                       logits="distinct", seed=T * 11 + E))


# one token routed inside each CTA by expert ranks: logits on a coarse grid (ties inside
# and across the top k), all equal (the k lowest experts win), E below one warp's width
@pytest.mark.parametrize("E,k,kind,H,I", [(64, 8, "coarse", 2048, 1408), (40, 6, "coarse", 256, 128),
                                          (64, 8, "flat", 256, 128), (17, 5, "flat", 128, 64),
                                          (33, 32, "coarse", 128, 64)])
def test_layer_one_token_tied_logits(E, k, kind, H, I):
    moe = need_gpu()
    d = make_layer_inputs(T=1, H=H, I=I, E=E, k=k, norm_topk_prob=True, dtype="bf16", logits="distinct",
                          seed=E + k)
    d["logits"] = (np.round(d["logits"] * 2) / 2 if kind == "coarse" else
                   np.full_like(d["logits"], 0.25)).astype(np.float32)
    _full_check(moe, d)


# the small-batch routing kernel waits for the kernel before it on the stream (which
# here writes the logits) before the FFN kernel, which reads the logits at once, may
# start: logits produced on the GPU just before each call, no synchronisation between
@pytest.mark.parametrize("T,E,k", [(1, 64, 8), (2, 32, 4), (5, 16, 2)])
def test_layer_logits_written_by_the_previous_kernel(T, E, k):
    moe = need_gpu()
    H, I = 256, 128
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=True, dtype="bf16", logits="distinct",
                          seed=T * 7 + E)
    hid, w13, w2 = to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16")
    g = torch.Generator(device=DEV)
    g.manual_seed(T + E)
    outs, logits_all = [], []
    for r in range(4):
        # a chain of device ops ending in the logits: the last one runs right before the call
        base = torch.randn((T, E), generator=g, device=DEV, dtype=torch.float64)
        logits = (base * 1.5 + 0.25 * r).to(torch.float32)
        outs.append(moe.moe_layer_forward(hid, logits, w13, w2, k, True))
        logits_all.append(logits)
    torch.cuda.synchronize()
    for out, logits in zip(outs, logits_all):
        lg = logits.cpu().numpy()
        ref = ffn.layer_forward(lg, d["hidden"], d["w13"], d["w2"], k, True, "bf16")["out"]
        assert_close_rel_max(to_np64(out), ref, layer_tolerance("bf16"), "layer out")


# CUDA-core path: float32, and bf16 shapes the tensor path does not take
@pytest.mark.parametrize("T,H,I,E,k,dtype", [
    (64, 128, 256, 8, 2, "f32"),
    (33, 40, 24, 3, 2, "f32"),
    (100, 72, 56, 6, 3, "bf16"),
    (1, 8, 8, 2, 2, "f32"),
])
def test_layer_cuda_core_shapes(T, H, I, E, k, dtype):
    moe = need_gpu()
    _full_check(moe, make_layer_inputs(T=T, H=H, I=I, E=E, k=k, norm_topk_prob=True, dtype=dtype,
                                       logits="distinct", seed=T))


def test_grouped_ffn_entry_point_with_oracle_routing():
    """moe_grouped_ffn fed the oracle's own align outputs."""
    moe = need_gpu()
    d = make_layer_inputs(T=400, H=256, I=320, E=12, k=3, norm_topk_prob=True, dtype="bf16",
                          logits="zipf", seed=5)
    w, i = gating.softmax_topk(d["logits"], 3, True)
    al = align.align_by_expert(i, w, 12)
    t = {k_: torch.from_numpy(np.ascontiguousarray(al[k_])).to(DEV)
         for k_ in ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")}
    out = moe.moe_grouped_ffn(to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16"),
                              3, t["counts"], t["offsets"], t["sorted_token_ids"], t["sorted_weights"],
                              t["reverse_indices"])
    torch.cuda.synchronize()
    ref = ffn.grouped_ffn(d["hidden"], d["w13"], d["w2"], "bf16", 3, al["counts"], al["offsets"],
                          al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"])
    assert_close_rel_max(to_np64(out), ref, 2e-2, "grouped ffn")


# Expert counts chosen so that every kind of last M tile occurs: none (a multiple of 256),
# swapped with 64 token columns (remainder 1..64), swapped with 128 (65..128), and a plain
# 256-row tile (129..255); k = 2 with even experts in slot 0 and odd experts in slot 1.
@pytest.mark.parametrize("H,I", [(320, 384), (256, 320)])
def test_grouped_ffn_every_last_tile_kind(H, I):
    moe = need_gpu()
    even = [256, 300, 64, 385, 0, 571]
    odd = [330, 384, 65, 129, 1, 667]
    T, E, k = sum(even), 12, 2
    assert sum(odd) == T
    rng = np.random.default_rng(H + I)
    idx = np.empty((T, k), np.int32)
    idx[:, 0] = rng.permutation(np.repeat(np.arange(0, E, 2), even))
    idx[:, 1] = rng.permutation(np.repeat(np.arange(1, E, 2), odd))
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=H * I)
    al = align.align_by_expert(idx, w, E)
    assert al["counts"][0::2].tolist() == even and al["counts"][1::2].tolist() == odd
    t = {k_: torch.from_numpy(np.ascontiguousarray(al[k_])).to(DEV)
         for k_ in ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")}
    out = moe.moe_grouped_ffn(to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16"),
                              k, t["counts"], t["offsets"], t["sorted_token_ids"], t["sorted_weights"],
                              t["reverse_indices"])
    torch.cuda.synchronize()
    ref = ffn.grouped_ffn(d["hidden"], d["w13"], d["w2"], "bf16", k, al["counts"], al["offsets"],
                          al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"])
    assert_close_rel_max(to_np64(out), ref, 2e-2, "grouped ffn, every last-tile kind")


# Remainders of every size (1, 31..33, 63..65, 129) after one to three full 256-row tiles,
# with enough tiles that each SM pair runs several in a row, so the two accumulator
# buffers alternate between full, swapped and ragged tiles.
@pytest.mark.parametrize("H,I", [(1024, 1024), (1216, 320)])
def test_grouped_ffn_remainders_after_full_tiles(H, I):
    moe = need_gpu()
    counts = [769, 800, 801, 832, 833, 768, 785, 816, 261, 316, 287, 385, 552, 0, 63, 256, 513, 577]
    E, k = len(counts), 1
    T = sum(counts)
    rng = np.random.default_rng(H - I)
    idx = rng.permutation(np.repeat(np.arange(E), counts)).astype(np.int32).reshape(T, 1)
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype="bf16", logits="distinct", seed=H + I)
    al = align.align_by_expert(idx, w, E)
    assert al["counts"].tolist() == counts
    t = {k_: torch.from_numpy(np.ascontiguousarray(al[k_])).to(DEV)
         for k_ in ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")}
    out = moe.moe_grouped_ffn(to_dev(d["hidden"], "bf16"), to_dev(d["w13"], "bf16"), to_dev(d["w2"], "bf16"),
                              k, t["counts"], t["offsets"], t["sorted_token_ids"], t["sorted_weights"],
                              t["reverse_indices"])
    torch.cuda.synchronize()
    ref = ffn.grouped_ffn(d["hidden"], d["w13"], d["w2"], "bf16", k, al["counts"], al["offsets"],
                          al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"])
    got = to_np64(out)
    assert_close_rel_max(got, ref, 2e-2, "grouped ffn, remainders after full tiles")
    # rows of the remainders alone, so a wrong remainder cannot hide under the global maximum
    off = al["offsets"]
    rem = np.concatenate([al["sorted_token_ids"][off[e] + (c // 256) * 256: off[e] + c]
                          for e, c in enumerate(counts) if c >= 256 and 0 < c % 256 <= 64])
    assert_close_rel_max(got[rem], ref[rem], 2e-2, "remainder rows")


@pytest.mark.parametrize("T,H,I,E,k", [(300, 256, 256, 8, 2), (40, 128, 128, 16, 4), (90, 40, 24, 5, 2),
                                       (1, 256, 256, 8, 6), (2, 128, 192, 16, 8)])
def test_grouped_ffn_dropped_slots_contribute_nothing(T, H, I, E, k):
    """Slots whose expert index is outside [0, E) are dropped by the align step; the FFN must
    ignore them even when the workspace holds stale data (filled with NaN bytes here)."""
    moe = need_gpu()
    dt = "bf16" if H % 64 == 0 else "f32"
    d = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, dtype=dt, logits="distinct", seed=T + k)
    w, idx = gating.softmax_topk(d["logits"], k, True)
    idx = idx.copy()
    rng = np.random.default_rng(T)
    drop = rng.random(idx.shape) < 0.2
    idx[drop] = np.where(rng.random(int(drop.sum())) < 0.5, -1, E + 3)
    al = align.align_by_expert(idx, w, E)
    assert al["valid_slots"] < T * k
    t = {k_: torch.from_numpy(np.ascontiguousarray(al[k_])).to(DEV)
         for k_ in ("counts", "offsets", "sorted_token_ids", "sorted_weights", "reverse_indices")}
    code = moe.MOE_BF16 if dt == "bf16" else moe.MOE_F32
    ws = torch.full((moe.moe_grouped_ffn_workspace_size(code, T, H, I, E, k),), 0xFF, dtype=torch.uint8, device=DEV)
    out = moe.moe_grouped_ffn(to_dev(d["hidden"], dt), to_dev(d["w13"], dt), to_dev(d["w2"], dt), k,
                              t["counts"], t["offsets"], t["sorted_token_ids"], t["sorted_weights"],
                              t["reverse_indices"], workspace=ws)
    torch.cuda.synchronize()
    ref = ffn.grouped_ffn(d["hidden"], d["w13"], d["w2"], dt, k, al["counts"], al["offsets"],
                          al["sorted_token_ids"], al["sorted_weights"], al["reverse_indices"])
    assert_close_rel_max(to_np64(out), ref, layer_tolerance(dt), "grouped ffn with dropped slots")


def test_layer_repeated_calls_are_identical():
    moe = need_gpu()
    d = make_layer_inputs(T=600, H=256, I=256, E=8, k=2, dtype="bf16", logits="distinct", seed=9)
    a, _, _ = _layer(moe, d)
    b, _, _ = _layer(moe, d)
    assert torch.equal(a, b)


def test_layer_status_stays_clear():
    moe = need_gpu()
    d = make_layer_inputs(T=300, H=128, I=128, E=8, k=2, dtype="bf16", logits="distinct", seed=2)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _layer(moe, d, status=st)
    assert int(st.item()) == 0


def _sample_tokens(ti_np, T, E, n, seed):
    rng = np.random.default_rng(seed)
    tok = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    counts = np.bincount(ti_np.reshape(-1), minlength=E)
    light = [e for e in np.argsort(counts, kind="stable") if counts[e] > 0][:8]
    for e in light:
        rows = np.nonzero((ti_np == e).any(axis=1))[0][:64]
        tok.update(rows.tolist())
    return np.array(sorted(tok), dtype=np.int64)


@pytest.mark.slow
@pytest.mark.parametrize("name,n", [("mixtral", 512), ("fine", 512), ("skew", 384)])
def test_full_size_workload_sampled(name, n):
    moe = need_gpu()
    d = make_layer_inputs(name)
    out, tw, ti = _layer(moe, d)
    w_ref, i_ref = gating.softmax_topk(d["logits"], d["k"], d["norm_topk_prob"])
    ti_np = ti.cpu().numpy()
    np.testing.assert_array_equal(ti_np, i_ref)
    np.testing.assert_allclose(tw.cpu().numpy(), w_ref, rtol=1e-6, atol=0)
    tok = _sample_tokens(ti_np, d["T"], d["E"], n, seed=1)
    ref = ffn.layer_rows(d["hidden"], d["w13"], d["w2"], d["dtype"], w_ref, i_ref, tok)
    got = to_np64(out[torch.from_numpy(tok).to(DEV)])
    assert_close_rel_max(got, ref, 2e-2, f"{name} sampled rows")
    assert np.isfinite(to_np64(out)).all()

"""Benchmark of the MoE layer forward path (one step = gating -> align -> grouped FFN -> combine).

Default (headline) workload: the skewed-load large-E prefill, bf16 (T=32768,
H=4096, I=1536, E=128, top_k=8, norm_topk_prob=True, Zipf(1.2) expert bias),
the largest configuration; synthetic seeded inputs resident in HBM. After it,
the JSON line's "workloads" object holds every other configuration (tiny f32,
Mixtral-shaped prefill, decode T = 1 / 8 / 64, fine-grained prefill), each
timed for at least 1 s and 200 steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0). Under torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (no data-path collective);
`value` is the total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_inputs import WORKLOADS  # noqa: E402

METRIC = "MoE layer tokens/sec; grouped-FFN TFLOPS & routing GB/s as % of GB300 peak"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="skew", choices=list(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations (each timed >= 1 s after the headline workload)")
    ap.add_argument("--no-routing", action="store_true", help="skip the large-T routing bandwidth section")
    ap.add_argument("--no-backward", action="store_true", help="skip the FFN backward section")
    ap.add_argument("--backward-only", action="store_true",
                    help="only the FFN backward section (for profiling captures)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's T (profiling captures)")
    ap.add_argument("--experts", type=int, default=None, help="override the workload's E (profiling captures)")
    ap.add_argument("--topk", type=int, default=None, help="override the workload's k (profiling captures)")
    ap.add_argument("--routing-only", action="store_true",
                    help="only the large-T routing bandwidth section (prints it as JSON; for profiling)")
    ap.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                    help="time the step as a CUDA graph replay (auto: on for decode batches, T <= 64)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (the slowest rank's time); x itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, world: int, steps: int, ms_total: float) -> float:
    """Tokens/s of the whole job: every rank runs its own replica of the workload, so the
    job processes tokens_per_rank * world tokens per step in the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms_total / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d.get("hbm_gbs", 6800.0), bf16_tflops=d.get("bf16_tflops", 1900.0),
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", 1700.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_device_inputs(wl, device, seed=0):
    """Seeded synthetic inputs drawn on the device (same recipes as moe_inputs, torch RNG):
    rows of the logits holding a repeated value are redrawn, as the recipes ask."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    hidden, logits = draw_tokens(wl, device, g, seed)
    H, I, E = wl.H, wl.I, wl.E
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    w13 = torch.empty((E, 2 * I, H), device=device, dtype=dt)
    w2 = torch.empty((E, H, I), device=device, dtype=dt)
    for e in range(E):   # one expert at a time keeps the fp32 temporaries small
        w13[e] = (torch.randn((2 * I, H), generator=g, device=device) / H ** 0.5).to(dt)
        w2[e] = (torch.randn((H, I), generator=g, device=device) / I ** 0.5).to(dt)
    return hidden, logits, w13, w2


def draw_tokens(wl, device, g, seed):
    """hidden [T, H] and router logits [T, E] of one batch from generator g."""
    import torch
    T, H, E = wl.T, wl.H, wl.E
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    hidden = torch.randn((T, H), generator=g, device=device, dtype=torch.float32).to(dt)
    bias = torch.zeros(E, device=device, dtype=torch.float32)
    if wl.logits == "jitter":
        bias = 1e-3 * torch.arange(E, device=device, dtype=torch.float32)
    elif wl.logits == "zipf":
        r = torch.arange(1, E + 1, dtype=torch.float64)
        p = r ** -1.2
        by_rank = (2.0 * torch.log(p / p.sum())).float()
        perm = torch.randperm(E, generator=torch.Generator().manual_seed(seed))
        b = torch.empty(E)
        b[perm] = by_rank
        bias = b.to(device)
    logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float32) + bias
    for _ in range(100):   # "distinct values": redraw rows with a repeated logit
        srt = torch.sort(logits, dim=1).values
        bad = torch.nonzero((srt[:, 1:] == srt[:, :-1]).any(dim=1)).flatten()
        if bad.numel() == 0:
            break
        logits[bad] = torch.randn((bad.numel(), E), generator=g, device=device, dtype=torch.float32) + bias
    return hidden, logits


# Decode batches (T <= DECODE_T) rotate over this many token batches, one per step, so
# that consecutive steps route to different experts, as consecutive decode steps do:
# with one batch repeated, the ~L2-sized set of expert rows a step reads would partly
# stay in L2 from the step before.
DECODE_T, DECODE_BATCHES = 64, 8


def routing_bandwidth(moe, wl, dev, peaks, reps=10, target_bytes=768 << 20):
    """Each routing kernel on a token count large enough that its inputs and outputs
    (>= 768 MiB) stream through HBM rather than L2: algorithmic bytes / CUDA-event time.

    Bytes per token (what the method must move at the least):
      gating 4E + 8k (bf16 logits: 2E + 8k); indices->multihot 8k + 9E;
      multihot->indices 8E + 8k (probs and indices out); align 8k in + 12k out (+ E-sized
      tables); group-limited top-k (DeepSeek-V3 shape E=256, 8 groups, keep 4, k=8) 4E + 8k.
    """
    import torch
    E, k = wl.E, wl.k
    per_tok = {"gating_softmax_topk": 4 * E + 8 * k, "gating_softmax_topk_bf16": 2 * E + 8 * k,
               "indices_to_multihot": 8 * k + 9 * E,
               "multihot_to_indices": 8 * E + 8 * k, "align_by_expert": 20 * k}
    T = max(1, int(target_bytes // (8 * E + 8 * k)))
    T = min(T, (1 << 31) // max(k, 1) - 1)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    logits = torch.randn((T, E), generator=g, device=dev)
    logits_bf16 = logits.to(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    w, idx = moe.moe_gating_softmax_topk(logits, k, wl.norm_topk_prob)
    mh, pm, pos = moe.moe_indices_to_multihot(idx, w, E)
    p2, i2 = moe.moe_multihot_to_indices(pm, pos, k)
    ws = torch.empty(max(1, moe.moe_align_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)
    al = moe.moe_align_by_expert(idx, w, E, workspace=ws)
    calls = {
        "gating_softmax_topk": lambda st: moe.moe_gating_softmax_topk(logits, k, wl.norm_topk_prob, weights=w,
                                                                      indices=idx, stream=st),
        "gating_softmax_topk_bf16": lambda st: moe.moe_gating_softmax_topk_bf16(
            logits_bf16, k, wl.norm_topk_prob, weights=w, indices=idx, stream=st),
        "indices_to_multihot": lambda st: moe.moe_indices_to_multihot(idx, w, E, multihot=mh, probs_in_multihot=pm,
                                                                      position_map=pos, stream=st),
        "multihot_to_indices": lambda st: moe.moe_multihot_to_indices(pm, pos, k, probs=p2, indices=i2, stream=st),
        "align_by_expert": lambda st: moe.moe_align_by_expert(idx, w, E, out=al, workspace=ws, stream=st),
    }
    res = {}
    inner = 10   # calls per captured graph: the timed launches run back to back, with no host gap

    def timed(fn, nbytes, tokens=T):
        for _ in range(2):
            fn(stream)
        torch.cuda.synchronize()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(gr, stream=side, capture_error_mode="thread_local"):
                for _ in range(inner):
                    fn(side)
        torch.cuda.synchronize()
        gr.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            gr.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / (reps * inner)
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"tokens": tokens, "us": ms * 1e3, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"], "bytes": nbytes,
                "timing": "CUDA graph of %d calls replayed %d times" % (inner, reps)}

    for name, fn in calls.items():
        res[name] = timed(fn, per_tok[name] * T)
    del logits, logits_bf16, mh, pm, pos, p2, i2, al, ws
    # DeepSeek-V3-shaped group-limited routing on sigmoid scores
    Eg, kg = 256, 8
    Tg = int(target_bytes // (4 * Eg + 8 * kg))
    sc = torch.sigmoid(torch.randn((Tg, Eg), generator=g, device=dev))
    bias = 0.05 * torch.randn((Eg,), generator=g, device=dev)
    gw, gi = moe.moe_group_limited_topk(sc, kg, 8, 4, "noaux_tc", bias=bias)
    res["group_limited_topk"] = timed(
        lambda st: moe.moe_group_limited_topk(sc, kg, 8, 4, "noaux_tc", bias=bias, weights=gw, indices=gi, stream=st),
        (4 * Eg + 8 * kg) * Tg, Tg)
    res["group_limited_topk"]["shape"] = "E=256, n_group=8, topk_group=4, k=8, noaux_tc"
    return res


def backward_bench(moe, wl, dev, hidden, logits, w13, w2, peaks, steps):
    """FFN backward (moe_grouped_ffn_backward) on the workload's own routing and a seeded
    N(0,1) upstream gradient: CUDA-event time per step (no per-kernel events), then a
    separate pass with per-kernel events. Routed flops per step: FC1 recomputed
    (2 S H 2I), dA (2 S H I), dX (2 S 2I H), dW2 (2 S H I), dW13 (2 S 2I H) = 16 S H I."""
    import torch
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    w, idx = moe.moe_gating_softmax_topk(logits, k, wl.norm_topk_prob)
    aws = torch.empty(max(1, moe.moe_align_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)
    al = moe.moe_align_by_expert(idx, w, E, workspace=aws)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    d_out = torch.randn((T, H), generator=g, device=dev).to(hidden.dtype)
    ws = torch.empty(moe.moe_grouped_ffn_backward_workspace_size(moe.MOE_BF16, T, H, I, E, k), dtype=torch.uint8,
                     device=dev)
    outs = dict(d_hidden=torch.empty_like(hidden), d_w13=torch.empty_like(w13), d_w2=torch.empty_like(w2),
                d_weights=torch.empty((T, k), dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream(dev)

    def step():
        moe.moe_grouped_ffn_backward(hidden, w13, w2, k, al["counts"], al["offsets"], al["sorted_token_ids"],
                                     al["sorted_weights"], al["reverse_indices"], d_out, workspace=ws,
                                     stream=stream, **outs)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    moe.profiler_enable(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    moe.profiler_enable(False)
    kern = {n: round(v["total_ms"] / steps, 4) for n, v in moe.profiler_report().items()}
    flops = 16.0 * T * k * H * I
    tf = flops / (ms / 1e3) / 1e12
    return {"ms_per_step": ms, "tflops": tf, "peak_tflops": peaks["bf16_tflops"],
            "frac": tf / peaks["bf16_tflops"], "flops_per_step": flops,
            "flops": "routed work 16*S*H*I (FC1 recomputed, dA, dX, dW2, dW13)", "kernels_ms": kern,
            "timing": "CUDA events over %d steps after 3 warm-up steps; kernels_ms from a second pass" % steps}


def kernel_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or None when the
    capture is for another workload or the kernel sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec["bytes_per_launch"] if h.hexdigest() == rec["source_sha256"] else None


def cpu_baseline(wl, hidden, logits, w13, w2, budget_s=20.0):
    """The oracle as it stands, on the host cores, over a bounded sample of tokens."""
    from oracle import ffn, gating
    import torch
    t0 = time.perf_counter()
    lg = logits.cpu().numpy()
    wts, idx = gating.softmax_topk(lg, wl.k, wl.norm_topk_prob)
    used = set(np.unique(idx[: min(wl.T, 64)]).tolist())

    def host(t):
        a = t.contiguous().cpu()
        return a.view(torch.int16).numpy().view(np.uint16) if a.dtype == torch.bfloat16 else a.numpy()

    hid = host(hidden)
    w13h = {e: host(w13[e]) for e in used}
    w2h = {e: host(w2[e]) for e in used}

    class Lazy:
        def __init__(self, d):
            self.d = d

        def __getitem__(self, e):
            return self.d[int(e)]

        def __len__(self):
            return wl.E

    copy_s = time.perf_counter() - t0
    n, tot, done = 8, 0.0, 0
    start = time.perf_counter()
    while done < min(wl.T, 64):
        tok = np.arange(done, min(done + n, wl.T, 64))
        t1 = time.perf_counter()
        ffn.layer_rows(hid, Lazy(w13h), Lazy(w2h), wl.dtype, wts, idx, tok)
        tot += time.perf_counter() - t1
        done += len(tok)
        if time.perf_counter() - start > budget_s:
            break
    # routing over the whole batch is part of every token's cost
    t2 = time.perf_counter()
    wts, idx = gating.softmax_topk(lg, wl.k, wl.norm_topk_prob)
    route_s = time.perf_counter() - t2
    per_tok = tot / max(done, 1) + route_s / wl.T
    return {"value": 1.0 / per_tok, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"numpy float64 oracle: routing over all {wl.T} tokens + FFN/combine of the "
                      f"first {done} tokens (host copy of {len(used)} experts' weights, {copy_s:.1f}s, "
                      f"not counted); BLAS threads = all host cores"}


def run_reference(args, wl, rank, world):
    """--impl reference: the oracle on the host cores, one bounded sample per step."""
    if rank != 0:
        return
    import torch
    from oracle import ffn, gating
    import moe_inputs as mi
    d = mi.make_layer_inputs(wl, with_weights=False)
    n_tok = max(1, min(8, 16 // wl.k))     # at most 16 experts' weights touched per step
    tok = np.arange(n_tok)
    w, i = gating.softmax_topk(d["logits"], wl.k, wl.norm_topk_prob)
    used = sorted(set(np.unique(i[:n_tok]).tolist()))
    # weights only for the experts the sample touches (same distribution, per-expert seeds)
    w13 = {e: mi.gen_normal(np.random.SeedSequence([wl.seed, 13, e]), (2 * wl.I, wl.H), 1 / np.sqrt(wl.H), wl.dtype)
           for e in used}
    w2 = {e: mi.gen_normal(np.random.SeedSequence([wl.seed, 2, e]), (wl.H, wl.I), 1 / np.sqrt(wl.I), wl.dtype)
          for e in used}

    class Lazy:
        def __init__(self, dd):
            self.d = dd

        def __getitem__(self, e):
            return self.d[int(e)]

        def __len__(self):
            return wl.E

    def step():
        ww, ii = gating.softmax_topk(d["logits"], wl.k, wl.norm_topk_prob)
        ffn.layer_rows(d["hidden"], Lazy(w13), Lazy(w2), wl.dtype, ww, ii, tok)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    # one step = routing of all T tokens + FFN of n_tok tokens; scale FFN to the whole batch
    t1 = time.perf_counter()
    gating.softmax_topk(d["logits"], wl.k, wl.norm_topk_prob)
    route = time.perf_counter() - t1
    per_tok = (dt - route) / n_tok + route / wl.T
    value = 1.0 / per_tok
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, world),
            "inputs": "seeded numpy PCG64 on the host (moe_inputs recipes; weights only of the experts the "
                      "sample touches, drawn per expert)",
            "timing": "wall clock over the steps on the host cores",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"each step: oracle routing of all {wl.T} tokens + FFN of {n_tok} tokens; "
                                       "tokens/s extrapolated per token"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def fp32_simt_peak_tflops():
    """FP32 FMA rate of the CUDA cores: 152 SMs x 128 lanes x 2 flop x 2.07 GHz."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def dominant_roofline(moe, wl, kern, logits, peaks, step_ms, prof_s=0.0):
    """Roofline of the kernel that bounds the workload, from the per-kernel CUDA-event times.

    The per-kernel times come from a pass of prof_s seconds of eager steps: a kernel timed
    inside a pass of 0.5 s or more ran under the power cap, so a tensor-bound kernel is
    held against the sustained bf16 peak there, and against the burst peak otherwise.

    decode, one kernel (T <= 2 inside the layer call): ffn_decode_layer streams every
    active expert's w13 and w2 rows; algorithmic bytes = those rows + the token rows +
    the activations written and read back + the output.
    decode, two kernels (T <= 64): ffn_fc1_gemv (T <= 2, CUDA-core matrix-vector
    products) or ffn_fc1_decode (tensor cores) streams the weight rows of the experts
    the batch routes to: algorithmic bytes = those rows + the token rows + the
    activations written. Both add the layer step's bandwidth over all active expert
    weights (w13 and w2).
    prefill bf16: ffn_fc1_tc, 2 S H 2I flops per launch against the measured bf16 burst peak.
    float32 (CUDA cores): ffn_fc1_simt, the same flops against the FP32 FMA rate.
    """
    import torch
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    S = T * k
    lay = kern.get("ffn_decode_layer")
    if lay and lay["launches"]:
        # one kernel for the whole FFN: every active expert's w13 and w2 rows, the
        # token rows, the activations written and read back, the output written
        _, ti = moe.moe_gating_softmax_topk(logits, k, wl.norm_topk_prob)
        active = int(torch.unique(ti).numel())
        nbytes = float(active * 3 * I * H * 2 + T * H * 2 + 2 * S * I * 2 + T * H * 2)
        lay_ms = lay["total_ms"] / lay["launches"]
        gbs = nbytes / (lay_ms / 1e3) / 1e9
        step_bytes = float(active * 3 * I * H * 2)
        return {"bound": "hbm", "kernel": "ffn_decode_layer", "achieved": gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": kernel_traffic("ffn_decode_layer", wl.name),
                "peak_source": peaks["source"] + " (copy bandwidth)", "active_experts": active,
                "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": lay_ms,
                "layer_step_weight_GBps": step_bytes / (step_ms / 1e3) / 1e9,
                "layer_step_weight_frac": step_bytes / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    dname = next((n for n in ("ffn_fc1_gemv", "ffn_fc1_decode") if kern.get(n) and kern[n]["launches"]), None)
    if dname:
        dec = kern[dname]
        _, ti = moe.moe_gating_softmax_topk(logits, k, wl.norm_topk_prob)
        active = int(torch.unique(ti).numel())
        nbytes = float(active * 2 * I * H * 2 + T * H * 2 + S * I * 2)
        dec_ms = dec["total_ms"] / dec["launches"]
        gbs = nbytes / (dec_ms / 1e3) / 1e9
        step_bytes = float(active * 3 * I * H * 2)
        return {"bound": "hbm", "kernel": dname, "achieved": gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": kernel_traffic(dname, wl.name),
                "peak_source": peaks["source"] + " (copy bandwidth)", "active_experts": active,
                "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": dec_ms,
                "layer_step_weight_GBps": step_bytes / (step_ms / 1e3) / 1e9,
                "layer_step_weight_frac": step_bytes / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    sustained = prof_s >= 0.5
    tc_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    tc_src = peaks["source"] + (" (sustained bf16, cuBLAS: per-kernel pass of %.1f s)" % prof_s if sustained
                                else " (burst bf16, cuBLAS)")
    for name, bound, peak, unit, src in (
            ("ffn_fc1_tc", "tensor", tc_peak, "TFLOP/s", tc_src),
            ("ffn_fc1_simt", "alu", fp32_simt_peak_tflops(), "TFLOP/s",
             "derived: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz")):
        r = kern.get(name)
        if r and r["launches"]:
            ms = r["total_ms"] / r["launches"]
            flops = 2.0 * S * H * (2 * I)
            ach = flops / (ms / 1e3) / 1e12
            return {"bound": bound, "kernel": name, "achieved": ach, "peak": peak, "unit": unit,
                    "frac": ach / peak, "traffic": kernel_traffic(name, wl.name), "peak_source": src,
                    "algorithmic_flops_per_launch": flops, "avg_launch_ms": ms}
    return None


def measure(moe, wl, dev, steps, warmup, graph_mode="auto", with_e2e=True, seed=0, world=1, clocks=False,
            min_seconds=0.0, min_steps=0):
    """One workload: device-timed layer steps, per-kernel times, end-to-end rate.

    steps: timed steps; when min_seconds / min_steps are given the count grows until the
    timed region lasts at least min_seconds (estimated from the warm-up) and min_steps.
    """
    import torch
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    hidden, logits, w13, w2 = make_device_inputs(wl, dev, seed=seed)
    nb = DECODE_BATCHES if T <= DECODE_T else 1
    hiddens, logitss = [hidden], [logits]
    for r in range(1, nb):
        g = torch.Generator(device=dev)
        g.manual_seed(seed * 1000 + r)
        h_r, l_r = draw_tokens(wl, dev, g, seed)
        hiddens.append(h_r)
        logitss.append(l_r)
    dcode = moe.MOE_BF16 if wl.dtype == "bf16" else moe.MOE_F32
    ws = torch.empty(moe.moe_layer_workspace_size(dcode, T, H, I, E, k), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=hidden.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    count = [0]

    def step(s=stream):
        r = count[0] % nb
        count[0] += 1
        moe.moe_layer_forward(hiddens[r], logitss[r], w13, w2, k, wl.norm_topk_prob, out=out, workspace=ws,
                              stream=s)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()

    use_graph = graph_mode == "on" or (graph_mode == "auto" and T <= 64)
    graphs, chain = [], None
    if use_graph:
        # each batch's layer step captured once, and the nb steps in turn captured once
        # more as one graph (what a decode loop does: the steps of a forward pass in one
        # graph); the timed region replays the chain, single steps only for a remainder
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for r in range(nb):
                count[0] = r
                step(side)
                torch.cuda.synchronize()
                gr = torch.cuda.CUDAGraph()
                count[0] = r
                with torch.cuda.graph(gr, stream=side, capture_error_mode="thread_local"):
                    step(side)
                graphs.append(gr)
            chain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(chain, stream=side, capture_error_mode="thread_local"):
                for r in range(nb):
                    count[0] = r
                    step(side)
        torch.cuda.synchronize()
        for gr in graphs + [chain]:
            gr.replay()
        torch.cuda.synchronize()
        count[0] = 0

    def replay_steps(n, single, whole):
        """n layer steps from graphs: the chain of all nb batches where a whole turn is left."""
        i = 0
        while i < n:
            if count[0] % nb == 0 and n - i >= nb:
                whole.replay()
                count[0] += nb
                i += nb
            else:
                single[count[0] % nb].replay()
                count[0] += 1
                i += 1

    def run(n):
        if use_graph:
            replay_steps(n, graphs, chain)
            return
        for _ in range(n):
            step()

    if min_seconds > 0 or min_steps > 0:   # size the timed region from a short probe
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run(5)
        b.record(stream)
        torch.cuda.synchronize()
        est = max(a.elapsed_time(b) / 5, 1e-3)
        steps = max(steps, min_steps, int(min_seconds * 1e3 / est) + 1)

    # per-kernel CUDA-event times (each kernel bracketed on its own stream): a timed
    # pass of eager steps just before the timed region
    clk = None
    if clocks:
        clk = ClockSampler(dev.index)
        clk.start()
        time.sleep(0.3)
    n_prof = min(steps, 200)
    moe.profiler_enable(True)
    for _ in range(n_prof):
        step()
    torch.cuda.synchronize()
    moe.profiler_enable(False)
    kern = moe.profiler_report()

    # ---- timed region: the steps, device events on the launching stream. No events
    # between the layer's kernels here: an event recorded between two launches
    # serialises the programmatic dependent launch of the second one.
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    run(steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk_rec = clk.stop() if clk else None
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms = ms_total / steps
    value = whole_job_rate(T, world, steps, ms_total)

    # ---- end to end through the public call: pinned host inputs in, output back to host.
    # Every step copies its inputs in and its output back; with two buffer sets the
    # copies of the neighbouring steps run on two copy streams while a step computes
    # (H2D of step i+1 and D2H of step i-1 overlap step i, as a serving loop would).
    e2e = None
    if with_e2e and use_graph:
        # decode batches: every step copies its inputs from pinned host memory, runs the
        # layer call and copies its output back. Two device buffer sets: in the captured
        # chain the H2D of step i+1 and the D2H of step i-1 run on two copy streams while
        # step i computes; single-step graphs (a remainder) run their copies in line.
        h_hidden = [h.cpu().pin_memory() for h in hiddens]
        h_logits = [x.cpu().pin_memory() for x in logitss]
        h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        d_hidden = [torch.empty_like(hidden) for _ in range(2)]
        d_logits = [torch.empty_like(logits) for _ in range(2)]
        d_out = [torch.empty_like(out) for _ in range(2)]
        gs, s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        gs.wait_stream(stream)

        def copy_in(r):
            d_hidden[r % 2].copy_(h_hidden[r], non_blocking=True)
            d_logits[r % 2].copy_(h_logits[r], non_blocking=True)

        def layer(r):
            moe.moe_layer_forward(d_hidden[r % 2], d_logits[r % 2], w13, w2, k, wl.norm_topk_prob,
                                  out=d_out[r % 2], workspace=ws, stream=gs)

        def copy_out(r):
            h_out[r % 2].copy_(d_out[r % 2], non_blocking=True)

        def e2e_once(r):
            copy_in(r)
            layer(r)
            copy_out(r)

        def e2e_chain():
            ev_in = [torch.cuda.Event() for _ in range(nb)]
            ev_comp = [torch.cuda.Event() for _ in range(nb)]
            ev_out = [torch.cuda.Event() for _ in range(nb)]
            s_in.wait_stream(gs)
            s_out.wait_stream(gs)
            for r in range(nb):
                with torch.cuda.stream(s_in):
                    if r >= 2:
                        s_in.wait_event(ev_comp[r - 2])   # step r-2 has read buffer set r % 2
                    copy_in(r)
                    ev_in[r].record(s_in)
                gs.wait_event(ev_in[r])
                if r >= 2:
                    gs.wait_event(ev_out[r - 2])          # step r-2's output has been read back
                layer(r)
                ev_comp[r].record(gs)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[r])
                    copy_out(r)
                    ev_out[r].record(s_out)
            gs.wait_stream(s_in)
            gs.wait_stream(s_out)

        g_e2e = []
        with torch.cuda.stream(gs):
            for r in range(nb):
                e2e_once(r)
                torch.cuda.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=gs, capture_error_mode="thread_local"):
                    e2e_once(r)
                g_e2e.append(gr)
            c_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(c_e2e, stream=gs, capture_error_mode="thread_local"):
                e2e_chain()
        torch.cuda.synchronize()
        for gr in g_e2e + [c_e2e]:
            gr.replay()
        torch.cuda.synchronize()
        count[0] = 0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        replay_steps(steps, g_e2e, c_e2e)
        b.record(stream)
        torch.cuda.synchronize()
        last = (steps - 1) % nb                   # the copied-back result is the last step's output
        moe.moe_layer_forward(hiddens[last], logitss[last], w13, w2, k, wl.norm_topk_prob, out=out,
                              workspace=ws, stream=stream)
        torch.cuda.synchronize()
        assert torch.equal(h_out[last % 2], out.cpu())
        e_ms = max_over_ranks(a.elapsed_time(b), dev)
        e2e = {"value": whole_job_rate(T, world, steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h_hidden[0].numel() * h_hidden[0].element_size() + h_logits[0].numel() * 4,
               "d2h_bytes_per_step": h_out[0].numel() * h_out[0].element_size(), "ms_per_step": e_ms / steps,
               "copies": "pinned host buffers; every step does the H2D copies of its hidden and logits, the "
                         "layer call and the D2H copy of its output, replayed from CUDA graphs as the timed "
                         "region's steps are; in the chain of %d steps the H2D of step i+1 and the D2H of "
                         "step i-1 overlap step i on two copy streams (two device buffer sets)" % nb}
    elif with_e2e:
        h_hidden = hidden.cpu().pin_memory()
        h_logits = logits.cpu().pin_memory()
        nb = 2
        h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nb)]
        d_hidden = [torch.empty_like(hidden) for _ in range(nb)]
        d_logits = [torch.empty_like(logits) for _ in range(nb)]
        d_out = [torch.empty_like(out) for _ in range(nb)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_comp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]

        def e2e_step(i):
            b = i % nb
            if i >= nb:
                s_in.wait_event(ev_comp[b])        # step i-2 has consumed input set b
            with torch.cuda.stream(s_in):
                d_hidden[b].copy_(h_hidden, non_blocking=True)
                d_logits[b].copy_(h_logits, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= nb:
                stream.wait_event(ev_out[b])       # step i-2's output has been read back
            moe.moe_layer_forward(d_hidden[b], d_logits[b], w13, w2, k, wl.norm_topk_prob, out=d_out[b],
                                  workspace=ws, stream=stream)
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                h_out[b].copy_(d_out[b], non_blocking=True)
            ev_out[b].record(s_out)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_stream(stream)
        for i in range(steps):
            e2e_step(i)
        stream.wait_stream(s_out)
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b), dev)
        e2e = {"value": whole_job_rate(T, world, steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h_hidden.numel() * h_hidden.element_size() + h_logits.numel() * 4,
               "d2h_bytes_per_step": h_out[0].numel() * h_out[0].element_size(),
               "ms_per_step": e_ms / steps,
               "copies": "pinned host buffers; the H2D of step i+1 and the D2H of step i-1 overlap step i "
                         "on two copy streams (two device buffer sets)"}

    peaks = measured_peaks()
    launches = sum(v["launches"] for v in kern.values()) / n_prof
    per_kernel = {n: {"launches_per_step": v["launches"] / n_prof, "avg_ms": v["total_ms"] / max(v["launches"], 1),
                      "share": v["total_ms"] / max(sum(x["total_ms"] for x in kern.values()), 1e-12)}
                  for n, v in kern.items()}
    res = {"value": value, "ms_per_step": ms, "steps": steps, "use_graph": use_graph,
           "layer_tflops": 6.0 * T * k * H * I / (ms / 1e3) / 1e12,
           "roofline": dominant_roofline(moe, wl, kern, logits, peaks, ms, prof_s=n_prof * ms / 1e3),
           "kernels": per_kernel,
           "gpu_launches_per_step": launches, "clocks": clk_rec, "e2e": e2e,
           "timing": ("CUDA graph replay: the %d token batches' layer steps in turn captured as one graph "
                      "(as a decode loop captures a forward pass), replayed steps // %d times, single-step "
                      "graphs for the remainder" % (nb, nb) if use_graph else "eager steps") +
                     "; per-kernel CUDA events (roofline, kernels) from a timed pass of %d eager steps just "
                     "before, since events between launches serialise the programmatic dependent launches" % n_prof,
           }
    return res, (hidden, logits, w13, w2)


def workload_config(wl, world):
    """The workload's configuration, identical for both arms (inputs and timing are reported beside it)."""
    weights_gb = wl.E * 3 * wl.I * wl.H * (2 if wl.dtype == "bf16" else 4) / 1e9
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
            "norm_topk_prob": wl.norm_topk_prob, "dtype": wl.dtype,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": ("inputs larger than L2 (weights %.2f GB)" % weights_gb +
                   ("; steps rotate over %d token batches, so consecutive steps route to different experts"
                    % DECODE_BATCHES if wl.T <= DECODE_T else ""))
                  if weights_gb > 0.2 else "inputs smaller than L2: L2-warm steps (latency-bound workload)"}


INPUTS_NOTE = "seeded torch RNG on device (N(0,1); weights N(0,1/sqrt(fan_in)); distinct logits)"


def main():
    args = parse()
    wl = WORKLOADS[args.workload]
    if args.tokens or args.experts or args.topk:
        import dataclasses
        wl = dataclasses.replace(wl, name=wl.name + "_reduced", T=args.tokens or wl.T, E=args.experts or wl.E,
                                 k=args.topk or wl.k)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    import torch
    import mixture_experts_routing_token_gb300 as moe
    from mixture_experts_routing_token_gb300.build import build
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(moe.LIB_PATH):
        build()
    if world > 1:
        dist.barrier()
    moe.lib()

    if args.routing_only:
        if rank == 0:
            print(json.dumps({"workload": wl.name, "routing": routing_bandwidth(moe, wl, dev, measured_peaks(),
                                                                                 reps=max(1, args.steps))}), flush=True)
        return
    if args.backward_only:
        hidden, logits, w13, w2 = make_device_inputs(wl, dev, seed=rank)
        if rank == 0:
            print(json.dumps({"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                              "backward": backward_bench(moe, wl, dev, hidden, logits, w13, w2, measured_peaks(),
                                                         max(3, min(args.steps, 10)))}), flush=True)
        return

    res, (hidden, logits, w13, w2) = measure(moe, wl, dev, args.steps, args.warmup, args.graph,
                                             with_e2e=not args.no_e2e, seed=rank, world=world, clocks=True)
    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peaks = measured_peaks()
    line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
            "config": workload_config(wl, world), "inputs": INPUTS_NOTE, "timing": res["timing"],
            "layer_tflops": res["layer_tflops"], "roofline": res["roofline"], "kernels": res["kernels"],
            "gpu_launches": res["gpu_launches_per_step"] * args.steps,
            "gpu_launches_per_step": res["gpu_launches_per_step"], "clocks": res["clocks"], "e2e": res["e2e"],
            "lib": moe.version()}
    if not args.no_routing:
        line["routing"] = routing_bandwidth(moe, wl, dev, peaks)
    if not args.no_backward and wl.dtype == "bf16" and wl.H % 64 == 0 and wl.I % 64 == 0:
        line["backward"] = backward_bench(moe, wl, dev, hidden, logits, w13, w2, peaks,
                                          max(3, min(args.steps, 10)))
    if not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline(wl, hidden, logits, w13, w2)
        except Exception as ex:   # the baseline is reported, never required
            line["cpu_baseline"] = {"error": repr(ex)}
    del hidden, logits, w13, w2
    torch.cuda.empty_cache()
    if not args.no_workloads and world == 1 and not (args.tokens or args.experts or args.topk):
        # every other configuration of the benchmark, each timed for >= 1 s and >= 200 steps
        others = {}
        for name, w in WORKLOADS.items():
            if name == wl.name:
                continue
            r, bufs = measure(moe, w, dev, 20, 5, "auto", with_e2e=True, seed=0, clocks=True,
                              min_seconds=1.0, min_steps=200)
            del bufs
            torch.cuda.empty_cache()
            others[name] = {"config": workload_config(w, 1), "timing": r["timing"],
                            "tokens_per_s": r["value"], "ms_per_step": r["ms_per_step"], "steps": r["steps"],
                            "layer_tflops": r["layer_tflops"], "e2e_tokens_per_s": (r["e2e"] or {}).get("value"),
                            "e2e_ms_per_step": (r["e2e"] or {}).get("ms_per_step"),
                            "roofline": r["roofline"], "kernels": r["kernels"],
                            "gpu_launches_per_step": r["gpu_launches_per_step"], "clocks": r["clocks"]}
        line["workloads"] = others
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

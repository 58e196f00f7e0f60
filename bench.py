"""Decode-step benchmark of the ResidualQuant path on GB300.

One step = what a looped model does to produce one token per sequence: for
every loop and every layer one attention call over the compressed cache (plus
the current token from the BF16 temporary buffer); each layer's last-loop call
(rq_decode_attention_append) also compresses that token, every loop of it,
into the cache.  Ouro-1.4B shape at 8k context: 24 layers x 4 loops = 96
attention calls per step, 24 of them appending, batch 4, 16 heads of width
128, INT4 anchor / INT2 residuals, g = 32.  The cache is kept at a fixed length (each step overwrites the same
next slot), so every step does the same work.

Prints one JSON line.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-attn tokens/s and effective HBM GB/s (% GB300 peak) at 8k/16k ctx"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _algo_bytes_per_token_call(w: synth.Workload, has_res: bool, chained_planes: int = 1) -> int:
    """Compressed bytes one attention call reads per cached token (K and V)."""
    d, ng = w.head_dim, w.head_dim // w.group_size
    anchor = d // 2 + 2 * ng
    res = d // 4 + 2 * ng + 2
    return 2 * (anchor + (res * chained_planes if has_res else 0))


def algorithmic_bytes_per_step(w: synth.Workload, batch: int, ctx: int, chained: bool = False) -> dict:
    """Bytes the step must move at minimum: every attention call reads its
    planes for all cached tokens, plus the current token, q and out; each
    append writes one token's records.  Shared anchor: loop l < P-1 reads the
    anchor and its own residual plane; chained: the anchor and the residual
    planes of loops l .. P-2."""
    P, L, H, d = w.loops_per_group, w.num_layers, w.num_heads, w.head_dim
    rows = batch * H
    small = rows * (3 * d * 2 + d * 4)                      # q, k_cur, v_cur (bf16) + out (fp32)
    per_loop = []
    for lp in range(P):
        planes = 0 if lp == P - 1 else (P - 1 - lp if chained else 1)
        per_loop.append(_algo_bytes_per_token_call(w, planes > 0, max(planes, 1)) * ctx * rows + small)
    per_call_res = per_loop[0] - small if P > 1 else 0
    per_call_anchor = per_loop[P - 1] - small
    calls = sum(per_loop)
    ng = d // w.group_size
    append = rows * 2 * ((d // 2 + 2 * ng) + (P - 1) * (d // 4 + 2 * ng + 2)) + rows * P * 2 * d * 2
    total = L * w.num_groups * (calls + append)
    return {"step": total, "call_res": per_call_res + small, "call_anchor": per_call_anchor + small,
            "per_loop": per_loop}


class ClockSampler:
    """nvidia-smi sampling during the timed region (SM clock, throttle reasons)."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.first = threading.Event()
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the timed region starts once the sampler delivers (its start-up takes a while);
            # the samples kept are the ones taken from then on
            self.first.wait(timeout=5.0)
            self.lines = []
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.first.set()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


class OracleSample:
    """The oracle as it stands, on the host cores: rebuild + attend for one
    (row, head) slice of an attention call at full context.  A step of the
    workload is batch * heads * calls such slices; timings are extrapolated."""

    def __init__(self, w: synth.Workload, ctx: int):
        import oracle
        self.oracle = oracle
        self.w, self.ctx = w, ctx
        d, P = w.head_dim, w.loops_per_group
        self.R = synth.rotation(d).astype(np.float32).astype(np.float64)
        self.geom = oracle.Geometry(1, P, 1, 1, d, w.group_size, 1, ctx)
        one = synth.Workload("row", 1, P, 1, 1, d, w.group_size, 1, ctx, w.alphas, w.anchor_is_base)
        self.buf = np.zeros(self.geom.total_bytes, dtype=np.uint8)
        _, kv = synth.looped_kv(123, one, batch=1, ntok=ctx)
        oracle.append(self.buf, self.geom, self.R, 0, 0, kv, [0])
        _, self.q = synth.queries(5, 1, 1, d)
        _, self.cur = synth.looped_kv(6, one, batch=1, ntok=1)
        self.scale = 1.0 / math.sqrt(d)
        self.n = 0

    def run(self, budget_s: float):
        """Row-calls for about budget_s seconds; returns (row_calls, seconds)."""
        P = self.w.loops_per_group
        n, t0 = 0, time.perf_counter()
        while True:
            loop = (self.n + n) % P
            self.oracle.decode_attention(self.buf, self.geom, self.R, 0, 0, loop, self.q,
                                         self.cur[loop, 0, :, :, 0], self.cur[loop, 1, :, :, 0],
                                         [self.ctx], self.scale)
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        self.n += n
        return n, el

    def row_calls_per_step(self, batch):
        return batch * self.w.num_heads * self.w.calls_per_step


def cpu_baseline(w: synth.Workload, batch: int, ctx: int, budget_s: float = 15.0) -> dict:
    smp = OracleSample(w, ctx)
    n, el = smp.run(budget_s)
    step_s = el / n * smp.row_calls_per_step(batch)
    return {"value": batch / step_s, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n} (row, head) attention calls at {ctx} tokens (float64 NumPy rebuild from the "
                      f"cache bytes + softmax), {el:.1f} s, extrapolated to "
                      f"{smp.row_calls_per_step(batch)} row-calls per step"}


def reduce_max_over_ranks(x: float, device=None) -> float:
    """Largest x over the ranks of the default process group (x itself without one):
    the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, batch: int, ms_step: float) -> float:
    """Whole-job tokens/s: each of `world` replicas decodes `batch` rows per step, and the
    step lasts `ms_step` milliseconds (the slowest rank's)."""
    return world * batch / (ms_step / 1e3)


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    budget = args.ref_budget or max(0.2, min(2.0, 150.0 / (args.steps + args.warmup)))
    smp = OracleSample(w, w.context)
    per_step = smp.row_calls_per_step(w.batch)
    # A step of this arm is a bounded sample of the decode step (about `budget`
    # seconds of its (row, head) attention calls): ms_per_step is the sample's
    # own time, and the throughput counts the fraction of a decode step done.
    times, total_n, total_s = [], 0, 0.0
    for i in range(args.warmup + args.steps):
        n, el = smp.run(budget)
        if i >= args.warmup:
            times.append(el)
            total_n += n
            total_s += el
    ms = 1000 * statistics.mean(times)
    val = w.batch * (total_n / per_step) / total_s
    sample = (f"each step: about {budget:.2f} s of (row, head) attention calls at {w.context} tokens "
              f"(float64 NumPy rebuild from the cache bytes + softmax) out of the {per_step} row-calls "
              f"of a decode step; {total_n} row-calls in {total_s:.1f} s over the timed steps "
              f"(a whole decode step would take {per_step * total_s / total_n:.0f} s)")
    line = {"metric": METRIC, "value": val, "unit": "tokens/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, args.chained),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _config(w, chained=False, hadamard=False, paged=False, query_heads=None):
    return {"workload": f"{w.name}: {w.num_layers} layers x {w.loops_per_group} loops x {w.num_groups} groups, "
                        f"{w.num_heads} KV heads x {w.head_dim}, batch {w.batch}, {w.context}-token context, "
                        f"INT4 anchor + INT2 residuals, group {w.group_size}, "
                        f"{'chained' if chained else 'shared'} anchor"
                        + (", Walsh-Hadamard rotation" if hadamard else "") + (", paged layout" if paged else "")
                        + (f", {query_heads} query heads (grouped-query)" if query_heads else ""),
            "global_batch": w.batch, "seq_len": w.context, "parallelism": "replicas",
            "l2": _l2_note(w, chained)}


L2_BYTES = 129e6   # GB300's L2


def _l2_note(w, chained=False):
    """How the timed steps meet the L2 rule: the compressed cache a step streams
    either exceeds the L2 or it does not (then the figure is a warm-cache one)."""
    if algorithmic_bytes_per_step(w, w.batch, w.context, chained)["step"] > L2_BYTES:
        return "inputs larger than L2 (every step streams the whole compressed cache)"
    return "inputs fit in L2: a warm-cache, launch-bound figure (the small parity case)"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="rq", choices=["rq", "reference"])
    ap.add_argument("--workload", default="ouro8k", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--group-size", type=int, default=None)
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16 comparator")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the main workload (the default run also times " + ", ".join(
                        ("ouro16k_b2", "ouro16k_b4", "huginn")) + " as sub-records)")
    ap.add_argument("--ref-budget", type=float, default=None,
                    help="seconds of oracle work per reference step (default: about 150 s per run)")
    ap.add_argument("--quiet", action="store_true")
    ap.add_argument("--chained", action="store_true", help="chained anchors (loop l coded against loop l+1)")
    ap.add_argument("--query-heads", type=int, default=None,
                    help="query heads per row (a multiple of the KV heads: grouped-query attention)")
    ap.add_argument("--paged", action="store_true",
                    help="paged cache layout: pages assigned through a shuffled block table")
    ap.add_argument("--hadamard", action="store_true",
                    help="Walsh-Hadamard rotation applied as a fast transform (head_dim 128)")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers than the workload (a small case for profiler captures)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.batch or args.group_size or args.layers:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch or w.batch, group_size=args.group_size or w.group_size,
                                num_layers=args.layers or w.num_layers)
    if args.impl == "reference":
        run_reference(args, w)
        return
    run_rq(args, w)


def _time_step(args, w, dev, rank, world, chained=False, hadamard=False, paged=False, query_heads=None):
    """Builds a cache of workload w on dev, fills it (prefill), captures one decode
    step in a CUDA graph and times args.steps replays (after args.warmup), then
    each kind of call on its own.  Returns the measurements and the live objects
    (graph, stream, per-step tensors, cache handle) for the end-to-end leg;
    _release frees them."""
    import torch
    import decode_attention_rq_gb300 as rq

    L, P, G, H, d, g, B, N = (w.num_layers, w.loops_per_group, w.num_groups, w.num_heads, w.head_dim,
                              w.group_size, w.batch, w.context)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    R32 = None if hadamard else torch.from_numpy(synth.rotation(d).astype(np.float32)).to(dev)
    Hq = query_heads or H   # grouped-query attention when Hq > H (the pages' models: Hq = H)
    cfg = rq.rq_config(L, P, G, H, d, g, B, N + 64, (rq.RQ_MODE_CHAINED if chained else rq.RQ_MODE_SHARED)
                       | (rq.RQ_MODE_HADAMARD if hadamard else 0), Hq)
    if paged:
        # every row's tiles on pages of a shuffled table (the pool holds exactly those pages)
        ntiles = -(-(N + 64) // 64)
        num_pages = B * ntiles
        perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(5 + rank))
        table = perm.reshape(B, ntiles).to(torch.int32).to(dev)
        nbytes = rq.rq_cache_paged_bytes(cfg, num_pages)
        cache_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        handle = rq.rq_cache_create_paged(cfg, num_pages, cache_buf, nbytes, table, ntiles, R32)
    else:
        table = None
        nbytes = rq.rq_cache_bytes(cfg)
        cache_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        handle = rq.rq_cache_create(cfg, cache_buf, nbytes, R32)
    ws_bytes = rq.rq_decode_workspace_bytes(cfg, B)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    status = ws[:16].view(torch.int32)
    seq0 = torch.zeros(B, dtype=torch.int32, device=dev)
    # prefill: compress N tokens per (layer, group)
    t0 = time.perf_counter()
    for layer in range(L):
        for grp in range(G):
            kv = synth.looped_kv_torch(gen, w, B, N, dev)
            rq.rq_append(handle, layer, grp, B, kv, seq0, N, status)
            del kv
    torch.cuda.synchronize()
    prefill_s = time.perf_counter() - t0
    seq = torch.full((B,), N, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(d)
    ncalls = L * G * P
    # per-step inputs: queries per call, the BF16 temporary buffer per (layer, group)
    q_all = torch.randn((ncalls, B, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
    temp_all = torch.stack([synth.looped_kv_torch(gen, w, B, 1, dev) for _ in range(L * G)])  # [LG,P,2,B,H,1,d]
    out_all = torch.empty((ncalls, B, Hq, d), dtype=torch.float32, device=dev)

    order = [(lp, layer, grp) for grp in range(G) for lp in range(P) for layer in range(L)]

    s = torch.cuda.Stream(device=dev)

    def call(i):
        lp, layer, grp = order[i]
        t = temp_all[layer * G + grp]
        if lp == P - 1:   # the anchor loop: attention, then the token joins the cache
            rq.rq_decode_attention_append(handle, layer, grp, B, q_all[i], t[..., 0, :], seq, scale, out_all[i],
                                          ws, ws_bytes, s.cuda_stream)
        else:
            rq.rq_decode_attention(handle, layer, grp, lp, B, q_all[i], t[lp, 0, :, :, 0], t[lp, 1, :, :, 0],
                                   seq, scale, out_all[i], ws, ws_bytes, s.cuda_stream)

    def step():
        for i in range(ncalls):
            call(i)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()   # eager once (also sets kernel attributes before capture)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    torch.cuda.synchronize()

    # warm-up (replay() launches on the current stream: make it s, where the events are)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    # timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(args.steps):
                graph.replay()
            e1.record(s)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    ms_total = reduce_max_over_ranks(e0.elapsed_time(e1), dev)
    ms_step = ms_total / args.steps
    st = status.cpu().numpy()
    if st.any():
        raise RuntimeError(f"device status word reports an error: {st.tolist()}")

    # time per call (its three kernels; decode_kernel dominates), CUDA events on its stream.
    # The step's own call sequence is replayed with events only where the kind of call
    # changes (a run of residual-loop calls, a run of anchor-loop calls): inside a run the
    # calls keep their programmatic-dependent overlap, as in the step, and a run's time
    # divided by its calls is the time per call.
    byts = algorithmic_bytes_per_step(w, B, N, chained)
    kinds = [lp < P - 1 for (lp, _, _) in order]
    bounds = [0] + [i for i in range(1, ncalls) if kinds[i] != kinds[i - 1]] + [ncalls]
    ev = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    t_res = t_anchor = 0.0
    n_res = n_anchor = bytes_res = 0
    with torch.cuda.stream(s):
        for r in range(4):
            ev[0].record(s)
            for k in range(len(bounds) - 1):
                for i in range(bounds[k], bounds[k + 1]):
                    call(i)
                ev[k + 1].record(s)
            torch.cuda.synchronize()
            if r == 0:
                continue   # warm-up pass
            for k in range(len(bounds) - 1):
                ms, n = ev[k].elapsed_time(ev[k + 1]), bounds[k + 1] - bounds[k]
                if kinds[bounds[k]]:
                    t_res, n_res = t_res + ms, n_res + n
                    bytes_res += sum(byts["per_loop"][order[i][0]] for i in range(bounds[k], bounds[k + 1]))
                else:
                    t_anchor, n_anchor = t_anchor + ms, n_anchor + n
    peak, peak_kind = _peaks()
    # the dominant launch: a residual-loop call (shared: anchor + one residual plane;
    # chained: anchor + the planes down to the loop), bytes and time summed over those calls
    per_launch_bytes = bytes_res / n_res
    avg_launch_ms = t_res / n_res
    achieved = per_launch_bytes / (avg_launch_ms / 1e3) / 1e9
    anchor_ms = t_anchor / n_anchor
    anchor_gbs = byts["call_anchor"] / (anchor_ms / 1e3) / 1e9
    step_gbs = byts["step"] / (ms_step / 1e3) / 1e9
    return {
        "ms_step": ms_step, "clocks": clk.summary(), "prefill_s": prefill_s, "step_gbs": step_gbs,
        "peak": peak, "peak_kind": peak_kind, "calls": ncalls,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "avg_launch_ms": avg_launch_ms, "bytes_per_launch": per_launch_bytes,
                     "anchor_loop_call": {"avg_ms": anchor_ms, "bytes": byts["call_anchor"],
                                          "includes_token_append": True, "achieved": anchor_gbs,
                                          "frac": anchor_gbs / peak}},
        "launches_per_step": 3 * ncalls,   # a call is qprep + decode + merge kernels (the append runs in the merge)
        "gen": gen, "scale": scale,
        "live": {"graph": graph, "stream": s, "q_all": q_all, "temp_all": temp_all, "out_all": out_all,
                 "handle": handle, "cache_buf": cache_buf, "ws": ws, "table": table, "R": R32},
    }


def _release(t):
    import torch
    import decode_attention_rq_gb300 as rq
    live = t.pop("live")
    torch.cuda.synchronize()
    rq.rq_cache_destroy(live["handle"])
    live.clear()
    torch.cuda.empty_cache()


# The configurations the default run also times, each as a sub-record of the
# JSON line: the two 16k-context batches of the Ouro throughput comparison and
# the Huginn shape (head width 96, 55 heads, 8 loop groups of 4).
EXTRA_CONFIGS = ("ouro16k_b2", "ouro16k_b4", "huginn")


def _sub_record(args, name, dev, rank, world):
    w = synth.WORKLOADS[name]
    t = _time_step(args, w, dev, rank, world)
    rec = {"config": _config(w), "ms_per_step": t["ms_step"],
           "tokens_per_s": job_throughput(world, w.batch, t["ms_step"]),
           "effective_gbps": t["step_gbs"], "frac_of_hbm_peak": t["step_gbs"] / t["peak"],
           "roofline": dict(t["roofline"], kernel="rq_decode_attention, residual-loop call",
                            peak_source=f"MEASURED_PEAKS.json hbm_gbs ({t['peak_kind']})"),
           "gpu_launches": t["launches_per_step"] * args.steps, "clocks": t["clocks"]}
    gen, scale = t["gen"], t["scale"]
    _release(t)
    if not args.no_bf16:
        rec["bf16_comparator"] = bench_bf16(args, w, dev, gen, scale)
        rec["speedup_vs_bf16"] = rec["bf16_comparator"]["ms_per_step_attention"] / rec["ms_per_step"]
    return rec


def run_rq(args, w):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    B = w.batch
    t = _time_step(args, w, dev, rank, world, args.chained, args.hadamard, args.paged, args.query_heads)
    ms_step = t["ms_step"]
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic_per_launch.json")
    if os.path.exists(tp):
        try:
            tj = json.load(open(tp))
            if (tj.get("workload") == w.name and tj.get("batch") == B and tj.get("group_size") == w.group_size
                    and not args.chained and not args.hadamard and not args.paged and not args.query_heads
                    and tj.get("kernel_source_hash") == _kernel_hash()):
                traffic = tj.get("bytes_per_launch")
        except Exception:
            traffic = None

    peak = t["peak"]
    value = job_throughput(world, B, ms_step)
    roof = t["roofline"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32/fp32", "data": "synthetic",
        "config": _config(w, args.chained, args.hadamard, args.paged, args.query_heads),
        "effective_gbps": t["step_gbs"], "frac_of_hbm_peak": t["step_gbs"] / peak,
        "roofline": {"bound": "hbm", "achieved": roof["achieved"], "peak": peak, "unit": "GB/s",
                     "frac": roof["frac"], "traffic": traffic,
                     "kernel": "rq_decode_attention, residual-loop call (qprep_kernel + "
                               "decode_kernel<d, g, 1> + merge_kernel)",
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({t['peak_kind']})",
                     "avg_launch_ms": roof["avg_launch_ms"], "bytes_per_launch": roof["bytes_per_launch"],
                     "anchor_loop_call": roof["anchor_loop_call"]},
        "gpu_launches": t["launches_per_step"] * args.steps,
        "clocks": t["clocks"],
        "prefill_s": t["prefill_s"],
    }
    if not args.no_e2e:
        live = t["live"]
        line["e2e"] = bench_e2e(args, live["graph"], live["stream"], live["q_all"], live["temp_all"],
                                live["out_all"], B)
    gen, scale = t["gen"], t["scale"]
    _release(t)
    # BF16 comparator: the same calls over uncompressed K/V
    if not args.no_bf16 and not args.query_heads:   # the BF16 comparator is multi-head
        line["bf16_comparator"] = bench_bf16(args, w, dev, gen, scale)
        # whole compressed step (appends included) against the BF16 attention calls alone
        line["speedup_vs_bf16"] = line["bf16_comparator"]["ms_per_step_attention"] / ms_step
    if not args.no_configs and w.name == "ouro8k" and not (args.batch or args.group_size or args.layers
                                                          or args.chained or args.hadamard or args.paged
                                                          or args.query_heads):
        line["configs"] = {name: _sub_record(args, name, dev, rank, world) for name in EXTRA_CONFIGS}
    if rank == 0 and not args.no_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, B, w.context, budget_s=15.0)
    if rank == 0:
        print(json.dumps(line))


def bench_bf16(args, w, dev, gen, scale):
    """The library's BF16 decode kernel over the same calls (K/V [B,H,N,d] per call)."""
    import torch
    import decode_attention_rq_gb300 as rq
    L, P, G, H, d, B, N = w.num_layers, w.loops_per_group, w.num_groups, w.num_heads, w.head_dim, w.batch, w.context
    ncalls = L * G * P
    # distinct K/V per call up to a memory budget; beyond it calls cycle over the buffers
    # (each call streams far more than the L2 holds, so reuse across calls hits DRAM)
    per_call = 2 * B * H * N * d * 2
    nbuf = max(2, min(ncalls, int(48e9 // per_call)))
    kv = torch.empty((nbuf, 2, B, H, N, d), dtype=torch.bfloat16, device=dev)
    kv.normal_(generator=gen)
    q = torch.randn((ncalls, B, H, d), generator=gen, device=dev).to(torch.bfloat16)
    cur = torch.randn((ncalls, 2, B, H, d), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    seq = torch.full((B,), N, dtype=torch.int32, device=dev)
    ws_bytes = rq.rq_bf16_workspace_bytes(B, H, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)

    def step(st):
        for i in range(ncalls):
            rq.rq_decode_attention_bf16(kv[i % nbuf, 0], kv[i % nbuf, 1], cur[i, 0], cur[i, 1], q[i], seq, B, H, d, N, scale,
                                        out, ws, ws_bytes, st)
    with torch.cuda.stream(s):
        step(s.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s.cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        e0.record(s)
        for _ in range(args.steps):
            graph.replay()
        e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    byts = ncalls * B * H * (N * 2 * d * 2 + 3 * d * 2 + d * 4)
    peak, _ = _peaks()
    del kv
    torch.cuda.empty_cache()
    return {"ms_per_step_attention": ms, "tokens_per_s": B / (ms / 1e3), "calls": ncalls,
            "effective_gbps": byts / (ms / 1e3) / 1e9, "frac_of_hbm_peak": byts / (ms / 1e3) / 1e9 / peak}


def bench_e2e(args, graph, s, q_all, temp_all, out_all, B):
    """Same step with its per-step inputs coming from pinned host memory and the
    step's attention outputs read back, copies inside the timed region."""
    import torch
    q_h = q_all.cpu().pin_memory()
    t_h = temp_all.cpu().pin_memory()
    o_h = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(args.steps):
            q_all.copy_(q_h, non_blocking=True)
            temp_all.copy_(t_h, non_blocking=True)
            graph.replay()
            o_h.copy_(out_all, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    wall = (time.perf_counter() - t0) / args.steps * 1e3
    h2d = q_all.numel() * q_all.element_size() + temp_all.numel() * temp_all.element_size()
    d2h = out_all.numel() * out_all.element_size()
    return {"value": B / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "wall_ms_per_step": wall}


def _kernel_hash():
    """Hash of the kernel sources with comments and blank lines dropped (a comment
    edit does not change the kernels the traffic counters were taken on)."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_rq_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()

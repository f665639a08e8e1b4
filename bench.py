"""Benchmark: one decode step of sparse attention over MXFP4 paged caches.

A step is the whole hot path on one batch: mx4_insert of the decode tokens'
K/V/index-K rows (when the workload inserts in the step), index_score over
every cached index key, topk_select, sparse_paged_decode (split + merge).
Inputs are resident in HBM when the timed region starts; the L2 is flushed
(a 256 MiB write, then a read of it so the write-back of its dirty lines
falls outside the step) between timed steps, outside the per-step CUDA events.

By default all five workloads are measured, each with its own block in the
JSON line (step time, tokens/s, per-kernel times, the scorer's, the decode's
and the hot path's HBM fractions, the end-to-end rate through the C entry points
with host buffers -- mx4_decode_steps, K steps with the copies of neighbouring steps
overlapped, and mx4_decode_step, one call a step -- clocks).  The headline -- `value`, `roofline`,
`e2e`, the extra legs and the CPU baselines -- is workload 4: 256 sequences,
lognormal contexts (median 8192, capped at 131072), one decode token each
inserted in the step, top-2048, the only workload whose step runs all four
kernels and the largest.  `--workload N` measures one workload only.

Clocks are sampled with nvidia-smi over a soak of about one second of the same
step right before the K timed steps and over the timed steps themselves.

Under torchrun (N > 1) every rank runs an independent replica of the same
workload (the path shards by sequence with no exchange step): weak scaling,
value = tokens of all ranks / the slowest rank's time.

`--impl reference` times the CPU oracle (plain C, float64) on this host's
cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mxfp4_sparse_paged_gb300 import workloads as W  # noqa: E402

METRIC = "sparse MXFP4 paged-decode tokens/s"
UNIT = "tokens/s"
FP8_INDEX_SCALE = 0.25  # per-cache scale of the fp8 index-K variant: |row| / 0.25 stays below 448


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _config(wl):
    L = wl.seq_lens
    return {"workload": wl.spec.name, "batch": wl.B, "decode_tokens_per_seq": wl.q,
            "decode_tokens": wl.T, "contexts": {"min": int(L.min()), "median": int(np.median(L)),
                                                "max": int(L.max()), "sum": int(L.sum())},
            "top_k": wl.k, "q_heads": W.Q_HEADS, "kv_heads": W.KV_HEADS, "head_dim": W.HEAD_DIM,
            "insert_in_step": wl.spec.insert_in_step, "seed": wl.spec.seed,
            "l2": "flushed between timed steps (256 MiB written then read back, outside the "
                  "step events, so no dirty lines of the flush are written back inside them)",
            "parallelism": "replicas (one independent batch per GPU)"}


# --------------------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi sampled every 50 ms during the timed region."""

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.f.read().splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.f.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- CPU oracle

class _OracleCache:
    """The oracle's page pools for a workload, filled per sequence on demand (untimed:
    the cache contents before the step)."""

    def __init__(self, wl):
        import oracle
        from mxfp4_sparse_paged_gb300.step import step_inputs_host
        oracle.build()
        self.oracle = oracle
        self.wl = wl
        self.host = step_inputs_host(wl)
        P = wl.num_pages
        self.kp = np.full((P, 1, 8704), 0xFF, np.uint8)
        self.vp = np.full_like(self.kp, 0xFF)
        self.ip = np.full((P, 8704), 0xFF, np.uint8)
        self.scale = 1 / math.sqrt(W.HEAD_DIM)

    def fill(self, s):
        wl, o = self.wl, self.oracle
        n = wl.prefilled(s)
        for a in range(0, n, 65536):
            b = min(n, a + 65536)
            o.mx4_insert(wl.rows(s, 0, a, b)[:, None], wl.rows(s, 1, a, b)[:, None],
                         wl.rows(s, 2, a, b), wl.slots(s, np.arange(a, b)), self.kp, self.vp,
                         self.ip)

    def step(self, s):
        """The oracle's step for sequence s: insert of its decode tokens (when the
        workload inserts in the step), scores, top-k, attention."""
        wl, o, host = self.wl, self.oracle, self.host
        tok = np.arange(s * wl.q, (s + 1) * wl.q)
        lens = wl.seq_lens[[s]]
        bt = wl.block_table[[s]]
        if wl.spec.insert_in_step:
            o.mx4_insert(host["k"][tok][:, None], host["v"][tok][:, None], host["idx_k"][tok],
                         host["slots"][tok], self.kp, self.vp, self.ip)
        sc = o.index_score(host["iq"][tok], wl.q, self.ip, bt, lens, int(lens[0]))
        sel = o.topk_select(sc, lens, wl.q, wl.k)
        o.sparse_paged_decode(host["q"][tok], wl.q, self.kp, self.vp, bt, lens, sel, self.scale)


def _sample_order(wl):
    return [int(s) for s in np.random.default_rng(1234).permutation(wl.B)]


def cpu_oracle_sample(wl, budget_s: float = 15.0, cache=None):
    """Time the oracle's step (insert of the step tokens, score, top-k, attention)
    on a bounded sample of sequences, one thread; returns (tokens/s, detail, seconds)."""
    c = cache or _OracleCache(wl)
    done_tok, spent, seqs = 0, 0.0, []
    for s in _sample_order(wl):
        c.fill(s)
        t0 = time.perf_counter()
        c.step(s)
        spent += time.perf_counter() - t0
        done_tok += wl.q
        seqs.append(s)
        if spent >= budget_s:
            break
    frac_ctx = float(wl.seq_lens[seqs].sum()) / float(wl.seq_lens.sum())
    detail = (f"{len(seqs)} of {wl.B} sequences ({done_tok} decode tokens, "
              f"{100 * frac_ctx:.1f}% of the step's cached tokens), single thread, "
              f"{spent:.1f} s; value = sampled decode tokens / oracle step time")
    return done_tok / spent, detail, spent


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_parallel(wl, budget_s: float = 15.0, workers: int | None = None, cache=None):
    """The same oracle step over a bounded sample of sequences, spread over the host's
    cores: one thread per core takes whole sequences (the oracle is a C library and
    its calls release the interpreter lock).  The sample size comes from a short
    single-thread probe of the seconds per sequence, to about budget_s of wall time;
    the cache fill is untimed.  Returns (tokens/s, detail, seconds, cores)."""
    from concurrent.futures import ThreadPoolExecutor
    workers = workers or host_cores()
    c = cache or _OracleCache(wl)
    order = _sample_order(wl)
    probe = order[:2]
    for s in probe:
        c.fill(s)
    t0 = time.perf_counter()
    for s in probe:
        c.step(s)
    per_seq = (time.perf_counter() - t0) / len(probe)
    n = int(min(wl.B, max(workers, round(budget_s * workers / per_seq))))
    seqs = order[:n]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(c.fill, seqs))
        t0 = time.perf_counter()
        list(ex.map(c.step, seqs))
        wall = time.perf_counter() - t0
    done_tok = len(seqs) * wl.q
    frac_ctx = float(wl.seq_lens[seqs].sum()) / float(wl.seq_lens.sum())
    detail = (f"{len(seqs)} of {wl.B} sequences ({done_tok} decode tokens, "
              f"{100 * frac_ctx:.1f}% of the step's cached tokens), {workers} threads over "
              f"whole sequences, {wall:.1f} s wall; value = sampled decode tokens / wall time")
    return done_tok / wall, detail, wall, workers


# --------------------------------------------------------------------------- ranks

def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest of the ranks' values (each rank's timed region; the job ends with
    the slowest rank).  A no-op for one rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank_step: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job decode tokens/s: every rank runs its own batch (replicas), so the
    job processes world x tokens per step, in the slowest rank's time."""
    return tokens_per_rank_step * world * steps / (total_ms / 1e3)


# --------------------------------------------------------------------------- GPU arm

def _flusher(dev):
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2(v):
        # Write a buffer twice the L2 size, then read it back: the read evicts the
        # written lines, so their write-back lands here rather than in the step.
        flush.fill_(v)
        flush.view(torch.int64).sum()
    return flush_l2


def _event_ms(pairs):
    return [a.elapsed_time(b) for a, b in pairs]


def _roof(name, nbytes, ms, peak, traffic=None, extra=None):
    gbs = nbytes / (ms / 1e3) / 1e9
    d = {"bound": "hbm", "kernel": name, "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
         "frac": round(gbs / peak, 4), "algorithmic_bytes_per_launch": int(nbytes),
         "traffic": traffic}
    if traffic:
        d["traffic_over_algorithmic"] = round(traffic / nbytes, 3)
        d["dram_gbs_at_traffic"] = round(traffic / (ms / 1e3) / 1e9, 1)
    if extra:
        d.update(extra)
    return d


def measure_workload(wid, args, dev, stream, flush_l2, world, barrier, headline=False):
    """Time one workload's decode step on this GPU: warm-up, a clock-sampled soak of
    about args.soak seconds of the same step, the timed steps (one event pair each,
    L2 flushed between them), a per-kernel event pass, and the step end to end
    through the C entry points with host buffers.  Returns the
    workload's block of the JSON line (and the live objects for the headline's
    extra legs)."""
    import torch

    import mxfp4_sparse_paged_gb300 as m
    from mxfp4_sparse_paged_gb300.step import DecodeStep, PagedCaches, step_inputs_host

    wl = W.make(wid)
    caches = PagedCaches(wl.num_pages, device=dev,
                         fp8_index_scale=FP8_INDEX_SCALE if headline else None)
    caches.fill(wl)
    step = DecodeStep(wl, caches, device=dev)
    host = step_inputs_host(wl)
    torch.cuda.synchronize()
    ab = W.algorithmic_bytes(wl)
    # The in-step insert rewrites the decode tokens' rows with the same values, so
    # every timed step does identical work.
    step.load_inputs(host)
    for _ in range(args.warmup):
        flush_l2(1)
        step.run(stream=stream)
    m.mx4_check_status()
    if not args.eager:
        step.capture()  # the step's kernels as one CUDA graph (same launches, same order)
        for _ in range(3):
            flush_l2(1)
            step.replay()

    def one_step():
        if args.eager:
            step.run(stream=stream)
        else:
            step.replay()

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    st = [(ev(), ev()) for _ in range(args.steps)]
    # clocks: sampled over a soak of the same step right before the timed steps and
    # over the timed steps (a timed region of K steps is far shorter than a sample)
    clocks = Clocks(int(dev.index or 0))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    soak_steps = 0
    while time.perf_counter() - t0 < args.soak:
        for _ in range(50):
            flush_l2(1)
            one_step()
        soak_steps += 50
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(i & 0xFF)
        st[i][0].record(stream)
        one_step()
        st[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    ck = clocks.stop()
    m.mx4_check_status()
    step_ms = _event_ms(st)
    # Per-kernel times: each entry point captured alone as a CUDA graph and replayed
    # with an event pair around each replay (GPU time only, no host launch cost),
    # the L2 flushed before each.  The selection is timed after the scorer has run, so
    # it reads the scores of this step.
    calls = step.stage_calls()  # on the current stream: the capture stream while capturing
    kern_ms = {}
    reps = min(args.steps, 200)
    for name, fn in calls.items():
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        evs = [(ev(), ev()) for _ in range(reps)]
        for i in range(reps):
            flush_l2(i & 0xFF)
            evs[i][0].record(stream)
            g.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        kern_ms[name] = statistics.mean(_event_ms(evs))
        del g
    m.mx4_check_status()
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_value(wl.T, world, args.steps, total_ms)

    # ---- end to end through the C ABI with host buffers: every step copies its
    # packed inputs from pinned host memory, runs the four stages and copies its
    # output back.  `e2e`: the K steps in one mx4_decode_steps call, the copies of
    # neighbouring steps overlapping the compute on two copy streams;
    # `e2e_one_call_a_step`: K mx4_decode_step calls, each copy in line with its step.
    pin = step.pack_inputs(host)
    h_out = torch.empty(tuple(step.out.shape), dtype=torch.float32).pin_memory()
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    step.run_host_steps(pin, h_out, 4, stream, h2d, d2h)
    for _ in range(3):
        step.run_host(pin, h_out, stream=stream)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = ev(), ev()
    e0.record(stream)
    step.run_host_steps(pin, h_out, args.steps, stream, h2d, d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    m.mx4_check_status()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step.run_host(pin, h_out, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    m.mx4_check_status()
    e2e1_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    io = {"h2d_bytes_per_step": int(pin.numel()),
          "d2h_bytes_per_step": int(h_out.numel() * h_out.element_size())}
    e2e = dict({"value": round(job_value(wl.T, world, args.steps, e2e_ms), 1), "unit": UNIT}, **io,
               mode="through the C entry point mx4_decode_steps: the K steps in one call, each "
                    "copying its packed inputs from pinned host memory and its output to "
                    "pinned host memory, the copies of neighbouring steps overlapping the "
                    "compute on two copy streams; no L2 flush")
    e2e_one = dict({"value": round(job_value(wl.T, world, args.steps, e2e1_ms), 1),
                    "unit": UNIT}, **io,
                   mode="K calls of the C entry point mx4_decode_step on one stream, each "
                        "step's copies in line with its compute; no L2 flush")

    peak, peak_kind = _peaks()
    sc_ms, dec_ms = kern_ms["index_score"], kern_ms["sparse_paged_decode"]
    hot = ab["index_score"] + ab["sparse_paged_decode"]
    hot_gbs = hot / ((sc_ms + dec_ms) / 1e3) / 1e9
    r_score = _roof("index_score", ab["index_score"], sc_ms, peak,
                    _ncu_traffic(wl.spec.name, "index_score_traffic.json"),
                    {"timing": "the scorer alone (index_score call); inside the step it is "
                               "the first kernel of index_topk"})
    r_dec = _roof("sparse_paged_decode (run kernel + merge kernel)", ab["sparse_paged_decode"],
                  dec_ms, peak, _ncu_traffic(wl.spec.name, "decode_split_traffic.json"),
                  {"traffic_kernel": "decode_split_kernel"})
    block = {
        "value": round(value, 1), "unit": UNIT, "ms_per_step": round(total_ms / args.steps, 4),
        "decode_tokens": wl.T, "cached_tokens": int(wl.seq_lens.astype(np.int64).sum()),
        "kernel_ms": {n: round(v, 5) for n, v in kern_ms.items()},
        "kernel_ms_timing": "each entry point captured alone as a CUDA graph, mean of event "
                            "pairs around its replays, L2 flushed before each; index_score and "
                            "topk_select are the pair index_topk combines",
        "roofline_index_score": r_score, "roofline_decode": r_dec,
        "hot_path_hbm": {"kernels": "index_score + sparse_paged_decode",
                         "algorithmic_bytes": int(hot), "achieved_gbs": round(hot_gbs, 1),
                         "frac": round(hot_gbs / peak, 4),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "hot_path_hbm_with_topk": {
            "kernels": "index_topk (scorer + selection) + sparse_paged_decode",
            "algorithmic_bytes": int(hot),
            "achieved_gbs": round(hot / ((kern_ms["index_topk"] + dec_ms) / 1e3) / 1e9, 1),
            "frac": round(hot / ((kern_ms["index_topk"] + dec_ms) / 1e3) / 1e9 / peak, 4)},
        "e2e": e2e, "e2e_one_call_a_step": e2e_one, "clocks": ck, "soak_steps": soak_steps,
        "gpu_launches": step.launches_per_step() * args.steps,
        "wall_s_timed_region": round(wall, 4),
    }
    return block, (wl, caches, step, host, kern_ms)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    stream = torch.cuda.current_stream()
    flush_l2 = _flusher(dev)
    head = args.workload if args.workload is not None else 4
    order = [head] if args.workload is not None else [0, 1, 2, 3, 4]
    blocks = {}
    for wid in order:
        blk, live = measure_workload(wid, args, dev, stream, flush_l2, world, barrier,
                                     headline=(wid == head))
        blocks[W.SPECS[wid].name] = blk
        if wid == head:
            head_blk, head_live = blk, live
        else:
            del live
            torch.cuda.empty_cache()
    wl, caches, step, host, kern_ms = head_live
    peak, _ = _peaks()

    # the headline's extra legs: the overlapped serving loop, the writer, the fp8 and
    # block-scaled scorers
    from mxfp4_sparse_paged_gb300.step import PipelinedSteps
    pipe = PipelinedSteps(wl, caches, device=dev)
    pin = pipe.pack_inputs(host)
    for _ in range(4):
        _, done = pipe.submit(pin)
    done.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.h2d)
    for _ in range(args.steps):
        _, done = pipe.submit(pin)
    pipe.h2d.wait_event(done)
    e1.record(pipe.h2d)
    torch.cuda.synchronize()
    pipe_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    writer = time_writer(wl, dev, stream, flush_l2, min(args.steps, 200))
    fp8 = time_fp8_scorer(wl, caches, step, stream, flush_l2, min(args.steps, 200))
    mxq = time_mxq_scorer(wl, caches, step, stream, flush_l2, min(args.steps, 200))

    # roofline of the step's dominant HBM-bound kernel (the one taking longer)
    dominant = "roofline_decode" if kern_ms["sparse_paged_decode"] > kern_ms["index_score"] \
        else "roofline_index_score"
    line = {
        "metric": METRIC, "value": head_blk["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head_blk["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic (seeded N(0,1) K/V/index-K rows quantised to MXFP4 pages; "
                "bf16 N(0,1) queries)",
        "config": _config(wl),
        "roofline": dict(head_blk[dominant], peak_source="measured (MEASURED_PEAKS.json hbm_gbs)"
                         if _peaks()[1] == "measured" else "fallback"),
        "roofline_index_score": head_blk["roofline_index_score"],
        "roofline_decode": head_blk["roofline_decode"],
        "hot_path_hbm": head_blk["hot_path_hbm"],
        "hot_path_hbm_with_topk": head_blk["hot_path_hbm_with_topk"],
        "kernel_ms": head_blk["kernel_ms"], "kernel_ms_timing": head_blk["kernel_ms_timing"],
        "step_launch": ("separate API calls" if args.eager else
                        "one CUDA-graph launch of the step's kernels (captured from the API calls)"),
        "e2e": head_blk["e2e"],
        "e2e_one_call_a_step": head_blk["e2e_one_call_a_step"],
        "e2e_pipelined": {"value": round(job_value(wl.T, world, args.steps, pipe_ms), 1),
                          "unit": UNIT, "h2d_bytes_per_step": int(pin.numel()),
                          "d2h_bytes_per_step": int(pipe.h_out[0].numel() * 4),
                          "mode": "the Python serving loop (PipelinedSteps): packed inputs and "
                                  "the output copied on their own streams, overlapping the "
                                  "neighbouring steps' compute; one CUDA-graph launch a step"},
        "norm_rope_writer": writer,
        "fp8_index_variant": dict(fp8, mxfp4_index_score_us=round(kern_ms["index_score"] * 1e3, 2),
                                  peak_gbs=peak, frac=round(fp8["achieved_gbs"] / peak, 4)),
        "block_scaled_index_variant": dict(
            mxq, mxfp4_index_score_us=round(kern_ms["index_score"] * 1e3, 2), peak_gbs=peak,
            frac=round(mxq["achieved_gbs"] / peak, 4),
            numerics="index-q converted to MXFP8 (OCP: per 32-dim block, shared exponent "
                     "floor(log2 amax) - 8, E4M3 elements); tcgen05 block-scaled MMA"),
        "gpu_launches": head_blk["gpu_launches"],
        "clocks": head_blk["clocks"],
        "wall_s_timed_region": head_blk["wall_s_timed_region"],
        "workloads": blocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        cache = _OracleCache(wl)
        v, detail, spent = cpu_oracle_sample(wl, args.cpu_budget, cache)
        pv, pdetail, pwall, cores = cpu_oracle_parallel(wl, args.cpu_budget, cache=cache)
        line["cpu_baseline_parallel"] = {"value": round(pv, 3), "unit": UNIT, "cores": cores,
                                         "kind": "oracle", "sample": pdetail}
        line["cpu_baseline"] = {"value": round(v, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": detail}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_fp8_scorer(wl, caches, step, stream, flush_l2, steps):
    """index_score_fp8 over the fp8 (E4M3) index-K cache, filled from the same rows as
    the MXFP4 one, with the step's index-q, block table and lengths: event-timed per
    launch on the launching stream after an L2 flush.  Algorithmic bytes: one 128-byte
    key row per cached token."""
    import torch

    import mxfp4_sparse_paged_gb300 as m
    if step.slots.numel():  # the decode tokens' own rows, as the step inserts them
        m.fp8_index_insert(step.idx_new, step.slots, caches.fp8_index_scale, caches.fp8_idx_pages,
                           stream=stream)

    def score():
        m.index_score_fp8(step.iq, wl.q, caches.fp8_idx_pages, step.block_table, step.seq_lens,
                          caches.fp8_index_scale, step.scores, stream=stream)

    for _ in range(3):
        flush_l2(1)
        score()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        flush_l2(i & 0xFF)
        evs[i][0].record(stream)
        score()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    m.mx4_check_status()
    us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    nbytes = int(W.HEAD_DIM * wl.seq_lens.astype(np.int64).sum())
    return {"kernel": "index_score_fp8", "scale": caches.fp8_index_scale, "us": round(us, 2),
            "algorithmic_bytes": nbytes, "achieved_gbs": round(nbytes / us / 1e3, 1),
            "timing": "mean of CUDA-event pairs on the launching stream, L2 flushed before each"}


def time_mxq_scorer(wl, caches, step, stream, flush_l2, steps):
    """index_score_mxq -- the block-scaled tensor-core scorer, index-q converted to
    MXFP8 -- over the step's own MXFP4 index-K cache, index-q, block table and
    lengths: event-timed per launch on the launching stream after an L2 flush.
    Algorithmic bytes as index_score's: one 68-byte key row per cached token."""
    import torch

    import mxfp4_sparse_paged_gb300 as m

    def score():
        m.index_score_mxq(step.iq, wl.q, caches.idx_pages, step.block_table, step.seq_lens,
                          step.scores, stream=stream)

    for _ in range(3):
        flush_l2(1)
        score()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        flush_l2(i & 0xFF)
        evs[i][0].record(stream)
        score()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    m.mx4_check_status()
    us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    nbytes = W.algorithmic_bytes(wl)["index_score"]
    return {"kernel": "index_score_mxq", "us": round(us, 2), "algorithmic_bytes": nbytes,
            "achieved_gbs": round(nbytes / us / 1e3, 1),
            "traffic": _ncu_traffic(wl.spec.name, "index_score_mxq_traffic.json"),
            "timing": "mean of CUDA-event pairs on the launching stream, L2 flushed before each"}


def time_writer(wl, dev, stream, flush_l2, steps):
    """The norm + rotary writer (mx4_norm_rope_insert) on the step's T new tokens,
    next to the plain mx4_insert of the same K/V/index-K rows; both on a scratch
    pool, event-timed on the launching stream after an L2 flush.  Positions are the
    decode tokens' own; the rotary table covers them."""
    import torch

    import mxfp4_sparse_paged_gb300 as m
    T, H, Hkv = wl.T, W.Q_HEADS, W.KV_HEADS
    pos = wl.positions()
    x = {n: torch.from_numpy(a).to(dev) for n, a in W.writer_inputs(T, H, Hkv, wl.spec.seed).items()}
    cs = torch.from_numpy(W.rope_table(int(pos.max()) + 1)).to(dev)
    P = (T + W.PAGE_TOKENS - 1) // W.PAGE_TOKENS
    kp = torch.full((P, Hkv, W.PAGE_BYTES), W.POISON, dtype=torch.uint8, device=dev)
    vp = torch.full_like(kp, W.POISON)
    ip = torch.full((P, W.PAGE_BYTES), W.POISON, dtype=torch.uint8, device=dev)
    slots = torch.arange(T, dtype=torch.int64, device=dev)
    posd = torch.from_numpy(pos).to(dev)
    q_out = torch.empty((T, H, W.HEAD_DIM), dtype=torch.bfloat16, device=dev)
    iq_out = torch.empty((T, W.HEAD_DIM), dtype=torch.bfloat16, device=dev)

    def writer():
        m.mx4_norm_rope_insert(x["q"], x["iq"], x["k"], x["v"], x["idx_k"], posd, cs, x["g_q"],
                               x["g_k"], x["g_iq"], x["g_ik"], 1e-6, slots, kp, vp, ip, q_out,
                               iq_out, stream=stream)

    def plain():
        m.mx4_insert(x["k"], x["v"], x["idx_k"], slots, kp, vp, ip, stream=stream)

    us = {}
    for name, fn in (("mx4_norm_rope_insert", writer), ("mx4_insert", plain)):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush_l2(i & 0xFF)
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        us[name] = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    m.mx4_check_status()
    row = W.PAGE_BYTES // W.PAGE_TOKENS
    # fp32 rows in, one rotary-table row and position and slot per token, bf16 q and
    # index-q out, K/V/index-K page rows out
    nbytes = T * ((H + 2 * Hkv + 2) * W.HEAD_DIM * 4 + W.HEAD_DIM * 4 + 16 +
                  (H + 1) * W.HEAD_DIM * 2 + (2 * Hkv + 1) * row)
    return {"kernel": "mx4_norm_rope_insert", "tokens": T, "us": round(us["mx4_norm_rope_insert"], 2),
            "plain_mx4_insert_us": round(us["mx4_insert"], 2), "algorithmic_bytes": nbytes,
            "achieved_gbs": round(nbytes / us["mx4_norm_rope_insert"] / 1e3, 1),
            "timing": "mean of CUDA-event pairs on the launching stream, L2 flushed before each"}


def _ncu_traffic(name, record="index_score_traffic.json"):
    """dram bytes (read + write) per launch of a kernel from its committed ncu record
    for this workload, or None when there is none or the kernel's sources changed
    since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", record)
    try:
        with open(p) as f:
            rec = json.load(f)[name]
        h = hashlib.sha256()
        for src in rec["kernel_sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != rec["kernel_sources_sha256_16"]:
            return None
        return int(rec["traffic_bytes_per_launch"])
    except Exception:
        return None


def run_reference(args):
    """The reference arm: the oracle (C, float64) on the host's cores.  A step is the
    oracle's step for one sequence -- the insert of its decode tokens, scores, top-k,
    attention -- taken in turn from a fixed random order that cycles through the whole
    workload.  The steps are independent, so the --warmup steps and then the --steps
    timed steps each run on one thread per core; value = timed decode tokens / wall
    time of the timed steps.  The cache fill is untimed."""
    from concurrent.futures import ThreadPoolExecutor
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = W.make(args.workload)
    L = wl.seq_lens.astype(np.int64)
    workers = host_cores()
    cache = _OracleCache(wl)
    order = _sample_order(wl)
    seq_of = [order[i % wl.B] for i in range(args.warmup + args.steps)]
    warm, timed = seq_of[:args.warmup], seq_of[args.warmup:]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(cache.fill, sorted(set(seq_of))))
        list(ex.map(cache.step, warm))
        t0 = time.perf_counter()
        list(ex.map(cache.step, timed))
        wall = time.perf_counter() - t0
    value = len(timed) * wl.q / wall
    seen = sorted(set(timed))
    frac = float(L[seen].sum()) / float(L.sum())
    sample = (f"{len(timed)} timed steps of one sequence each, cycling through a fixed random "
              f"order ({len(seen)} of {wl.B} sequences, {100 * frac:.1f}% of the cached "
              f"tokens), {workers} threads, {wall:.1f} s wall; value = decode tokens / wall time")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * wall / len(timed), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(wl),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": workers,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile_step(args):
    """One eager decode step of the workload (each entry point once) and one launch of
    each extra leg (the norm/rotary writer, the fp8 index-K insert and scorer, the
    block-scaled scorer), inside
    the NVTX range "mx4_step", after the cache fill and a few warm-up steps outside it;
    for an ncu capture of every library kernel of a step (--nvtx --nvtx-include
    "mx4_step/").  Prints nothing to time."""
    import torch

    import mxfp4_sparse_paged_gb300 as m
    from mxfp4_sparse_paged_gb300.step import DecodeStep, PagedCaches, step_inputs_host
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    wl = W.make(args.workload if args.workload is not None else 4)
    caches = PagedCaches(wl.num_pages, device=dev, fp8_index_scale=FP8_INDEX_SCALE)
    caches.fill(wl)
    step = DecodeStep(wl, caches, device=dev)
    step.load_inputs(step_inputs_host(wl))
    for _ in range(args.warmup):
        step.run(stream=stream, fused=False)
    flush_l2 = _flusher(dev)
    flush_l2(1)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("mx4_step")
    step.run(stream=stream, fused=False)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("mx4_step")
    time_writer(wl, dev, stream, lambda v: None, 1)
    time_fp8_scorer(wl, caches, step, stream, lambda v: None, 1)
    time_mxq_scorer(wl, caches, step, stream, lambda v: None, 1)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    m.mx4_check_status()
    print(f"profile step done: {wl.spec.name}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=None, choices=range(5),
                    help="one workload only (default: all five, the last, 4, as the headline)")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of the same step run, clock-sampled, before the timed steps")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the cpu_baseline legs of the GPU arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-step", action="store_true",
                    help="one step and one launch of each extra leg inside the NVTX range "
                         "mx4_step, for an ncu capture; no timing")
    ap.add_argument("--eager", action="store_true",
                    help="time the step as separate API calls instead of one CUDA-graph launch")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.workload is None:
            args.workload = 4
        run_reference(args)
    elif args.profile_step:
        profile_step(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

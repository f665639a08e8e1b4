"""Benchmark: one decode step of sparse attention over MXFP4 paged caches.

A step is the whole hot path on one batch: mx4_insert of the decode tokens'
K/V/index-K rows (when the workload inserts in the step), index_score over
every cached index key, topk_select, sparse_paged_decode (split + merge).
Inputs are resident in HBM when the timed region starts; the L2 is flushed
(a 256 MiB write, then a read of it so the write-back of its dirty lines
falls outside the step) between timed steps, outside the per-step CUDA events.

Default workload: 256 sequences, lognormal contexts (median 8192, capped at
131072), one decode token each inserted in the step, top-2048 -- the only
workload whose step runs all four kernels.  `--workload 0..4` picks another.

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

def run_gpu(args):
    import torch
    import torch.distributed as dist

    import mxfp4_sparse_paged_gb300 as m
    from mxfp4_sparse_paged_gb300.step import DecodeStep, PagedCaches, PipelinedSteps, step_inputs_host

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

    wl = W.make(args.workload)
    # The fill also writes the fp8 index-K cache variant from the same rows; the timed
    # step reads only the MXFP4 pools.
    caches = PagedCaches(wl.num_pages, device=dev, fp8_index_scale=FP8_INDEX_SCALE)
    caches.fill(wl)
    step = DecodeStep(wl, caches, device=dev)
    host = step_inputs_host(wl)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2(v):
        # Write a buffer twice the L2 size, then read it back: the read evicts the
        # written lines, so their write-back lands here rather than in the step.
        flush.fill_(v)
        flush.view(torch.int64).sum()
    ab = W.algorithmic_bytes(wl)

    # The in-step insert rewrites the decode tokens' rows with the same values, so
    # every timed step does identical work.
    names = (["mx4_insert"] if wl.spec.insert_in_step else []) + \
        ["index_score", "topk_select", "sparse_paged_decode"]
    step.load_inputs(host)
    for _ in range(args.warmup):
        flush_l2(1)
        step.run(stream=stream)
    m.mx4_check_status()

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    st = [(ev(), ev()) for _ in range(args.steps)]
    if not args.eager:
        step.capture()  # the step's kernels as one CUDA graph (same launches, same order)
        for _ in range(3):
            flush_l2(1)
            step.replay()
    clocks = Clocks(local)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(i & 0xFF)
        st[i][0].record(stream)
        if args.eager:
            step.run(stream=stream)
        else:
            step.replay()
        st[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    ck = clocks.stop()
    m.mx4_check_status()
    step_ms = [a.elapsed_time(b) for a, b in st]
    # Per-kernel times: the same steps again with an event pair around each entry
    # point (events between kernels stop a kernel from starting early under the
    # previous one, so they are kept out of the step timing above).
    per = {n: [(ev(), ev()) for _ in range(args.steps)] for n in names}
    for i in range(args.steps):
        flush_l2(i & 0xFF)
        step.run(stream=stream, events={n: per[n][i] for n in names})
    torch.cuda.synchronize()
    m.mx4_check_status()
    kern_ms = {n: statistics.mean(a.elapsed_time(b) for a, b in per[n]) for n in names}
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(wl.T, world, args.steps, total_ms)

    # ---- end to end through the public API: host inputs -> device -> step -> host
    # output for every step, with the transfers of neighbouring steps overlapped
    # (PipelinedSteps).  No flush here: each step streams the 204 MB index cache and
    # writes and reads 134 MB of scores, more than the 129 MB L2.
    pipe = PipelinedSteps(wl, caches, device=dev)
    pin = pipe.pack_inputs(host)
    h2d = pin.numel()
    d2h = pipe.h_out[0].numel() * pipe.h_out[0].element_size()
    for _ in range(4):
        _, done = pipe.submit(pin)
    done.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(pipe.h2d)
    for _ in range(args.steps):
        _, done = pipe.submit(pin)
    pipe.h2d.wait_event(done)
    e1.record(pipe.h2d)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = job_value(wl.T, world, args.steps, e2e_ms)
    m.mx4_check_status()

    writer = time_writer(wl, dev, stream, flush_l2, min(args.steps, 200))
    fp8 = time_fp8_scorer(wl, caches, step, stream, flush_l2, min(args.steps, 200))

    peak, peak_kind = _peaks()
    score_s = kern_ms["index_score"] / 1e3
    achieved = ab["index_score"] / score_s / 1e9
    dec_s = kern_ms["sparse_paged_decode"] / 1e3
    hot_bytes = ab["index_score"] + ab["sparse_paged_decode"]
    hot_gbs = hot_bytes / (score_s + dec_s) / 1e9
    traffic = _ncu_traffic(wl.spec.name)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic (seeded N(0,1) K/V/index-K rows quantised to MXFP4 pages; "
                "bf16 N(0,1) queries)",
        "config": _config(wl),
        "roofline": {"bound": "hbm", "kernel": "index_score", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": ab["index_score"],
                     "traffic": traffic},
        "roofline_decode": {
            "bound": "hbm", "kernel": "sparse_paged_decode (split + merge kernels)",
            "achieved": round(ab["sparse_paged_decode"] / dec_s / 1e9, 1), "peak": peak,
            "unit": "GB/s", "frac": round(ab["sparse_paged_decode"] / dec_s / 1e9 / peak, 4),
            "algorithmic_bytes_per_launch": ab["sparse_paged_decode"],
            "traffic": _ncu_traffic(wl.spec.name, "decode_split_traffic.json"),
            "traffic_kernel": "decode_split_kernel"},
        "hot_path_hbm": {"kernels": "index_score + sparse_paged_decode",
                         "algorithmic_bytes": hot_bytes, "achieved_gbs": round(hot_gbs, 1),
                         "frac": round(hot_gbs / peak, 4)},
        "kernel_ms": {n: round(v, 5) for n, v in kern_ms.items()},
        "step_launch": ("separate API calls" if args.eager else
                        "one CUDA-graph launch of the step's kernels (captured from the API calls)"),
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "mode": "every step copies its inputs from pinned host memory and reads its "
                        "output back; the copies of neighbouring steps overlap the compute "
                        "(two buffer sets, three streams, one packed input copy and one CUDA-graph "
                        "launch a step); no L2 flush (a step moves more than the L2 holds)"},
        "norm_rope_writer": writer,
        "fp8_index_variant": dict(fp8, mxfp4_index_score_us=round(kern_ms["index_score"] * 1e3, 2),
                                  peak_gbs=peak,
                                  frac=round(fp8["achieved_gbs"] / peak, 4)),
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": ck,
        "wall_s_timed_region": round(wall, 3),
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4, choices=range(5))
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the cpu_baseline legs of the GPU arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time the step as separate API calls instead of one CUDA-graph launch")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

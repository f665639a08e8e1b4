"""Resident MXFP4 page caches and one decode step through the C ABI.

`PagedCaches` owns the three page pools of one layer (K and V [pages, 1, 8704],
index-K [pages, 8704]) in device memory, poisoned with 0xFF so a read of a
never-written row shows up as NaN, and fills them from a workload with
mx4_insert through the shared page-128 slot mapping ("vllm.models.minimax_m3.
amd.mono.dispatch", _slots_shared).  Optionally it also holds the fp8 index-K
cache [pages, 16384] of the other revision, filled from the same rows.

`DecodeStep` holds the per-step buffers and workspaces and issues, on one
stream, the hot path of a decode step: [mx4_insert of the new tokens] ->
index_topk (score and select in one call; fused=False issues index_score and
topk_select instead) -> sparse_paged_decode.  It allocates nothing per step.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import (FP8_PAGE_BYTES, fp8_index_insert, index_score, index_topk, mx4_decode_step,
               mx4_decode_steps,
               mx4_decode_step_input_layout, mx4_insert, sparse_paged_decode,
               sparse_paged_decode_workspace, topk_select, topk_select_workspace)
from . import workloads as W


class PagedCaches:
    """Resident page pools: MXFP4 K, V and index-K, and optionally the fp8 (E4M3)
    index-K cache variant with its per-cache scale, filled from the same rows."""

    def __init__(self, num_pages: int, device="cuda", kv_heads: int = 1,
                 fp8_index_scale: float | None = None):
        self.num_pages = num_pages
        self.k_pages = torch.full((num_pages, kv_heads, W.PAGE_BYTES), W.POISON, dtype=torch.uint8,
                                  device=device)
        self.v_pages = torch.full_like(self.k_pages, W.POISON)
        self.idx_pages = torch.full((num_pages, W.PAGE_BYTES), W.POISON, dtype=torch.uint8,
                                    device=device)
        self.fp8_index_scale = fp8_index_scale
        self.fp8_idx_pages = None
        if fp8_index_scale is not None:
            self.fp8_idx_pages = torch.full((num_pages, FP8_PAGE_BYTES), W.POISON,
                                            dtype=torch.uint8, device=device)

    def nbytes(self) -> int:
        fp8 = 0 if self.fp8_idx_pages is None else self.num_pages * FP8_PAGE_BYTES
        return 3 * self.num_pages * W.PAGE_BYTES + fp8

    def insert_rows(self, k, v, idx_k, slots, stream=None, fp8=True):
        """Insert into the MXFP4 pools and (fp8=True, if present) the fp8 index cache."""
        mx4_insert(k, v, idx_k, slots, self.k_pages, self.v_pages, self.idx_pages, stream=stream)
        if fp8 and self.fp8_idx_pages is not None:
            fp8_index_insert(idx_k, slots, self.fp8_index_scale, self.fp8_idx_pages, stream=stream)

    def fill(self, wl: W.Workload, chunk: int = 32768, sequences=None):
        """Insert tokens 0 .. prefilled(s)-1 of every (or the given) sequence."""
        dev = self.k_pages.device
        seqs = range(wl.B) if sequences is None else sequences
        for s in seqs:
            n = wl.prefilled(s)
            for a in range(0, n, chunk):
                b = min(n, a + chunk)
                k = torch.from_numpy(wl.rows(s, W.K_ROWS, a, b)).to(dev).view(b - a, 1, W.HEAD_DIM)
                v = torch.from_numpy(wl.rows(s, W.V_ROWS, a, b)).to(dev).view(b - a, 1, W.HEAD_DIM)
                ik = torch.from_numpy(wl.rows(s, W.IDX_ROWS, a, b)).to(dev)
                slots = torch.from_numpy(wl.slots(s, np.arange(a, b))).to(dev)
                self.insert_rows(k, v, ik, slots)


def _layout(specs):
    """Byte offsets (256-byte aligned) of named tensors packed into one buffer."""
    out, off = {}, 0
    for name, shape, dtype in specs:
        nb = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        out[name] = (off, nb, tuple(shape), dtype)
        off += (nb + 255) // 256 * 256
    out["bytes"] = max(off, 256)
    return out


def _views(buf: torch.Tensor, layout: dict) -> dict:
    return {name: buf[o:o + nb].view(dt).view(shape)
            for name, (o, nb, shape, dt) in ((k, v) for k, v in layout.items() if k != "bytes")}


def step_inputs_host(wl: W.Workload):
    """Host (numpy) inputs of one decode step: q/iq bf16 bits, the new tokens'
    rows and slots (empty unless the workload inserts in the step)."""
    q_bits, iq_bits = W.queries_bf16(wl)
    if wl.spec.insert_in_step:
        pos = wl.positions()
        s_of_t = np.repeat(np.arange(wl.B), wl.q)
        k = np.stack([wl.rows(int(s), W.K_ROWS, int(p), int(p) + 1)[0] for s, p in zip(s_of_t, pos)])
        v = np.stack([wl.rows(int(s), W.V_ROWS, int(p), int(p) + 1)[0] for s, p in zip(s_of_t, pos)])
        ik = np.stack([wl.rows(int(s), W.IDX_ROWS, int(p), int(p) + 1)[0]
                       for s, p in zip(s_of_t, pos)])
        slots = wl.step_slots()
    else:
        k = v = ik = np.zeros((0, W.HEAD_DIM), np.float32)
        slots = np.zeros(0, np.int64)
    return {"q": q_bits, "iq": iq_bits, "k": k, "v": v, "idx_k": ik, "slots": slots}


class DecodeStep:
    """Buffers and the kernel sequence of one decode step of workload `wl`."""

    def __init__(self, wl: W.Workload, caches: PagedCaches, device="cuda", fused=True):
        self.wl = wl
        self.caches = caches
        self.fused = fused
        T, k = wl.T, wl.k
        self.ld = int(wl.max_len)
        self.scale = 1.0 / math.sqrt(W.HEAD_DIM)
        self.block_table = torch.from_numpy(wl.block_table).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        n_ins = T if wl.spec.insert_in_step else 0
        # the step's inputs live in one device buffer (one host -> device copy a step)
        self.input_layout = _layout([
            ("q", (T, W.Q_HEADS, W.HEAD_DIM), torch.bfloat16),
            ("iq", (T, W.HEAD_DIM), torch.bfloat16),
            ("k", (n_ins, 1, W.HEAD_DIM), torch.float32),
            ("v", (n_ins, 1, W.HEAD_DIM), torch.float32),
            ("idx_k", (n_ins, W.HEAD_DIM), torch.float32),
            ("slots", (n_ins,), torch.int64)])
        offs, nbytes = mx4_decode_step_input_layout(T, n_ins)
        assert nbytes == self.input_layout["bytes"] and offs == [
            self.input_layout[n][0] for n in ("q", "iq", "k", "v", "idx_k", "slots")], \
            "packed input layout differs from the C step entry's"
        self.inputs = torch.empty(self.input_layout["bytes"], dtype=torch.uint8, device=device)
        views = _views(self.inputs, self.input_layout)
        self.q, self.iq = views["q"], views["iq"]
        self.k_new, self.v_new, self.idx_new = views["k"], views["v"], views["idx_k"]
        self.slots = views["slots"]
        self.graph = None
        self.scores = torch.empty((T, self.ld), dtype=torch.float32, device=device)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=device)
        self.out = torch.empty((T, W.Q_HEADS, W.HEAD_DIM), dtype=torch.float32, device=device)
        tws = topk_select_workspace(T, k, self.ld)
        self.topk_ws = torch.empty(max(tws, 16), dtype=torch.uint8, device=device) if tws else None
        self.dec_ws = torch.empty(sparse_paged_decode_workspace(T, k), dtype=torch.uint8,
                                  device=device)

    def pack_inputs(self, host: dict) -> torch.Tensor:
        """One step's host inputs (numpy, as from step_inputs_host) packed into a pinned
        buffer with the layout of the device input buffer."""
        buf = torch.empty(self.input_layout["bytes"], dtype=torch.uint8).pin_memory()
        views = _views(buf, self.input_layout)
        for name in ("q", "iq", "k", "v", "idx_k", "slots"):
            a = host[name]
            a = a.view(np.int16) if a.dtype == np.uint16 else a
            t = torch.from_numpy(np.ascontiguousarray(a))
            dst = views[name]
            if t.dtype == torch.int16:
                t = t.view(torch.bfloat16)
            dst.copy_(t.view(dst.shape))
        return buf

    def load_packed(self, packed: torch.Tensor, non_blocking=False):
        """Copy a packed pinned input buffer (pack_inputs) to the device: one copy."""
        self.inputs.copy_(packed, non_blocking=non_blocking)

    def capture(self):
        """Record run() (all kernels of the step) as a CUDA graph; replay() then
        launches the whole step at once.  The eager run that precedes the capture
        (first-call set-up) inserts nothing: its slots are set to -1, and the input
        buffer is restored afterwards."""
        saved = self.inputs.clone()
        self.slots.fill_(-1)
        self.run()
        self.inputs.copy_(saved)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(stream=torch.cuda.current_stream())
        self.graph = g
        return g

    def replay(self):
        """Launch the captured step on the current stream."""
        self.graph.replay()

    def load_inputs(self, host: dict, non_blocking=False):
        """Copy one step's host inputs (numpy or pinned torch) into the device buffers."""
        def put(dst, src, view_dtype=None):
            if isinstance(src, np.ndarray):
                src = torch.from_numpy(src)
            if view_dtype is not None:
                src = src.view(view_dtype)
            dst.copy_(src.view(dst.shape), non_blocking=non_blocking)
        put(self.q, host["q"].view(np.int16) if isinstance(host["q"], np.ndarray) else host["q"],
            torch.bfloat16)
        put(self.iq, host["iq"].view(np.int16) if isinstance(host["iq"], np.ndarray) else host["iq"],
            torch.bfloat16)
        if self.slots.numel():
            put(self.k_new, host["k"])
            put(self.v_new, host["v"])
            put(self.idx_new, host["idx_k"])
            put(self.slots, host["slots"])

    def stage_calls(self, stream=None) -> dict:
        """Each entry point of the step as a callable (name -> fn), for timing them one
        at a time: the insert (when the workload inserts), index_topk, and the pair it
        combines (index_score, topk_select), and sparse_paged_decode."""
        c, wl = self.caches, self.wl
        calls = {}
        if self.slots.numel():
            calls["mx4_insert"] = lambda: c.insert_rows(self.k_new, self.v_new, self.idx_new,
                                                        self.slots, stream=stream, fp8=False)
        calls["index_topk"] = lambda: index_topk(self.iq, wl.q, c.idx_pages, self.block_table,
                                                 self.seq_lens, self.scores, wl.k, self.topk_idx,
                                                 self.topk_ws, stream=stream)
        calls["index_score"] = lambda: index_score(self.iq, wl.q, c.idx_pages, self.block_table,
                                                   self.seq_lens, self.scores, stream=stream)
        calls["topk_select"] = lambda: topk_select(self.scores, self.seq_lens, wl.q, wl.k,
                                                   self.topk_idx, self.topk_ws, stream=stream)
        calls["sparse_paged_decode"] = lambda: sparse_paged_decode(
            self.q, wl.q, c.k_pages, c.v_pages, self.block_table, self.seq_lens, self.topk_idx,
            self.scale, self.out, self.dec_ws, stream=stream)
        return calls

    def run(self, stream=None, events=None, fused=None):
        """Enqueue the step on `stream`.  `events` (optional dict name -> (start, end)
        CUDA events) brackets each entry point for per-kernel timing; `fused`
        overrides the step's choice of index_topk or index_score + topk_select."""
        fused = self.fused if fused is None else fused
        c = self.caches
        wl = self.wl

        def timed(name, fn):
            if events and name in events:
                events[name][0].record(stream)
                fn()
                events[name][1].record(stream)
            else:
                fn()

        if self.slots.numel():
            timed("mx4_insert", lambda: c.insert_rows(self.k_new, self.v_new, self.idx_new,
                                                      self.slots, stream=stream, fp8=False))
        if fused:
            timed("index_topk", lambda: index_topk(self.iq, wl.q, c.idx_pages, self.block_table,
                                                   self.seq_lens, self.scores, wl.k, self.topk_idx,
                                                   self.topk_ws, stream=stream))
        else:
            timed("index_score", lambda: index_score(self.iq, wl.q, c.idx_pages,
                                                     self.block_table, self.seq_lens, self.scores,
                                                     stream=stream))
            timed("topk_select", lambda: topk_select(self.scores, self.seq_lens, wl.q, wl.k,
                                                     self.topk_idx, self.topk_ws, stream=stream))
        timed("sparse_paged_decode", lambda: sparse_paged_decode(
            self.q, wl.q, c.k_pages, c.v_pages, self.block_table, self.seq_lens, self.topk_idx,
            self.scale, self.out, self.dec_ws, stream=stream))

    def run_host(self, h_inputs: torch.Tensor, h_out: torch.Tensor, stream=None):
        """The whole step from host memory to host memory through the C entry point
        mx4_decode_step: the packed host inputs (pack_inputs; the same layout as the
        device input buffer) are copied in, the four stages run, and the output is
        copied into the host tensor h_out [T, 16, 128] fp32.  Asynchronous."""
        wl, c = self.wl, self.caches
        mx4_decode_step(h_inputs, self.slots.numel(), self.inputs, c.k_pages, c.v_pages,
                        c.idx_pages, self.block_table, self.seq_lens, wl.q, wl.k, self.scale,
                        self.scores, self.topk_idx, self.topk_ws, self.dec_ws, self.out, h_out,
                        stream=stream)

    def run_host_steps(self, h_inputs: torch.Tensor, h_out: torch.Tensor, n_steps: int,
                       stream: torch.cuda.Stream, h2d: torch.cuda.Stream,
                       d2h: torch.cuda.Stream):
        """n_steps steps from host memory to host memory through the C entry point
        mx4_decode_steps: the copies of neighbouring steps overlap the compute
        (inputs on h2d, outputs on d2h, kernels on stream).  h_inputs: one packed
        pinned buffer used by every step ([bytes]) or one per step ([n_steps, bytes]);
        h_out: pinned fp32 [T, 16, 128] (every step's output in turn) or
        [n_steps, T, 16, 128].  The second staging and output sets are allocated on
        first use.  Asynchronous; `stream` waits for the last output copy."""
        wl, c = self.wl, self.caches
        if getattr(self, "_staging2", None) is None:
            set_bytes = (self.input_layout["bytes"] + 255) // 256 * 256
            self._staging2 = torch.empty(2 * set_bytes, dtype=torch.uint8, device=self.out.device)
            self._out2 = torch.empty((2,) + tuple(self.out.shape), dtype=torch.float32,
                                     device=self.out.device)
        mx4_decode_steps(n_steps, h_inputs, self.slots.numel(), self._staging2, c.k_pages,
                         c.v_pages, c.idx_pages, self.block_table, self.seq_lens, wl.q, wl.k,
                         self.scale, self.scores, self.topk_idx, self.topk_ws, self.dec_ws,
                         self._out2, h_out, stream, h2d, d2h, same_inputs=(h_inputs.dim() == 1))

    def launches_per_step(self) -> int:
        """Kernels this library launches per step: insert; the scorer; the top-k
        selection (threshold and segment filter when a row can exceed the candidate
        capacity, then select); decode run kernel + merge."""
        sel = 3 if self.topk_ws is not None else 1
        return (1 if self.slots.numel() else 0) + 1 + sel + 2


class PipelinedSteps:
    """Back-to-back decode steps with the host transfers overlapped.

    A serving loop's step copies its inputs (q, iq, the new tokens' rows and slots)
    from pinned host memory and reads its output back.  Here step i+1's inputs
    (one packed buffer, one copy) go to the device on one stream while step i
    computes, and step i's output is read back on another while step i+1
    computes.  Each step is one CUDA-graph launch of all its kernels.  Two
    DecodeStep buffer sets alternate; the page caches are shared and the steps run
    in order on the compute stream, so every insert lands before the next step's
    reads.
    """

    def __init__(self, wl: W.Workload, caches: PagedCaches, device="cuda"):
        self.steps = [DecodeStep(wl, caches, device=device), DecodeStep(wl, caches, device=device)]
        for st in self.steps:
            st.capture()
        self.compute = torch.cuda.Stream(device=device)
        self.h2d = torch.cuda.Stream(device=device)
        self.d2h = torch.cuda.Stream(device=device)
        self.h_out = [torch.empty(s.out.shape, dtype=torch.float32).pin_memory() for s in self.steps]
        ev = lambda: torch.cuda.Event()  # noqa: E731
        self.inputs_ready = [ev(), ev()]
        self.compute_done = [ev(), ev()]
        self.out_done = [ev(), ev()]
        self.n = 0

    def pack_inputs(self, host: dict) -> torch.Tensor:
        return self.steps[0].pack_inputs(host)

    def submit(self, packed: torch.Tensor):
        """Enqueue one step on a packed pinned input buffer (pack_inputs); returns
        (pinned output tensor, event recorded when it holds this step's result)."""
        b = self.n & 1
        st = self.steps[b]
        with torch.cuda.stream(self.h2d):
            if self.n >= 2:
                self.h2d.wait_event(self.compute_done[b])  # step n-2 is done with buffers b
            st.load_packed(packed, non_blocking=True)
            self.inputs_ready[b].record(self.h2d)
        self.compute.wait_event(self.inputs_ready[b])
        if self.n >= 2:
            self.compute.wait_event(self.out_done[b])  # step n-2's output has been read back
        with torch.cuda.stream(self.compute):
            st.replay()
        self.compute_done[b].record(self.compute)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.compute_done[b])
            self.h_out[b].copy_(st.out, non_blocking=True)
            self.out_done[b].record(self.d2h)
        self.n += 1
        return self.h_out[b], self.out_done[b]

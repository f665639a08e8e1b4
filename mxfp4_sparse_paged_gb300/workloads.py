"""Seeded synthetic inputs for sparse-attention decode over MXFP4 paged caches.

This module only draws random inputs and lays out the tables that address
them.  It holds none of the method's arithmetic (no quantisation, no scoring,
no selection, no attention), so both the CUDA path and the CPU oracle can be
fed from it.

The five workloads follow the head geometry of one tensor-parallel rank of
the MiniMax-M3 sparse-attention layer ("vllm.models.minimax_m3.amd.mono.weights",
_build_cp_qkv: q(2048) | k(128) | v(128) | index_q(128) | index_k(128) rows,
i.e. 16 query heads, one KV head, one index head, head_dim 128) and the
page-128 cache of "vllm.models.minimax_m3.amd.ops.mxfp4_pages".

Every random draw comes from a numpy PCG64 generator keyed by
(workload seed, purpose, sequence, chunk), so any slice of any sequence can be
regenerated on its own, on any machine, without drawing the rest.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_TOKENS = 128
HEAD_DIM = 128
Q_HEADS = 16
KV_HEADS = 1
PAGE_BYTES = 8704
POISON = 0xFF  # bytes of never-written rows and pages (scale 0xFF reads as NaN)

K_ROWS, V_ROWS, IDX_ROWS = 0, 1, 2
_CHUNK = 4096  # tokens per independently seeded chunk of rows

# purposes of the seeded streams
_P_ROWS, _P_QUERY, _P_LENS, _P_PERM, _P_OUTLIER, _P_WRITER = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Spec:
    """One synthetic decode workload."""
    name: str
    batch: int                 # sequences B
    q: int                     # decode tokens per sequence
    lens: tuple                # ("fixed", L) | ("uniform", lo, hi) | ("lognormal", median, sigma, cap)
    k: int                     # top-k per decode token
    shuffle_pages: bool        # physical page ids a random permutation of the pool
    outlier_scale: float       # 1.0, or the factor applied to the outlier channels
    outlier_frac: float        # fraction of channels scaled (rounded, per tensor)
    insert_in_step: bool       # the decode token's rows are inserted inside the step
    seed: int
    spare_pages: int = 2       # never-used pages in the pool (poisoned)


SPECS = {
    0: Spec("tiny-b1-ctx512", 1, 1, ("fixed", 512), 128, False, 1.0, 0.0, False, 0),
    1: Spec("b8-ctx8192", 8, 1, ("fixed", 8192), 2048, True, 1.0, 0.0, False, 1),
    2: Spec("b64-ctx4096-65536", 64, 1, ("uniform", 4096, 65536), 2048, True, 1.0, 0.0,
            False, 2),
    3: Spec("b16-ctx131072-q4", 16, 4, ("fixed", 131072), 2048, True, 1.0, 0.0, False, 3),
    4: Spec("b256-lognormal8192-insert", 256, 1, ("lognormal", 8192, 1.0, 131072), 2048,
            True, 20.0, 0.01, True, 4),
}


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


@dataclass
class Workload:
    """Shapes, tables and lengths of one workload (contents are drawn lazily)."""
    spec: Spec
    seq_lens: np.ndarray        # int32 [B]
    block_table: np.ndarray     # int32 [B, W]; -1 past a sequence's pages
    num_pages: int
    outlier_channels: tuple = field(default=())  # one tuple of channels per row kind

    @property
    def B(self) -> int:
        return self.spec.batch

    @property
    def q(self) -> int:
        return self.spec.q

    @property
    def T(self) -> int:
        return self.spec.batch * self.spec.q

    @property
    def k(self) -> int:
        return self.spec.k

    @property
    def bt_width(self) -> int:
        return self.block_table.shape[1]

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max())

    def positions(self) -> np.ndarray:
        """Position of each decode token t = s*q + j: seq_len - q + j."""
        L = self.seq_lens.astype(np.int64)
        j = np.arange(self.q, dtype=np.int64)
        return (L[:, None] - self.q + j[None, :]).reshape(-1)

    def prefilled(self, s: int) -> int:
        """Tokens of sequence s already in the cache before the timed step."""
        L = int(self.seq_lens[s])
        return L - 1 if self.spec.insert_in_step else L

    def slots(self, s: int, positions) -> np.ndarray:
        """Page-128 slot of each given position of sequence s: the physical page
        from the block table times 128, plus the row in the page."""
        positions = np.asarray(positions, dtype=np.int64)
        pages = self.block_table[s, positions // PAGE_TOKENS].astype(np.int64)
        return pages * PAGE_TOKENS + positions % PAGE_TOKENS

    def step_slots(self) -> np.ndarray:
        """Slot mapping of the decode tokens (int64 [T])."""
        pos = self.positions().reshape(self.B, self.q)
        return np.concatenate([self.slots(s, pos[s]) for s in range(self.B)])

    # ---------------------------------------------------------------- contents

    def rows(self, s: int, kind: int, start: int, stop: int) -> np.ndarray:
        """fp32 [stop-start, 128] rows (K, V or index-K) of tokens start..stop-1
        of sequence s, drawn N(0,1), outlier channels multiplied."""
        out = np.empty((stop - start, HEAD_DIM), np.float32)
        c0 = start // _CHUNK
        c1 = (stop - 1) // _CHUNK if stop > start else c0 - 1
        for c in range(c0, c1 + 1):
            lo, hi = c * _CHUNK, (c + 1) * _CHUNK
            blk = _rng(self.spec.seed, _P_ROWS, s, kind, c).standard_normal(
                (_CHUNK, HEAD_DIM), dtype=np.float32)
            a, b = max(lo, start), min(hi, stop)
            out[a - start:b - start] = blk[a - lo:b - lo]
        if self.outlier_channels:
            for ch in self.outlier_channels[kind]:
                out[:, ch] *= np.float32(self.spec.outlier_scale)
        return out

    def queries_f32(self):
        """(q fp32 [T, 16, 128], iq fp32 [T, 128]) drawn N(0,1); the caller rounds
        them to bf16 (torch's round-to-nearest-even conversion)."""
        g = _rng(self.spec.seed, _P_QUERY)
        qf = g.standard_normal((self.T, Q_HEADS, HEAD_DIM), dtype=np.float32)
        iqf = g.standard_normal((self.T, HEAD_DIM), dtype=np.float32)
        return qf, iqf


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values, rounded by torch."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def queries_bf16(wl: Workload):
    """(q bits uint16 [T,16,128], iq bits uint16 [T,128])."""
    qf, iqf = wl.queries_f32()
    return to_bf16_bits(qf), to_bf16_bits(iqf)


def make(config: int, *, batch: int | None = None, lens=None) -> Workload:
    """Build workload `config` (0..4); `batch`/`lens` shrink it for tests
    (same generator keys, so the first sequences are identical)."""
    spec = SPECS[config]
    if batch is not None or lens is not None:
        spec = Spec(spec.name + "-reduced", batch or spec.batch, spec.q, lens or spec.lens,
                    spec.k, spec.shuffle_pages, spec.outlier_scale, spec.outlier_frac,
                    spec.insert_in_step, spec.seed, spec.spare_pages)
    B = spec.batch
    kind = spec.lens[0]
    if kind == "fixed":
        L = np.full(B, spec.lens[1], np.int64)
    elif kind == "uniform":
        L = _rng(spec.seed, _P_LENS).integers(spec.lens[1], spec.lens[2], size=B,
                                              endpoint=True)
    elif kind == "lognormal":
        med, sigma, cap = spec.lens[1:]
        x = _rng(spec.seed, _P_LENS).normal(math.log(med), sigma, size=B)
        L = np.clip(np.rint(np.exp(x)), 1, cap).astype(np.int64)
    else:
        raise ValueError(kind)
    L = np.maximum(L, spec.q)
    pages_per_seq = (L + PAGE_TOKENS - 1) // PAGE_TOKENS
    W = int(pages_per_seq.max())
    used = int(pages_per_seq.sum())
    num_pages = used + spec.spare_pages
    ids = np.arange(num_pages, dtype=np.int64)
    if spec.shuffle_pages:
        ids = _rng(spec.seed, _P_PERM).permutation(num_pages)
    bt = np.full((B, W), -1, np.int32)
    o = 0
    for s in range(B):
        n = int(pages_per_seq[s])
        bt[s, :n] = ids[o:o + n]
        o += n
    channels = ()
    if spec.outlier_scale != 1.0:
        n_out = max(1, int(round(spec.outlier_frac * HEAD_DIM)))
        g = _rng(spec.seed, _P_OUTLIER)
        channels = tuple(tuple(int(c) for c in g.choice(HEAD_DIM, n_out, replace=False))
                         for _ in range(3))
    return Workload(spec, L.astype(np.int32), bt, num_pages, channels)


def algorithmic_bytes(wl: Workload) -> dict:
    """Bytes the page layout forces per step: 68 B per cached token row read.

    index_score reads each sequence's index rows once (all q decode tokens of a
    sequence share the pass); sparse_paged_decode reads one K and one V row per
    selected token; mx4_insert writes three rows per inserted token."""
    row = PAGE_BYTES // PAGE_TOKENS
    L = wl.seq_lens.astype(np.int64)
    pos = wl.positions()
    sel = np.minimum(pos + 1, wl.k)
    ins = wl.T if wl.spec.insert_in_step else 0
    return {
        "index_score": int(row * L.sum()),
        "sparse_paged_decode": int(2 * row * sel.sum()),
        "mx4_insert": int(3 * row * ins),
        "selected_tokens": int(sel.sum()),
    }


def rope_table(max_pos: int, base: float = 10000.0) -> np.ndarray:
    """Rotary table fp32 [max_pos, 128]: column i < 64 is cos(p * base^(-i/64)) at
    row p, column 64 + i the matching sine.  It is an input of the writer like any
    other (the usual rotary frequencies; any table is a valid one)."""
    inv = base ** (-np.arange(HEAD_DIM // 2, dtype=np.float64) / (HEAD_DIM // 2))
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def writer_inputs(T: int, H: int, Hkv: int, seed: int) -> dict:
    """Pre-norm fp32 rows of T new tokens for the norm + rotary writer: q [T, H, 128],
    iq [T, 128], k and v [T, Hkv, 128], idx_k [T, 128] (N(0,1) rows, each row
    times 2^u with u uniform in [-8, 8)), and the four norm weights g_q, g_k, g_iq,
    g_ik [128] drawn 1 + 0.2 N(0,1)."""
    g = _rng(seed, _P_WRITER)

    def rows(*shape):
        x = g.standard_normal(shape + (HEAD_DIM,))
        return (x * np.exp2(g.uniform(-8, 8, shape + (1,)))).astype(np.float32)

    out = {"q": rows(T, H), "iq": rows(T), "k": rows(T, Hkv), "v": rows(T, Hkv),
           "idx_k": rows(T)}
    for n in ("g_q", "g_k", "g_iq", "g_ik"):
        out[n] = (1.0 + 0.2 * g.standard_normal(HEAD_DIM)).astype(np.float32)
    return out

"""Both sides of a parity check, built from the same seeded inputs.

The oracle side quantises the workload's fp32 rows itself (its own pages) and
computes scores, selections and attention outputs for a chosen subset of
sequences; nothing on it comes from the CUDA path.  The GPU side fills device
pages with mx4_insert and runs the decode step through the C ABI.
"""
import math

import numpy as np

import oracle
from mxfp4_sparse_paged_gb300 import workloads as W

SCORE_REL = 4e-6   # fp32 dot of 128 terms: <= ~34 roundings of u = 2^-24 on sum |terms|
TOPK_BAND = 1e-5   # tokens this close (relative) to the k-th score may swap
ATTN_ABS = 2e-3    # max-abs error of attention outputs


class OracleSide:
    """Oracle pages of the sequences `seqs` (same physical page ids as the GPU)."""

    def __init__(self, wl: W.Workload, seqs, host):
        self.wl = wl
        self.seqs = list(seqs)
        P = wl.num_pages
        self.kp = np.full((P, 1, 8704), W.POISON, np.uint8)
        self.vp = np.full((P, 1, 8704), W.POISON, np.uint8)
        self.ip = np.full((P, 8704), W.POISON, np.uint8)
        for s in self.seqs:
            n = wl.prefilled(s)
            for a in range(0, n, 65536):
                b = min(n, a + 65536)
                oracle.mx4_insert(wl.rows(s, W.K_ROWS, a, b)[:, None],
                                  wl.rows(s, W.V_ROWS, a, b)[:, None],
                                  wl.rows(s, W.IDX_ROWS, a, b), wl.slots(s, np.arange(a, b)),
                                  self.kp, self.vp, self.ip)
        tok = np.concatenate([np.arange(s * wl.q, (s + 1) * wl.q) for s in self.seqs])
        self.tok = tok
        if wl.spec.insert_in_step:
            oracle.mx4_insert(host["k"][tok][:, None], host["v"][tok][:, None],
                              host["idx_k"][tok], host["slots"][tok], self.kp, self.vp, self.ip)
        self.lens = wl.seq_lens[self.seqs]
        self.bt = wl.block_table[self.seqs]
        self.ld = int(wl.max_len)
        self.iq = host["iq"][tok]
        self.q = host["q"][tok]

    def pages_of(self, s):
        n = (int(self.wl.seq_lens[s]) + 127) // 128
        return self.wl.block_table[s, :n]

    def scores(self):
        return oracle.index_score(self.iq, self.wl.q, self.ip, self.bt, self.lens, self.ld,
                                  want_mag=True)

    def topk(self, scores):
        return oracle.topk_select(scores, self.lens, self.wl.q, self.wl.k)

    def attend(self, sel):
        return oracle.sparse_paged_decode(self.q, self.wl.q, self.kp, self.vp, self.bt, self.lens,
                                          sel, 1 / math.sqrt(128))


def check_scores(got, want, mag, n_valid):
    """got fp32 [T, ld] vs oracle float64; entries 0..L-1 of each row compared."""
    for t in range(want.shape[0]):
        n = n_valid[t]
        g = got[t, :n].astype(np.float64)
        w = want[t, :n]
        fin = np.isfinite(w)
        assert np.array_equal(np.isfinite(g), fin), f"token {t}: -inf pattern differs"
        err = np.abs(g[fin] - w[fin])
        tol = SCORE_REL * mag[t, :n][fin] + 1e-30
        bad = np.nonzero(err > tol)[0]
        assert bad.size == 0, (f"token {t}: {bad.size} scores off, worst at i={bad[0]}: "
                               f"{g[fin][bad[0]]} vs {w[fin][bad[0]]} (tol {tol[bad[0]]})")


def check_topk(got, want, scores, n_sel_rows):
    """Selections equal except tokens within TOPK_BAND (relative) of the k-th score."""
    for t in range(want.shape[0]):
        g, w = got[t], want[t]
        gv, wv = g[g >= 0], w[w >= 0]
        assert len(gv) == len(wv), f"token {t}: {len(gv)} vs {len(wv)} selected"
        assert np.all(np.diff(gv) > 0), f"token {t}: not ascending"
        assert np.all(g[len(gv):] == -1)
        if np.array_equal(gv, wv):
            continue
        row = scores[t, :n_sel_rows[t]]
        tau = np.sort(row)[::-1][len(wv) - 1]
        band = TOPK_BAND * max(abs(tau), float(np.sqrt(np.mean(row ** 2))))
        diff = np.setxor1d(gv, wv)
        assert np.all(np.abs(row[diff] - tau) <= band), \
            f"token {t}: selections differ outside the near-tie band"

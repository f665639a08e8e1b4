"""Parity of the block-scaled tensor-core scorer (index_score_mxq) with the
oracle's MXFP8-query mode (index_score_mxq in oracle/: the bf16 index-q row
converted to MXFP8 per the OCP MX rules, dotted with the dequantised MXFP4 key).

The query's E4M3 codes are an integer decision taken in fp32 on both sides (a
power-of-two scaling, exact, then nearest-even), so the only difference left is
the tensor core's fp32 accumulation, held to the same bound as the other scorers:
SCORE_REL of the sum of |terms|.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp4_sparse_paged_gb300 as m
from mxfp4_sparse_paged_gb300 import workloads as W
from mxfp4_sparse_paged_gb300.step import DecodeStep, PagedCaches, step_inputs_host

from _sides import OracleSide, check_scores

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _dev_bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)


def _paged_case(lens, rng, scale_lo=112, scale_hi=142):
    """Random MXFP4 pages (any byte is a valid e2m1 pair) for sequences of `lens`,
    pages scattered through a pool with a spare page, block table padded with -1."""
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    npg = (lens + 127) // 128
    P = int(npg.sum()) + 3
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((B, int(npg.max()) + 1), -1, np.int32)
    o = 0
    for s in range(B):
        bt[s, :npg[s]] = perm[o:o + npg[s]]
        o += npg[s]
    pages = rng.integers(0, 256, (P, 8704), dtype=np.uint8)
    pages[:, 8192:] = rng.integers(scale_lo, scale_hi, (P, 512), dtype=np.uint8)
    return lens, bt, pages


def _query_rows(n, rng):
    """bf16 index-q rows with the MXFP8 conversion's edge cases spread over blocks:
    magnitudes from 2^-20 to 2^20 per row, all-zero blocks, blocks below the
    normal range (shared exponent clamped to -127), blocks whose largest element
    lands in (448, 512) after scaling (saturates to 448), and a one-hot block."""
    x = rng.standard_normal((n, 128)) * 2.0 ** rng.uniform(-20, 20, (n, 1))
    for r in range(n):
        b = 32 * (r % 4)
        kind = r % 5
        if kind == 1:
            x[r, b:b + 32] = 0.0
        elif kind == 2:
            x[r, b:b + 32] = rng.standard_normal(32) * 2.0 ** -128
        elif kind == 3:
            x[r, b:b + 32] = rng.uniform(-1, 1, 32)
            x[r, b + 5] = 1.9375                       # / 2^-8 = 496 -> saturates
        elif kind == 4:
            x[r, b:b + 32] = 0.0
            x[r, b + 31] = -3.0
    return _bf16_bits(x.astype(np.float32))


def _run_both(iq_bits, q, pages, bt, lens, ld):
    want, mag = oracle.index_score_mxq(iq_bits, q, pages, bt, lens, ld, want_mag=True)
    got = torch.full((len(lens) * q, ld), 7.0, dtype=torch.float32, device=DEV)
    m.index_score_mxq(_dev_bf16(iq_bits), q, torch.from_numpy(pages).to(DEV),
                      torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV), got)
    m.mx4_check_status()
    return got.cpu().numpy(), want, mag


def _worst_rel(got, want, mag, L_tok):
    w = 0.0
    for t in range(want.shape[0]):
        n = int(L_tok[t])
        fin = np.isfinite(want[t, :n])
        e = np.abs(got[t, :n][fin].astype(np.float64) - want[t, :n][fin])
        mm = mag[t, :n][fin]
        nz = mm > 0
        if nz.any():
            w = max(w, float((e[nz] / mm[nz]).max()))
    return w


@pytest.mark.parametrize("q", [1, 2, 3, 5, 8])
def test_index_score_mxq_ragged_against_oracle(q):
    rng = np.random.default_rng(500 + q)
    lens, bt, pages = _paged_case([q, 127, 128, 129, 700, 1500, 2049, 4100, 9000], rng)
    iq_bits = _query_rows(len(lens) * q, rng)
    ld = int(lens.max()) + 5
    got, want, mag = _run_both(iq_bits, q, pages, bt, lens, ld)
    L_tok = np.repeat(lens, q)
    print(f"q={q}: worst |err| / sum|terms| = {_worst_rel(got, want, mag, L_tok):.3g}")
    check_scores(got, want, mag, L_tok)
    for t in range(len(L_tok)):                        # nothing written past seq_len
        assert np.all(got[t, L_tok[t]:] == 7.0)


def test_index_score_mxq_many_pages_per_cta():
    # Enough pages that every CTA streams several through its stage ring (and
    # wraps it), with sequence changes inside a CTA's range of pages.
    rng = np.random.default_rng(606)
    q = 2
    lens, bt, pages = _paged_case([70001, 3, 65536, 40000, 129, 90000], rng)
    assert int(((lens + 127) // 128).sum()) > 4 * 3 * 160
    iq_bits = _query_rows(len(lens) * q, rng)
    ld = int(lens.max())
    got, want, mag = _run_both(iq_bits, q, pages, bt, lens, ld)
    L_tok = np.repeat(lens, q)
    print(f"worst |err| / sum|terms| = {_worst_rel(got, want, mag, L_tok):.3g}")
    check_scores(got, want, mag, L_tok)


def test_index_score_mxq_key_scale_extremes():
    # Key scale bytes across the E8M0 range (2^-100 .. 2^100 with queries that keep
    # the products finite in fp32), one row whose codes are all zero, and a
    # sequence whose length is not a multiple of 128 with q = 4.
    rng = np.random.default_rng(77)
    q = 4
    lens, bt, pages = _paged_case([300, 1000], rng, 27, 228)
    pages[bt[0, 0], 5 * 64:6 * 64] = 0
    iq_bits = _bf16_bits((rng.standard_normal((2 * q, 128)) * 2.0 ** -30).astype(np.float32))
    got, want, mag = _run_both(iq_bits, q, pages, bt, lens, 1000)
    L_tok = np.repeat(lens, q)
    print(f"worst |err| / sum|terms| = {_worst_rel(got, want, mag, L_tok):.3g}")
    check_scores(got, want, mag, L_tok)


def test_index_score_mxq_close_to_the_bf16_scorer():
    # The mode's documented difference from index_score: each query element moves
    # by at most half an E4M3 step of its block (2^-4 relative to the block's
    # scale step) or the saturation error, so |mxq - bf16| <= sum_j |k_j| * delta_j.
    rng = np.random.default_rng(91)
    q = 2
    lens, bt, pages = _paged_case([2000, 517], rng)
    iq_bits = _query_rows(len(lens) * q, rng)
    ld = 2000
    got, _, _ = _run_both(iq_bits, q, pages, bt, lens, ld)
    ref = torch.empty((len(lens) * q, ld), dtype=torch.float32, device=DEV)
    m.index_score(_dev_bf16(iq_bits), q, torch.from_numpy(pages).to(DEV),
                  torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV), ref)
    ref = ref.cpu().numpy().astype(np.float64)
    x = torch.from_numpy(iq_bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    delta = np.empty_like(x)                              # per-element bound on the query change
    for t in range(x.shape[0]):
        for b in range(4):
            blk = x[t, 32 * b:32 * b + 32]
            E = oracle.mxfp8_block_exponent(float(np.abs(blk).max()))
            step = 2.0 ** (E - 3) * 2.0 ** np.floor(np.log2(np.maximum(np.abs(blk) * 2.0 ** -E, 2.0 ** -6)))
            delta[t, 32 * b:32 * b + 32] = np.maximum(step / 2, np.abs(blk) - 448 * 2.0 ** E)
    # sum_j |k_j| delta_j from the oracle's dequantised keys, for a sample of rows
    for s, L in enumerate(lens):
        for i in rng.choice(int(L), 40, replace=False):
            krow = oracle.dequant_row(pages[bt[s, i // 128]], int(i % 128))
            for j in range(q):
                t = s * q + j
                if i > L - q + j:
                    continue
                bound = float(np.abs(krow) @ delta[t])
                magx = float(np.abs(krow) @ np.abs(x[t]))     # both scorers' fp32 error scale
                assert abs(got[t, i] - ref[t, i]) <= bound + 1e-5 * magx + 1e-30


def test_index_score_mxq_full_size_sampled():
    # The b256 lognormal workload (2.98 M cached tokens): the whole batch scored in
    # block-scaled mode after the step's insert, sampled sequences against the
    # oracle's own pages.
    wl = W.make(4)
    caches = PagedCaches(wl.num_pages, device=DEV)
    caches.fill(wl)
    step = DecodeStep(wl, caches, device=DEV)
    host = step_inputs_host(wl)
    step.load_inputs(host)
    step.run()
    sc = torch.empty_like(step.scores)
    m.index_score_mxq(step.iq, wl.q, caches.idx_pages, step.block_table, step.seq_lens, sc)
    m.mx4_check_status()
    L = wl.seq_lens
    short = int(np.nonzero(L < 2048)[0][0])
    seqs = sorted({short, int(np.argmax(L)), int(np.argmin(L)), 9, 77, 140, 201, 255})
    assert len(seqs) >= 8
    orc = OracleSide(wl, seqs, host)
    want, mag = oracle.index_score_mxq(orc.iq, wl.q, orc.ip, orc.bt, orc.lens, orc.ld,
                                       want_mag=True)
    got = sc.cpu().numpy()[orc.tok]
    L_tok = np.repeat(orc.lens, wl.q)
    print(f"worst |err| / sum|terms| = {_worst_rel(got, want, mag, L_tok):.3g}")
    check_scores(got, want, mag, L_tok)

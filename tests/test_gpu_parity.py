"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Page bytes and top-k sets are compared bit for bit (top-k: except tokens within
1e-5 relative of the k-th score); scores within the fp32 rounding bound of a
128-term dot product; attention outputs within max-abs 2e-3.  Small workloads
are compared in full, the full-size ones on sampled sequences, in the launch
configuration the benchmark times (DecodeStep).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import mxfp4_sparse_paged_gb300 as m
from mxfp4_sparse_paged_gb300 import workloads as W
from mxfp4_sparse_paged_gb300.step import DecodeStep, PagedCaches, PipelinedSteps, step_inputs_host

from _sides import ATTN_ABS, OracleSide, check_scores, check_topk

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"


def _gpu_step(wl):
    caches = PagedCaches(wl.num_pages, device=DEV)
    caches.fill(wl)
    step = DecodeStep(wl, caches, device=DEV)
    host = step_inputs_host(wl)
    step.load_inputs(host)
    step.run()
    m.mx4_check_status()
    return caches, step, host


def _compare(wl, seqs, caches, step, host):
    orc = OracleSide(wl, seqs, host)
    kp, vp, ip = (caches.k_pages.cpu().numpy(), caches.v_pages.cpu().numpy(),
                  caches.idx_pages.cpu().numpy())
    for s in seqs:
        pg = orc.pages_of(s)
        assert np.array_equal(kp[pg], orc.kp[pg]), f"K pages of sequence {s}"
        assert np.array_equal(vp[pg], orc.vp[pg]), f"V pages of sequence {s}"
        assert np.array_equal(ip[pg], orc.ip[pg]), f"index pages of sequence {s}"
    sc, mag = orc.scores()
    tok = orc.tok
    L_tok = np.repeat(orc.lens, wl.q).astype(np.int64)
    n_tok = wl.positions()[tok] + 1
    check_scores(step.scores.cpu().numpy()[tok], sc, mag, L_tok)
    sel = orc.topk(sc)
    g_sel = step.topk_idx.cpu().numpy()[tok]
    check_topk(g_sel, sel, sc, n_tok)
    want = orc.attend(sel)
    # chain output where the selections agree exactly
    g_out = step.out.cpu().numpy()[tok]
    same = [i for i in range(len(tok)) if np.array_equal(g_sel[i], sel[i])]
    assert len(same) >= len(tok) // 2
    err = max(float(np.abs(g_out[i] - want[i]).max()) for i in same)
    assert err <= ATTN_ABS, f"chain attention max-abs {err}"
    # the GPU decode fed the oracle's selection: every sampled token
    idx = step.topk_idx.clone()
    idx[torch.as_tensor(tok, device=DEV)] = torch.as_tensor(sel, device=DEV)
    out = torch.empty_like(step.out)
    m.sparse_paged_decode(step.q, wl.q, caches.k_pages, caches.v_pages, step.block_table,
                          step.seq_lens, idx, step.scale, out, step.dec_ws)
    m.mx4_check_status()
    err2 = float(np.abs(out.cpu().numpy()[tok] - want).max())
    assert err2 <= ATTN_ABS, f"decode max-abs {err2}"
    return err, err2


# ----------------------------------------------------------------- workloads

def test_config0_tiny_full():
    wl = W.make(0)
    _compare(wl, [0], *_gpu_step(wl))


def test_config1_full():
    wl = W.make(1)
    _compare(wl, range(wl.B), *_gpu_step(wl))


def test_config2_sampled():
    wl = W.make(2)
    L = wl.seq_lens
    seqs = sorted({int(np.argmin(L)), int(np.argmax(L)), 3, 7, 19, 33, 45, 58, 63})
    assert len(seqs) >= 8
    _compare(wl, seqs, *_gpu_step(wl))


def test_config3_sampled_multi_token():
    wl = W.make(3)
    _compare(wl, [0, 2, 4, 6, 9, 11, 13, 15], *_gpu_step(wl))  # 8 of 16 sequences, 32 tokens


def test_config4_sampled_with_insert():
    wl = W.make(4)
    L = wl.seq_lens
    short = int(np.nonzero(L < 2048)[0][0])
    seqs = sorted({short, int(np.argmax(L)), int(np.argmin(L)), 5, 30, 60, 100, 150, 200, 250})
    assert len(seqs) >= 8
    _compare(wl, seqs, *_gpu_step(wl))


def _custom(lens, q, k, seed, insert=False, outliers=False):
    lens = np.asarray(lens, np.int64)
    base = W.SPECS[4 if outliers else 1]
    spec = dataclasses.replace(base, name="custom", batch=len(lens), q=q, k=k, seed=seed,
                               insert_in_step=insert, lens=("fixed", 0))
    pages = (lens + 127) // 128
    P = int(pages.sum()) + 3
    ids = np.random.default_rng(seed).permutation(P)
    bt = np.full((len(lens), int(pages.max())), -1, np.int32)
    o = 0
    for s, n in enumerate(pages):
        bt[s, :n] = ids[o:o + n]
        o += n
    ch = ()
    if outliers:
        ch = ((3,), (64,), (127,))
    return W.Workload(spec, lens.astype(np.int32), bt, P, ch)


@pytest.mark.parametrize("q", [1, 2, 3, 4])
def test_ragged_lengths_all_tokens(q):
    # lengths around page and split boundaries, k above and below the context
    wl = _custom([q, 127, 128, 129, 255, 256, 257, 700, 1500], q=q, k=300, seed=40 + q)
    _compare(wl, range(wl.B), *_gpu_step(wl))


def test_ragged_with_insert_and_outliers():
    wl = _custom([1, 2, 129, 1000, 3000], q=1, k=2048, seed=77, insert=True, outliers=True)
    _compare(wl, range(wl.B), *_gpu_step(wl))


# ----------------------------------------------------------------- insert edges

def _insert_both(rows):
    """Insert rows (fp32 [n, 128]) as index keys on both sides; return both pools."""
    n = rows.shape[0]
    P = (n + 127) // 128
    slots = np.arange(n, dtype=np.int64)
    ip_o = np.full((P, 8704), 0xFF, np.uint8)
    oracle.mx4_insert(None, None, rows, slots, None, None, ip_o)
    kp = torch.full((P, 1, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    vp = torch.full_like(kp, 0xFF)
    ip = torch.full((P, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    r = torch.from_numpy(rows).to(DEV)
    m.mx4_insert(r.view(n, 1, 128), r.view(n, 1, 128), r, torch.from_numpy(slots).to(DEV),
                 kp, vp, ip)
    m.mx4_check_status()
    return ip.cpu().numpy(), ip_o


def test_insert_special_values_bit_exact():
    rows = np.zeros((64, 128), np.float32)
    f32 = np.finfo(np.float32)
    rows[1, :] = -0.0
    rows[2, 0] = f32.tiny                       # smallest normal
    rows[3, 0] = np.float32(2.0 ** -149)        # smallest subnormal
    rows[3, 1] = -np.float32(2.0 ** -140)
    rows[4, :32] = f32.max
    rows[4, 1] = -f32.max
    rows[5, :32] = np.float32(3e38) * np.linspace(-1, 1, 32, dtype=np.float32)
    # exact ties after scaling by 2^E (block amax 6 -> E = 0)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    rows[6, :7], rows[6, 7] = ties, 6.0
    rows[6, 32:39], rows[6, 39] = -ties, -6.0
    rows[7, :7], rows[7, 7] = ties * 2.0 ** -20, 6.0 * 2.0 ** -20
    rows[8, :] = np.float32(7.999)              # saturation
    rows[9, :] = np.float32(np.nextafter(np.float32(2), np.float32(0)))
    rng = np.random.default_rng(1)
    rows[10:] = (rng.standard_normal((54, 128)) *
                 2.0 ** rng.integers(-140, 120, (54, 1))).astype(np.float32)
    got, want = _insert_both(rows)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("q", [1, 3])
def test_index_score_special_scale_bytes(q):
    # Index keys whose scale byte is 0 with non-zero codes (block amax just above
    # 2^-126), all-zero blocks (byte 0, codes 0), and one row poisoned to scale
    # 0xFF inside the valid range: finite scores match, the poisoned one is
    # non-finite on both sides.
    rng = np.random.default_rng(21)
    n = 300
    rows = rng.standard_normal((n, 128)).astype(np.float32)
    rows[10:20, :32] = rng.uniform(-1.5, 1.5, (10, 32)).astype(np.float32) * np.float32(2.0 ** -126)
    rows[20:30, 32:64] = 0.0
    rows[30:35] = 0.0
    ip, ip_o = _insert_both(rows)
    assert np.array_equal(ip, ip_o)
    assert (ip_o[0, 8192 + 10 * 4] == 0) and (ip_o[0, 10 * 64] != 0)
    ip_o[0, 8192 + 40 * 4:8192 + 41 * 4] = 0xFF
    ip[0, 8192 + 40 * 4:8192 + 41 * 4] = 0xFF
    iq32 = rng.standard_normal((q, 128)).astype(np.float32)
    iq = torch.from_numpy(iq32).to(torch.bfloat16)
    iq_bits = iq.view(torch.int16).numpy().view(np.uint16)
    lens = np.array([n], np.int32)
    bt = np.arange(3, dtype=np.int32)[None, :]
    want, mag = oracle.index_score(iq_bits, q, ip_o, bt, lens, n, want_mag=True)
    got = torch.empty((q, n), dtype=torch.float32, device=DEV)
    m.index_score(iq.to(DEV), q, torch.from_numpy(ip).to(DEV), torch.from_numpy(bt).to(DEV),
                  torch.from_numpy(lens).to(DEV), got)
    m.mx4_check_status()
    g = got.cpu().numpy()
    check_scores(g, want, mag, np.full(q, n))
    assert not np.isfinite(g[:, 40]).any() and not np.isfinite(want[:, 40]).any()


def test_insert_dense_sweep_of_scaled_values():
    # Every 257th fp32 bit pattern in [0, 8) (both signs), 31 per block next to an
    # anchor of 4.0 so the block exponent is 0 and y = x.
    pats = np.arange(0, np.float32(8.0).view(np.uint32), 257, dtype=np.uint32)
    vals = pats.view(np.float32)
    vals = np.concatenate([vals, -vals])
    nb = (len(vals) + 30) // 31
    blocks = np.zeros((nb, 32), np.float32)
    blocks[:, 0] = 4.0
    flat = np.zeros(nb * 31, np.float32)
    flat[:len(vals)] = vals
    blocks[:, 1:] = flat.reshape(nb, 31)
    nrow = (nb + 3) // 4
    rows = np.zeros((nrow * 4, 32), np.float32)
    rows[:nb] = blocks
    rows = rows.reshape(nrow, 128)
    for a in range(0, nrow, 1 << 16):
        got, want = _insert_both(np.ascontiguousarray(rows[a:a + (1 << 16)]))
        assert np.array_equal(got, want)


def test_insert_every_pattern_near_each_rounding_threshold():
    # Both encoders are monotone step functions of |y| (the kernel counts threshold
    # comparisons; the oracle takes the nearest grid value), so they agree everywhere
    # once they agree on every fp32 pattern around each of the 7 midpoints and on a
    # sweep in between (the test above).  Here: all patterns within 4096 ulps of each
    # midpoint, both signs, next to an anchor of 4.0 so the block exponent is 0.
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    u = mids.view(np.int32)
    pats = (u[:, None] + np.arange(-4096, 4097, dtype=np.int32)[None, :]).reshape(-1)
    vals = pats.view(np.float32)
    vals = np.concatenate([vals, -vals])
    nb = (len(vals) + 30) // 31
    blocks = np.zeros((nb, 32), np.float32)
    blocks[:, 0] = 4.0
    flat = np.zeros(nb * 31, np.float32)
    flat[:len(vals)] = vals
    blocks[:, 1:] = flat.reshape(nb, 31)
    nrow = (nb + 3) // 4
    rows = np.zeros((nrow * 4, 32), np.float32)
    rows[:nb] = blocks
    got, want = _insert_both(rows.reshape(nrow, 128))
    assert np.array_equal(got, want)


# ----------------------------------------------------------------- top-k exact

def test_topk_bit_exact_on_shared_scores():
    # Same fp32 scores on both sides: the selection must be identical.  Rows with
    # heavy ties, negative values, +/-0, k below/at/above the context.
    rng = np.random.default_rng(5)
    B, q = 12, 2
    lens = np.array([1, 2, 5, 300, 2047, 2048, 2049, 4097, 10000, 65536, 3, 131072], np.int32)
    lens = np.maximum(lens, q)
    ld = int(lens.max())
    sc = np.full((B * q, ld), -np.inf, np.float32)
    for t in range(B * q):
        n = int(lens[t // q]) - q + t % q + 1
        kind = t % 4
        if kind == 0:
            row = rng.standard_normal(n).astype(np.float32) * 10
        elif kind == 1:
            row = rng.integers(-3, 4, n).astype(np.float32)          # heavy ties
        elif kind == 2:
            row = np.where(rng.random(n) < 0.5, 0.0, -0.0).astype(np.float32)
        else:
            row = -np.abs(rng.standard_normal(n)).astype(np.float32)
        sc[t, :n] = row
    lens_ok = lens
    for k in (1, 7, 2048, 20000):
        want = oracle.topk_select(sc.astype(np.float64), lens_ok, q, k)
        d_sc = torch.from_numpy(sc).to(DEV)
        out = torch.empty((B * q, k), dtype=torch.int32, device=DEV)
        ws_n = m.topk_select_workspace(B * q, k, ld)
        ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=DEV)
        m.topk_select(d_sc, torch.from_numpy(lens_ok).to(DEV), q, k, out, ws)
        m.mx4_check_status()
        assert np.array_equal(out.cpu().numpy(), want), f"k={k}"


def test_topk_segment_filter_paths():
    # Rows longer than one filter segment: candidates spread evenly, concentrated
    # in the last segment (recency-biased scores), all in one segment, k above the
    # candidate capacity (workspace-free exact path), and an odd row stride
    # (scalar loads).
    rng = np.random.default_rng(11)
    lens = np.array([40000, 131072, 70001, 16385, 99999, 8193, 200000], np.int32)
    B, q = len(lens), 1
    for ld_pad, ks in ((0, (2048, 9000)), (1, (2048,))):
        ld = int(lens.max()) + ld_pad
        sc = np.full((B, ld), -np.inf, np.float32)
        for t in range(B):
            n = int(lens[t])
            row = rng.standard_normal(n).astype(np.float32)
            if t % 3 == 1:
                row += np.linspace(0, 6, n, dtype=np.float32)      # recency bias
            elif t % 3 == 2:
                a = rng.integers(0, max(1, n - 3000))
                row[a:a + 3000] += 8                               # one hot window
            sc[t, :n] = row
        d_sc = torch.from_numpy(sc).to(DEV)
        d_lens = torch.from_numpy(lens).to(DEV)
        for k in ks:
            want = oracle.topk_select(sc.astype(np.float64), lens, q, k)
            out = torch.empty((B, k), dtype=torch.int32, device=DEV)
            ws_n = m.topk_select_workspace(B, k, ld)
            ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=DEV)
            m.topk_select(d_sc, d_lens, q, k, out, ws)
            m.mx4_check_status()
            assert np.array_equal(out.cpu().numpy(), want), f"k={k} ld={ld}"


def _sample_rank(n, k, kcand=8192, ksample=2048):
    """The selection kernel's documented threshold rank for a row of n > kcand scores:
    the sample key at rank m + 4 sqrt(m) + 8 (m = k * ksample / n), lowered to
    2r + 64 when the candidates fall short.  Used only to build rows that reach each
    branch; the expected selection always comes from the oracle."""
    m_ = k * ksample / n
    r0 = min(ksample - 1, int(m_ + 4.0 * math.sqrt(m_)) + 8)
    ranks = [r0]
    while ranks[-1] < ksample - 1:
        ranks.append(min(ksample - 1, 2 * ranks[-1] + 64))
    return ranks


def _retry_row(n, k, level, rng, kcand=8192):
    """A row of n scores whose evenly spaced 2048-key sample (positions j*n//2048) is
    1000 - j, so the threshold at sample rank r is 1000 - r, and whose other keys sit
    near -2000.  `level` = how many threshold reductions the selection needs: the keys
    put between the thresholds of levels `level` - 1 and `level` make up the
    candidates only from that level on.
    level -1: 1800 sample keys are 100 and 248 are -5000, so the reductions fall
    short until the threshold drops to -5000 and the candidates exceed the capacity.
    level -2: every sample key is 100 (k > 2048), so the reductions run out of sample
    ranks and the threshold is dropped altogether."""
    row = (rng.standard_normal(n) - 2000.0).astype(np.float32)
    pos = (np.arange(2048, dtype=np.int64) * n) // 2048
    rest = np.setdiff1d(np.arange(n), pos)
    if level == -1:
        row[pos] = np.where(np.arange(2048) < 1800, 100.0, -5000.0).astype(np.float32)
        return row
    if level == -2:
        assert k > 2048
        row[pos] = 100.0
        return row
    ranks = _sample_rank(n, k, kcand)
    hi = 1000.0 - ranks[level - 1]          # threshold of the level before: must fall short
    lo = 1000.0 - ranks[level]              # threshold of this level
    row[pos] = 1000.0 - np.arange(2048, dtype=np.float32)
    target = min(kcand, k + 500)
    need = target - (ranks[level] + 1)       # sample keys >= lo: ranks[level] + 1
    pick = rng.choice(rest, size=need, replace=False)
    row[pick] = rng.uniform(lo + 0.01, hi - 0.01, need).astype(np.float32)
    return row


@pytest.mark.parametrize("k", [2048, 8192])
def test_topk_threshold_retry_paths(k):
    # Rows on which the sampled threshold leaves fewer than k candidates, so the
    # selection lowers it once (level 1) or twice (level 2) before the candidates
    # fit, runs out of sample ranks and takes the exact path (level -1), or gets
    # more than the candidate capacity at once (the sample all below the rest).
    # Bit-exact against the oracle on the same fp32 scores; no status bits.
    rng = np.random.default_rng(2024 + k)
    n_rows = [131072, 131072, 65536, 40000, 131072, 9000]
    levels = [1, 2, 1, 2, -1, 1]
    if k == 8192:
        n_rows, levels = [131072, 131072, 65536, 131072, 131072], [1, 2, 1, -1, -2]
    rows = [_retry_row(n, k, lev, rng) for n, lev in zip(n_rows, levels)]
    # sample far below the rest: threshold takes the whole row (> capacity)
    n_low = 100000
    low = rng.standard_normal(n_low).astype(np.float32)
    low[(np.arange(2048, dtype=np.int64) * n_low) // 2048] = -100.0
    rows.append(low)
    lens = np.array([len(r) for r in rows], np.int32)
    ld = int(lens.max())
    sc = np.full((len(rows), ld), -np.inf, np.float32)
    for t, r in enumerate(rows):
        sc[t, :len(r)] = r
    want = oracle.topk_select(sc.astype(np.float64), lens, 1, k)
    out = torch.empty((len(rows), k), dtype=torch.int32, device=DEV)
    ws_n = m.topk_select_workspace(len(rows), k, ld)
    assert ws_n > 0  # the rows take the segment filter first
    ws = torch.empty(ws_n, dtype=torch.uint8, device=DEV)
    m.topk_select(torch.from_numpy(sc).to(DEV), torch.from_numpy(lens).to(DEV), 1, k, out, ws)
    assert m.mx4_check_status() == 0
    got = out.cpu().numpy()
    for t in range(len(rows)):
        assert np.array_equal(got[t], want[t]), f"row {t} (n={lens[t]}, k={k})"


@pytest.mark.parametrize("wid", [2, 3, 4])
def test_index_topk_matches_the_separate_calls(wid):
    # index_topk (scorer with key histograms + selection from them) against
    # index_score + topk_select on the full workload: scores and selections
    # bit-identical (the same fp32 scores, the same exact selection rule).
    wl = W.make(wid)
    caches, step, host = _gpu_step(wl)  # the step runs index_topk
    sc_f, idx_f = step.scores.clone(), step.topk_idx.clone()
    step.run(fused=False)
    m.mx4_check_status()
    n = wl.positions() + 1
    sc_s = step.scores.cpu().numpy()
    sf = sc_f.cpu().numpy()
    for t in range(wl.T):
        assert np.array_equal(sf[t, :n[t]], sc_s[t, :n[t]]), f"scores of token {t}"
    assert torch.equal(idx_f, step.topk_idx)


def test_index_topk_heavy_ties_and_short_rows():
    # Index keys with a few distinct rows: the scores take a handful of values, so
    # thousands of keys tie with the k-th largest and the lowest indices among them
    # are taken; rows of one CTA, of a cluster, and longer than a cluster covers.
    # Bit-exact against the oracle's selection of the oracle's scores (equal-valued
    # keys give equal fp32 scores).
    rng = np.random.default_rng(8)
    lens = np.array([20000, 8192, 300, 131072, 140000], np.int32)
    B, q, k = len(lens), 1, 2048
    pages = (lens + 127) // 128
    P = int(pages.sum())
    ids = rng.permutation(P).astype(np.int32)
    bt = np.full((B, int(pages.max())), -1, np.int32)
    o = 0
    for s_, n_ in enumerate(pages):
        bt[s_, :n_] = ids[o:o + n_]
        o += n_
    base = rng.standard_normal((4, 128)).astype(np.float32)
    ip_o = np.full((P, 8704), 0xFF, np.uint8)
    ip = torch.full((P, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    kv = torch.full((P, 1, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    for s_ in range(B):
        L = int(lens[s_])
        rows = base[rng.integers(0, 4, L)]
        pos = np.arange(L)
        slots = (bt[s_, pos // 128].astype(np.int64) * 128 + pos % 128)
        oracle.mx4_insert(None, None, rows, slots, None, None, ip_o)
        r = torch.from_numpy(rows).to(DEV)
        m.mx4_insert(r.view(L, 1, 128), r.view(L, 1, 128), r, torch.from_numpy(slots).to(DEV),
                     kv, kv.clone(), ip)
    m.mx4_check_status()
    assert np.array_equal(ip.cpu().numpy(), ip_o)
    iq = torch.from_numpy(rng.standard_normal((B, 128)).astype(np.float32)).to(torch.bfloat16)
    iq_bits = iq.view(torch.int16).numpy().view(np.uint16)
    ld = int(lens.max())
    want_sc = oracle.index_score(iq_bits, q, ip_o, bt, lens, ld)
    want = oracle.topk_select(want_sc, lens, q, k)
    scores = torch.empty((B, ld), dtype=torch.float32, device=DEV)
    out = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = torch.full((m.index_topk_workspace(B, k, ld),), 0xAB, dtype=torch.uint8, device=DEV)
    for _ in range(2):  # the workspace's contents on entry do not matter
        m.index_topk(iq.to(DEV), q, ip, torch.from_numpy(bt).to(DEV),
                     torch.from_numpy(lens).to(DEV), scores, k, out, ws)
        assert m.mx4_check_status() == 0
        assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("q", [1, 4])
def test_index_topk_ragged_long_rows_against_oracle(q):
    # rows around the candidate capacity and the segment size, q decode tokens each
    wl = _custom([8191, 8192, 8193, 16385, 40000, 70001], q=q, k=2048, seed=90 + q)
    _compare(wl, range(wl.B), *_gpu_step(wl))


@pytest.mark.parametrize("wid", [1, 4])
def test_pipelined_steps_match_a_plain_step(wid):
    # The overlapped serving loop (packed inputs, one CUDA-graph launch a step)
    # gives, step after step, the plain step's output.
    wl = W.make(wid)
    caches, step, host = _gpu_step(wl)
    want = step.out.cpu().numpy()
    pipe = PipelinedSteps(wl, caches, device=DEV)
    pin = pipe.pack_inputs(host)
    for _ in range(5):
        h_out, done = pipe.submit(pin)
        done.synchronize()
        assert np.array_equal(h_out.numpy(), want)
    outs = [pipe.submit(pin) for _ in range(4)]
    torch.cuda.synchronize()
    for h_out, _ in outs[-2:]:
        assert np.array_equal(h_out.numpy(), want)
    m.mx4_check_status()


@pytest.mark.parametrize("wid", [0, 4])
def test_host_to_host_step_matches_a_plain_step(wid):
    # mx4_decode_step (host inputs -> device -> the four stages -> host output, one C
    # call) gives the plain step's output, call after call.
    wl = W.make(wid)
    caches, step, host = _gpu_step(wl)
    want = step.out.cpu().numpy()
    pin = step.pack_inputs(host)
    h_out = torch.full(tuple(step.out.shape), float("nan"), dtype=torch.float32).pin_memory()
    for _ in range(3):
        h_out.fill_(float("nan"))
        step.run_host(pin, h_out)
        torch.cuda.current_stream().synchronize()
        assert np.array_equal(h_out.numpy(), want)
    m.mx4_check_status()


@pytest.mark.parametrize("wid", [1, 4])
def test_multi_step_host_call_matches_plain_steps(wid):
    # mx4_decode_steps (5 steps in one C call, inputs and outputs in host memory, the
    # copies of neighbouring steps overlapped on two copy streams) gives every step
    # the plain step's output; with per-step buffers and with one shared buffer.
    wl = W.make(wid)
    caches, step, host = _gpu_step(wl)
    want = step.out.cpu().numpy()
    pin = step.pack_inputs(host)
    n = 5
    per_step = torch.stack([pin] * n).pin_memory()
    h_outs = torch.full((n,) + tuple(step.out.shape), float("nan"), dtype=torch.float32)
    h_outs = h_outs.pin_memory()
    cs = torch.cuda.Stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    step.run_host_steps(per_step, h_outs, n, cs, h2d, d2h)
    cs.synchronize()
    for i in range(n):
        assert np.array_equal(h_outs[i].numpy(), want), f"step {i}"
    h_out = torch.full(tuple(step.out.shape), float("nan"), dtype=torch.float32).pin_memory()
    step.run_host_steps(pin, h_out, n, cs, h2d, d2h)
    cs.synchronize()
    assert np.array_equal(h_out.numpy(), want)
    m.mx4_check_status()


# ----------------------------------------------------------------- decode edges

def test_decode_single_selected_token_is_exact_value_row():
    wl = _custom([300], q=1, k=8, seed=3)
    caches, step, host = _gpu_step(wl)
    orc = OracleSide(wl, [0], host)
    for i in (0, 127, 128, 299):
        idx = torch.full((1, 8), -1, dtype=torch.int32, device=DEV)
        idx[0, 0] = i
        out = torch.empty_like(step.out)
        m.sparse_paged_decode(step.q, 1, caches.k_pages, caches.v_pages, step.block_table,
                              step.seq_lens, idx, step.scale, out, step.dec_ws)
        pg = int(wl.block_table[0, i // 128])
        vrow = oracle.dequant_row(orc.vp[pg, 0], i % 128)
        assert np.array_equal(out.cpu().numpy()[0].astype(np.float64),
                              np.broadcast_to(vrow, (16, 128)))


def test_decode_output_invariant_to_split_boundaries():
    # The same selection written in one list, or padded so it crosses split
    # boundaries differently, gives the same result within fp32 rounding.
    wl = _custom([3000], q=1, k=2048, seed=9)
    caches, step, host = _gpu_step(wl)
    sel = step.topk_idx.clone()
    out1 = torch.empty_like(step.out)
    m.sparse_paged_decode(step.q, 1, caches.k_pages, caches.v_pages, step.block_table,
                          step.seq_lens, sel, step.scale, out1, step.dec_ws)
    wide = torch.full((1, 4096), -1, dtype=torch.int32, device=DEV)
    valid = sel[0][sel[0] >= 0]
    wide[0, 100:100 + valid.numel()] = valid
    ws = torch.empty(m.sparse_paged_decode_workspace(1, 4096), dtype=torch.uint8, device=DEV)
    out2 = torch.empty_like(step.out)
    m.sparse_paged_decode(step.q, 1, caches.k_pages, caches.v_pages, step.block_table,
                          step.seq_lens, wide, step.scale, out2, ws)
    m.mx4_check_status()
    assert float((out1 - out2).abs().max()) <= 1e-5


# ----------------------------------------------------------------- bad data

def test_bad_slot_page_and_index_are_flagged_not_faulted():
    wl = _custom([200, 300], q=1, k=64, seed=11)
    caches, step, host = _gpu_step(wl)
    P = wl.num_pages
    # slot beyond the pool
    r = torch.zeros((1, 1, 128), device=DEV)
    with pytest.raises(m.Mx4Error) as ei:
        m.mx4_insert(r, r, r[:, 0], torch.tensor([P * 128], device=DEV), caches.k_pages,
                     caches.v_pages, caches.idx_pages)
        m.mx4_check_status()
    assert ei.value.bits & 0x1
    # a block-table entry outside the pool
    bt = step.block_table.clone()
    bt[1, 0] = P + 5
    with pytest.raises(m.Mx4Error) as ei:
        m.index_score(step.iq, 1, caches.idx_pages, bt, step.seq_lens, step.scores)
        m.mx4_check_status()
    assert ei.value.bits & 0x2
    # a top-k index beyond the token's position
    idx = step.topk_idx.clone()
    idx[0, 0] = 250
    with pytest.raises(m.Mx4Error) as ei:
        m.sparse_paged_decode(step.q, 1, caches.k_pages, caches.v_pages, step.block_table,
                              step.seq_lens, idx, step.scale, step.out, step.dec_ws)
        m.mx4_check_status()
    assert ei.value.bits & 0x8
    # a sequence length beyond the block table
    sl = step.seq_lens.clone()
    sl[0] = 10 ** 6
    with pytest.raises(m.Mx4Error) as ei:
        m.index_score(step.iq, 1, caches.idx_pages, step.block_table, sl, step.scores)
        m.mx4_check_status()
    assert ei.value.bits & 0x4
    m.mx4_check_status()  # cleared


def test_empty_batch_is_a_no_op():
    z = torch.empty((0, 128), dtype=torch.bfloat16, device=DEV)
    pages = torch.zeros((1, 8704), dtype=torch.uint8, device=DEV)
    m.index_score(z, 1, pages, torch.zeros((0, 1), dtype=torch.int32, device=DEV),
                  torch.zeros(0, dtype=torch.int32, device=DEV),
                  torch.zeros((0, 1), dtype=torch.float32, device=DEV))
    r = torch.empty((0, 1, 128), device=DEV)
    kv = torch.zeros((1, 1, 8704), dtype=torch.uint8, device=DEV)
    m.mx4_insert(r, r, r[:, 0], torch.empty(0, dtype=torch.int64, device=DEV), kv, kv.clone(),
                 pages)
    m.mx4_check_status()


# ----------------------------------------------------------------- norm + rotary writer
#
# The writer's fp32 arithmetic (sum of squares, IEEE square root and divide, the
# turn) lands within 2e-6 (|z_i| + |z_partner|) of the float64 definition, z the
# normed row before the turn.  Page bytes must equal the exact quantiser's bytes
# for fl32(float64 row), or else be what it gives some row inside that band (a
# value within the band of an E2M1 rounding midpoint or of a power-of-two block
# maximum); bf16 outputs must lie between the roundings of the band's ends.

_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _signed_codes(data):
    codes = np.empty(128, np.int64)
    codes[0::2], codes[1::2] = data & 15, data >> 4
    return np.where(codes & 8, -1.0, 1.0) * _E2M1_MAG[codes & 7]


def _quantised_value(x, E):
    """Signed E2M1 value the exact quantiser gives each x (float64) at block exponent E."""
    a = np.minimum(np.abs(x) * 2.0 ** -E, 6.0)
    mag = np.array([oracle.e2m1_value(oracle.round_magnitude(v)) for v in a])
    return np.sign(x) * mag


def _row_in_band(data, scale, y, tol):
    lo, hi = y - tol, y + tol
    got = _signed_codes(data)
    for b in range(4):
        sl = slice(32 * b, 32 * b + 32)
        l, h = lo[sl], hi[sl]
        amin = np.where((l <= 0) & (h >= 0), 0.0, np.minimum(np.abs(l), np.abs(h))).max()
        amax = np.maximum(np.abs(l), np.abs(h)).max()
        E = int(scale[b]) - 127
        if not oracle.block_exponent(amin) <= E <= oracle.block_exponent(amax):
            return False
        if not (np.all(_quantised_value(l, E) <= got[sl]) and
                np.all(got[sl] <= _quantised_value(h, E))):
            return False
    return True


def _check_quantised(got, want, slots, y, tol, what):
    """got/want: [P, 8704] pages; row i of y/tol goes to slots[i] (skipped if < 0)."""
    n_diff = 0
    gm, wm = got.copy(), want.copy()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        pg, r = divmod(int(s), 128)
        d, sc = slice(64 * r, 64 * r + 64), slice(8192 + 4 * r, 8196 + 4 * r)
        if not (np.array_equal(got[pg, d], want[pg, d]) and
                np.array_equal(got[pg, sc], want[pg, sc])):
            n_diff += 1
            assert _row_in_band(got[pg, d], got[pg, sc], y[i], tol[i]), f"{what} of token {i}"
        for a in (gm, wm):
            a[pg, d], a[pg, sc] = 0, 0
    assert np.array_equal(gm, wm), f"{what}: rows outside the slots were touched"
    return n_diff


def _check_bf16(got, y, tol, what):
    g = got.float().numpy().reshape(y.shape).astype(np.float64)
    lo = torch.from_numpy(y - tol).to(torch.bfloat16).double().numpy()
    hi = torch.from_numpy(y + tol).to(torch.bfloat16).double().numpy()
    assert np.all((lo <= g) & (g <= hi)), f"{what}: bf16 outside the band"
    exact = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.mean(g == exact) >= 0.99, f"{what}: too many band-edge roundings"


def _norm_rope_band(x, g, cs, pos, eps):
    y = oracle.norm_rope(x.reshape(-1, 128), g, cs, pos, eps)
    z = oracle.norm_rope(x.reshape(-1, 128), g, cs, pos, eps, rope=False)
    return y, 2e-6 * (np.abs(z) + np.abs(np.roll(z, 64, axis=1)))


def _writer_gpu(x, pos, cs, eps, slots, P, H, Hkv):
    d = {n: torch.from_numpy(a).to(DEV) for n, a in x.items()}
    T = pos.shape[0]
    kp = torch.full((P, Hkv, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    vp = torch.full_like(kp, 0xFF)
    ip = torch.full((P, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    q_out = torch.zeros((T, H, 128), dtype=torch.bfloat16, device=DEV)
    iq_out = torch.zeros((T, 128), dtype=torch.bfloat16, device=DEV)
    m.mx4_norm_rope_insert(d["q"], d["iq"], d["k"], d["v"], d["idx_k"],
                           torch.from_numpy(pos).to(DEV), torch.from_numpy(cs).to(DEV), d["g_q"],
                           d["g_k"], d["g_iq"], d["g_ik"], eps, torch.from_numpy(slots).to(DEV),
                           kp, vp, ip, q_out, iq_out)
    return kp, vp, ip, q_out, iq_out


@pytest.mark.parametrize("H,Hkv", [(16, 1), (4, 2)])
def test_norm_rope_insert_against_oracle(H, Hkv):
    T, P, max_pos = 300, 4, 4096
    x = W.writer_inputs(T, H, Hkv, seed=31 + H)
    rng = np.random.default_rng(32 + Hkv)
    pos = rng.integers(0, max_pos, T).astype(np.int64)
    pos[0], pos[1] = 0, max_pos - 1          # identity turn; last table row
    for n in ("q", "iq", "k", "idx_k"):
        x[n][2] = 0.0                        # a zero row stays zero (eps > 0)
    cs = W.rope_table(max_pos)
    eps = float(np.float32(1e-6))
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    slots[5] = slots[17] = -1                # tokens that are not cached
    yq, tq = _norm_rope_band(x["q"], x["g_q"], cs, np.repeat(pos, H), eps)
    yiq, tiq = _norm_rope_band(x["iq"], x["g_iq"], cs, pos, eps)
    yk, tk = _norm_rope_band(x["k"], x["g_k"], cs, np.repeat(pos, Hkv), eps)
    yik, tik = _norm_rope_band(x["idx_k"], x["g_ik"], cs, pos, eps)
    kp_o = np.full((P, Hkv, 8704), 0xFF, np.uint8)
    vp_o = kp_o.copy()
    ip_o = np.full((P, 8704), 0xFF, np.uint8)
    oracle.mx4_insert(yk.astype(np.float32).reshape(T, Hkv, 128), x["v"],
                      yik.astype(np.float32), slots, kp_o, vp_o, ip_o)

    kp, vp, ip, q_out, iq_out = _writer_gpu(x, pos, cs, eps, slots, P, H, Hkv)
    m.mx4_check_status()
    assert np.array_equal(vp.cpu().numpy(), vp_o)            # V goes in unchanged
    _check_bf16(q_out.cpu(), yq, tq, "q")
    _check_bf16(iq_out.cpu(), yiq, tiq, "index-q")
    assert not q_out[2].any() and not iq_out[2].any()
    kpn, ipn = kp.cpu().numpy(), ip.cpu().numpy()
    yk, tk = yk.reshape(T, Hkv, 128), tk.reshape(T, Hkv, 128)
    nd = sum(_check_quantised(kpn[:, h], kp_o[:, h], slots, yk[:, h], tk[:, h], f"K head {h}")
             for h in range(Hkv))
    nd += _check_quantised(ipn, ip_o, slots, yik, tik, "index-K")
    # rows whose bytes differ from the exact quantiser's for fl32(y): each is inside
    # the band; the count is printed so a drift toward the ceiling shows in the logs
    print(f"writer (H={H}, Hkv={Hkv}): {nd} of {T * (Hkv + 1)} K / index-K rows differ "
          f"from the exact quantiser's bytes (ceiling 2 %)")
    assert nd <= 0.02 * T * (Hkv + 1)


def test_norm_rope_insert_bad_position_is_flagged_and_skipped():
    H, Hkv, P, max_pos = 16, 1, 1, 64
    x = W.writer_inputs(4, H, Hkv, seed=3)
    cs = W.rope_table(max_pos)
    pos = np.array([0, 63, 64, -1], np.int64)
    slots = np.arange(4, dtype=np.int64)
    kp, vp, ip, q_out, iq_out = _writer_gpu(x, pos, cs, 1e-6, slots, P, H, Hkv)
    with pytest.raises(m.Mx4Error) as ei:
        m.mx4_check_status()
    assert ei.value.bits & 0x8
    vp_o = np.full((P, Hkv, 8704), 0xFF, np.uint8)
    oracle.mx4_insert(None, x["v"][:2], None, slots[:2], vp_o.copy(), vp_o, None)
    assert np.array_equal(vp.cpu().numpy(), vp_o)           # tokens 2, 3 left alone
    assert q_out[:2].any() and not q_out[2:].any() and not iq_out[2:].any()
    # no tokens: nothing to do, nothing flagged
    e = {n: a[:0] if a.ndim > 1 else a for n, a in x.items()}
    _writer_gpu(e, pos[:0], cs, 1e-6, slots[:0], P, H, Hkv)
    m.mx4_check_status()


# ----------------------------------------------------------------- fp8 index cache variant

FP8_PAGE = 16384


def _bf16_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)


def _fp8_insert_both(rows, slots, scale, P):
    want = np.full((P, FP8_PAGE), 0xFF, np.uint8)
    oracle.fp8_index_insert(rows, slots, scale, want)
    got = torch.full((P, FP8_PAGE), 0xFF, dtype=torch.uint8, device=DEV)
    m.fp8_index_insert(torch.from_numpy(rows).to(DEV), torch.from_numpy(slots).to(DEV), scale, got)
    m.mx4_check_status()
    return got, want


@pytest.mark.parametrize("scale", [1.0, 0.37, 2.0 ** -20])
def test_fp8_index_insert_bit_exact(scale):
    # Quotients on every E4M3 rounding midpoint and just off it, zeros of both
    # signs, subnormal and smallest-normal inputs, the saturation edge, and rows
    # across 30 binades; scattered slots with two skipped tokens.
    f32 = np.finfo(np.float32)
    finite = np.array([oracle.e4m3_value(c) for c in range(128) if c != 0x7F])
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0)), finite.astype(np.float32)])
    vals = np.concatenate([vals, -vals])
    nrow = (len(vals) + 127) // 128
    rows = np.zeros((nrow + 70, 128), np.float32)
    rows.reshape(-1)[:len(vals)] = vals * np.float32(scale)
    r = nrow
    rows[r + 1] = -0.0
    rows[r + 2, :6] = np.array([448, 449, 464, 465, 1e30, -1e30]) * scale
    rows[r + 2, 6] = -f32.max
    rows[r + 3] = f32.tiny
    rows[r + 4] = np.float32(2.0 ** -149)
    rows[r + 5, :4] = np.array([2.0 ** -10, -2.0 ** -10, 2.0 ** -12, -2.0 ** -12]) * scale
    rng = np.random.default_rng(17)
    k = rows.shape[0] - (r + 6)
    rows[r + 6:] = (rng.standard_normal((k, 128)) * np.exp2(rng.uniform(-12, 10, (k, 1))) *
                    scale).astype(np.float32)
    n = rows.shape[0]
    P = (n + 127) // 128 + 1
    slots = rng.permutation(P * 128)[:n].astype(np.int64)
    slots[3] = slots[40] = -1
    got, want = _fp8_insert_both(rows, slots, scale, P)
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("q", [1, 3])
def test_index_score_fp8_ragged_and_topk_chain(q):
    rng = np.random.default_rng(40 + q)
    lens = np.array([q, 127, 128, 129, 700, 1500, 2049, 4100], np.int32)
    B = len(lens)
    npg = (lens + 127) // 128
    P = int(npg.sum()) + 2
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((B, int(npg.max())), -1, np.int32)
    o = 0
    for s in range(B):
        bt[s, :npg[s]] = perm[o:o + npg[s]]
        o += npg[s]
    scale = 0.37
    rows = [(rng.standard_normal((int(L), 128)) * 3).astype(np.float32) for L in lens]
    rows[5][::97] *= 40                                   # a few outlier rows
    slots = np.concatenate([bt[s, np.arange(L) // 128].astype(np.int64) * 128 + np.arange(L) % 128
                            for s, L in enumerate(lens)])
    got_pages, want_pages = _fp8_insert_both(np.concatenate(rows), slots, scale, P)
    assert np.array_equal(got_pages.cpu().numpy(), want_pages)
    iq_bits = W.to_bf16_bits(rng.standard_normal((B * q, 128)).astype(np.float32))
    ld = int(lens.max()) + 5
    want, mag = oracle.index_score_fp8(iq_bits, q, want_pages, bt, lens, scale, ld, want_mag=True)
    d_bt, d_lens = torch.from_numpy(bt).to(DEV), torch.from_numpy(lens).to(DEV)
    sc = torch.full((B * q, ld), 7.0, dtype=torch.float32, device=DEV)
    m.index_score_fp8(_bf16_dev(iq_bits), q, got_pages, d_bt, d_lens, scale, sc)
    m.mx4_check_status()
    g = sc.cpu().numpy()
    L_tok = np.repeat(lens, q)
    check_scores(g, want, mag, L_tok)
    assert np.all(g[:, -5:][np.repeat(lens, q) < ld - 5] == 7.0)   # nothing past seq_len
    # the selection from these scores, against the oracle's selection from its own
    k = 256
    sel = oracle.topk_select(want, lens, q, k)
    out = torch.empty((B * q, k), dtype=torch.int32, device=DEV)
    ws = torch.empty(max(m.topk_select_workspace(B * q, k, ld), 16), dtype=torch.uint8, device=DEV)
    m.topk_select(sc, d_lens, q, k, out, ws)
    m.mx4_check_status()
    n_tok = np.array([int(lens[t // q]) - q + t % q + 1 for t in range(B * q)])
    check_topk(out.cpu().numpy(), sel, want, n_tok)
    # a poisoned key row (0xFF bytes: E4M3 NaN) gives a non-finite score on both sides
    pg, row = int(bt[4, 0]), 10
    want_pages[pg, row * 128:(row + 1) * 128] = 0xFF
    got_pages[pg, row * 128:(row + 1) * 128] = 0xFF
    want, mag = oracle.index_score_fp8(iq_bits, q, want_pages, bt, lens, scale, ld, want_mag=True)
    m.index_score_fp8(_bf16_dev(iq_bits), q, got_pages, d_bt, d_lens, scale, sc)
    m.mx4_check_status()
    g = sc.cpu().numpy()
    check_scores(g, want, mag, L_tok)
    assert not np.isfinite(g[4 * q:5 * q, row]).any()


def test_index_score_fp8_full_size_sampled():
    # The b256 lognormal workload (2.98 M cached tokens) in the launch configuration
    # the benchmark times: the whole batch scored from the fp8 cache, sampled
    # sequences checked against the oracle's own fp8 pages.
    wl = W.make(4)
    scale = 0.25
    caches = PagedCaches(wl.num_pages, device=DEV, fp8_index_scale=scale)
    caches.fill(wl)
    step = DecodeStep(wl, caches, device=DEV)
    host = step_inputs_host(wl)
    step.load_inputs(host)
    step.run()
    m.fp8_index_insert(step.idx_new, step.slots, scale, caches.fp8_idx_pages)  # decode tokens
    m.index_score_fp8(step.iq, wl.q, caches.fp8_idx_pages, step.block_table, step.seq_lens,
                      scale, step.scores)
    m.mx4_check_status()
    L = wl.seq_lens
    short = int(np.nonzero(L < 2048)[0][0])
    seqs = sorted({short, int(np.argmax(L)), int(np.argmin(L)), 7, 131})
    pages = np.full((wl.num_pages, FP8_PAGE), 0xFF, np.uint8)
    for s in seqs:
        n = wl.prefilled(s)
        for a in range(0, n, 65536):
            b = min(n, a + 65536)
            oracle.fp8_index_insert(wl.rows(s, W.IDX_ROWS, a, b), wl.slots(s, np.arange(a, b)),
                                    scale, pages)
    tok = np.concatenate([np.arange(s * wl.q, (s + 1) * wl.q) for s in seqs])
    oracle.fp8_index_insert(host["idx_k"][tok], host["slots"][tok], scale, pages)
    lens = wl.seq_lens[seqs]
    want, mag = oracle.index_score_fp8(host["iq"][tok], wl.q, pages, wl.block_table[seqs], lens,
                                       scale, int(wl.max_len), want_mag=True)
    g = step.scores.cpu().numpy()[tok]
    check_scores(g, want, mag, np.repeat(lens, wl.q))

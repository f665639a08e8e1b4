"""GPU parity at the limits include/mx4sp.h states, each against the oracle.

- the longest scored row: ld_scores = 8388608 (2^23 tokens, 65536 pages, 512 filter
  segments), through index_topk and through topk_select;
- the largest top-k width: k = 65536, in topk_select (the exact path past the
  candidate capacity) and in sparse_paged_decode (a 65536-entry selection);
- the most KV heads a page pool holds in mx4_insert: Hkv = 8.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import mxfp4_sparse_paged_gb300 as m

from _sides import ATTN_ABS, check_scores, check_topk

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda"
MAX_LD = 8388608  # ld_scores limit of index_topk / topk_select (512 segments of 16384)


def _block_table(rng, lens):
    pages = (np.asarray(lens, np.int64) + 127) // 128
    P = int(pages.sum())
    ids = rng.permutation(P).astype(np.int32)
    bt = np.full((len(lens), int(pages.max())), -1, np.int32)
    o = 0
    for s, n in enumerate(pages):
        bt[s, :n] = ids[o:o + n]
        o += n
    return bt, P


def _random_pages(rng, P):
    """P MXFP4 pages of random codes with scale bytes 120..134 (finite, moderate)."""
    pg = np.empty((P, 8704), np.uint8)
    pg[:, :8192] = rng.integers(0, 256, (P, 8192), dtype=np.uint8)
    pg[:, 8192:] = rng.integers(120, 135, (P, 512), dtype=np.uint8)
    return pg


def test_index_topk_at_the_longest_context():
    # one sequence of 2^23 cached tokens (the longest row index_topk takes) and one of
    # 100000, one decode token each, top-2048: scores within the fp32 bound of the
    # oracle's, selections equal up to near-ties of the k-th score, and bit-exact
    # against the oracle's selection of the kernel's own scores
    rng = np.random.default_rng(71)
    lens = np.array([MAX_LD, 100000], np.int32)
    B, q, k = 2, 1, 2048
    bt, P = _block_table(rng, lens)
    ip = _random_pages(rng, P)
    iq = torch.from_numpy(rng.standard_normal((B, 128)).astype(np.float32)).to(torch.bfloat16)
    iq_bits = iq.view(torch.int16).numpy().view(np.uint16)
    ld = MAX_LD
    scores = torch.empty((B, ld), dtype=torch.float32, device=DEV)
    out = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = torch.empty(max(m.index_topk_workspace(B, k, ld), 16), dtype=torch.uint8, device=DEV)
    m.index_topk(iq.to(DEV), q, torch.from_numpy(ip).to(DEV), torch.from_numpy(bt).to(DEV),
                 torch.from_numpy(lens).to(DEV), scores, k, out, ws)
    assert m.mx4_check_status() == 0
    got_sc = scores.cpu().numpy()
    got = out.cpu().numpy()
    want_sc, mag = oracle.index_score(iq_bits, q, ip, bt, lens, ld, want_mag=True)
    check_scores(got_sc, want_sc, mag, lens)
    check_topk(got, oracle.topk_select(want_sc, lens, q, k), want_sc, lens)
    assert np.array_equal(got, oracle.topk_select(got_sc.astype(np.float64), lens, q, k))


def test_topk_at_the_longest_row_and_the_largest_k():
    # rows of 2^23 scores: N(0,1); a recency trend (the candidates pile up in the last
    # segments); five distinct values (a tie group far past the candidate capacity).
    # k = 2048 and 8192 (the filter's capacity) and 65536 (the exact global path)
    rng = np.random.default_rng(72)
    n = MAX_LD
    x = rng.standard_normal(n).astype(np.float32)
    sc = np.stack([x, x + np.linspace(0.0, 3.0, n, dtype=np.float32),
                   rng.integers(-2, 3, n).astype(np.float32)])
    T = sc.shape[0]
    lens = np.full(T, n, np.int32)
    d_sc = torch.from_numpy(sc).to(DEV)
    d_lens = torch.from_numpy(lens).to(DEV)
    sc64 = sc.astype(np.float64)
    for k in (2048, 8192, 65536):
        want = oracle.topk_select(sc64, lens, 1, k)
        out = torch.empty((T, k), dtype=torch.int32, device=DEV)
        ws = torch.empty(max(m.topk_select_workspace(T, k, n), 16), dtype=torch.uint8,
                         device=DEV)
        m.topk_select(d_sc, d_lens, 1, k, out, ws)
        assert m.mx4_check_status() == 0
        assert np.array_equal(out.cpu().numpy(), want), f"k={k}"


def test_decode_with_the_largest_k():
    # k = 65536: sequence 0 (70000 cached tokens) selects positions 0..65535, sequence
    # 1 (1000 tokens) every position then -1 padding; K/V written by mx4_insert
    # (bit-exact against the oracle's pages); outputs against the float64 oracle, and
    # the allocation-free entry point equal to the workspace one
    rng = np.random.default_rng(73)
    lens = np.array([70000, 1000], np.int32)
    B, q, k, H = 2, 1, 65536, 16
    bt, P = _block_table(rng, lens)
    kp_o = np.full((P, 1, 8704), 0xFF, np.uint8)
    vp_o = np.full((P, 1, 8704), 0xFF, np.uint8)
    kp = torch.full((P, 1, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    vp = torch.full((P, 1, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    ip = torch.full((P, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    for s in range(B):
        L = int(lens[s])
        kr = rng.standard_normal((L, 1, 128)).astype(np.float32)
        vr = rng.standard_normal((L, 1, 128)).astype(np.float32)
        pos = np.arange(L)
        slots = bt[s, pos // 128].astype(np.int64) * 128 + pos % 128
        oracle.mx4_insert(kr, vr, None, slots, kp_o, vp_o, None)
        m.mx4_insert(torch.from_numpy(kr).to(DEV), torch.from_numpy(vr).to(DEV),
                     torch.from_numpy(kr[:, 0]).to(DEV), torch.from_numpy(slots).to(DEV),
                     kp, vp, ip)
    assert m.mx4_check_status() == 0
    assert np.array_equal(kp.cpu().numpy(), kp_o) and np.array_equal(vp.cpu().numpy(), vp_o)
    sel = np.full((B, k), -1, np.int32)
    sel[0] = np.arange(k)
    sel[1, :lens[1]] = np.arange(lens[1])
    qf = torch.from_numpy(rng.standard_normal((B, H, 128)).astype(np.float32)).to(torch.bfloat16)
    q_bits = qf.view(torch.int16).numpy().view(np.uint16)
    scale = 1.0 / math.sqrt(128.0)
    want = oracle.sparse_paged_decode(q_bits, q, kp_o, vp_o, bt, lens, sel, scale)
    d_q, d_bt = qf.to(DEV), torch.from_numpy(bt).to(DEV)
    d_lens, d_sel = torch.from_numpy(lens).to(DEV), torch.from_numpy(sel).to(DEV)
    out = torch.empty((B, H, 128), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.sparse_paged_decode_workspace(B, k), dtype=torch.uint8, device=DEV)
    m.sparse_paged_decode(d_q, q, kp, vp, d_bt, d_lens, d_sel, scale, out, ws)
    assert m.mx4_check_status() == 0
    err = float(np.abs(out.cpu().numpy() - want).max())
    assert err <= ATTN_ABS, f"max-abs {err}"
    out2 = torch.empty_like(out)
    m.sparse_paged_decode_noalloc(d_q, q, kp, vp, d_bt, d_lens, d_sel, scale, out2)
    assert m.mx4_check_status() == 0
    assert torch.equal(out, out2)


def test_insert_with_the_most_kv_heads():
    # Hkv = 8 (the most the insert takes): 4096 tokens, K/V pools with a head stride
    # above the page size, some slots negative (skipped), K rows spanning wide
    # magnitudes; every page byte equal to the oracle's
    rng = np.random.default_rng(74)
    T, Hkv = 4096, 8
    P = 40
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    slots[rng.random(T) < 0.05] = -1
    kr = (rng.standard_normal((T, Hkv, 128)) * np.exp(rng.normal(0, 4, (T, Hkv, 1)))).astype(np.float32)
    vr = rng.standard_normal((T, Hkv, 128)).astype(np.float32)
    ir = rng.standard_normal((T, 128)).astype(np.float32)
    kp_o = np.full((P, Hkv, 8704), 0xFF, np.uint8)
    vp_o = np.full((P, Hkv, 8704), 0xFF, np.uint8)
    ip_o = np.full((P, 8704), 0xFF, np.uint8)
    oracle.mx4_insert(kr, vr, ir, slots, kp_o, vp_o, ip_o)
    kv = torch.full((2, P, Hkv, 8704 + 128), 0xFF, dtype=torch.uint8, device=DEV)
    ip = torch.full((P, 8704), 0xFF, dtype=torch.uint8, device=DEV)
    m.mx4_insert(torch.from_numpy(kr).to(DEV), torch.from_numpy(vr).to(DEV),
                 torch.from_numpy(ir).to(DEV), torch.from_numpy(slots).to(DEV),
                 kv[0, :, :, :8704], kv[1, :, :, :8704], ip)
    assert m.mx4_check_status() == 0
    got = kv.cpu().numpy()
    assert np.array_equal(got[0, :, :, :8704], kp_o) and np.array_equal(got[1, :, :, :8704], vp_o)
    assert np.all(got[:, :, :, 8704:] == 0xFF)  # the gap between heads is not written
    assert np.array_equal(ip.cpu().numpy(), ip_o)

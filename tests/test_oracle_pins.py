"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one oracle function to something independent of it: values
written out by hand from the format definitions (tests/golden/), closed-form
invariants, special cases that reduce to a library routine, or brute force on
tiny inputs.  The cases are chosen so that a plausible slip anywhere in the
oracle (a swapped nibble, a wrong scale offset, an off-by-one in the causal
bound, a dropped sign, K used for V, a transposed block table) fails one.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from mxfp4_sparse_paged_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.split("#", 1)[0].strip()
            if ln:
                yield ln


# ---------------------------------------------------------------- formats

def test_e2m1_table_all_codes():
    seen = 0
    for ln in _lines("e2m1_values.txt"):
        code, val = ln.split()
        got = oracle.e2m1_value(int(code))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code
        seen += 1
    assert seen == 16


def test_e8m0_values():
    for ln in _lines("e8m0_values.txt"):
        b, val = ln.split()
        got = oracle.e8m0_value(int(b))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val), b


def test_e2m1_rounding_midpoints():
    n = 0
    for ln in _lines("e2m1_rounding.txt"):
        y, code = ln.split()
        assert oracle.round_magnitude(float(y)) == int(code), y
        n += 1
    assert n >= 28


def test_block_exponent_special_cases():
    # power-of-two amax: floor(log2) exact
    assert oracle.block_exponent(1.0) == -2
    assert oracle.block_exponent(2.0) == -1
    assert oracle.block_exponent(4.0) == 0
    # just below a power of two
    assert oracle.block_exponent(float(np.nextafter(np.float32(2.0), np.float32(0)))) == -2
    assert oracle.block_exponent(6.0) == 0
    assert oracle.block_exponent(7.99) == 0
    assert oracle.block_exponent(8.0) == 1
    assert oracle.block_exponent(0.0) == -127
    # smallest fp32 normal / subnormal clamp to -127
    assert oracle.block_exponent(2.0 ** -126) == -127
    assert oracle.block_exponent(2.0 ** -140) == -127
    assert oracle.block_exponent(2.0 ** -125) == -127   # -125 - 2 = -127: at the bound
    assert oracle.block_exponent(2.0 ** -124) == -126   # inside the range
    # largest finite fp32: floor(log2) = 127 -> 125
    assert oracle.block_exponent(float(np.finfo(np.float32).max)) == 125


def test_block_exponent_generic_range():
    # E = floor(log2 a) - 2 for random normal magnitudes, checked with exact ints
    rng = np.random.default_rng(7)
    for e in range(-120, 127, 7):
        for f in rng.uniform(1.0, 2.0, 5):
            a = float(np.float32(f * 2.0 ** e))
            if a >= 2.0 ** (e + 1):
                continue
            assert oracle.block_exponent(a) == max(-127, e - 2)


def _parse_blocks():
    cases, cur = [], None
    for ln in _lines("quantize_blocks.txt"):
        key, rest = ln.split(None, 1)
        if key == "case":
            cur = {"name": rest, "x": np.zeros(128, np.float32)}
            cases.append(cur)
        elif key == "x":
            for item in rest.split():
                i, v = item.split("=")
                cur["x"][int(i)] = np.float32(float(v))
        elif key == "scale":
            cur["scale"] = [int(h, 16) for h in rest.split()]
        elif key == "data":
            d = [int(h, 16) for h in rest.split()]
            cur["data"] = d + [0] * (64 - len(d))
    return cases


@pytest.mark.parametrize("case", _parse_blocks(), ids=lambda c: c["name"])
def test_hand_worked_rows(case):
    data, scale = oracle.quantize_row(case["x"])
    assert list(scale) == case["scale"]
    assert list(data) == case["data"]


def test_error_bound_closed_form():
    # |y - q(y)| <= half the local grid spacing: 0.25 on [0,2], 0.5 on (2,4],
    # 1 on (4,6], < 2 in saturation (6,8); y = x / 2^E.
    rng = np.random.default_rng(11)
    for trial in range(300):
        sc = float(2.0 ** rng.integers(-30, 30))
        x = (rng.standard_normal(32) * sc).astype(np.float32)
        if trial % 3 == 0:
            x[rng.integers(32)] *= 20
        codes, sb = oracle.quantize_block(x)
        E = sb - 127
        for xi, c in zip(x, codes):
            y = abs(float(xi)) / 2.0 ** E
            qv = abs(oracle.e2m1_value(int(c)))
            bound = 0.25 if y <= 2 else 0.5 if y <= 4 else 1.0 if y <= 6 else 2.0
            assert abs(y - qv) <= bound
            assert y < 8
            if qv != 0:
                assert (int(c) >> 3) == (1 if xi < 0 else 0)


def test_representable_values_roundtrip_exactly():
    # A block whose values are grid values times 2^E, with the largest magnitude in
    # [4, 6] so floor(log2 amax) = E + 2, quantises to exactly those codes.
    rng = np.random.default_rng(5)
    grid = np.array([oracle.e2m1_value(c) for c in range(16)])
    for trial in range(200):
        E = int(rng.integers(-100, 100))
        codes = rng.integers(0, 16, 32)
        codes[rng.integers(32)] = rng.choice([6, 7, 14, 15])
        x = (grid[codes] * 2.0 ** E).astype(np.float32)
        got, sb = oracle.quantize_block(x)
        assert sb == E + 127
        # zero may come back with either sign only if the input zero had that sign
        assert np.array_equal(got, codes.astype(np.uint8))


def test_nonfinite_rejected():
    x = np.zeros(32, np.float32)
    x[3] = np.inf
    with pytest.raises(ValueError):
        oracle.quantize_block(x)
    x[3] = np.nan
    with pytest.raises(ValueError):
        oracle.quantize_block(x)


# ---------------------------------------------------------------- page layout

def test_page_geometry_constants():
    # [128 tokens x 64 B data][128 tokens x 4 B scale] = 8704 B = 128 x 68 B
    assert oracle.PAGE_BYTES == 8704 == 128 * 68 == W.PAGE_BYTES
    assert oracle._load().orc_page_bytes() == 8704


def test_insert_writes_exactly_the_row_bytes():
    # Insert one token into page 2, row 37 of a 4-page, 2-head cache and check that
    # only bytes row*64..row*64+63 (data view) and 8192+row*4..+3 (scale view) of
    # that page and head changed.
    P, H = 4, 2
    rng = np.random.default_rng(3)
    kp = np.full((P, H, 8704), 0xAA, np.uint8)
    vp = np.full((P, H, 8704), 0xAA, np.uint8)
    ip = np.full((P, 8704), 0xAA, np.uint8)
    k = rng.standard_normal((1, H, 128)).astype(np.float32)
    v = rng.standard_normal((1, H, 128)).astype(np.float32)
    ik = rng.standard_normal((1, 128)).astype(np.float32)
    slot = np.array([2 * 128 + 37], np.int64)
    oracle.mx4_insert(k, v, ik, slot, kp, vp, ip)
    for arr, src, heads in ((kp, k, H), (vp, v, H), (ip, ik, 0)):
        for h in range(max(heads, 1)):
            page = arr[2, h] if heads else arr[2]
            x = src[0, h] if heads else src[0]
            data, scale = oracle.quantize_row(x)
            assert np.array_equal(page[37 * 64:38 * 64], data)
            assert np.array_equal(page[8192 + 37 * 4:8192 + 38 * 4], scale)
            mask = np.ones(8704, bool)
            mask[37 * 64:38 * 64] = False
            mask[8192 + 37 * 4:8192 + 38 * 4] = False
            assert np.all(page[mask] == 0xAA)
        others = [p for p in range(P) if p != 2]
        assert np.all(arr[others] == 0xAA)


def test_negative_slot_skips_and_out_of_pool_is_rejected():
    kp = np.zeros((2, 1, 8704), np.uint8)
    vp = np.zeros((2, 1, 8704), np.uint8)
    ip = np.zeros((2, 8704), np.uint8)
    x = np.ones((1, 1, 128), np.float32)
    oracle.mx4_insert(x, x, x[:, 0], np.array([-1], np.int64), kp, vp, ip)
    assert not kp.any() and not vp.any() and not ip.any()
    with pytest.raises(ValueError):
        oracle.mx4_insert(x, x, x[:, 0], np.array([2 * 128], np.int64), kp, vp, ip)


def test_nibble_order_and_dequant():
    page = np.zeros(8704, np.uint8)
    page[5 * 64 + 0] = 0x92        # elements 0,1 of row 5: codes 2 (1.0), 9 (-0.5)
    page[5 * 64 + 63] = 0x7F       # elements 126,127: codes 15 (-6), 7 (6)
    page[8192 + 5 * 4 + 0] = 128   # block 0 scale 2
    page[8192 + 5 * 4 + 3] = 125   # block 3 scale 0.25
    d = oracle.dequant_row(page, 5)
    assert d[0] == 2.0 and d[1] == -1.0
    assert d[126] == -1.5 and d[127] == 1.5
    assert np.all(d[2:126] == 0)
    page[8192 + 5 * 4 + 1] = 255   # NaN scale poisons exactly block 1
    d = oracle.dequant_row(page, 5)
    assert np.all(np.isnan(d[32:64])) and not np.isnan(d[:32]).any()


# ---------------------------------------------------------------- scoring

def _grid_rows(rng, n, E_range=(-4, 3)):
    """Rows of exactly representable values (so dequant(quant(x)) == x)."""
    grid = np.array([oracle.e2m1_value(c) for c in range(16)])
    rows = np.zeros((n, 128), np.float32)
    for i in range(n):
        for b in range(4):
            E = int(rng.integers(*E_range))
            codes = rng.integers(0, 16, 32)
            codes[rng.integers(32)] = rng.choice([6, 7, 14, 15])
            rows[i, 32 * b:32 * b + 32] = grid[codes] * 2.0 ** E
    return rows


def _fill(pages_shape_P, bt, lens, rows):
    ip = np.full((pages_shape_P, 8704), 0xFF, np.uint8)
    for s, L in enumerate(lens):
        pos = np.arange(L)
        slots = bt[s, pos // 128].astype(np.int64) * 128 + pos % 128
        oracle.mx4_insert(None, None, rows[s], slots, None, None, ip)
    return ip


def test_representable_rows_roundtrip_through_pages():
    rng = np.random.default_rng(9)
    rows = _grid_rows(rng, 300)
    bt = np.array([[2, 0, 1]], np.int32)
    ip = _fill(3, bt, [300], [rows])
    back = oracle.dequant_tokens(ip, bt[0], 300)
    assert np.array_equal(back, rows.astype(np.float64))


def test_index_score_exact_small_case_and_causal_bound():
    # Two sequences, q = 2 decode tokens each, physical pages permuted.  Values are
    # exactly representable and the queries are small integers, so the exact
    # score is a rational number computed here with Fractions.
    rng = np.random.default_rng(21)
    lens = [130, 7]
    bt = np.array([[3, 1], [0, -1]], np.int32)
    rows = [_grid_rows(rng, L) for L in lens]
    ip = _fill(4, bt, lens, rows)
    q = 2
    iqf = rng.integers(-3, 4, (4, 128)).astype(np.float32)
    iq = W.to_bf16_bits(iqf)
    ld = 140
    sc = oracle.index_score(iq, q, ip, bt, np.array(lens, np.int32), ld)
    for s in range(2):
        for j in range(q):
            t = s * q + j
            p = lens[s] - q + j
            for i in range(ld):
                if i > p:
                    assert sc[t, i] == -np.inf
                    continue
                exact = sum(Fraction(int(iqf[t, d])) * Fraction(float(rows[s][i, d]))
                            for d in range(128))
                assert sc[t, i] == float(exact)


def test_index_score_unit_query_reads_one_element():
    rng = np.random.default_rng(2)
    rows = _grid_rows(rng, 256)
    bt = np.array([[1, 0]], np.int32)
    ip = _fill(2, bt, [256], [rows])
    for d in (0, 1, 31, 32, 77, 127):
        iqf = np.zeros((1, 128), np.float32)
        iqf[0, d] = 1.0
        sc = oracle.index_score(W.to_bf16_bits(iqf), 1, ip, bt, np.array([256], np.int32), 256)
        assert np.array_equal(sc[0], rows[:, d].astype(np.float64))


def test_index_score_invariant_to_physical_page_permutation():
    rng = np.random.default_rng(4)
    L = 500
    x = rng.standard_normal((L, 128)).astype(np.float32)
    iq = W.to_bf16_bits(rng.standard_normal((1, 128)).astype(np.float32))
    bt1 = np.array([[0, 1, 2, 3]], np.int32)
    bt2 = np.array([[3, 0, 2, 1]], np.int32)
    s1 = oracle.index_score(iq, 1, _fill(4, bt1, [L], [x]), bt1, np.array([L], np.int32), L)
    s2 = oracle.index_score(iq, 1, _fill(4, bt2, [L], [x]), bt2, np.array([L], np.int32), L)
    assert np.array_equal(s1, s2)


# ---------------------------------------------------------------- top-k

def test_topk_hand_cases():
    for ln in _lines("topk_cases.txt"):
        sc, k, want = [p.split() for p in ln.split(";")]
        scores = np.array([[float(v) for v in sc]])
        got = oracle.topk_select(scores, np.array([len(sc)], np.int32), 1, int(k[0]))
        assert list(got[0]) == [int(v) for v in want], ln


def test_topk_brute_force_small_rows():
    # Brute force: the chosen set must be the lexicographically-best k-subset under
    # (score desc, index asc), i.e. every chosen element ranks before every
    # unchosen one.  Ties are forced by drawing scores from a few values.
    rng = np.random.default_rng(13)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 45))
        scores = rng.integers(-3, 4, n).astype(np.float64) * 0.5
        got = oracle.topk_select(scores[None], np.array([n], np.int32), 1, k)[0]
        chosen = [int(i) for i in got if i >= 0]
        assert chosen == sorted(chosen) and len(chosen) == min(n, k)
        assert all(i == -1 for i in got[len(chosen):])
        rest = [i for i in range(n) if i not in chosen]
        for a in chosen:
            for b in rest:
                assert scores[a] > scores[b] or (scores[a] == scores[b] and a < b)


def test_topk_multi_token_causal_lengths():
    # q = 3 decode tokens of one sequence of length 5: token j sees 5 - 3 + j + 1.
    scores = np.array([[9, 8, 7, -np.inf, -np.inf],
                       [1, 2, 3, 4, -np.inf],
                       [5, 5, 5, 5, 6]], np.float64)
    got = oracle.topk_select(scores, np.array([5], np.int32), 3, 4)
    assert list(got[0]) == [0, 1, 2, -1]
    assert list(got[1]) == [0, 1, 2, 3]
    assert list(got[2]) == [0, 1, 2, 4]


# ---------------------------------------------------------------- attention

def _kv_setup(rng, L, bt, outlier=False):
    k = rng.standard_normal((L, 1, 128)).astype(np.float32)
    v = rng.standard_normal((L, 1, 128)).astype(np.float32)
    if outlier:
        v[:, 0, 5] *= 20
    P = int(bt.max()) + 1
    kp = np.full((P, 1, 8704), 0xFF, np.uint8)
    vp = np.full((P, 1, 8704), 0xFF, np.uint8)
    pos = np.arange(L)
    slots = bt[0, pos // 128].astype(np.int64) * 128 + pos % 128
    oracle.mx4_insert(k, v, None, slots, kp, vp, None)
    return kp, vp


def test_decode_full_selection_equals_dense_sdpa():
    # top-k = context -> dense softmax attention; compared with torch's float64
    # scaled_dot_product_attention over the oracle-dequantised K and V.
    rng = np.random.default_rng(17)
    L = 300
    bt = np.array([[2, 0, 1]], np.int32)
    kp, vp = _kv_setup(rng, L, bt, outlier=True)
    qb = W.to_bf16_bits(rng.standard_normal((1, 16, 128)).astype(np.float32))
    sel = np.arange(512, dtype=np.int32)[None]
    sel[0, L:] = -1
    scale = 1 / math.sqrt(128)
    out = oracle.sparse_paged_decode(qb, 1, kp, vp, bt, np.array([L], np.int32), sel, scale)
    K = torch.from_numpy(oracle.dequant_tokens(kp, bt[0], L, head=0))
    V = torch.from_numpy(oracle.dequant_tokens(vp, bt[0], L, head=0))
    qf = torch.from_numpy(qb.astype(np.uint32) << 16).view(torch.float32).double()
    ref = torch.nn.functional.scaled_dot_product_attention(
        qf.view(1, 16, 1, 128), K.expand(1, 16, L, 128), V.expand(1, 16, L, 128), scale=scale)
    assert np.allclose(out[0], ref.view(16, 128).numpy(), rtol=1e-12, atol=1e-12)


def test_decode_single_token_returns_its_value_row():
    rng = np.random.default_rng(19)
    L = 200
    bt = np.array([[1, 0]], np.int32)
    kp, vp = _kv_setup(rng, L, bt)
    qb = W.to_bf16_bits(rng.standard_normal((1, 16, 128)).astype(np.float32))
    for i in (0, 127, 128, 199):
        sel = np.full((1, 8), -1, np.int32)
        sel[0, 0] = i
        out = oracle.sparse_paged_decode(qb, 1, kp, vp, bt, np.array([L], np.int32), sel, 0.1)
        vrow = oracle.dequant_row(vp[bt[0, i // 128], 0], i % 128)
        assert np.array_equal(out[0], np.broadcast_to(vrow, (16, 128)))


def test_decode_zero_query_gives_mean_of_selected_values():
    rng = np.random.default_rng(23)
    L = 256
    bt = np.array([[0, 1]], np.int32)
    kp, vp = _kv_setup(rng, L, bt)
    qb = np.zeros((1, 16, 128), np.uint16)
    sel = np.array([[3, 50, 129, 255, -1, -1]], np.int32)
    out = oracle.sparse_paged_decode(qb, 1, kp, vp, bt, np.array([L], np.int32), sel, 0.3)
    V = oracle.dequant_tokens(vp, bt[0], L, head=0)
    want = V[[3, 50, 129, 255]].mean(axis=0)
    assert np.allclose(out[0], np.broadcast_to(want, (16, 128)), rtol=1e-14, atol=1e-15)


def test_decode_rejects_index_beyond_position():
    rng = np.random.default_rng(1)
    bt = np.array([[0]], np.int32)
    kp, vp = _kv_setup(rng, 100, bt)
    qb = np.zeros((1, 16, 128), np.uint16)
    with pytest.raises(ValueError):
        oracle.sparse_paged_decode(qb, 1, kp, vp, bt, np.array([100], np.int32),
                                   np.array([[100]], np.int32), 1.0)


def test_decode_gqa_uses_kv_head_group():
    # With Hkv = 2 and H = 4, heads 0,1 read KV head 0 and heads 2,3 read KV head 1.
    rng = np.random.default_rng(29)
    L = 10
    k = rng.standard_normal((L, 2, 128)).astype(np.float32)
    v = rng.standard_normal((L, 2, 128)).astype(np.float32)
    kp = np.zeros((1, 2, 8704), np.uint8)
    vp = np.zeros((1, 2, 8704), np.uint8)
    oracle.mx4_insert(k, v, None, np.arange(L, dtype=np.int64), kp, vp, None)
    qb = np.zeros((1, 4, 128), np.uint16)
    sel = np.arange(L, dtype=np.int32)[None]
    out = oracle.sparse_paged_decode(qb, 1, kp, vp, np.array([[0]], np.int32),
                                     np.array([L], np.int32), sel, 1.0)
    for h in range(4):
        V = np.stack([oracle.dequant_row(vp[0, h // 2], i) for i in range(L)])
        assert np.allclose(out[0, h], V.mean(axis=0), rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------- norm + rotary (R10)

def _cos_sin(angles):
    """One rotary row per angle vector (64 angles): [cos(64) | sin(64)], fp32."""
    a = np.asarray(angles, np.float64).reshape(-1, 64)
    return np.concatenate([np.cos(a), np.sin(a)], axis=1).astype(np.float32)


def test_norm_rope_hand_row():
    # x = (3, 4, 0, ...): mean of squares 25/128, so z = x * sqrt(128) / 5; no turn
    x = np.zeros((1, 128), np.float32)
    x[0, 0], x[0, 1] = 3, 4
    y = oracle.norm_rope(x, np.ones(128, np.float32), _cos_sin(np.zeros(64)), [0], 0.0)
    want = np.zeros(128)
    want[0], want[1] = 3 * math.sqrt(128) / 5, 4 * math.sqrt(128) / 5
    assert np.allclose(y[0], want, rtol=0, atol=1e-12)


def test_norm_rope_constant_row_gives_the_weight():
    g = np.linspace(-2, 2, 128).astype(np.float32)
    for c in (1e-3, 7.0, -5.0):
        x = np.full((1, 128), c, np.float32)
        y = oracle.norm_rope(x, g, _cos_sin(np.zeros(64)), [0], 0.0, rope=False)
        assert np.allclose(y[0], np.sign(c) * g.astype(np.float64), rtol=1e-12, atol=0)


def test_norm_rope_quarter_turn_direction():
    # cos 0, sin 1: (z_i, z_{i+64}) -> (-z_{i+64}, z_i)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 128)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    cs = np.zeros((1, 128), np.float32)
    cs[0, 64:] = 1.0
    z = oracle.norm_rope(x, g, cs, [0, 0], 1e-6, rope=False)
    y = oracle.norm_rope(x, g, cs, [0, 0], 1e-6)
    assert np.array_equal(y[:, :64], -z[:, 64:]) and np.array_equal(y[:, 64:], z[:, :64])


def test_norm_rope_turn_keeps_pair_norms_and_position_picks_the_row():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 128)).astype(np.float32)
    g = np.ones(128, np.float32)
    ang = rng.uniform(-math.pi, math.pi, (7, 64))
    cs = _cos_sin(ang)
    pos = np.array([0, 3, 6, 3, 1])
    z = oracle.norm_rope(x, g, cs, pos, 0.0, rope=False)
    y = oracle.norm_rope(x, g, cs, pos, 0.0)
    assert np.allclose(y[:, :64] ** 2 + y[:, 64:] ** 2, z[:, :64] ** 2 + z[:, 64:] ** 2,
                       rtol=1e-6, atol=1e-12)
    c, s = cs[pos, :64].astype(np.float64), cs[pos, 64:].astype(np.float64)
    assert np.allclose(y[:, 0], z[:, 0] * c[:, 0] - z[:, 64] * s[:, 0], rtol=1e-14, atol=0)
    # unit weight, no eps: the normed row has mean square 1
    assert np.allclose((z ** 2).mean(axis=1), 1.0, rtol=1e-12)


def test_norm_rope_zero_row_and_bad_position():
    x = np.zeros((1, 128), np.float32)
    cs = _cos_sin(np.zeros((2, 64)))
    y = oracle.norm_rope(x, np.ones(128, np.float32), cs, [1], 1e-6)
    assert np.array_equal(y, np.zeros((1, 128)))
    with pytest.raises(Exception):
        oracle.norm_rope(x, np.ones(128, np.float32), cs, [2], 1e-6)


# ---------------------------------------------------------------- fp8 index cache (E4M3)

def test_e4m3_hand_values():
    # OCP E4M3: bias 7, subnormals m/8 * 2^-6, S.1111.111 NaN, largest normal 448
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
            0x0F: 1.875 * 2.0 ** -6, 0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0,
            0x77: 240.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, v in hand.items():
        assert oracle.e4m3_value(code) == v, hex(code)
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) == -1.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_values_match_torch_float8():
    # A library decode of the same format: all 256 codes.
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(mine))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], mine[ok])
    assert np.array_equal(np.signbit(lib[ok]), np.signbit(mine[ok]))


def test_e4m3_encode_ties_and_saturation():
    hand = [(1.0625, 0x38), (1.1875, 0x3A), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
            (2.0 ** -6 * (1 + 1 / 16), 0x08), (15 * 2.0 ** -10, 0x08), (448.0, 0x7E),
            (449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),
            (float(np.finfo(np.float32).max), 0x7E), (-0.0, 0x80), (-(2.0 ** -12), 0x80),
            (0.0, 0x00), (0.1, 0x1D), (-3.3, 0xC5)]
    for y, code in hand:
        assert oracle.e4m3_encode(y) == code, (y, hex(code), hex(oracle.e4m3_encode(y)))
    # every finite code round-trips
    for c in range(256):
        if (c & 0x7F) != 0x7F:
            assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, hex(c)


def test_e4m3_encode_matches_torch_float8_in_range():
    # torch rounds to nearest even but does not saturate: compare below 464.
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(20000) * np.exp2(rng.uniform(-14, 9, 20000))).astype(np.float32)
    finite = np.array([oracle.e4m3_value(c) for c in range(256) if (c & 0x7F) != 0x7F])
    mids = (np.sort(finite)[1:] + np.sort(finite)[:-1]) / 2
    x = np.concatenate([x, mids.astype(np.float32),
                        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                        np.nextafter(mids.astype(np.float32), np.float32(-np.inf))])
    x = x[np.abs(x) < 464]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    # torch may drop the sign of a value that rounds to zero: compare magnitudes there
    z = (lib & 0x7F) == 0
    assert np.array_equal(mine[~z], lib[~z])
    assert np.all((mine[z] & 0x7F) == 0)


def _fp8_fill(P, bt, lens, rows, scale):
    pages = np.full((P, oracle.FP8_PAGE_BYTES), 0xFF, np.uint8)
    for s, L in enumerate(lens):
        slots = np.array([bt[s, i // 128] * 128 + i % 128 for i in range(L)], np.int64)
        oracle.fp8_index_insert(rows[s], slots, scale, pages)
    return pages


def test_fp8_insert_layout_scale_and_slots():
    pages = np.full((2, oracle.FP8_PAGE_BYTES), 0xFF, np.uint8)
    x = np.zeros((3, 128), np.float32)
    x[0, 0], x[0, 5], x[0, 127] = 3.0, -0.5, 896.0
    x[1, 1] = 1.0
    oracle.fp8_index_insert(x, np.array([130, -1, 127]), 2.0, pages)
    row = pages[1, 2 * 128:3 * 128]                       # slot 130: page 1, row 2
    assert row[0] == 0x3C and row[5] == 0xA8 and row[127] == 0x7E   # 1.5, -0.25, 448
    assert np.all(np.delete(row, [0, 5, 127]) == 0)
    assert np.all(pages[0, 127 * 128:] == 0)              # slot 127: the zero row x[2]
    untouched = np.ones_like(pages, bool)
    untouched[1, 256:384] = False
    untouched[0, 127 * 128:] = False
    assert np.all(pages[untouched] == 0xFF)              # slot -1 wrote nothing
    with pytest.raises(ValueError):
        oracle.fp8_index_insert(x[:1], np.array([256]), 1.0, pages)
    with pytest.raises(ValueError):
        oracle.fp8_index_insert(x[:1], np.array([0]), 0.0, pages)


def test_fp8_index_score_exact_small_case_and_causal_bound():
    # Keys decoded by torch's float8 type, queries small integers, scale a power of
    # two: the exact score is a rational number computed here with Fractions.
    rng = np.random.default_rng(23)
    lens = [130, 9]
    bt = np.array([[2, 0], [1, -1]], np.int32)
    scale = 0.25
    rows = [(rng.standard_normal((L, 128)) * 4).astype(np.float32) for L in lens]
    pages = _fp8_fill(3, bt, lens, rows, scale)
    q = 2
    iqf = rng.integers(-3, 4, (4, 128)).astype(np.float32)
    ld = 140
    sc = oracle.index_score_fp8(W.to_bf16_bits(iqf), q, pages, bt, np.array(lens, np.int32),
                                scale, ld)
    dec = torch.from_numpy(pages).view(torch.float8_e4m3fn).double().numpy()
    for s in range(2):
        for j in range(q):
            t = s * q + j
            p = lens[s] - q + j
            for i in range(ld):
                if i > p:
                    assert sc[t, i] == -np.inf
                    continue
                pg = bt[s, i // 128]
                key = dec[pg, (i % 128) * 128:(i % 128 + 1) * 128]
                exact = sum(Fraction(int(iqf[t, d])) * Fraction(float(key[d])) * Fraction(scale)
                            for d in range(128))
                assert sc[t, i] == float(exact)


def test_fp8_index_score_unit_query_reads_one_element_times_scale():
    rng = np.random.default_rng(3)
    rows = [(rng.standard_normal((200, 128)) * 100).astype(np.float32)]
    bt = np.array([[1, 0]], np.int32)
    pages = _fp8_fill(2, bt, [200], rows, 8.0)
    dec = torch.from_numpy(pages).view(torch.float8_e4m3fn).double().numpy()
    for d in (0, 3, 64, 127):
        iqf = np.zeros((1, 128), np.float32)
        iqf[0, d] = 1.0
        sc = oracle.index_score_fp8(W.to_bf16_bits(iqf), 1, pages, bt, np.array([200], np.int32),
                                    8.0, 200)
        want = [dec[bt[0, i // 128], (i % 128) * 128 + d] * 8.0 for i in range(200)]
        assert np.array_equal(sc[0], want)


# ---------------------------------------------------------------- block-scaled score mode (MXFP8 query)

def test_mxfp8_hand_worked_block():
    # amax 1 -> E = 0 - 8 = -8 (byte 0x77); y = x * 2^8: 256 -> 0x78, 76.8 -> 80 -> 0x6A,
    # -5.12 -> -5 -> 0xCA; zeros stay zero
    x = np.zeros(32, np.float32)
    x[:3] = [1.0, 0.3, -0.02]
    codes, sb = oracle.mxfp8_quantize_block(x)
    assert sb == 0x77
    assert list(codes[:3]) == [0x78, 0x6A, 0xCA] and not codes[3:].any()
    codes, sb = oracle.mxfp8_quantize_block(np.zeros(32, np.float32))
    assert sb == 0 and not codes.any()


def test_mxfp8_block_exponent_and_saturation_edge():
    assert oracle.mxfp8_block_exponent(1.0) == -8
    assert oracle.mxfp8_block_exponent(2.0) == -7
    assert oracle.mxfp8_block_exponent(float(np.nextafter(np.float32(2), np.float32(0)))) == -8
    assert oracle.mxfp8_block_exponent(2.0 ** -130) == -127
    assert oracle.mxfp8_block_exponent(float(np.finfo(np.float32).max)) == 127 - 8
    # an amax just below 2^(E+9) scales to just below 512: it saturates to 448
    x = np.zeros(32, np.float32)
    x[0] = np.nextafter(np.float32(2), np.float32(0))
    x[1] = -x[0]
    codes, sb = oracle.mxfp8_quantize_block(x)
    assert sb == 127 - 8 and codes[0] == 0x7E and codes[1] == 0xFE


def test_mxfp8_elements_match_torch_float8_at_the_block_exponent():
    # With E fixed by the block maximum, an element's code is the library's E4M3
    # conversion of x * 2^-E wherever that stays below 464 (torch does not saturate).
    rng = np.random.default_rng(12)
    for trial in range(200):
        x = (rng.standard_normal(32) * 2.0 ** rng.integers(-30, 30)).astype(np.float32)
        x[rng.integers(32)] *= rng.choice([1.0, 0.0, 1e-8])
        codes, sb = oracle.mxfp8_quantize_block(x)
        E = sb - 127
        assert E == oracle.mxfp8_block_exponent(float(np.abs(x).max()))
        y = x.astype(np.float64) * 2.0 ** -E
        assert np.abs(y).max() < 512
        ok = np.abs(y) < 464
        lib = torch.from_numpy(y[ok].astype(np.float32)).to(torch.float8_e4m3fn)
        lib = lib.view(torch.uint8).numpy()
        z = (lib & 0x7F) == 0
        assert np.array_equal(codes[ok][~z], lib[~z])
        assert np.all((codes[ok][z] & 0x7F) == 0)
        assert np.all(codes[~ok] & 0x7F == 0x7E)


def test_index_score_mxq_exact_against_rationals_and_error_bound():
    # Keys of exactly representable MXFP4 values; the query's MXFP8 values come from
    # torch's E4M3 decode of the oracle's codes times 2^E; the score is their exact
    # rational dot.  And the difference to the bf16-query score stays within
    # sum_j |k_j| * (E4M3 half-step of q_j at its block exponent).
    rng = np.random.default_rng(31)
    lens = [200, 5]
    bt = np.array([[1, 2], [0, -1]], np.int32)
    rows = [_grid_rows(rng, L) for L in lens]
    ip = _fill(3, bt, lens, rows)
    q = 1
    iqf = (rng.standard_normal((2, 128)) * np.exp2(rng.integers(-6, 6, (2, 128)))).astype(np.float32)
    iq = W.to_bf16_bits(iqf)
    iqv = torch.from_numpy(iq.view(np.int16)).view(torch.bfloat16).double().numpy()
    sc = oracle.index_score_mxq(iq, q, ip, bt, np.array(lens, np.int32), 200)
    ref = oracle.index_score(iq, q, ip, bt, np.array(lens, np.int32), 200)
    for t in range(2):
        qhat, half = np.zeros(128), np.zeros(128)
        for b in range(4):
            codes, sb = oracle.mxfp8_quantize_block(iqv[t, 32 * b:32 * b + 32].astype(np.float32))
            dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
            qhat[32 * b:32 * b + 32] = dec * 2.0 ** (sb - 127)
            # half an E4M3 step at each element's binade (2^-10 below 2^-6), or the
            # distance to 448 where the scaled element saturates; times 2^E
            y = np.abs(iqv[t, 32 * b:32 * b + 32]) * 2.0 ** -(sb - 127)
            e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
            half[32 * b:32 * b + 32] = np.maximum(2.0 ** (e - 4), y - 448.0) * 2.0 ** (sb - 127)
        for i in range(lens[t]):
            key = rows[t][i].astype(np.float64)
            exact = sum(Fraction(float(qhat[d])) * Fraction(float(key[d])) for d in range(128))
            assert sc[t, i] == float(exact)
            assert abs(sc[t, i] - ref[t, i]) <= float(np.abs(key) @ half) * (1 + 1e-12)
        assert np.all(sc[t, lens[t]:] == -np.inf)


def test_encoders_are_monotone_step_functions():
    # The e2m1 rounding and the E4M3 encoder never decrease as |y| grows, and change
    # value only at the grid midpoints: over dense sorted inputs the decoded value is
    # non-decreasing and every step of it straddles a midpoint.
    y = np.linspace(0.0, 7.999, 20001)
    mag = np.array([oracle.e2m1_value(oracle.round_magnitude(v)) for v in y])
    assert np.all(np.diff(mag) >= 0)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    mids = (grid[1:] + grid[:-1]) / 2
    for i in np.nonzero(np.diff(mag))[0]:
        assert np.any((y[i] <= mids) & (mids <= y[i + 1])), (y[i], y[i + 1])
    z = np.linspace(-500.0, 500.0, 40001).astype(np.float32)
    val = np.array([oracle.e4m3_value(oracle.e4m3_encode(v)) for v in z])
    assert np.all(np.diff(val) >= 0)

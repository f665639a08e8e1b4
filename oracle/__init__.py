"""CPU oracle for sparse-attention decode over an MXFP4 paged KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the benchmark's CPU-baseline leg import this package.  The CUDA library
does not import, link or call it, and it shares no code with the library.

The arithmetic lives in ``mx4_oracle.c`` (plain C, float64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.  Every function
below mirrors one C function; their docstrings restate what it computes and
the source it follows (see the C file's header for the page citations and the
readings R1..R17 taken where the pages are silent).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

PAGE_TOKENS = 128
ROW_ELEMS = 128
DATA_BYTES = 64
SCALE_BYTES = 4
PAGE_BYTES = PAGE_TOKENS * (DATA_BYTES + SCALE_BYTES)


def build(force: bool = False) -> str:
    """Compile mx4_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-Wall", "-Wextra",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        lib.orc_e2m1_value.restype = ctypes.c_double
        lib.orc_e2m1_value.argtypes = [i32]
        lib.orc_e8m0_value.restype = ctypes.c_double
        lib.orc_e8m0_value.argtypes = [i32]
        lib.orc_block_exponent.restype = i32
        lib.orc_block_exponent.argtypes = [ctypes.c_double]
        lib.orc_e2m1_round_magnitude.restype = i32
        lib.orc_e2m1_round_magnitude.argtypes = [ctypes.c_double]
        lib.orc_quantize_block.restype = i32
        lib.orc_quantize_block.argtypes = [P, P, P]
        lib.orc_quantize_row.restype = i32
        lib.orc_quantize_row.argtypes = [P, P, P]
        lib.orc_dequant_row.restype = None
        lib.orc_dequant_row.argtypes = [P, i32, P]
        lib.orc_mx4_insert.restype = i32
        lib.orc_mx4_insert.argtypes = [P, P, P, i64, i32, P, P, P, i64, i64, P, i64, i64]
        lib.orc_index_score.restype = i32
        lib.orc_index_score.argtypes = [P, i64, i32, P, i64, i64, P, i64, P, P, P, i64]
        lib.orc_topk_select.restype = i32
        lib.orc_topk_select.argtypes = [P, i64, P, i64, i32, i32, P]
        lib.orc_norm_rope.restype = i32
        lib.orc_norm_rope.argtypes = [P, i64, P, P, i64, P, ctypes.c_double, i32, P]
        lib.orc_sparse_paged_decode.restype = i32
        lib.orc_sparse_paged_decode.argtypes = [P, i64, i32, i32, i32, P, P, i64, i64, i64,
                                                P, i64, P, P, i32, ctypes.c_double, P]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [i32]
        lib.orc_e4m3_encode.restype = i32
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_fp8_index_insert.restype = i32
        lib.orc_fp8_index_insert.argtypes = [P, i64, P, ctypes.c_float, P, i64, i64]
        lib.orc_index_score_fp8.restype = i32
        lib.orc_index_score_fp8.argtypes = [P, i64, i32, P, i64, i64, P, i64, P, ctypes.c_float,
                                            P, P, i64]
        lib.orc_mxfp8_block_exponent.restype = i32
        lib.orc_mxfp8_block_exponent.argtypes = [ctypes.c_double]
        lib.orc_mxfp8_quantize_block.restype = i32
        lib.orc_mxfp8_quantize_block.argtypes = [P, P, P]
        lib.orc_index_score_mxq.restype = i32
        lib.orc_index_score_mxq.argtypes = [P, i64, i32, P, i64, i64, P, i64, P, P, P, i64]
        lib.orc_page_bytes.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# --------------------------------------------------------------------------
# element / scale types
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (OCP MX v1.0 FP4 E2M1)."""
    return _load().orc_e2m1_value(int(code))


def e8m0_value(byte: int) -> float:
    """Value of an E8M0 scale byte, 2^(byte-127); NaN for 0xFF."""
    return _load().orc_e8m0_value(int(byte))


def block_exponent(amax: float) -> int:
    """Shared exponent floor(log2(amax)) - 2, clamped to [-127, 127]."""
    return _load().orc_block_exponent(float(amax))


def round_magnitude(ay: float) -> int:
    """Nearest E2M1 magnitude code to |y|, ties to the even mantissa."""
    return _load().orc_e2m1_round_magnitude(float(ay))


def quantize_block(x):
    """32 fp32 values -> (codes uint8[32], scale byte)."""
    x = _c(x, np.float32)
    assert x.shape == (32,)
    codes = np.zeros(32, np.uint8)
    sb = np.zeros(1, np.uint8)
    _check(_load().orc_quantize_block(_ptr(x), _ptr(codes), _ptr(sb)), "quantize_block")
    return codes, int(sb[0])


def quantize_row(x):
    """128 fp32 values -> (data uint8[64], scale uint8[4])."""
    x = _c(x, np.float32)
    assert x.shape == (128,)
    data = np.zeros(64, np.uint8)
    scale = np.zeros(4, np.uint8)
    _check(_load().orc_quantize_row(_ptr(x), _ptr(data), _ptr(scale)), "quantize_row")
    return data, scale


def dequant_row(page, row: int):
    """Dequantised token row `row` (0..127) of one 8704-byte page, float64[128]."""
    page = _c(page, np.uint8)
    assert page.shape == (PAGE_BYTES,)
    out = np.zeros(128, np.float64)
    _load().orc_dequant_row(_ptr(page), int(row), _ptr(out))
    return out


def dequant_tokens(pages, block_table_row, n, head=None):
    """Dequantised rows of logical tokens 0..n-1 of one sequence, float64[n,128].

    pages: [P, 8704] (index cache) or [P, Hkv, 8704] with `head` given."""
    out = np.zeros((n, 128), np.float64)
    for i in range(n):
        pg = int(block_table_row[i // PAGE_TOKENS])
        page = pages[pg] if head is None else pages[pg, head]
        out[i] = dequant_row(page, i % PAGE_TOKENS)
    return out


# --------------------------------------------------------------------------
# the four steps
# --------------------------------------------------------------------------

def mx4_insert(k, v, idx_k, slot_mapping, k_pages, v_pages, idx_pages):
    """Quantise-on-insert into numpy page arrays, in place.

    k, v: fp32 [T, Hkv, 128] (or None); idx_k: fp32 [T, 128] (or None);
    slot_mapping: int64 [T]; k_pages, v_pages: uint8 [P, Hkv, 8704];
    idx_pages: uint8 [P, 8704]."""
    lib = _load()
    slot_mapping = _c(slot_mapping, np.int64)
    T = slot_mapping.shape[0]
    Hkv = 1 if k_pages is None else k_pages.shape[1]
    for arr in (k_pages, v_pages, idx_pages):
        if arr is not None:
            assert arr.dtype == np.uint8 and arr.flags.c_contiguous
    k = None if k is None else _c(k, np.float32)
    v = None if v is None else _c(v, np.float32)
    idx_k = None if idx_k is None else _c(idx_k, np.float32)
    kv_ps = 0 if k_pages is None else k_pages.strides[0]
    kv_hs = 0 if k_pages is None else k_pages.strides[1]
    idx_ps = 0 if idx_pages is None else idx_pages.strides[0]
    P = (k_pages if k_pages is not None else idx_pages).shape[0]
    rc = lib.orc_mx4_insert(_ptr(k), _ptr(v), _ptr(idx_k), T, Hkv, _ptr(slot_mapping),
                            _ptr(k_pages), _ptr(v_pages), kv_ps, kv_hs, _ptr(idx_pages),
                            idx_ps, P)
    _check(rc, "mx4_insert")


def norm_rope(x, g, cos_sin, positions, eps, rope=True):
    """RMS-norm with weight g, then (rope) the rotary turn of dims (i, i+64) by
    cos_sin[pos]: float64 [n, 128] from fp32 rows x [n, 128]."""
    lib = _load()
    x = _c(x, np.float32).reshape(-1, 128)
    n = x.shape[0]
    g = _c(g, np.float32)
    cos_sin = _c(cos_sin, np.float32)
    positions = _c(np.broadcast_to(np.asarray(positions, np.int64), (n,)), np.int64)
    out = np.empty((n, 128), np.float64)
    rc = lib.orc_norm_rope(_ptr(x), n, _ptr(g), _ptr(cos_sin), cos_sin.shape[0], _ptr(positions),
                           ctypes.c_double(eps), int(bool(rope)), _ptr(out))
    _check(rc, "norm_rope")
    return out


def index_score(iq_bits, q_per_seq, idx_pages, block_table, seq_lens, ld, want_mag=False):
    """Index scores, float64 [T, ld] (and sum of |terms| if want_mag).

    iq_bits: bf16 bit patterns, uint16 [T, 128]."""
    lib = _load()
    iq_bits = _c(iq_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B = seq_lens.shape[0]
    T = iq_bits.shape[0]
    assert T == B * q_per_seq
    scores = np.empty((T, ld), np.float64)
    mag = np.empty((T, ld), np.float64) if want_mag else None
    rc = lib.orc_index_score(_ptr(iq_bits), B, int(q_per_seq), _ptr(idx_pages),
                             idx_pages.strides[0], idx_pages.shape[0], _ptr(block_table),
                             block_table.shape[1], _ptr(seq_lens), _ptr(scores), _ptr(mag), ld)
    _check(rc, "index_score")
    return (scores, mag) if want_mag else scores


def topk_select(scores, seq_lens, q_per_seq, k):
    """Top-k token indices per decode token, int32 [T, k], ascending, -1 padded."""
    lib = _load()
    scores = _c(scores, np.float64)
    seq_lens = _c(seq_lens, np.int32)
    T, ld = scores.shape
    out = np.empty((T, k), np.int32)
    rc = lib.orc_topk_select(_ptr(scores), ld, _ptr(seq_lens), seq_lens.shape[0],
                             int(q_per_seq), int(k), _ptr(out))
    _check(rc, "topk_select")
    return out


def sparse_paged_decode(q_bits, q_per_seq, k_pages, v_pages, block_table, seq_lens, topk,
                        scale):
    """Attention output over the selected tokens, float64 [T, H, 128].

    q_bits: bf16 bit patterns uint16 [T, H, 128]; k/v_pages uint8 [P, Hkv, 8704];
    topk: int32 [T, kw] (-1 entries ignored)."""
    lib = _load()
    q_bits = _c(q_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    topk = _c(topk, np.int32)
    T, H, _ = q_bits.shape
    B = seq_lens.shape[0]
    assert T == B * q_per_seq
    assert k_pages.strides == v_pages.strides and k_pages.shape == v_pages.shape
    out = np.zeros((T, H, 128), np.float64)
    rc = lib.orc_sparse_paged_decode(_ptr(q_bits), B, int(q_per_seq), H, k_pages.shape[1],
                                     _ptr(k_pages), _ptr(v_pages), k_pages.strides[0],
                                     k_pages.strides[1], k_pages.shape[0], _ptr(block_table),
                                     block_table.shape[1], _ptr(seq_lens), _ptr(topk),
                                     topk.shape[1], float(scale), _ptr(out))
    _check(rc, "sparse_paged_decode")
    return out


# --------------------------------------------------------------------------
# the fp8 index cache variant
# --------------------------------------------------------------------------

FP8_ROW_BYTES = 128
FP8_PAGE_BYTES = PAGE_TOKENS * FP8_ROW_BYTES


def e4m3_value(code: int) -> float:
    """Value of an FP8 E4M3 code (OCP); NaN for S.1111.111."""
    return _load().orc_e4m3_value(int(code))


def e4m3_encode(y: float) -> int:
    """E4M3 code of the fp32 value y: nearest, ties to even, saturating at 448."""
    return _load().orc_e4m3_encode(float(y))


def fp8_index_insert(idx_k, slot_mapping, scale, pages):
    """Insert index-K rows (fp32 [T, 128]) into fp8 pages (uint8 [P, 16384]), in
    place: code E4M3(fl32(x / scale)) per element."""
    idx_k = _c(idx_k, np.float32).reshape(-1, ROW_ELEMS)
    slot_mapping = _c(slot_mapping, np.int64)
    assert pages.dtype == np.uint8 and pages.flags.c_contiguous
    assert pages.shape[1] == FP8_PAGE_BYTES
    rc = _load().orc_fp8_index_insert(_ptr(idx_k), idx_k.shape[0], _ptr(slot_mapping),
                                      ctypes.c_float(scale), _ptr(pages), pages.strides[0],
                                      pages.shape[0])
    _check(rc, "fp8_index_insert")


def index_score_fp8(iq_bits, q_per_seq, pages, block_table, seq_lens, scale, ld,
                    want_mag=False):
    """Index scores over the fp8 cache, float64 [T, ld] (and sum of |terms| if
    want_mag).  iq_bits: bf16 bit patterns, uint16 [T, 128]."""
    lib = _load()
    iq_bits = _c(iq_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B = seq_lens.shape[0]
    T = iq_bits.shape[0]
    assert T == B * q_per_seq
    scores = np.empty((T, ld), np.float64)
    mag = np.empty((T, ld), np.float64) if want_mag else None
    rc = lib.orc_index_score_fp8(_ptr(iq_bits), B, int(q_per_seq), _ptr(pages), pages.strides[0],
                                 pages.shape[0], _ptr(block_table), block_table.shape[1],
                                 _ptr(seq_lens), ctypes.c_float(scale), _ptr(scores), _ptr(mag),
                                 ld)
    _check(rc, "index_score_fp8")
    return (scores, mag) if want_mag else scores


# --------------------------------------------------------------------------
# block-scaled score mode: the index-q row in MXFP8
# --------------------------------------------------------------------------

def mxfp8_block_exponent(amax: float) -> int:
    """Shared exponent of an MXFP8 (E4M3) block: floor(log2(amax)) - 8, clamped."""
    return _load().orc_mxfp8_block_exponent(float(amax))


def mxfp8_quantize_block(x):
    """32 fp32 values -> (E4M3 codes uint8[32], E8M0 scale byte)."""
    x = _c(x, np.float32)
    assert x.shape == (32,)
    codes = np.zeros(32, np.uint8)
    sb = np.zeros(1, np.uint8)
    _check(_load().orc_mxfp8_quantize_block(_ptr(x), _ptr(codes), _ptr(sb)), "mxfp8_quantize_block")
    return codes, int(sb[0])


def index_score_mxq(iq_bits, q_per_seq, idx_pages, block_table, seq_lens, ld, want_mag=False):
    """Index scores with each index-q row first converted to MXFP8, float64 [T, ld]."""
    lib = _load()
    iq_bits = _c(iq_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B = seq_lens.shape[0]
    T = iq_bits.shape[0]
    assert T == B * q_per_seq
    scores = np.empty((T, ld), np.float64)
    mag = np.empty((T, ld), np.float64) if want_mag else None
    rc = lib.orc_index_score_mxq(_ptr(iq_bits), B, int(q_per_seq), _ptr(idx_pages),
                                 idx_pages.strides[0], idx_pages.shape[0], _ptr(block_table),
                                 block_table.shape[1], _ptr(seq_lens), _ptr(scores), _ptr(mag), ld)
    _check(rc, "index_score_mxq")
    return (scores, mag) if want_mag else scores

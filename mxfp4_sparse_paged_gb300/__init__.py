"""Sparse-attention decode over an MXFP4 paged KV cache, native to GB300.

Thin Python binding of the C ABI in include/mx4sp.h (libmx4sp.so, hand-written
sm_103a CUDA kernels).  Every function here has the name of the C entry point
it calls and only marshals arguments: torch tensors become device pointers,
byte strides and the current CUDA stream.  All computation runs in the CUDA
library; there is no fallback, and a missing library raises.

Page tensors are uint8 with a contiguous 8704-byte last axis: K/V pages
[pages, heads, 8704], index-K pages [pages, 8704] (the page of
"vllm.models.minimax_m3.amd.ops.mxfp4_pages").
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["mx4_insert", "mx4_norm_rope_insert", "fp8_index_insert", "index_score_fp8", "index_score", "index_score_mxq",
           "index_topk", "index_topk_workspace", "topk_select", "sparse_paged_decode",
           "topk_select_workspace", "sparse_paged_decode_workspace", "mx4_check_status",
           "sparse_paged_decode_noalloc", "NOALLOC_SCRATCH_BYTES", "mx4_decode_step", "mx4_decode_steps",
           "mx4_decode_step_input_layout",
           "mx4_last_error", "mx4_page_bytes", "library_path", "Mx4Error", "PAGE_BYTES",
           "PAGE_TOKENS", "HEAD_DIM"]

PAGE_BYTES = 8704
FP8_PAGE_BYTES = 16384
PAGE_TOKENS = 128
HEAD_DIM = 128
NOALLOC_SCRATCH_BYTES = 32 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libmx4sp.so")
_lock = threading.Lock()
_lib = None

STATUS_BITS = {0x1: "bad-slot", 0x2: "bad-page", 0x4: "bad-seq-len", 0x8: "bad-topk-index",
               0x10: "non-finite-input"}


class Mx4Error(RuntimeError):
    def __init__(self, code: int, msg: str, bits: int = 0):
        super().__init__(f"mx4 status {code}: {msg}")
        self.code = code
        self.bits = bits


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.mx4_last_error.restype = ctypes.c_char_p
        lib.mx4_last_error.argtypes = []
        lib.mx4_page_bytes.restype = sz
        lib.mx4_page_bytes.argtypes = []
        lib.mx4_insert.restype = i32
        lib.mx4_insert.argtypes = [P, P, P, i64, i32, P, P, P, i64, i64, P, i64, i64, P]
        lib.mx4_norm_rope_insert.restype = i32
        lib.mx4_norm_rope_insert.argtypes = [P, P, P, P, P, i64, i32, i32, P, P, i64, P, P, P, P,
                                             ctypes.c_float, P, P, P, i64, i64, P, i64, i64, P,
                                             P, P]
        lib.fp8_index_insert.restype = i32
        lib.fp8_index_insert.argtypes = [P, i64, P, ctypes.c_float, P, i64, i64, P]
        lib.index_score_fp8.restype = i32
        lib.index_score_fp8.argtypes = [P, i64, i32, P, i64, i64, P, i64, i64, P, ctypes.c_float,
                                        P, i64, P]
        lib.index_score.restype = i32
        lib.index_score.argtypes = [P, i64, i32, P, i64, i64, P, i64, i64, P, P, i64, P]
        lib.index_score_mxq.restype = i32
        lib.index_score_mxq.argtypes = [P, i64, i32, P, i64, i64, P, i64, i64, P, P, i64, P]
        lib.index_topk.restype = i32
        lib.index_topk.argtypes = [P, i64, i32, P, i64, i64, P, i64, i64, P, P, i64, i32, P, P,
                                   sz, P]
        lib.index_topk_workspace.restype = sz
        lib.index_topk_workspace.argtypes = [i64, i32, i64]
        lib.topk_select.restype = i32
        lib.topk_select.argtypes = [P, i64, P, i64, i32, i32, P, P, sz, P]
        lib.topk_select_workspace.restype = sz
        lib.topk_select_workspace.argtypes = [i64, i32, i64]
        lib.sparse_paged_decode.restype = i32
        lib.sparse_paged_decode.argtypes = [P, i64, i32, i32, i32, P, P, i64, i64, i64, P, i64,
                                            i64, P, P, i32, ctypes.c_float, P, P, sz, P]
        lib.sparse_paged_decode_workspace.restype = sz
        lib.sparse_paged_decode_workspace.argtypes = [i64, i32]
        lib.sparse_paged_decode_noalloc.restype = i32
        lib.sparse_paged_decode_noalloc.argtypes = [P, i64, i32, i32, i32, P, P, i64, i64, i64, P,
                                                    i64, i64, P, P, i32, ctypes.c_float, P, P]
        lib.mx4_decode_step_input_bytes.restype = sz
        lib.mx4_decode_step_input_bytes.argtypes = [i64, i64]
        lib.mx4_decode_step_input_offsets.restype = None
        lib.mx4_decode_step_input_offsets.argtypes = [i64, i64, ctypes.POINTER(sz)]
        lib.mx4_decode_step.restype = i32
        lib.mx4_decode_step.argtypes = [P, i64, P, sz, P, P, i64, i64, P, i64, i64, P, i64, i64,
                                        P, i32, i32, ctypes.c_float, P, i64, P, P, sz, P, sz, P,
                                        P, P]
        lib.mx4_decode_steps.restype = i32
        lib.mx4_decode_steps.argtypes = [i64, P, sz, i64, P, sz, P, P, i64, i64, P, i64, i64, P,
                                         i64, i64, P, i32, i32, ctypes.c_float, P, i64, P, P, sz,
                                         P, sz, P, P, sz, P, P, P]
        lib.mx4_check_status.restype = i32
        lib.mx4_check_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        _lib = lib
        return lib


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    # Every tensor handed to the library passes here: a host tensor would be read
    # on the device, so it is refused before the call.
    if t is None:
        return None
    if t.device.type != "cuda":
        raise ValueError(f"every tensor argument must be a CUDA tensor, got a {t.device} tensor "
                         f"of shape {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _check(rc: int):
    if rc != 0:
        raise Mx4Error(rc, _load().mx4_last_error().decode())


def _need(t, dtype, name, contiguous=True):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _dims(t, name, *sizes):
    """t must have len(sizes) dims; a size of None matches any extent."""
    if t.dim() != len(sizes) or any(w is not None and int(e) != w for e, w in zip(t.shape, sizes)):
        want = ", ".join("*" if w is None else str(w) for w in sizes)
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected [{want}]")


def _rows_at_least(t, n, name):
    if int(t.shape[0]) < n:
        raise ValueError(f"{name} has {int(t.shape[0])} rows, needs at least {n}")


def _pages(t, name, ndim):
    _need(t, torch.uint8, name, contiguous=False)
    if t.dim() != ndim or t.shape[-1] != PAGE_BYTES or t.stride(-1) != 1:
        raise ValueError(f"{name}: uint8 pages need shape [...] x {PAGE_BYTES} with a "
                         f"contiguous byte axis, got {tuple(t.shape)} strides {t.stride()}")


def mx4_last_error() -> str:
    return _load().mx4_last_error().decode()


def mx4_page_bytes() -> int:
    return int(_load().mx4_page_bytes())


def mx4_insert(k, v, idx_k, slot_mapping, k_pages, v_pages, idx_pages, stream=None):
    """Quantise new tokens' K [T,Hkv,128], V [T,Hkv,128] and index-K [T,128] (fp32)
    into their page rows through slot_mapping (int64 [T]); pages are written in place."""
    _need(k, torch.float32, "k")
    _need(v, torch.float32, "v")
    _need(idx_k, torch.float32, "idx_k")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _pages(k_pages, "k_pages", 3)
    _pages(v_pages, "v_pages", 3)
    _pages(idx_pages, "idx_pages", 2)
    if k_pages.stride() != v_pages.stride() or k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape and strides")
    _dims(k, "k", None, None, HEAD_DIM)
    T, Hkv = int(k.shape[0]), int(k.shape[1])
    _dims(v, "v", T, Hkv, HEAD_DIM)
    _dims(idx_k, "idx_k", T, HEAD_DIM)
    _dims(slot_mapping, "slot_mapping", T)
    if int(k_pages.shape[1]) != Hkv:
        raise ValueError(f"k_pages has {int(k_pages.shape[1])} KV heads, k has {Hkv}")
    _check(_load().mx4_insert(_ptr(k), _ptr(v), _ptr(idx_k), T, Hkv, _ptr(slot_mapping),
                              _ptr(k_pages), _ptr(v_pages), k_pages.stride(0), k_pages.stride(1),
                              _ptr(idx_pages), idx_pages.stride(0), int(k_pages.shape[0]),
                              _stream(stream)))


def mx4_norm_rope_insert(q, iq, k, v, idx_k, positions, cos_sin, g_q, g_k, g_iq, g_ik, eps,
                         slot_mapping, k_pages, v_pages, idx_pages, q_out, iq_out, stream=None):
    """RMS-norm (weights g_*) and rotary turn (cos_sin [max_pos, 128] = [cos | sin],
    row positions[t]) of the new tokens' q [T,H,128] and index-q [T,128] heads
    -> bf16 q_out, iq_out; of their K and index-K heads -> MXFP4 page rows, with V
    inserted unchanged (all fp32 inputs)."""
    for t, name in ((q, "q"), (iq, "iq"), (k, "k"), (v, "v"), (idx_k, "idx_k"),
                    (cos_sin, "cos_sin"), (g_q, "g_q"), (g_k, "g_k"), (g_iq, "g_iq"),
                    (g_ik, "g_ik")):
        _need(t, torch.float32, name)
    _need(positions, torch.int64, "positions")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(q_out, torch.bfloat16, "q_out")
    _need(iq_out, torch.bfloat16, "iq_out")
    _pages(k_pages, "k_pages", 3)
    _pages(v_pages, "v_pages", 3)
    _pages(idx_pages, "idx_pages", 2)
    if k_pages.stride() != v_pages.stride() or k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape and strides")
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be [T, H, 128] and k [T, Hkv, 128]")
    T, H, Hkv = int(q.shape[0]), int(q.shape[1]), int(k.shape[1])
    want = {"q": (q, (T, H, 128)), "iq": (iq, (T, 128)), "k": (k, (T, Hkv, 128)),
            "v": (v, (T, Hkv, 128)), "idx_k": (idx_k, (T, 128)), "positions": (positions, (T,)),
            "slot_mapping": (slot_mapping, (T,)), "q_out": (q_out, (T, H, 128)),
            "iq_out": (iq_out, (T, 128)), "g_q": (g_q, (128,)), "g_k": (g_k, (128,)),
            "g_iq": (g_iq, (128,)), "g_ik": (g_ik, (128,))}
    for name, (t, shape) in want.items():
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    if cos_sin.dim() != 2 or cos_sin.shape[1] != 128:
        raise ValueError("cos_sin must be [max_pos, 128] (cosines | sines)")
    if int(k_pages.shape[1]) != Hkv:
        raise ValueError(f"k_pages has {int(k_pages.shape[1])} KV heads, k has {Hkv}")
    _check(_load().mx4_norm_rope_insert(
        _ptr(q), _ptr(iq), _ptr(k), _ptr(v), _ptr(idx_k), T, H, Hkv, _ptr(positions),
        _ptr(cos_sin), int(cos_sin.shape[0]), _ptr(g_q), _ptr(g_k), _ptr(g_iq), _ptr(g_ik),
        float(eps), _ptr(slot_mapping), _ptr(k_pages), _ptr(v_pages), k_pages.stride(0),
        k_pages.stride(1), _ptr(idx_pages), idx_pages.stride(0), int(k_pages.shape[0]),
        _ptr(q_out), _ptr(iq_out), _stream(stream)))


def _fp8_pages(t, name):
    _need(t, torch.uint8, name, contiguous=False)
    if t.dim() != 2 or t.shape[1] != FP8_PAGE_BYTES or t.stride(1) != 1:
        raise ValueError(f"{name}: uint8 pages need shape [P, {FP8_PAGE_BYTES}] with a "
                         f"contiguous byte axis, got {tuple(t.shape)} strides {t.stride()}")


def fp8_index_insert(idx_k, slot_mapping, scale, pages, stream=None):
    """Quantise new tokens' index-K rows (fp32 [T, 128]) into the fp8 (E4M3) index
    cache pages [P, 16384] through slot_mapping (int64 [T]), code E4M3(x / scale)."""
    _need(idx_k, torch.float32, "idx_k")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _fp8_pages(pages, "pages")
    _dims(idx_k, "idx_k", None, HEAD_DIM)
    _dims(slot_mapping, "slot_mapping", int(idx_k.shape[0]))
    _check(_load().fp8_index_insert(_ptr(idx_k), int(idx_k.shape[0]), _ptr(slot_mapping),
                                    float(scale), _ptr(pages), pages.stride(0),
                                    int(pages.shape[0]), _stream(stream)))


def index_score_fp8(iq, q_per_seq, pages, block_table, seq_lens, scale, scores, stream=None):
    """index_score over the fp8 index cache: scale * iq . E4M3 row, fp32 [T, ld]."""
    _need(iq, torch.bfloat16, "iq")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(scores, torch.float32, "scores")
    _fp8_pages(pages, "pages")
    _dims(seq_lens, "seq_lens", None)
    B = int(seq_lens.shape[0])
    _dims(iq, "iq", B * int(q_per_seq), HEAD_DIM)
    _dims(block_table, "block_table", None, None)
    _rows_at_least(block_table, B, "block_table")
    _dims(scores, "scores", None, None)
    _rows_at_least(scores, B * int(q_per_seq), "scores")
    _check(_load().index_score_fp8(_ptr(iq), int(iq.shape[0]), int(q_per_seq), _ptr(pages),
                                   pages.stride(0), int(pages.shape[0]), _ptr(block_table), B,
                                   int(block_table.shape[1]), _ptr(seq_lens), float(scale),
                                   _ptr(scores), scores.stride(0), _stream(stream)))


def index_score(iq, q_per_seq, idx_pages, block_table, seq_lens, scores, stream=None):
    """scores[t, i] = iq[t] . dequant(indexK[s, i]) for i <= position (fp32 [T, ld])."""
    _score_call("index_score", iq, q_per_seq, idx_pages, block_table, seq_lens, scores, stream)


def index_score_mxq(iq, q_per_seq, idx_pages, block_table, seq_lens, scores, stream=None):
    """index_score with iq[t] converted to MXFP8 first (block-scaled tensor-core mode)."""
    _score_call("index_score_mxq", iq, q_per_seq, idx_pages, block_table, seq_lens, scores,
                stream)


def _score_call(name, iq, q_per_seq, idx_pages, block_table, seq_lens, scores, stream):
    _need(iq, torch.bfloat16, "iq")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(scores, torch.float32, "scores")
    _pages(idx_pages, "idx_pages", 2)
    _dims(seq_lens, "seq_lens", None)
    B = int(seq_lens.shape[0])
    _dims(iq, "iq", B * int(q_per_seq), HEAD_DIM)
    _dims(block_table, "block_table", None, None)
    _rows_at_least(block_table, B, "block_table")
    _dims(scores, "scores", None, None)
    _rows_at_least(scores, B * int(q_per_seq), "scores")
    _check(getattr(_load(), name)(_ptr(iq), int(iq.shape[0]), int(q_per_seq), _ptr(idx_pages),
                                  idx_pages.stride(0), int(idx_pages.shape[0]), _ptr(block_table),
                                  B, int(block_table.shape[1]), _ptr(seq_lens), _ptr(scores),
                                  scores.stride(0), _stream(stream)))


def index_topk_workspace(T, k, ld_scores) -> int:
    return int(_load().index_topk_workspace(int(T), int(k), int(ld_scores)))


def index_topk(iq, q_per_seq, idx_pages, block_table, seq_lens, scores, k, topk_idx, ws,
               stream=None):
    """index_score then topk_select in one call: scores (fp32 [T, ld]) and
    topk_idx (int32 [T, k]); ws is a uint8 workspace of index_topk_workspace(T, k, ld)
    bytes (None when that is 0)."""
    _need(iq, torch.bfloat16, "iq")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(scores, torch.float32, "scores")
    _need(topk_idx, torch.int32, "topk_idx")
    _pages(idx_pages, "idx_pages", 2)
    _dims(seq_lens, "seq_lens", None)
    B = int(seq_lens.shape[0])
    T = B * int(q_per_seq)
    _dims(iq, "iq", T, HEAD_DIM)
    _dims(block_table, "block_table", None, None)
    _rows_at_least(block_table, B, "block_table")
    _dims(scores, "scores", None, None)
    _rows_at_least(scores, T, "scores")
    _dims(topk_idx, "topk_idx", None, int(k))
    _rows_at_least(topk_idx, T, "topk_idx")
    _check(_load().index_topk(_ptr(iq), T, int(q_per_seq), _ptr(idx_pages), idx_pages.stride(0),
                              int(idx_pages.shape[0]), _ptr(block_table), B,
                              int(block_table.shape[1]), _ptr(seq_lens), _ptr(scores),
                              scores.stride(0), int(k), _ptr(topk_idx), _ptr(ws),
                              0 if ws is None else ws.numel() * ws.element_size(),
                              _stream(stream)))


def topk_select_workspace(T, k, ld_scores) -> int:
    return int(_load().topk_select_workspace(int(T), int(k), int(ld_scores)))


def topk_select(scores, seq_lens, q_per_seq, k, topk_idx, ws=None, stream=None):
    """topk_idx[t] = the min(k, n) best indices (ties -> lower index), ascending, -1 padded."""
    _need(scores, torch.float32, "scores")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(topk_idx, torch.int32, "topk_idx")
    _dims(seq_lens, "seq_lens", None)
    T = int(seq_lens.shape[0]) * int(q_per_seq)
    _dims(scores, "scores", None, None)
    _rows_at_least(scores, T, "scores")
    _dims(topk_idx, "topk_idx", None, int(k))
    _rows_at_least(topk_idx, T, "topk_idx")
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(_load().topk_select(_ptr(scores), scores.stride(0), _ptr(seq_lens),
                               int(seq_lens.shape[0]), int(q_per_seq), int(k), _ptr(topk_idx),
                               _ptr(ws), ws_bytes, _stream(stream)))


def sparse_paged_decode_workspace(T, k) -> int:
    return int(_load().sparse_paged_decode_workspace(int(T), int(k)))


def sparse_paged_decode(q, q_per_seq, k_pages, v_pages, block_table, seq_lens, topk_idx, scale,
                        out, ws, stream=None):
    """out[t, h] = softmax(scale * q[t,h] . K_sel) V_sel over the selected tokens (fp32)."""
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(out, torch.float32, "out")
    _pages(k_pages, "k_pages", 3)
    _pages(v_pages, "v_pages", 3)
    if k_pages.stride() != v_pages.stride() or k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape and strides")
    _dims(q, "q", None, None, HEAD_DIM)
    T, H = int(q.shape[0]), int(q.shape[1])
    _dims(seq_lens, "seq_lens", None)
    B = int(seq_lens.shape[0])
    if T != B * int(q_per_seq):
        raise ValueError(f"q has {T} tokens, seq_lens gives {B} x {int(q_per_seq)}")
    _dims(out, "out", T, H, HEAD_DIM)
    _dims(topk_idx, "topk_idx", T, None)
    _dims(block_table, "block_table", None, None)
    _rows_at_least(block_table, B, "block_table")
    ws_bytes = ws.numel() * ws.element_size()
    _check(_load().sparse_paged_decode(
        _ptr(q), T, int(q_per_seq), H, int(k_pages.shape[1]), _ptr(k_pages), _ptr(v_pages),
        k_pages.stride(0), k_pages.stride(1), int(k_pages.shape[0]), _ptr(block_table),
        int(seq_lens.shape[0]), int(block_table.shape[1]), _ptr(seq_lens), _ptr(topk_idx),
        int(topk_idx.shape[1]), float(scale), _ptr(out), _ptr(ws), ws_bytes, _stream(stream)))


def sparse_paged_decode_noalloc(q, q_per_seq, k_pages, v_pages, block_table, seq_lens, topk_idx,
                                scale, out, stream=None):
    """sparse_paged_decode for callers that cannot allocate device memory: the run
    workspace is the library's own fixed NOALLOC_SCRATCH_BYTES array, so no
    workspace argument is taken and nothing is allocated.  Calls on one device
    share that array and must not overlap on the GPU."""
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(out, torch.float32, "out")
    _pages(k_pages, "k_pages", 3)
    _pages(v_pages, "v_pages", 3)
    if k_pages.stride() != v_pages.stride() or k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape and strides")
    _dims(q, "q", None, None, HEAD_DIM)
    T, H = int(q.shape[0]), int(q.shape[1])
    _dims(seq_lens, "seq_lens", None)
    B = int(seq_lens.shape[0])
    if T != B * int(q_per_seq):
        raise ValueError(f"q has {T} tokens, seq_lens gives {B} x {int(q_per_seq)}")
    _dims(out, "out", T, H, HEAD_DIM)
    _dims(topk_idx, "topk_idx", T, None)
    _dims(block_table, "block_table", None, None)
    _rows_at_least(block_table, B, "block_table")
    _check(_load().sparse_paged_decode_noalloc(
        _ptr(q), T, int(q_per_seq), H, int(k_pages.shape[1]), _ptr(k_pages), _ptr(v_pages),
        k_pages.stride(0), k_pages.stride(1), int(k_pages.shape[0]), _ptr(block_table),
        int(seq_lens.shape[0]), int(block_table.shape[1]), _ptr(seq_lens), _ptr(topk_idx),
        int(topk_idx.shape[1]), float(scale), _ptr(out), _stream(stream)))


def _host_ptr(t, name):
    # The step's input and output buffers live in host memory (page-locked for an
    # asynchronous copy); a device tensor here would be read as a host address.
    if t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host (CPU) tensor")
    return ctypes.c_void_p(t.data_ptr())


def mx4_decode_step_input_layout(T, n_new):
    """(offsets of q, iq, k_new, v_new, idx_k_new, slots in the packed input buffer,
    its total bytes) for mx4_decode_step."""
    off = (ctypes.c_size_t * 6)()
    _load().mx4_decode_step_input_offsets(int(T), int(n_new), off)
    return [int(x) for x in off], int(_load().mx4_decode_step_input_bytes(int(T), int(n_new)))


def _step_args(n_new, k_pages, v_pages, idx_pages, block_table, seq_lens, q_per_seq, k, scale,
               d_scores, d_topk_idx, topk_ws, dec_ws, d_out, out_sets):
    """Checks shared by the step entry points; returns (T, the marshalled cache,
    table and workspace arguments between the staging size and d_out)."""
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(d_scores, torch.float32, "d_scores")
    _need(d_topk_idx, torch.int32, "d_topk_idx")
    _need(d_out, torch.float32, "d_out")
    _pages(k_pages, "k_pages", 3)
    _pages(v_pages, "v_pages", 3)
    _pages(idx_pages, "idx_pages", 2)
    if k_pages.stride() != v_pages.stride() or k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape and strides")
    B = int(seq_lens.shape[0])
    T = B * int(q_per_seq)
    if out_sets == 1:
        _dims(d_out, "d_out", T, 16, HEAD_DIM)
    else:
        _dims(d_out, "d_out", out_sets, T, 16, HEAD_DIM)
    _dims(d_topk_idx, "d_topk_idx", T, int(k))
    _dims(d_scores, "d_scores", None, None)
    _rows_at_least(d_scores, T, "d_scores")
    _rows_at_least(block_table, B, "block_table")
    tws = 0 if topk_ws is None else topk_ws.numel() * topk_ws.element_size()
    args = (_ptr(k_pages), _ptr(v_pages), k_pages.stride(0), k_pages.stride(1), _ptr(idx_pages),
            idx_pages.stride(0), int(k_pages.shape[0]), _ptr(block_table), B,
            int(block_table.shape[1]), _ptr(seq_lens), int(q_per_seq), int(k), float(scale),
            _ptr(d_scores), d_scores.stride(0), _ptr(d_topk_idx), _ptr(topk_ws), tws,
            _ptr(dec_ws), dec_ws.numel() * dec_ws.element_size())
    return T, args


def mx4_decode_step(h_inputs, n_new, d_staging, k_pages, v_pages, idx_pages, block_table,
                    seq_lens, q_per_seq, k, scale, d_scores, d_topk_idx, topk_ws, dec_ws, d_out,
                    h_out, stream=None):
    """One decode step from host memory to host memory: copy the packed host inputs
    (uint8 CPU tensor, layout mx4_decode_step_input_layout) to d_staging, insert the
    n_new new tokens, score, select, attend, and copy the output (fp32 [T, 16, 128])
    into the host tensor h_out.  Asynchronous on `stream`."""
    _need(h_inputs, torch.uint8, "h_inputs")
    _need(h_out, torch.float32, "h_out")
    _need(d_staging, torch.uint8, "d_staging")
    T, args = _step_args(n_new, k_pages, v_pages, idx_pages, block_table, seq_lens, q_per_seq,
                         k, scale, d_scores, d_topk_idx, topk_ws, dec_ws, d_out, 1)
    _, nbytes = mx4_decode_step_input_layout(T, n_new)
    if h_inputs.numel() < nbytes or d_staging.numel() < nbytes:
        raise ValueError(f"input buffers need {nbytes} bytes")
    _dims(h_out, "h_out", T, 16, HEAD_DIM)
    _check(_load().mx4_decode_step(
        _host_ptr(h_inputs, "h_inputs"), int(n_new), _ptr(d_staging), d_staging.numel(), *args,
        _ptr(d_out), _host_ptr(h_out, "h_out"), _stream(stream)))


def mx4_decode_steps(n_steps, h_inputs, n_new, d_staging, k_pages, v_pages, idx_pages,
                     block_table, seq_lens, q_per_seq, k, scale, d_scores, d_topk_idx, topk_ws,
                     dec_ws, d_out, h_out, stream, h2d_stream, d2h_stream, same_inputs=False):
    """n_steps decode steps in order, host memory to host memory, the copies of
    neighbouring steps overlapping the compute on two copy streams.  h_inputs: uint8
    CPU tensor [n_steps, bytes] of packed inputs (or [bytes] with same_inputs=True:
    the same inputs every step); d_staging: uint8 device buffer of two input sets;
    d_out: fp32 device [2, T, 16, 128]; h_out: fp32 CPU [n_steps, T, 16, 128] (or
    [T, 16, 128], every step's output in turn).  Asynchronous on `stream`, which
    waits for the last output copy."""
    _need(h_inputs, torch.uint8, "h_inputs")
    _need(h_out, torch.float32, "h_out")
    _need(d_staging, torch.uint8, "d_staging")
    for name, st in (("h2d_stream", h2d_stream), ("d2h_stream", d2h_stream)):
        if not isinstance(st, torch.cuda.Stream):
            raise ValueError(f"{name} must be a torch.cuda.Stream")
    T, args = _step_args(n_new, k_pages, v_pages, idx_pages, block_table, seq_lens, q_per_seq,
                         k, scale, d_scores, d_topk_idx, topk_ws, dec_ws, d_out, 2)
    _, nbytes = mx4_decode_step_input_layout(T, n_new)
    set_bytes = (nbytes + 255) // 256 * 256
    n_steps = int(n_steps)
    if same_inputs:
        _dims(h_inputs, "h_inputs", None)
        in_stride = 0
    else:
        _dims(h_inputs, "h_inputs", n_steps, None)
        in_stride = int(h_inputs.shape[1])
    if h_inputs.shape[-1] < nbytes or d_staging.numel() < 2 * set_bytes:
        raise ValueError(f"h_inputs rows need {nbytes} bytes, d_staging {2 * set_bytes}")
    if h_out.dim() == 3:
        _dims(h_out, "h_out", T, 16, HEAD_DIM)
        out_stride = 0
    else:
        _dims(h_out, "h_out", n_steps, T, 16, HEAD_DIM)
        out_stride = T * 16 * HEAD_DIM * 4
    _check(_load().mx4_decode_steps(
        n_steps, _host_ptr(h_inputs, "h_inputs"), in_stride, int(n_new), _ptr(d_staging),
        d_staging.numel(), *args, _ptr(d_out), _host_ptr(h_out, "h_out"), out_stride,
        _stream(stream), _stream(h2d_stream), _stream(d2h_stream)))


def mx4_check_status(stream=None) -> int:
    """Synchronise the stream; raise Mx4Error if a kernel flagged bad data (clears it)."""
    bits = ctypes.c_uint32(0)
    rc = _load().mx4_check_status(_stream(stream), ctypes.byref(bits))
    if rc != 0:
        raise Mx4Error(rc, _load().mx4_last_error().decode(), bits.value)
    return 0

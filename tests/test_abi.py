"""The C-ABI library builds for sm_103a, loads, and exports every entry point
declared in include/mx4sp.h; host-side argument checks answer without a GPU
(they return before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mx4sp.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from mxfp4_sparse_paged_gb300 import build
    path = build.build()
    import mxfp4_sparse_paged_gb300 as m
    m._load()
    return ctypes.CDLL(path)


def test_header_declares_the_four_steps():
    names = _declared()
    for n in ("mx4_insert", "index_score", "topk_select", "sparse_paged_decode",
              "topk_select_workspace", "sparse_paged_decode_workspace", "mx4_check_status",
              "mx4_last_error", "mx4_page_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_page_bytes(lib):
    import mxfp4_sparse_paged_gb300 as m
    assert m.mx4_page_bytes() == 8704 == 128 * 68


def test_library_is_sm103a_only():
    from mxfp4_sparse_paged_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _err(m):
    return m.mx4_last_error()


def test_host_validation_without_gpu(lib):
    import mxfp4_sparse_paged_gb300 as m
    L = m._load()
    # negative T
    assert L.mx4_insert(None, None, None, -1, 1, None, None, None, 8704, 8704, None, 8704, 1,
                        None) == -1
    assert "T" in _err(m)
    # unsupported KV head count
    assert L.mx4_insert(None, None, None, 1, 0, None, None, None, 8704, 8704, None, 8704, 1,
                        None) == -2
    # T == 0 is a no-op
    assert L.mx4_insert(None, None, None, 0, 1, None, None, None, 8704, 8704, None, 8704, 1,
                        None) == 0
    # NULL pointers
    assert L.mx4_insert(None, None, None, 4, 1, None, None, None, 8704, 8704, None, 8704, 1,
                        None) == -1
    # index_score: q out of range, T mismatch, empty batch
    assert L.index_score(None, 1, 9, None, 8704, 1, None, 1, 1, None, None, 1, None) == -2
    assert L.index_score(None, 3, 1, None, 8704, 1, None, 2, 1, None, None, 1, None) == -1
    assert L.index_score(None, 0, 1, None, 8704, 1, None, 0, 1, None, None, 1, None) == 0
    # topk: k out of range
    assert L.topk_select(None, 1, None, 1, 1, 0, None, None, 0, None) == -2
    # decode: unsupported head geometry, workspace too small
    assert L.sparse_paged_decode(None, 1, 1, 8, 1, None, None, 8704, 8704, 1, None, 1, 1, None,
                                 None, 16, ctypes.c_float(0.1), None, None, 0, None) == -2
    assert "16 query heads" in _err(m)
    need = L.sparse_paged_decode_workspace(1, 2048)
    assert need > 0
    assert L.sparse_paged_decode(None, 1, 1, 16, 1, None, None, 8704, 8704, 1, None, 1, 1, None,
                                 None, 2048, ctypes.c_float(0.1), None, None, need - 1,
                                 None) == -3
    assert L.sparse_paged_decode(None, 1, 1, 16, 1, None, None, 8704, 8704, 1, None, 1, 1, None,
                                 None, 2048, ctypes.c_float(float("nan")), None, None, need,
                                 None) == -1


def _decode_ws(T, k, sms):
    # one partial record (16 heads x 128 outputs, then 16 maxima and 16 sums, fp32)
    # per (warp, token) run: at most one per warp plus one per token, with one CTA of
    # 8 warps per SM, fewer CTAs when the warps would get fewer than 4 tiles of 16
    # entries each
    tiles = T * ((k + 15) // 16)
    warps = 8 * max(1, min(sms, tiles // 32))
    return (warps + T) * (16 * 128 + 32) * 4


def test_workspace_sizes(lib):
    import mxfp4_sparse_paged_gb300 as m
    # without a GPU the SM count cannot be read: the size assumes 1024 SMs (a bound)
    assert m.sparse_paged_decode_workspace(64, 2048) == _decode_ws(64, 2048, 1024)
    assert m.sparse_paged_decode_workspace(1, 1) == _decode_ws(1, 1, 1024) == 9 * 8320
    assert m.sparse_paged_decode_workspace(0, 2048) == 0
    # count [T] | threshold [T] | (offset, count) per 16384-score segment | kCand = 8192
    # keys and indices, each section padded to 16 bytes
    assert m.topk_select_workspace(64, 2048, 131072) == 2 * 64 * 4 + 64 * 8 * 8 + 2 * 64 * 8192 * 4
    assert m.topk_select_workspace(3, 2048, 20000) == 2 * 16 + 48 + 2 * 3 * 8192 * 4
    assert m.topk_select_workspace(64, 2048, 8192) == 0      # no row exceeds the capacity
    assert m.topk_select_workspace(64, 9000, 131072) == 0    # k above the capacity
    assert m.index_topk_workspace(64, 2048, 131072) == m.topk_select_workspace(64, 2048, 131072)


def test_bindings_refuse_host_tensors_before_any_call():
    # A host pointer handed to a kernel would be read on the device: the binding
    # refuses it first (no library call, no GPU needed).
    import torch
    import mxfp4_sparse_paged_gb300 as m
    r = torch.zeros((2, 1, 128))
    pages = torch.zeros((1, 1, 8704), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        m.mx4_insert(r, r, r[:, 0], torch.zeros(2, dtype=torch.int64), pages, pages.clone(),
                     pages[:, 0])
    with pytest.raises(ValueError, match="CUDA tensor"):
        m.mx4_norm_rope_insert(torch.zeros((2, 16, 128)), r[:, 0], r, r, r[:, 0],
                               torch.zeros(2, dtype=torch.int64), torch.zeros((4, 128)),
                               *(torch.ones(128) for _ in range(4)), 1e-6,
                               torch.zeros(2, dtype=torch.int64), pages, pages.clone(),
                               pages[:, 0], torch.zeros((2, 16, 128), dtype=torch.bfloat16),
                               torch.zeros((2, 128), dtype=torch.bfloat16))


def _cpu_args():
    import torch
    T, H, B, k, ld = 4, 16, 4, 8, 300
    f32, bf, i32, i64, u8 = torch.float32, torch.bfloat16, torch.int32, torch.int64, torch.uint8
    return {
        "k": torch.zeros((T, 1, 128)), "v": torch.zeros((T, 1, 128)),
        "idx_k": torch.zeros((T, 128)), "slots": torch.zeros(T, dtype=i64),
        "kp": torch.zeros((3, 1, 8704), dtype=u8), "vp": torch.zeros((3, 1, 8704), dtype=u8),
        "ip": torch.zeros((3, 8704), dtype=u8), "fp8": torch.zeros((3, 16384), dtype=u8),
        "iq": torch.zeros((T, 128), dtype=bf), "q": torch.zeros((T, H, 128), dtype=bf),
        "bt": torch.zeros((B, 3), dtype=i32), "sl": torch.ones(B, dtype=i32),
        "scores": torch.zeros((T, ld), dtype=f32), "idx": torch.zeros((T, k), dtype=i32),
        "out": torch.zeros((T, H, 128), dtype=f32), "ws": torch.zeros(64, dtype=u8),
    }


def _calls(a, m):
    return {
        "mx4_insert": lambda: m.mx4_insert(a["k"], a["v"], a["idx_k"], a["slots"], a["kp"],
                                           a["vp"], a["ip"]),
        "index_score": lambda: m.index_score(a["iq"], 1, a["ip"], a["bt"], a["sl"], a["scores"]),
        "index_score_fp8": lambda: m.index_score_fp8(a["iq"], 1, a["fp8"], a["bt"], a["sl"], 0.5,
                                                     a["scores"]),
        "fp8_index_insert": lambda: m.fp8_index_insert(a["idx_k"], a["slots"], 1.0, a["fp8"]),
        "topk_select": lambda: m.topk_select(a["scores"], a["sl"], 1, a["idx"].shape[1], a["idx"],
                                             a["ws"]),
        "sparse_paged_decode": lambda: m.sparse_paged_decode(a["q"], 1, a["kp"], a["vp"], a["bt"],
                                                             a["sl"], a["idx"], 0.1, a["out"],
                                                             a["ws"]),
        "sparse_paged_decode_noalloc": lambda: m.sparse_paged_decode_noalloc(
            a["q"], 1, a["kp"], a["vp"], a["bt"], a["sl"], a["idx"], 0.1, a["out"]),
    }


def test_bindings_with_consistent_host_tensors_stop_at_the_device_check(lib):
    import mxfp4_sparse_paged_gb300 as m
    for name, call in _calls(_cpu_args(), m).items():
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


@pytest.mark.parametrize("bad", [
    ("mx4_insert", "v", (4, 2, 128)), ("mx4_insert", "idx_k", (3, 128)),
    ("mx4_insert", "slots", (5,)), ("mx4_insert", "k", (4, 2, 128)),
    ("index_score", "iq", (3, 128)), ("index_score", "bt", (3, 3)),
    ("index_score", "scores", (3, 300)), ("index_score_fp8", "bt", (2, 3)),
    ("index_score_fp8", "iq", (4, 64)), ("fp8_index_insert", "slots", (3,)),
    ("topk_select", "scores", (2, 300)), ("topk_select", "idx", (3, 8)),
    ("sparse_paged_decode", "out", (4, 8, 128)), ("sparse_paged_decode", "idx", (3, 8)),
    ("sparse_paged_decode", "bt", (3, 3)), ("sparse_paged_decode", "q", (5, 16, 128)),
    ("sparse_paged_decode_noalloc", "out", (4, 16, 64)),
])
def test_bindings_refuse_inconsistent_shapes(lib, bad):
    # A table shorter than the batch, an output with too few rows or a K/V head count
    # the pages do not have would let a kernel read or write past the buffer.
    import torch
    import mxfp4_sparse_paged_gb300 as m
    call, key, shape = bad
    a = _cpu_args()
    a[key] = torch.zeros(shape, dtype=a[key].dtype)
    with pytest.raises(ValueError) as ei:
        _calls(a, m)[call]()
    assert "CUDA tensor" not in str(ei.value), str(ei.value)


def test_decode_step_host_validation_and_layout(lib):
    # The whole-step call refuses NULL buffers and a short staging buffer before it
    # enqueues anything; its packed input layout is q | iq | k | v | idx_k | slots,
    # each section 256-byte aligned.
    import mxfp4_sparse_paged_gb300 as m
    L = m._load()
    offs, nbytes = m.mx4_decode_step_input_layout(256, 256)
    sizes = [256 * 16 * 128 * 2, 256 * 128 * 2, 256 * 512, 256 * 512, 256 * 512, 256 * 8]
    want, o = [], 0
    for sz in sizes:
        want.append(o)
        o += (sz + 255) // 256 * 256
    assert offs == want and nbytes == o
    assert m.mx4_decode_step_input_layout(4, 0)[0][2:] == [4 * 16 * 128 * 2 + 1024] * 4
    f = ctypes.c_float(0.1)
    args = [None, 0, None, 0, None, None, 8704, 8704, None, 8704, 1, None, 2, 1, None, 1, 16, f,
            None, 64, None, None, 0, None, 0, None, None, None]
    assert L.mx4_decode_step(*args) == -1 and "NULL" in _err(m)
    buf = ctypes.create_string_buffer(64)
    args[0] = args[26] = ctypes.cast(buf, ctypes.c_void_p)
    args[2] = ctypes.c_void_p(4096)
    args[3] = 16  # staging far below the packed inputs
    assert L.mx4_decode_step(*args) == -3 and "staging" in _err(m)


def test_decode_steps_host_validation(lib):
    # The multi-step call refuses a negative step count, a missing copy stream or two
    # equal streams and
    # a staging buffer below two input sets before it enqueues anything; zero steps
    # is a no-op.
    import mxfp4_sparse_paged_gb300 as m
    L = m._load()
    f = ctypes.c_float(0.1)
    buf = ctypes.create_string_buffer(64)
    host = ctypes.cast(buf, ctypes.c_void_p)
    s1, s2, s3 = ctypes.c_void_p(16), ctypes.c_void_p(32), ctypes.c_void_p(48)
    _, nbytes = m.mx4_decode_step_input_layout(2, 0)
    args = [1, host, 0, 0, ctypes.c_void_p(4096), 2 * nbytes - 256, None, None, 8704, 8704,
            None, 8704, 1, None, 2, 1, None, 1, 16, f, None, 64, None, None, 0, None, 0,
            ctypes.c_void_p(8192), host, 0, s1, s2, s3]
    a = list(args); a[0] = -1
    assert L.mx4_decode_steps(*a) == -1 and "n_steps" in _err(m)
    a = list(args); a[0] = 0
    assert L.mx4_decode_steps(*a) == 0
    a = list(args); a[32] = s2
    assert L.mx4_decode_steps(*a) == -1 and "streams" in _err(m)
    a = list(args); a[31] = None
    assert L.mx4_decode_steps(*a) == -1 and "streams" in _err(m)
    a = list(args); a[30] = None   # the compute stream may be the default one
    assert L.mx4_decode_steps(*a) == -3 and "staging" in _err(m)
    assert L.mx4_decode_steps(*args) == -3 and "staging" in _err(m)

"""sparse_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a host framework that owns all device memory and hands
an extension only the operation's inputs and outputs, or a C or
foreign-language runtime with no device allocator).  It keeps the run
workspace in the library's own fixed device array instead of a caller buffer.

Checked through the C ABI against sparse_paged_decode (caller workspace) on the
same inputs, on two calls in a row, within the attention tolerance of the
other parity tests.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import mxfp4_sparse_paged_gb300 as m
from mxfp4_sparse_paged_gb300 import workloads as W
from mxfp4_sparse_paged_gb300.step import DecodeStep, PagedCaches, step_inputs_host

ATTN_ABS = 2e-3

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def test_noalloc_matches_workspace_entry_point_twice():
    wl = W.make(1)  # 8 sequences x 8192 tokens, top-2048
    caches = PagedCaches(wl.num_pages, device="cuda")
    caches.fill(wl)
    step = DecodeStep(wl, caches, device="cuda")
    step.load_inputs(step_inputs_host(wl))
    step.run()
    m.mx4_check_status()
    ref = step.out.clone()
    assert m.sparse_paged_decode_workspace(wl.T, wl.k) <= m.NOALLOC_SCRATCH_BYTES
    for call in range(2):
        out = torch.full_like(step.out, float("nan"))
        m.sparse_paged_decode_noalloc(step.q, wl.q, caches.k_pages, caches.v_pages,
                                      step.block_table, step.seq_lens, step.topk_idx, step.scale,
                                      out)
        m.mx4_check_status()
        err = float((out - ref).abs().max())
        assert np.isfinite(err) and err <= ATTN_ABS, f"call {call}: max-abs {err}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # (8 warps per SM + T) partial records of 8320 bytes above 32 MiB: refused before
    # any launch
    T, k = 4096, 16
    assert m.sparse_paged_decode_workspace(T, k) > m.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((T, 16, 128), dtype=torch.bfloat16, device="cuda")
    pages = torch.zeros((1, 1, 8704), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((T, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones(T, dtype=torch.int32, device="cuda")
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros((T, 16, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(m.Mx4Error) as ei:
        m.sparse_paged_decode_noalloc(q, 1, pages, pages.clone(), bt, sl, idx, 0.1, out)
    assert ei.value.code == -3 and "scratch" in str(ei.value)

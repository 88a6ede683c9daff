"""The allocation-free split-KV decode entry point, fa_fwd_varlen_noalloc.

It serves callers that cannot allocate device memory when they run
attention -- custom ops handed only their inputs and outputs, serving loops
whose memory is fixed at start-up, request paths that must not call
cudaMalloc -- by keeping the split partials in the library's own static
device scratch array.  These tests call it through the C ABI and check it
against fa_fwd_varlen with a caller-provided workspace, on two calls in a row
(the second on different inputs, so stale partials left in the shared scratch
by the first call must not leak into it).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import fa_inputs as fi
import flashattention_forward_gb300 as fa
from flashattention_forward_gb300 import build as fa_build
from fa_testlib import LSE_TOL, OUT_TOL, compare, host, run_gpu, to_device


def _noalloc(p, t, splits):
    out = torch.empty((p.total_q, p.hq, p.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.hq, p.total_q), dtype=torch.float32, device="cuda")
    return fa.fwd_varlen_noalloc(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], out, lse,
                                 max_seqlen_q=p.max_seqlen_q, max_seqlen_k=p.max_seqlen_k,
                                 total_k=p.total_k, block_table=t.get("bt"), page_size=p.page_size,
                                 softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
                                 num_splits=splits)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa_build.build()
    first = fi.config3()                                   # 64 seqs, paged, GQA 32/8, 16 splits
    second = fi.make_problem([2] * 9, [40, 700, 1500, 64, 65, 3000, 1, 900, 2222], hq=8, hkv=2, dk=128,
                             seed=21, page_size=32, spare_pages=4, causal=True)
    for p, splits in ((first, 0), (second, 5)):
        t = to_device(p)
        want = splits or fa.default_splits(p.num_seqs, p.max_seqlen_q, p.max_seqlen_k, p.hq, p.hkv, p.page_size,
                                           p.total_k)
        assert want > 1
        ref_o, ref_l = host(*run_gpu(p, t, num_splits=want))     # existing entry, torch workspace
        got_o, got_l = host(*_noalloc(p, t, splits))
        compare(got_o, got_l, ref_o, ref_l, OUT_TOL, LSE_TOL)
    assert fa.device_error() == 0


def test_noalloc_rejects_oversized_scratch_before_launch():
    """A request whose partials exceed the static scratch fails on the host."""
    fa_build.build()
    L = fa.lib()
    T, Hq, D = 4096, 16, 128                     # 4096 rows * 16 heads * 128 * 4 B * 64 splits >> 32 MiB

    def desc(dt, shape):
        d = fa.Tensor()
        d.data, d.dtype, d.ndim = 1 << 20, dt, len(shape)
        s = 1
        for i in reversed(range(len(shape))):
            d.shape[i], d.stride[i] = shape[i], s
            s *= shape[i]
        return d

    q = desc(fa.FA_BF16, [T, Hq, D])
    k = desc(fa.FA_BF16, [T * 64, 1, D])
    launch = fa.Launch(num_seqs=T, max_seqlen_q=1, max_seqlen_k=64 * 512, num_splits=64, total_q=T,
                       total_k=T * 64)
    st = L.fa_fwd_varlen_noalloc(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), None, None, None, None,
                                 None, None, None, 0.1, 0, 0, None, None, None, 0, ctypes.byref(launch), None)
    assert st == fa.FA_ERR_UNSUPPORTED
    assert b"exceeds the static" in L.fa_last_error()

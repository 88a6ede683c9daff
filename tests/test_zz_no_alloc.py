"""The allocation-free split-KV decode entry point, fa_fwd_varlen_noalloc.

It serves callers that cannot allocate device memory when they run
attention -- custom ops handed only their inputs and outputs, serving loops
whose memory is fixed at start-up, request paths that must not call
cudaMalloc -- by keeping the split partials (and a Q add's per-key terms) in
the library's own static device scratch array.  These tests call it through
the C ABI on several calls in a row, each on different inputs (so stale
contents left in the shared scratch by one call must not leak into the
next), and check every result two ways: bit for bit against fa_fwd_varlen
with a caller-provided workspace (the same kernels run), and against the
fp64 oracle at the contract's tolerances.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import fa_inputs as fi
import flashattention_forward_gb300 as fa
import oracle
from flashattention_forward_gb300 import build as fa_build
from fa_testlib import LSE_TOL, OUT_TOL, compare, host, run_gpu, to_device


def _noalloc(p, t, splits):
    out = torch.empty((p.total_q, p.hq, p.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.hq, p.total_q), dtype=torch.float32, device="cuda")
    return fa.fwd_varlen_noalloc(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], out, lse,
                                 max_seqlen_q=p.max_seqlen_q, max_seqlen_k=p.max_seqlen_k,
                                 total_k=p.total_k, block_table=t.get("bt"), page_size=p.page_size,
                                 k_scale=t.get("k_scale"), v_scale=t.get("v_scale"),
                                 softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
                                 score_mod=p.mod_kind, alibi_slope=p.alibi_slope, softcap=p.softcap,
                                 block_mask=t.get("bm"), num_splits=splits, prologue=p.prologue)


def _calls():
    """(problem, num_splits) pairs run back to back; 0 = the library's default."""
    lens9 = [40, 700, 1500, 64, 65, 3000, 1, 900, 2222]
    return [
        (fi.config3(), 0),                                              # 64 seqs, paged, GQA 32/8
        (fi.make_problem([2] * 9, lens9, hq=8, hkv=2, dk=128, seed=21, page_size=32, spare_pages=4,
                         causal=True), 5),
        (fi.make_problem([1] * 6, [90, 1000, 4000, 17, 2500, 640], hq=16, hkv=4, dk=128, seed=22, page_size=64,
                         spare_pages=3, kv_dtype="e4m3"), 3),           # e4m3 KV, per-token scales
        (fi.make_problem([1] * 5, [300, 2000, 129, 4000, 1000], hq=8, hkv=2, dk=64, seed=23, page_size=16,
                         spare_pages=2, mod="softcap", softcap=6.0, window=700), 4),
        (fi.make_problem([1] * 4, [500, 3000, 1200, 260], hq=8, hkv=8, dk=128, seed=24,
                         block_mask_density=0.6, mod="alibi", alibi_slope=0.02), 2),   # packed, block mask
        (fi.make_problem([1] * 4, [700, 64, 2049, 1], hq=8, hkv=2, dk=128, seed=25, page_size=16, spare_pages=2,
                         kv_dtype="int8").replace(prologue={"q": [("add", 0.3)], "k": [("sub", 0.1)],
                                                            "v": [("mul", 0.5)]}), 3),
    ]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_and_oracle_on_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa_build.build()
    for p, splits in _calls():
        t = to_device(p)
        want = splits or fa.default_splits(p.num_seqs, p.max_seqlen_q, p.max_seqlen_k, p.hq, p.hkv, p.page_size,
                                           p.total_k)
        assert want > 1
        ref_o, ref_l = host(*run_gpu(p, t, num_splits=want))     # existing entry, torch workspace
        got_o, got_l = host(*_noalloc(p, t, splits))
        assert np.array_equal(got_o, ref_o), p.name
        assert np.array_equal(got_l, ref_l), p.name
        ro, rl = oracle.forward(p)
        compare(got_o, got_l, ro, rl, OUT_TOL, LSE_TOL)
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


def test_noalloc_checks_rows_against_total_q_before_sizing():
    """q.shape[0] must equal launch->total_q: the scratch is sized from q's
    rows, so an understated total_q cannot slip past the size check."""
    fa_build.build()
    L = fa.lib()
    q = fa.Tensor()
    q.data, q.dtype, q.ndim = 1 << 20, fa.FA_BF16, 3
    for i, (n, st) in enumerate(((64, 32 * 128), (32, 128), (128, 1))):
        q.shape[i], q.stride[i] = n, st
    k = fa.Tensor()
    k.data, k.dtype, k.ndim = 1 << 21, fa.FA_BF16, 3
    for i, (n, st) in enumerate(((4096, 8 * 128), (8, 128), (128, 1))):
        k.shape[i], k.stride[i] = n, st
    launch = fa.Launch(num_seqs=64, max_seqlen_q=1, max_seqlen_k=64, num_splits=4, total_q=1, total_k=4096)
    st = L.fa_fwd_varlen_noalloc(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), None, None, None, None,
                                 None, None, None, 0.1, 0, 0, None, None, None, 0, ctypes.byref(launch), None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert b"total_q" in L.fa_last_error()

"""GPU parity for paged caches whose pages hold fewer than 16 keys (1, 2, 4, 8):
the K/V rows are gathered one key at a time with 16-byte copies instead of TMA
boxes, on every path that reads a paged cache -- the ping-pong prefill (Dk 64
and 128), the chunked-ring prefill (Dk 192 bf16, e4m3 and int8 caches) and the
split-KV decode (bf16 and byte caches).

Two checks per case: the fp64 oracle within the contract's tolerances, and
bit-identity with the same tokens stored in pages of 16 keys (the draws of
Q, K and V come before the page permutation, so only the page layout
differs): the gather writes the same bytes into the same shared-memory layout
as the boxes, so every later step sees identical operands.
"""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import compare, compare_units, host, run_gpu, sample_units

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from flashattention_forward_gb300 import build
    build.build()
    yield
    import flashattention_forward_gb300 as fa
    assert fa.device_error() == 0


CASES = {
    "d128_noncausal": dict(lens_q=[70, 300, 1, 129], lens_k=[200, 300, 1000, 129], hq=8, hkv=2, dk=128),
    "d128_causal": dict(lens_q=[70, 300, 1, 129], lens_k=[200, 300, 1000, 129], hq=8, hkv=2, dk=128, causal=True),
    "d64_window_gqa": dict(lens_q=[200, 3], lens_k=[260, 500], hq=8, hkv=1, dk=64, causal=True, window=90),
    "d192_bf16_causal": dict(lens_q=[300, 129, 1], lens_k=[700, 129, 300], hq=4, hkv=2, dk=192, dv=128,
                             causal=True),
    "e4m3_d128": dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, hkv=2, dk=128, kv_dtype="e4m3"),
    "e4m3_d192_causal": dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=1, dk=192, dv=128, kv_dtype="e4m3",
                             causal=True),
    "int8_d128_causal": dict(lens_q=[200, 64], lens_k=[333, 64], hq=4, hkv=2, dk=128, kv_dtype="int8", causal=True),
    "alibi_d128": dict(lens_q=[150], lens_k=[400], hq=4, hkv=4, dk=128, mod="alibi", alibi_slope=0.05),
}


def _problem(name, page_size):
    kw = dict(CASES[name])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k")
    return fi.make_problem(lens_q, lens_k, seed=300 + sorted(CASES).index(name), page_size=page_size,
                           spare_pages=7, **kw)


@pytest.mark.parametrize("page_size", [1, 2, 4, 8])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_small_pages(name, page_size):
    p = _problem(name, page_size)
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)
    o16, l16 = host(*run_gpu(_problem(name, 16)))
    assert np.array_equal(o, o16) and np.array_equal(l, l16)


DECODE = {
    "bf16_d128": dict(hq=8, hkv=2, dk=128),
    "bf16_d64_rows2": dict(hq=8, hkv=2, dk=64, sq=2),
    "e4m3_d128": dict(hq=8, hkv=2, dk=128, kv_dtype="e4m3"),
    "e4m3_d128_rows8": dict(hq=8, hkv=2, dk=128, kv_dtype="e4m3", sq=2),
    "int8_d128_rows16": dict(hq=8, hkv=2, dk=128, kv_dtype="int8", sq=4),
    "int8_d64": dict(hq=4, hkv=4, dk=64, kv_dtype="int8"),
}


def _decode_problem(name, page_size):
    kw = dict(DECODE[name])
    sq = kw.pop("sq", 1)
    lens_k = [1, 63, 64, 65, 700, 2049]
    return fi.make_problem([sq] * len(lens_k), lens_k, seed=400 + sorted(DECODE).index(name), page_size=page_size,
                           spare_pages=9, causal=sq > 1, **kw)


@pytest.mark.parametrize("page_size", [1, 4, 8])
@pytest.mark.parametrize("name", sorted(DECODE))
def test_decode_small_pages(name, page_size):
    p = _decode_problem(name, page_size)
    o, l = host(*run_gpu(p, num_splits=3))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)
    o16, l16 = host(*run_gpu(_decode_problem(name, 16), num_splits=3))
    assert np.array_equal(o, o16) and np.array_equal(l, l16)


def test_config4_geometry_with_one_key_pages():
    """The paged e4m3 Q/K 192, V/O 128 causal workload (16 sequences of
    U{1..4096} tokens, H 16) stored one key per page -- the lookup-bound
    layout -- on sampled rows."""
    p = fi.config4()
    p1 = fi.make_problem([int(x) for x in p.seqlens_q], [int(x) for x in p.seqlens_k], hq=16, hkv=16, dk=192,
                         dv=128, seed=1, page_size=1, spare_pages=64, kv_dtype="e4m3", causal=True,
                         name="config4_page1")
    o, l = host(*run_gpu(p1))
    units = sample_units(p1, 2000, seed=9)
    ro, rl = oracle.forward(p1, units=units)
    compare_units(o, l, units, ro, rl)

"""GPU parity of the split-KV decode on byte caches (e4m3 and int8 with
per-token scales) against the fp64 oracle.

The config-3 geometry (64 sequences, Sq = 1, Sk U{512..8192}, Hq 32, Hkv 8,
D 128, page 16, shuffled and NaN-poisoned pages) with e4m3 and int8 caches,
for several split counts, plus packed caches, D = 64, windows and several query
rows per sequence.  Tolerances are the contract's (|dout| <= 1e-2,
|dLSE| <= 1e-3): the kernel reads the cached values exactly as f16 and keeps
the scales in fp32; only Q (per-row power-of-two factor) and P * v_scale are
rounded to f16.
"""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import compare, host, run_gpu

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


def config3_bytes(kv_dtype, seed=0):
    rng = np.random.default_rng(seed)
    lens_k = [int(x) for x in rng.integers(512, 8193, size=64)]
    return fi.make_problem([1] * 64, lens_k, hq=32, hkv=8, dk=128, seed=seed + 1, page_size=16,
                           spare_pages=64, max_pages=512, kv_dtype=kv_dtype, name=f"decode_{kv_dtype}")


@pytest.mark.parametrize("kv_dtype", ["e4m3", "int8"])
@pytest.mark.parametrize("splits", [1, 4, None])
def test_config3_geometry_byte_cache(kv_dtype, splits):
    p = config3_bytes(kv_dtype)
    o, l = host(*run_gpu(p, num_splits=splits))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


CASES = {
    "packed_e4m3_d128": dict(lens_q=[1, 1, 1], lens_k=[700, 64, 3000], hq=8, hkv=2, dk=128, kv_dtype="e4m3"),
    "packed_int8_d64": dict(lens_q=[1, 1], lens_k=[129, 2000], hq=4, hkv=4, dk=64, kv_dtype="int8"),
    "paged_e4m3_d64_p64": dict(lens_q=[1, 1, 1, 1], lens_k=[1, 65, 640, 1500], hq=16, hkv=4, dk=64,
                               kv_dtype="e4m3", page_size=64, spare_pages=5),
    "paged_e4m3_window_causal": dict(lens_q=[2, 4], lens_k=[900, 1200], hq=8, hkv=2, dk=128, kv_dtype="e4m3",
                                     page_size=16, spare_pages=3, causal=True, window=100),
    "paged_int8_rows4_causal": dict(lens_q=[4, 2], lens_k=[333, 1024], hq=8, hkv=2, dk=128, kv_dtype="int8",
                                    page_size=32, spare_pages=2, causal=True),
    "paged_e4m3_p1024": dict(lens_q=[1, 1], lens_k=[2500, 100], hq=8, hkv=8, dk=128, kv_dtype="e4m3",
                             page_size=1024, spare_pages=1),
    # exactly 8 query rows per kv head (2 tokens x 4 heads) and fewer: the transposed P V form
    "paged_e4m3_rows8_causal": dict(lens_q=[2, 1, 2], lens_k=[500, 77, 1300], hq=8, hkv=2, dk=128,
                                    kv_dtype="e4m3", page_size=16, spare_pages=4, causal=True),
    "paged_int8_rows8_alibi": dict(lens_q=[2, 2], lens_k=[640, 129], hq=16, hkv=4, dk=128, kv_dtype="int8",
                                   page_size=64, spare_pages=2, causal=True, mod="alibi"),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("splits", [2, 7])
def test_byte_cache_decode_edge_cases(name, splits):
    kw = dict(CASES[name])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k")
    p = fi.make_problem(lens_q, lens_k, seed=900 + sorted(CASES).index(name), **kw)
    o, l = host(*run_gpu(p, num_splits=splits))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_byte_cache_single_key_rows_are_the_scaled_values():
    """Sk = 1: P = 1, so out = v * v_scale; the kernel rounds P * v_scale to
    f16 (2^-11 relative) and the output to bf16, so out is within one bf16
    ulp of the oracle's v * v_scale."""
    p = fi.make_problem([1, 1, 1], [1, 1, 1], hq=4, hkv=2, dk=128, seed=31, kv_dtype="e4m3", page_size=16,
                        spare_pages=2)
    o, l = host(*run_gpu(p, num_splits=2))
    ro, rl = oracle.forward(p)
    assert np.all(np.abs(o - ro) <= 2.0 ** -8 * np.abs(ro) + 1e-30)
    compare(o, l, ro, rl)

"""GPU parity of byte caches (e4m3, int8) in the vectorized 5-D page layouts,
K [N_pg, Hkv, Dk/16, P_s, 16] and V [N_pg, Hkv, P_s/16, Dv, 16] (FlyDSL PR
#1066: paged FP8 with vectorized-5D KV; the review's permutes (0, 3, 1, 2, 4)
and (0, 2, 4, 1, 3) recover the token-major pages).  The same tokens in the
token-major pages must give bit-identical results, and both the oracle's
within the contract's tolerances."""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import compare, host, run_gpu, to_device

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


def vec5_tensors(p):
    t = to_device(p)
    k5, v5 = fi.vectorize_pages(p.k.view(np.uint8), p.v.view(np.uint8))
    kvt = torch.int8 if p.kv_dtype == "int8" else torch.float8_e4m3fn
    t["k"] = torch.from_numpy(k5).view(kvt).cuda()
    t["v"] = torch.from_numpy(v5).view(kvt).cuda()
    return t


def check_both(p, **kw):
    o1, l1 = host(*run_gpu(p, **kw))
    o5, l5 = host(*run_gpu(p, vec5_tensors(p), **kw))
    assert np.array_equal(o5, o1) and np.array_equal(l5, l1)
    compare(o5, l5, *oracle.forward(p))


CASES = [
    dict(lens_q=[300, 129, 1], lens_k=[700, 129, 300], hq=4, hkv=2, dk=192, dv=128, page_size=64, causal=True),
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, dk=128, page_size=16, spare_pages=4),
    dict(lens_q=[200, 64, 3], lens_k=[260, 64, 500], hq=8, hkv=1, dk=64, page_size=32, causal=True, window=90),
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128, page_size=1024),
    dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, dk=128, page_size=128, mod="softcap", softcap=5.0),
    dict(lens_q=[200, 330], lens_k=[200, 330], hq=4, dk=128, page_size=64, block_mask_density=0.5),
]


@pytest.mark.parametrize("kv_dtype", ["e4m3", "int8"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_vec5_prefill_bit_identical_to_token_major(case, kv_dtype):
    kw = dict(CASES[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k")
    check_both(fi.make_problem(lens_q, lens_k, seed=700 + case, kv_dtype=kv_dtype, **kw))


@pytest.mark.parametrize("kv_dtype", ["e4m3", "int8"])
@pytest.mark.parametrize("page_size,dk", [(16, 128), (64, 64), (1024, 128)])
def test_vec5_split_kv_decode_bit_identical_to_token_major(page_size, dk, kv_dtype):
    lens_k = [1, 63, 700, 2049, 16, 1025]
    p = fi.make_problem([1] * 6, lens_k, hq=8, hkv=2, dk=dk, seed=710, page_size=page_size, spare_pages=3,
                        kv_dtype=kv_dtype)
    check_both(p, num_splits=3)


def test_vec5_config4_geometry():
    """Config 4 (16 sequences of U{1..4096}, H 16, Q/K 192, V/O 128, e4m3,
    page 64, causal) from 5-D pages."""
    check_both(fi.config4())

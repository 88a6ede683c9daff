"""GPU parity of the folded prologue (element maps x -> mul * x + add on Q, K
and V as read; fkl_python PR #7, prologue-fusion commit) against the fp64
oracle, which applies the maps to the values literally.  The kernels fold
them: q_mul * k_mul into the score scale, k_add into the LSE, v_mul and v_add
into the output normalisation.  Tolerances are the contract's (|dout| <=
1e-2, |dLSE| <= 1e-3), absolute, so the maps keep scaled scores of the
order of the plain runs' and |v_mul| <= 1: bf16 outputs of magnitude 2 or
more would round by up to 2^-7 alone.
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


MAPS = {
    "all": (0.75, 0.0, -1.5, 0.3, -0.75, 0.25),     # negative scale product: the general score path
    "scale_only": (1.25, 0.0, 0.8, 0.0, 1.0, 0.0),
    "shift_v": (1.0, 0.0, 1.0, -0.4, 0.5, 1.0),
}

CASES = {
    "d128_causal": dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, dk=128, causal=True),
    "d64_paged_gqa_window": dict(lens_q=[200, 3], lens_k=[260, 500], hq=8, hkv=2, dk=64, causal=True,
                                 window=90, page_size=32, spare_pages=3),
    "d192_bf16": dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128, causal=True),
    "e4m3_d128": dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, hkv=2, dk=128, kv_dtype="e4m3",
                      page_size=64, spare_pages=2),
    "alibi_d128": dict(lens_q=[150, 64], lens_k=[400, 64], hq=4, dk=128, mod="alibi", alibi_slope=0.05),
    "blocksparse_d128": dict(lens_q=[300, 129], lens_k=[330, 400], hq=4, hkv=2, dk=128, block_mask_density=0.5),
}


@pytest.mark.parametrize("maps", sorted(MAPS))
@pytest.mark.parametrize("name", sorted(CASES))
def test_prologue_prefill(name, maps):
    kw = dict(CASES[name])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k")
    p = fi.make_problem(lens_q, lens_k, seed=600 + sorted(CASES).index(name), **kw).replace(prologue=MAPS[maps])
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_prologue_softcap_scale_only():
    """The soft-cap takes the scale maps (k_add would not cancel under it)."""
    p = fi.make_problem([200, 64], [300, 64], hq=4, dk=128, seed=620, mod="softcap", softcap=5.0,
                        causal=True).replace(prologue=(1.5, 0.0, 0.5, 0.0, 0.75, 0.5))
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("maps", sorted(MAPS))
def test_prologue_split_kv_decode(kv_dtype, maps):
    lens_k = [1, 63, 700, 2049]
    p = fi.make_problem([1] * 4, lens_k, hq=8, hkv=2, dk=128, seed=630, page_size=16, spare_pages=4,
                        kv_dtype=kv_dtype).replace(prologue=MAPS[maps])
    o, l = host(*run_gpu(p, num_splits=3))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_prologue_config2_lengths():
    """The packed varlen workload of the headline step (8 sequences of
    U{0..2048} tokens, H 16, D 128) with every foldable map."""
    p = fi.config2(causal=False).replace(prologue=MAPS["all"])
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_identity_prologue_is_bit_identical_to_none():
    p = fi.make_problem([300, 129], [300, 400], hq=4, dk=128, seed=640, causal=True)
    o0, l0 = host(*run_gpu(p))
    o1, l1 = host(*run_gpu(p.replace(prologue=(1.0, 0.0, 1.0, 0.0, 1.0, 0.0))))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)

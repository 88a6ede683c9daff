"""GPU parity of the int8 KV path (per-token scales, value = int8 * scale;
the converter-warp kernel with f16 operands) against the fp64 oracle."""
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


def check(p, **kw):
    o, l = host(*run_gpu(p, **kw))
    ro, rl = oracle.forward(p)
    return compare(o, l, ro, rl)


I8_CASES = [
    dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, hkv=4, dk=192, dv=128, page_size=64, causal=True),
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, dk=128, page_size=16, spare_pages=4),
    dict(lens_q=[200, 64, 3], lens_k=[260, 64, 500], hq=8, hkv=1, dk=64, page_size=32, causal=True, window=90),
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128),                        # packed
    dict(lens_q=[130, 260], lens_k=[130, 260], hq=4, dk=128, page_size=128, mod="alibi"),
    dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, dk=128, page_size=64, mod="softcap", softcap=5.0),
    dict(lens_q=[0, 5, 0], lens_k=[7, 0, 0], hq=2, dk=64, page_size=16),                             # empty rows
    dict(lens_q=[200, 330], lens_k=[200, 330], hq=4, dk=128, page_size=1024, block_mask_density=0.5),
]


@pytest.mark.parametrize("case", range(len(I8_CASES)))
def test_int8_cases(case):
    kw = dict(I8_CASES[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    check(fi.make_problem(lens_q, lens_k, seed=400 + case, kv_dtype="int8", **kw))


def test_int8_single_key_all_values_bit_exact():
    """V holds every int8 value, scales 1, one visible key per row: out must
    equal the value exactly (exact int8 -> f16 operand)."""
    p = fi.make_problem([64, 64], [64, 64], hq=4, hkv=2, dk=128, dv=128, seed=9, kv_dtype="int8",
                        page_size=16, causal=True, window=1)
    vals = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    v = p.v.copy()
    n = v.shape[0] * v.shape[1] * v.shape[2]
    v.reshape(n, -1)[:] = np.resize(vals, (n, v.shape[-1]))
    p = p.replace(v=v, v_scale=np.where(np.isnan(p.v_scale), np.nan, np.float32(1.0)).astype(np.float32))
    o, _ = run_gpu(p)
    torch.cuda.synchronize()
    got = o.view(torch.int16).cpu().numpy().view(np.uint16)
    ro, _ = oracle.forward(p)
    assert np.array_equal(got, fi.bf16_bits(ro.astype(np.float32)))


def test_int8_config4_shape_sampled():
    """The config-4 geometry (16 ragged sequences, Q/K 192, V/O 128, page 64,
    causal) with an int8 cache."""
    p = fi.config4().replace()
    p = fi.make_problem(list(np.diff(p.cu_seqlens_q)), hq=16, hkv=16, dk=192, dv=128, seed=1, page_size=64,
                        kv_dtype="int8", causal=True, name="config4_int8")
    o, l = host(*run_gpu(p))
    units = sample_units(p, 2500, seed=4)
    ro, rl = oracle.forward(p, units=units)
    compare_units(o, l, units, ro, rl)

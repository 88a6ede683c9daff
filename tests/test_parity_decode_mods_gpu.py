"""GPU parity of the split-KV decode with score mods and block masks (ALiBi,
soft-cap, 128 x 128 block sparsity; fkl_python PR #7, flex commit) against
the fp64 oracle: bf16 and byte caches, GQA, several query rows per
sequence, windows.  Tolerances are the contract's (|dout| <= 1e-2,
|dLSE| <= 1e-3).
"""
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


LENS_K = [1, 63, 200, 700, 2049, 3000]

MODS = {
    "alibi": dict(mod="alibi", alibi_slope=0.05),
    "softcap": dict(mod="softcap", softcap=5.0),
    "softcap_tight": dict(mod="softcap", softcap=0.7, softmax_scale=0.5),
    "blocksparse": dict(block_mask_density=0.5),
    "alibi_blocksparse_window": dict(mod="alibi", alibi_slope=0.02, block_mask_density=0.6, window=900),
}


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3", "int8"])
@pytest.mark.parametrize("name", sorted(MODS))
def test_decode_with_mods(name, kv_dtype):
    p = fi.make_problem([1] * len(LENS_K), LENS_K, hq=8, hkv=2, dk=128, seed=700 + sorted(MODS).index(name),
                        page_size=16, spare_pages=5, kv_dtype=kv_dtype, **MODS[name])
    o, l = host(*run_gpu(p, num_splits=3))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


@pytest.mark.parametrize("name", ["alibi", "softcap", "blocksparse"])
def test_decode_with_mods_rows_and_causal(name):
    """Two query rows per sequence (causal, bottom-right) and a group of 4:
    eight rows per CTA."""
    p = fi.make_problem([2] * 4, [70, 300, 1000, 2500], hq=8, hkv=2, dk=64, seed=720, page_size=32,
                        spare_pages=3, causal=True, **MODS[name])
    o, l = host(*run_gpu(p, num_splits=4))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_default_splits_take_mods():
    """Decode shapes with a score mod now take the split-KV kernel by default."""
    import flashattention_forward_gb300 as fa
    p = fi.make_problem([1] * 8, [4000] * 8, hq=32, hkv=8, dk=128, seed=730, page_size=16, spare_pages=4,
                        mod="softcap", softcap=5.0)
    assert fa.default_splits(p.num_seqs, 1, p.max_seqlen_k, 32, 8, 16, p.total_k) > 1
    o, l = host(*run_gpu(p, num_splits=None))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)

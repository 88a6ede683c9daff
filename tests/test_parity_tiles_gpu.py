"""The bf16 ping-pong prefill with one 128-row query tile per CTA (two CTAs
per SM) and with two: each form forced for a whole process through
FA_GB300_PREFILL_VARIANT (read once per process), on ragged, causal,
windowed, masked and score-modded cases.  A query tile walks the same key
tiles in the same order either way, so the two forms must agree bit for bit,
and both with the fp64 oracle -- except under ALiBi, where the one-tile form
adds the bias's linear part inside the QK contraction (other roundings):
there both forms are held to the oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import compare

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CASES = [
    dict(lens_q=[1, 127, 128, 129, 300], hq=4, dk=64, causal=True),
    dict(lens_q=[5, 0, 77, 256, 700], lens_k=[300, 0, 77, 500, 700], hq=4, hkv=2, dk=128, causal=True),
    dict(lens_q=[200, 64], lens_k=[100, 10], hq=2, dk=128, causal=True),
    dict(lens_q=[130, 900], lens_k=[400, 900], hq=8, hkv=1, dk=128, causal=True, window=100),
    dict(lens_q=[300, 513], lens_k=[300, 600], hq=4, dk=128, mod="alibi", alibi_slope=0.0625, causal=True),
    dict(lens_q=[300, 700], lens_k=[500, 700], hq=4, dk=64, mod="alibi", alibi_slope=0.0625),    # straddling tiles
    dict(lens_q=[300, 640], lens_k=[300, 700], hq=4, dk=128, mod="softcap", softcap=5.0),
    dict(lens_q=[300, 650], lens_k=[330, 650], hq=4, hkv=2, dk=128, block_mask_density=0.5),
    dict(lens_q=[70, 300, 1, 400], lens_k=[200, 300, 1000, 400], hq=8, hkv=2, dk=128, page_size=64,
         spare_pages=5, causal=True),
]

CHILD = r"""
import sys, numpy as np
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import fa_inputs as fi
from fa_testlib import host, run_gpu
import test_parity_tiles_gpu as T
out = {{}}
for i, kw in enumerate(T.CASES):
    kw = dict(kw); lq = kw.pop("lens_q"); lk = kw.pop("lens_k", None)
    p = fi.make_problem(lq, lk, seed=700 + i, **kw)
    o, l = host(*run_gpu(p))
    out["o%d" % i], out["l%d" % i] = o, l
import flashattention_forward_gb300 as fa
assert fa.device_error() == 0
np.savez({path!r}, **out)
"""


def _run(variant, path):
    env = dict(os.environ, FA_GB300_PREFILL_VARIANT=str(variant))
    code = CHILD.format(root=ROOT, tests=HERE, path=path)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return np.load(path)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from flashattention_forward_gb300 import build
    build.build()


def test_one_and_two_tiles_per_cta_agree_bit_for_bit_and_with_the_oracle(tmp_path):
    one = _run(2, str(tmp_path / "one.npz"))
    two = _run(3, str(tmp_path / "two.npz"))
    for i, kw in enumerate(CASES):
        if kw.get("mod") != "alibi":
            assert np.array_equal(one["o%d" % i], two["o%d" % i]), i
            assert np.array_equal(one["l%d" % i], two["l%d" % i]), i
        kw = dict(kw)
        lq = kw.pop("lens_q")
        lk = kw.pop("lens_k", None)
        p = fi.make_problem(lq, lk, seed=700 + i, **kw)
        ro, rl = oracle.forward(p)
        compare(one["o%d" % i], one["l%d" % i], ro, rl)
        compare(two["o%d" % i], two["l%d" % i], ro, rl)

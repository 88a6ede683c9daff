"""GPU parity of the opt-in e4m3 P * V mode (FA_FLAG_PV_E4M3: e4m3 Q, K and
V with per-token scales; QK and P * V both kind::f8f6f4; FlyDSL PR #1066,
Technical Details and Test Result: direct FP8 P x V at V head dim 128)
against the fp64 oracle.

Each attention weight goes to e4m3 as p * v_scale / 2^e (2^e above the
sequence's largest V scale), so it carries up to 2^-4 relative rounding; an
output element then differs from the exact attention by at most about
2^-4 * max |v| over its keys (one dominant key), and far less when many keys
share the weight.  The row sums, and so the LSE, stay fp32 and exact to the
default 1e-3.  The tests hold:
  * weights that are exact in e4m3 (all scores equal, V scales 2^-7: every
    weight is 2^-1) to the default contract, |dout| <= 1e-2 -- the layout
    checks of the transposed V, the P tile and the scale folding;
  * random inputs to max |dout| <= 2^-4 * max |v| + 1e-2, mean |dout| <= 1e-2,
    |dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import compare, host, to_device

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


def run_pv8(p, t=None):
    import flashattention_forward_gb300 as fa
    t = to_device(p) if t is None else t
    return host(*fa.fwd_varlen(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                               max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, block_table=t.get("bt"),
                               page_size=p.page_size, k_scale=t.get("k_scale"), v_scale=t.get("v_scale"),
                               softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
                               score_mod=p.mod_kind, alibi_slope=p.alibi_slope, softcap=p.softcap,
                               block_mask=t.get("bm"), num_splits=0, pv_e4m3=True))


def v_max_abs(p):
    """max |v| over the cache (spare page slots hold NaN: left out)."""
    v = torch.from_numpy(p.v.copy()).view(torch.float8_e4m3fn).float().numpy()
    a = np.abs(v * p.v_scale[..., None])
    return float(np.max(a[np.isfinite(a)]))


def compare_pv8(p, o, l):
    ro, rl = oracle.forward(p)
    tol = 2.0 ** -4 * v_max_abs(p) + 1e-2
    eo, el = compare(o, l, ro, rl, out_tol=tol)
    fin = ~np.isneginf(rl.T)
    mean = float(np.mean(np.abs(o - ro)[fin])) if fin.any() else 0.0
    assert mean <= 1e-2, f"mean |dout| = {mean}"
    return eo, el, mean


CASES = [
    dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, hkv=2),                                # packed
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, page_size=16, spare_pages=4, causal=True),
    dict(lens_q=[200, 64, 3], lens_k=[260, 64, 500], hq=8, hkv=1, page_size=32, causal=True, window=90),
    dict(lens_q=[130, 260], lens_k=[130, 260], hq=4, page_size=128, mod="alibi"),
    dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, page_size=256, mod="softcap", softcap=5.0, causal=True),
    dict(lens_q=[0, 5, 0], lens_k=[7, 0, 0], hq=2, page_size=16),                                     # empty rows
    dict(lens_q=[200, 330], lens_k=[200, 330], hq=4, page_size=1024, block_mask_density=0.5),
    dict(lens_q=[300, 40], lens_k=[100, 40], hq=2, page_size=64, causal=True),                        # Sk < Sq
]


@pytest.mark.parametrize("dk", [128, 192])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_pv8_random(case, dk):
    kw = dict(CASES[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    p = fi.make_problem(lens_q, lens_k, seed=560 + case, dk=dk, dv=128, kv_dtype="e4m3", q_dtype="e4m3", **kw)
    compare_pv8(p, *run_pv8(p))


@pytest.mark.parametrize("dk", [128, 192])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_pv8_exact_weights(case, dk):
    """Q = 0 (every score 0, soft-capped or not) and V scales 2^-7 (so that
    the outputs, means of |v| <= 3.5, stay below 4, where a bf16 rounding is below 1e-2): every
    weight is exactly 2^-1 in e4m3, so the output is the exact mean of the
    allowed V rows and must meet the default contract."""
    kw = dict(CASES[case])
    if kw.get("mod") == "alibi":
        kw.pop("mod")
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    p = fi.make_problem(lens_q, lens_k, seed=580 + case, dk=dk, dv=128, kv_dtype="e4m3", q_dtype="e4m3", **kw)
    pow2 = np.where(np.isnan(p.v_scale), np.nan, np.float32(2.0 ** -7)).astype(np.float32)
    p = p.replace(q=np.zeros_like(p.q), v_scale=pow2)
    o, l = run_pv8(p)
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_pv8_config4_geometry_every_row():
    """Config 4 (16 sequences of U{1..4096} tokens, H 16, Q/K 192, V/O 128,
    page 64, causal) with e4m3 Q and e4m3 P * V: every (token, head) row."""
    base = fi.config4()
    p = fi.make_problem(list(np.diff(base.cu_seqlens_q)), hq=16, hkv=16, dk=192, dv=128, seed=1, page_size=64,
                        kv_dtype="e4m3", q_dtype="e4m3", spare_pages=16, causal=True)
    eo, el, mean = compare_pv8(p, *run_pv8(p))
    print(f"config 4, e4m3 P*V: max |dout| {eo:.3g}, mean {mean:.3g}, max |dLSE| {el:.3g}")

"""GPU parity of the backward pass (fa_bwd_varlen) against the fp64 oracle.

Each case runs the CUDA forward for out and LSE, the CUDA backward for
dq, dk, dv with a seeded dout, and the oracle's backward on the same bf16
inputs.  Tolerance, per gradient tensor: max |gpu - oracle| <= 2% of
max |oracle| + 1e-3.  Derivation: the kernels round P and dS to bf16 before
the accumulating MMAs (relative 2^-9 each), Delta comes from the forward's
bf16 output (relative 2^-9 per element), and the outputs are rounded to bf16
(relative 2^-9); a few such roundings against the largest element stay near
1%, and 2% leaves a margin while still catching a dropped term, a wrong
scale or a wrong index (those give errors of order 100%).
"""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import host, run_gpu, to_device

pytestmark = pytest.mark.gpu

REL_TOL, ABS_TOL = 0.02, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from flashattention_forward_gb300 import build
    build.build()
    yield
    import flashattention_forward_gb300 as fa
    assert fa.device_error() == 0


def _dout(p, seed):
    rng = np.random.default_rng(seed)
    return fi.bf16_bits(rng.standard_normal((p.total_q, p.hq, p.dv), dtype=np.float32))


def run_bwd(p, seed=11):
    import flashattention_forward_gb300 as fa
    t = to_device(p)
    out, lse = run_gpu(p, t)
    dob = _dout(p, seed)
    dout = torch.from_numpy(dob.view(np.int16).copy()).view(torch.bfloat16).cuda()
    dq, dk, dv = fa.bwd_varlen(t["q"], t["k"], t["v"], out, dout, lse, t["cu_q"], t["cu_k"],
                               max_seqlen_q=p.max_seqlen_q, max_seqlen_k=p.max_seqlen_k,
                               softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
                               score_mod=p.mod_kind, alibi_slope=p.alibi_slope, softcap=p.softcap,
                               block_mask=t.get("bm"))
    torch.cuda.synchronize()
    g = [x.float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv)]
    return g, fi.bf16_to_f32(dob).astype(np.float64)


def check(p, seed=11):
    (dq, dk, dv), dout = run_bwd(p, seed)
    rq, rk, rv = oracle.backward(p, dout)
    errs = {}
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert g.shape == r.shape, (name, g.shape, r.shape)
        assert np.isfinite(g).all(), f"non-finite {name}"
        e = float(np.abs(g - r).max()) if g.size else 0.0
        lim = REL_TOL * float(np.abs(r).max() if r.size else 0.0) + ABS_TOL
        errs[name] = e
        print(f"{name}: max|d| {e:.3e} (limit {lim:.3e}, max|ref| {np.abs(r).max():.3e})")
        assert e <= lim, f"{name}: max |d| = {e:.3e} > {lim:.3e}"
    return errs


CASES = {
    "config1_b2_h4_s128_d64_causal": dict(lens_q=[128, 128], hq=4, dk=64, causal=True, softmax_scale=0.125),
    "ragged_d128_causal": dict(lens_q=[0, 300, 129, 1, 64], hq=4, dk=128, causal=True),
    "ragged_d128_noncausal": dict(lens_q=[0, 300, 129, 1, 64], hq=4, dk=128),
    "gqa_d64_causal": dict(lens_q=[257, 40], hq=8, hkv=2, dk=64, causal=True),
    "gqa_d128_noncausal": dict(lens_q=[200, 77], hq=6, hkv=3, dk=128),
    "sq_lt_sk_causal": dict(lens_q=[100, 5], lens_k=[300, 260], hq=4, dk=128, causal=True),
    "sq_gt_sk_causal": dict(lens_q=[200, 64], lens_k=[100, 10], hq=2, dk=64, causal=True),
    "window_causal": dict(lens_q=[600, 130], hq=2, dk=128, causal=True, window=100),
    "window_noncausal": dict(lens_q=[400], lens_k=[500], hq=2, dk=64, window=70),
    "long_multi_tile": dict(lens_q=[900], hq=2, dk=128, causal=True),
    # score mods: ALiBi leaves dS as it is, the soft-cap scales it by 1 - tanh^2
    "alibi_causal_d128": dict(lens_q=[300, 129], hq=4, dk=128, causal=True, mod="alibi", alibi_slope=0.05),
    "alibi_gqa_sq_lt_sk_d64": dict(lens_q=[70, 200], lens_k=[260, 333], hq=8, hkv=2, dk=64, mod="alibi",
                                   alibi_slope=0.02),
    "softcap_causal_d128": dict(lens_q=[257, 64], hq=4, dk=128, causal=True, mod="softcap", softcap=2.0,
                                softmax_scale=0.25),
    "softcap_window_gqa_d64": dict(lens_q=[400], lens_k=[500], hq=4, hkv=2, dk=64, window=90, mod="softcap",
                                   softcap=5.0),
    "softcap_saturated_d64": dict(lens_q=[200, 130], hq=4, dk=64, mod="softcap", softcap=0.5, softmax_scale=1.0),
    # 128 x 128 block sparsity: skipped blocks add nothing; rows whose blocks
    # are all skipped have LSE = -inf and zero gradients
    "blocksparse_d128": dict(lens_q=[300, 129], lens_k=[330, 400], hq=4, hkv=2, dk=128, block_mask_density=0.5),
    "blocksparse_causal_d64": dict(lens_q=[520, 70], hq=4, dk=64, causal=True, block_mask_density=0.4),
    "blocksparse_alibi_gqa": dict(lens_q=[260, 390], hq=8, hkv=2, dk=128, mod="alibi", alibi_slope=0.03,
                                  block_mask_density=0.6),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bwd_matches_oracle(name):
    kw = dict(CASES[name])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    check(fi.make_problem(lens_q, lens_k, seed=700 + sorted(CASES).index(name), **kw))


def test_bwd_is_deterministic():
    p = fi.make_problem([700, 33], hq=4, hkv=2, dk=128, seed=5, causal=True)
    a, _ = run_bwd(p)
    b, _ = run_bwd(p)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_single_key_rows():
    """Sk = 1: every row sees one key, P = 1, so dq = dk = 0 and dv = sum of dout.

    P is recomputed from the fp32 LSE as exp2(s*c - LSE*log2 e), 1 within a
    few fp32 ulps, so dq and dk are zero up to ~1e-6 rather than exactly."""
    p = fi.make_problem([5, 130], [1, 1], hq=2, dk=64, seed=8)
    (dq, dk, dv), dout = run_bwd(p)
    assert np.abs(dq).max() <= 1e-4 and np.abs(dk).max() <= 1e-4
    ref = np.stack([dout[0:5].sum(0), dout[5:135].sum(0)])
    assert np.abs(dv - ref).max() <= REL_TOL * np.abs(ref).max() + ABS_TOL

"""GPU parity of the e4m3-Q path (e4m3 Q, K and V with per-token K/V scales;
QK on the e4m3 bytes by kind::f8f6f4 with the key scale applied per score
column, V converted to f16, PV kind::f16) against the fp64 oracle."""
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


Q8_CASES = [
    dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, hkv=2),                                # packed
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, page_size=16, spare_pages=4, causal=True),
    dict(lens_q=[200, 64, 3], lens_k=[260, 64, 500], hq=8, hkv=1, page_size=32, causal=True, window=90),
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=4, page_size=64, window=100),
    dict(lens_q=[130, 260], lens_k=[130, 260], hq=4, page_size=128, mod="alibi"),
    dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, page_size=256, mod="softcap", softcap=5.0, causal=True),
    dict(lens_q=[0, 5, 0], lens_k=[7, 0, 0], hq=2, page_size=16),                                     # empty rows
    dict(lens_q=[200, 330], lens_k=[200, 330], hq=4, page_size=1024, block_mask_density=0.5),
    dict(lens_q=[300, 40], lens_k=[100, 40], hq=2, page_size=64, causal=True),                        # Sk < Sq
    dict(lens_q=[513], lens_k=[1100], hq=2, hkv=1, page_size=512, causal=True, mod="alibi"),
]


@pytest.mark.parametrize("case", range(len(Q8_CASES)))
def test_q8_cases(case):
    kw = dict(Q8_CASES[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    check(fi.make_problem(lens_q, lens_k, seed=500 + case, dk=128, dv=128, kv_dtype="e4m3", q_dtype="e4m3", **kw))


Q8_D192_CASES = [
    dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, hkv=2),                                # packed
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, page_size=16, spare_pages=4, causal=True),
    dict(lens_q=[200, 64, 3], lens_k=[260, 64, 500], hq=8, hkv=1, page_size=64, causal=True, window=90),
    dict(lens_q=[130, 260], lens_k=[130, 260], hq=4, page_size=128, mod="alibi"),
    dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, page_size=64, mod="softcap", softcap=5.0, causal=True),
    dict(lens_q=[0, 5, 0], lens_k=[7, 0, 0], hq=2, page_size=16),                                     # empty rows
    dict(lens_q=[200, 330], lens_k=[200, 330], hq=4, page_size=1024, block_mask_density=0.5),
    dict(lens_q=[300, 40], lens_k=[100, 40], hq=2, page_size=64, causal=True),                        # Sk < Sq
]


@pytest.mark.parametrize("case", range(len(Q8_D192_CASES)))
def test_q8_d192_cases(case):
    """e4m3 Q at Q/K 192, V/O 128: a key row spans two 128-column chunks,
    the second half-empty (TMA zero-fills columns 192..255)."""
    kw = dict(Q8_D192_CASES[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    check(fi.make_problem(lens_q, lens_k, seed=520 + case, dk=192, dv=128, kv_dtype="e4m3", q_dtype="e4m3", **kw))


def test_q8_config4_geometry_every_row():
    """Config 4 (16 sequences of U{1..4096} tokens, H 16, Q/K 192, V/O 128,
    page 64, causal) with e4m3 Q: every (token, head) row against the oracle."""
    base = fi.config4()
    p = fi.make_problem(list(np.diff(base.cu_seqlens_q)), hq=16, hkv=16, dk=192, dv=128, seed=1, page_size=64,
                        kv_dtype="e4m3", q_dtype="e4m3", spare_pages=16, causal=True, name="config4_e4m3q")
    check(p)


def test_q8_key_scales_spread():
    """Key scales spread over 2^-4 .. 2^4 of their quantiser's value (scores
    then span a wide range): each score column must carry its own key's
    scale.  Keys are used as stored, so scales beyond the f16 range of a
    converted key are fine too."""
    p = fi.make_problem([200, 77], [333, 77], hq=4, hkv=2, dk=128, dv=128, seed=31, page_size=16,
                        kv_dtype="e4m3", q_dtype="e4m3", causal=True, spare_pages=2)
    rng = np.random.default_rng(5)
    f = np.exp2(rng.integers(-4, 5, size=p.k_scale.shape)).astype(np.float32)
    p = p.replace(k_scale=(p.k_scale * f).astype(np.float32))
    check(p)
    big = p.replace(k_scale=np.where(np.isnan(p.k_scale), np.nan, np.float32(300.0)).astype(np.float32),
                    softmax_scale=p.softmax_scale / 300.0)
    check(big)


def test_q8_zero_key_scale_gives_uniform_scores():
    """All key scales 0: every score is 0, so each row averages its visible V."""
    p = fi.make_problem([150, 90], [150, 90], hq=2, hkv=1, dk=128, dv=128, seed=32, page_size=32,
                        kv_dtype="e4m3", q_dtype="e4m3", causal=True)
    p = p.replace(k_scale=np.where(np.isnan(p.k_scale), np.nan, np.float32(0.0)).astype(np.float32))
    check(p)


def test_q8_matches_bf16_q_run_closely():
    """The same seeded problem with bf16 Q through the converter kernel and
    with e4m3 Q through the byte QK: both within the oracle tolerance of their
    own inputs, and close to each other (Q quantisation only)."""
    kw = dict(hq=4, hkv=2, dk=128, dv=128, seed=33, page_size=64, kv_dtype="e4m3", causal=True)
    pb = fi.make_problem([400, 100], [400, 300], **kw)
    pe = fi.make_problem([400, 100], [400, 300], q_dtype="e4m3", **kw)
    ob, lb = host(*run_gpu(pb))
    oe, le = host(*run_gpu(pe))
    compare(oe, le, *oracle.forward(pe))
    assert np.max(np.abs(oe - ob)) < 0.1 and np.max(np.abs(le - lb)) < 0.1


def test_q8_headline_geometry_sampled():
    """The packed varlen workload of the main benchmark (ragged lengths,
    Hq = Hkv = 16 at Dk = Dv = 128) with e4m3 Q/K/V, on sampled rows."""
    base = fi.config2(causal=False)
    p = fi.make_problem(list(np.diff(base.cu_seqlens_q)), hq=base.hq, hkv=base.hkv, dk=128, dv=128, seed=3,
                        kv_dtype="e4m3", q_dtype="e4m3", name="varlen_e4m3q")
    o, l = host(*run_gpu(p))
    units = sample_units(p, 2500, seed=6)
    ro, rl = oracle.forward(p, units=units)
    compare_units(o, l, units, ro, rl)


def test_q8_plan_and_graph_replay():
    """Prepared plan and CUDA-graph replay give the direct call's bytes."""
    import flashattention_forward_gb300 as fa
    from fa_testlib import to_device
    p = fi.make_problem([300, 129], [300, 400], hq=4, hkv=2, dk=128, dv=128, seed=34, page_size=16,
                        kv_dtype="e4m3", q_dtype="e4m3", causal=True)
    t = to_device(p)
    o1, l1 = run_gpu(p, t)
    plan = fa.FwdPlan(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                      max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, block_table=t["bt"], page_size=p.page_size,
                      k_scale=t["k_scale"], v_scale=t["v_scale"], softmax_scale=p.softmax_scale, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.run(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    plan.out.zero_()
    with torch.cuda.graph(g, stream=s):
        plan.run(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(plan.out.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(plan.lse, l1)

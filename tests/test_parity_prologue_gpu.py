"""GPU parity of the prologue (op chains of Mul, Add, Sub and Div by scalars
on Q, K and V as read; fkl_python PR #7, prologue-fusion commit) against the
fp64 oracle, which applies each op of each chain to the values literally, one
after the other.  The chains go through the public call as given; the library
composes them and folds the maps: the scale product into the score scale,
the row term into the LSE (or into the capped score under the soft-cap), a
Q add's per-key term through a pre-pass over the keys, and the V map into
the output normalisation.

Tolerances are the contract's (|dout| <= 1e-2, |dLSE| <= 1e-3), absolute, so
the chains keep scaled scores of the order of the plain runs' and |a_v| <= 1:
bf16 outputs of magnitude 2 or more would round by up to 2^-7 alone.
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


CHAINS = {
    # every kind of op on every tensor; a_q * a_k < 0 takes the general score path
    "all": {"q": [("add", 0.3), ("mul", 0.8)], "k": [("sub", 0.2), ("mul", -1.5), ("div", 1.25)],
            "v": [("mul", -0.75), ("add", 0.25)]},
    "q_add": {"q": [("sub", 0.25)]},
    "scale_only": {"q": [("mul", 1.25)], "k": [("div", 1.25)]},
    "shift_kv": {"k": [("add", -0.4)], "v": [("div", 2.0), ("add", 1.0)]},
}

CASES = {
    "d128_causal": dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, dk=128, causal=True),
    "d64_paged_gqa_window": dict(lens_q=[200, 3], lens_k=[260, 500], hq=8, hkv=2, dk=64, causal=True,
                                 window=90, page_size=32, spare_pages=3),
    "d192_bf16": dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128, causal=True),
    "e4m3_d128": dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, hkv=2, dk=128, kv_dtype="e4m3",
                      page_size=64, spare_pages=2),
    "e4m3_d192_paged": dict(lens_q=[200, 65], lens_k=[200, 400], hq=4, hkv=4, dk=192, dv=128, kv_dtype="e4m3",
                            page_size=64, spare_pages=2, causal=True),
    "int8_d128": dict(lens_q=[150, 9], lens_k=[150, 300], hq=4, hkv=2, dk=128, kv_dtype="int8", page_size=16,
                      spare_pages=2),
    "alibi_d128": dict(lens_q=[150, 64], lens_k=[400, 64], hq=4, dk=128, mod="alibi", alibi_slope=0.05),
    "softcap_d128": dict(lens_q=[200, 64], lens_k=[300, 64], hq=4, dk=128, mod="softcap", softcap=5.0,
                         causal=True),
    "blocksparse_d128": dict(lens_q=[300, 129], lens_k=[330, 400], hq=4, hkv=2, dk=128, block_mask_density=0.5),
    "pages_of_4": dict(lens_q=[100, 30], lens_k=[100, 250], hq=4, hkv=2, dk=128, page_size=4, spare_pages=2,
                       causal=True),
}


def problem(name, chain, seed_base=600):
    kw = dict(CASES[name])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k")
    return fi.make_problem(lens_q, lens_k, seed=seed_base + sorted(CASES).index(name), **kw).replace(
        prologue=CHAINS[chain])


@pytest.mark.parametrize("chain", sorted(CHAINS))
@pytest.mark.parametrize("name", sorted(CASES))
def test_prologue_prefill(name, chain):
    p = problem(name, chain)
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3", "int8"])
@pytest.mark.parametrize("chain", sorted(CHAINS))
def test_prologue_split_kv_decode(kv_dtype, chain):
    lens_k = [1, 63, 700, 2049]
    p = fi.make_problem([1] * 4, lens_k, hq=8, hkv=2, dk=128, seed=630, page_size=16, spare_pages=4,
                        kv_dtype=kv_dtype).replace(prologue=CHAINS[chain])
    o, l = host(*run_gpu(p, num_splits=3))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


@pytest.mark.parametrize("mod", ["softcap", "alibi"])
def test_prologue_split_kv_decode_with_score_mods(mod):
    """Under the soft-cap the row term (a K add) and the per-key term (a Q
    add) both enter the capped score."""
    p = fi.make_problem([1, 2, 1], [90, 700, 1500], hq=8, hkv=4, dk=64, seed=631, page_size=32, spare_pages=2,
                        mod=mod, softcap=4.0, alibi_slope=0.03, causal=True).replace(prologue=CHAINS["all"])
    o, l = host(*run_gpu(p, num_splits=4))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_prologue_softcap_with_shifts_on_q_and_k():
    """Soft-cap s = cap tanh(u / cap) is not shift-invariant: the row and key
    terms of the adds must be inside the cap."""
    p = fi.make_problem([200, 64], [300, 64], hq=4, hkv=2, dk=128, seed=620, mod="softcap", softcap=2.0,
                        causal=True).replace(prologue={"q": [("add", 0.4)], "k": [("mul", 0.5), ("sub", 0.3)],
                                                       "v": [("mul", 0.75), ("add", 0.5)]})
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_prologue_config2_lengths():
    """The packed varlen workload of config 2 (8 sequences of U{0..2048}
    tokens, H 16, D 128) with every kind of op."""
    p = fi.config2(causal=False).replace(prologue=CHAINS["all"])
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_identity_prologue_is_bit_identical_to_none():
    p = fi.make_problem([300, 129], [300, 400], hq=4, dk=128, seed=640, causal=True)
    o0, l0 = host(*run_gpu(p))
    o1, l1 = host(*run_gpu(p.replace(prologue={"q": [("mul", 1.0)], "k": [("add", 0.0)], "v": [("div", 1.0)]})))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_prologue_plan_and_graph_replay_with_a_q_add():
    """A prepared call with a Q add (its key-term pre-pass is part of the
    plan), launched twice and replayed from a CUDA graph."""
    import flashattention_forward_gb300 as fa
    from fa_testlib import to_device
    p = problem("d128_causal", "all")
    t = to_device(p)
    plan = fa.FwdPlan(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                      max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, softmax_scale=p.softmax_scale,
                      causal=p.causal, prologue=p.prologue)
    ro, rl = oracle.forward(p)
    plan.run()
    o1, l1 = host(plan.out.clone(), plan.lse.clone())
    compare(o1, l1, ro, rl)
    plan.out.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        plan.run(stream=s)            # warm-up on the capture stream
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            plan.run(stream=s)
    plan.out.zero_()
    g.replay()
    o2, l2 = host(plan.out, plan.lse)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)

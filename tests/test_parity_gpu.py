"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs.  Tolerances: max |dout| <= 1e-2, |dLSE| <= 1e-3,
-inf LSE and zero rows matched exactly, indexing bit-exact."""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle
from fa_testlib import compare, compare_units, host, run_gpu, sample_units, to_device

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


# ----------------------------------------------------------- configurations --

def test_config1_dense_causal():
    p = fi.config1()
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)
    # [T, H, D] packed == [2, 128, 4, 64]; LSE [H, T] viewed as [2, 4, 128]
    assert o.reshape(2, 128, 4, 64).shape == (2, 128, 4, 64)
    assert l.reshape(4, 2, 128).transpose(1, 0, 2).shape == (2, 4, 128)


@pytest.mark.parametrize("causal", [True, False])
def test_config2_varlen_prefill(causal):
    check(fi.config2(causal=causal))


def test_config3_paged_decode_split_kv():
    p = fi.config3()
    o, l = host(*run_gpu(p, num_splits=None))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


@pytest.mark.parametrize("run", fi.CONFIG5_RUNS)
def test_config5_flex_sampled(run):
    """Config 5 (B 4, H 16, S 8192, D 128): every head of every row at a
    128-row tile boundary or a sequence end, plus 4096 seeded random rows."""
    p = fi.config5(run)
    o, l = host(*run_gpu(p))
    units = sample_units(p, 4096, seed=5)
    assert len(units) >= 4096 + 4 * 128 * 16
    ro, rl = oracle.forward(p, units=units)
    compare_units(o, l, units, ro, rl)


# --------------------------------------------------------------- edge cases --

EDGE = [
    dict(lens_q=[1, 127, 128, 129, 300], hq=4, dk=64),
    dict(lens_q=[5, 0, 77, 256], lens_k=[300, 0, 77, 500], hq=4, hkv=2, dk=128, causal=True),
    dict(lens_q=[200, 64], lens_k=[100, 10], hq=2, dk=128, causal=True),          # Sq > Sk: masked rows
    dict(lens_q=[0, 0, 3], lens_k=[0, 5, 0], hq=2, dk=64),                        # empty sequences
    dict(lens_q=[130, 260], lens_k=[400, 260], hq=8, hkv=1, dk=128, causal=True, window=100),
    dict(lens_q=[130, 260], lens_k=[400, 260], hq=4, dk=64, window=70),
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, dk=128, mod="alibi", alibi_slope=0.0625, causal=True),
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, dk=128, mod="softcap", softcap=2.0),
    dict(lens_q=[300, 129], lens_k=[330, 400], hq=4, hkv=2, dk=128, block_mask_density=0.5),
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=4, dk=192, dv=128, causal=True),
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128, page_size=64, spare_pages=3),
    dict(lens_q=[300, 70], lens_k=[300, 200], hq=4, dk=128, softmax_scale=-0.05, causal=True),  # negative scale
    dict(lens_q=[513, 40, 900], lens_k=[513, 700, 900], hq=8, hkv=2, dk=64, causal=True),       # 3 pairs, GQA
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128, mod="softcap", softcap=3.0,
         causal=True),                                                                           # soft-cap, Dk 192
    dict(lens_q=[200, 130], hq=4, dk=64, mod="softcap", softcap=0.5, softmax_scale=1.0),        # tanh saturated
]


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_edge_cases_packed_and_paged(case):
    kw = dict(EDGE[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    check(fi.make_problem(lens_q, lens_k, seed=100 + case, **kw))


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256, 512, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_page_sizes_with_poisoned_slots(page_size, causal):
    p = fi.make_problem([70, 300, 1, 129], [200, 300, 1000, 129], hq=8, hkv=2, dk=128, seed=7,
                        page_size=page_size, spare_pages=5, causal=causal)
    check(p)


@pytest.mark.parametrize("splits", [1, 2, 7, 33])
@pytest.mark.parametrize("sq,paged", [(1, True), (2, True), (4, False), (1, False)])
def test_decode_split_counts(splits, sq, paged):
    lens_k = [1, 63, 64, 65, 700, 2049, 3000]
    p = fi.make_problem([sq] * len(lens_k), lens_k, hq=8, hkv=2, dk=128, seed=splits,
                        page_size=16 if paged else 0, spare_pages=4, causal=sq > 1)
    check(p, num_splits=splits)


def test_decode_d64_window():
    p = fi.make_problem([1, 1, 1], [500, 90, 1300], hq=16, hkv=1, dk=64, seed=3, page_size=32, window=200)
    check(p, num_splits=4)


def test_combine_entry_point_matches_oracle_merge():
    import flashattention_forward_gb300 as fa
    rng = np.random.default_rng(0)
    S, n, H, D = 5, 37, 3, 128
    # partial outputs are convex combinations of V rows: keep them in [-1, 1]
    o_part = rng.uniform(-1.0, 1.0, (S, n, H, D)).astype(np.float32)
    lse_part = (rng.standard_normal((S, H, n)) * 3).astype(np.float32)
    lse_part[1, 0, :] = -np.inf
    lse_part[:, 2, 5] = -np.inf                  # a row with every split empty
    out, lse = fa.combine(torch.from_numpy(o_part).cuda(), torch.from_numpy(lse_part).cuda())
    out, lse = host(out, lse)
    # oracle merge works on [S, rows, D] with rows = (t, h) in t-major order
    ro, rl = oracle.combine(o_part.reshape(S, n * H, D).astype(np.float64),
                            lse_part.transpose(0, 2, 1).reshape(S, n * H).astype(np.float64))
    compare(out, lse, ro.reshape(n, H, D), rl.reshape(n, H).T)


# -------------------------------------------------------- indexing bit-exact --

def _integer_values(p):
    """V rows filled with small integers that encode (token, head, dim):
    exactly representable in bf16, so a single visible key reproduces them bit-for-bit."""
    shape = p.v.shape
    idx = np.indices(shape).reshape(len(shape), -1)
    vals = ((idx[0] * 7 + idx[-2] * 3 + idx[-1]) % 200 - 100).astype(np.float32).reshape(shape)
    return p.replace(v=fi.bf16_bits(vals))


@pytest.mark.parametrize("paged", [False, True])
def test_single_visible_key_is_bit_exact(paged):
    """Causal window 1 leaves only key i' for each row: out must equal that V row exactly."""
    p = fi.make_problem([40, 300, 7], [90, 300, 520], hq=8, hkv=2, dk=128, seed=11, causal=True,
                        window=1, page_size=16 if paged else 0, spare_pages=6)
    p = _integer_values(p)
    o, l = run_gpu(p)
    torch.cuda.synchronize()
    got = o.view(torch.int16).cpu().numpy().view(np.uint16)
    ro, _ = oracle.forward(p)
    exp = fi.bf16_bits(ro.astype(np.float32))
    assert np.array_equal(got, exp)


def test_decode_single_key_bit_exact():
    p = fi.make_problem([1] * 6, [1] * 6, hq=8, hkv=2, dk=128, seed=12, page_size=16, spare_pages=3)
    p = _integer_values(p)
    for splits in (1, 3):
        o, _ = run_gpu(p, num_splits=splits)
        torch.cuda.synchronize()
        got = o.view(torch.int16).cpu().numpy().view(np.uint16)
        ro, _ = oracle.forward(p)
        assert np.array_equal(got, fi.bf16_bits(ro.astype(np.float32)))


def test_permuted_block_table_is_bit_identical():
    """Permuting pages together with the block table gives bit-identical output."""
    p = fi.make_problem([100, 260], [700, 260], hq=4, hkv=2, dk=128, seed=13, page_size=16, spare_pages=8,
                        causal=True)
    o1, l1 = host(*run_gpu(p))
    rng = np.random.default_rng(1)
    perm = rng.permutation(p.k.shape[0])          # new position of each old page
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    k2 = np.empty_like(p.k)
    v2 = np.empty_like(p.v)
    k2[perm] = p.k
    v2[perm] = p.v
    bt2 = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    o2, l2 = host(*run_gpu(p.replace(k=k2, v=v2, block_table=bt2)))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ------------------------------------------------ streams, guards, determinism --

def test_side_stream_and_determinism():
    p = fi.make_problem([300, 129, 64], [300, 500, 64], hq=8, hkv=2, dk=128, seed=14, causal=True)
    t = to_device(p)
    o1, l1 = host(*run_gpu(p, t))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)             # keep the side stream busy first
        o2, l2 = run_gpu(p, t, stream=s)
    s.synchronize()
    o2, l2 = host(o2, l2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_guard_bands_untouched():
    p = fi.make_problem([129, 0, 77], [300, 5, 77], hq=4, hkv=4, dk=64, seed=15, causal=True)
    t = to_device(p)
    big_o = torch.full((p.total_q + 3, p.hq, p.dv), 1024.0, dtype=torch.bfloat16, device="cuda")
    big_l = torch.full((p.hq + 1, p.total_q), 777.0, dtype=torch.float32, device="cuda")
    o, l = run_gpu(p, t, out=big_o[:p.total_q], lse=big_l[:p.hq])
    torch.cuda.synchronize()
    assert torch.all(big_o[p.total_q:] == 1024.0)
    assert torch.all(big_l[p.hq:] == 777.0)
    ro, rl = oracle.forward(p)
    compare(*host(o, l), ro, rl)


@pytest.mark.parametrize("causal", [False, True])
def test_two_pass_softmax_variant(monkeypatch, causal):
    """The 10-warp two-pass softmax (used when the register split does not fit)."""
    monkeypatch.setenv("FA_GB300_PREFILL_VARIANT", "1")
    check(fi.make_problem([300, 129, 700], [300, 400, 700], hq=4, hkv=2, dk=128, seed=31, causal=causal))
    check(fi.make_problem([200, 64], [500, 64], hq=4, dk=64, seed=32, causal=causal, mod="alibi"))


# ------------------------------------------------------------- prepared call --

@pytest.mark.parametrize("case", ["prefill_paged_causal", "decode_split", "fp8_alibi"])
def test_fwd_plan_matches_call_and_oracle(case):
    """FwdPlan (descriptors marshalled once, re-issued by run()) gives the
    bit-identical result of fwd_varlen, on every re-run, and matches the oracle."""
    import flashattention_forward_gb300 as fa
    if case == "prefill_paged_causal":
        p = fi.make_problem([300, 0, 129], [700, 5, 129], hq=8, hkv=2, dk=128, seed=41, causal=True,
                            page_size=64)
    elif case == "decode_split":
        p = fi.make_problem([1] * 6, [3000, 1, 257, 4096, 0, 900], hq=16, hkv=2, dk=128, seed=42,
                            page_size=16)
    else:
        p = fi.make_problem([200, 77], [450, 300], hq=4, hkv=2, dk=128, seed=43, kv_dtype="e4m3",
                            mod="alibi")
    t = to_device(p)
    plan = fa.FwdPlan(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                      max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, block_table=t.get("bt"),
                      page_size=p.page_size, k_scale=t.get("k_scale"), v_scale=t.get("v_scale"),
                      softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
                      score_mod=p.mod_kind, alibi_slope=p.alibi_slope, softcap=p.softcap,
                      block_mask=t.get("bm"))
    if case == "decode_split":
        assert plan.launch.num_splits > 1
    ref_o, ref_l = host(*run_gpu(p, t, num_splits=plan.launch.num_splits))
    for _ in range(3):
        o, l = host(*plan.run())
        assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l)
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


def test_graph_capture_of_call_and_plan():
    """The forward enqueues kernels only (no allocation, copy or sync inside),
    so both the plain call and a prepared plan can be captured in a CUDA graph
    and replayed on new inputs written into the same buffers."""
    import flashattention_forward_gb300 as fa
    p = fi.make_problem([300, 129, 64], [300, 500, 64], hq=8, hkv=2, dk=128, seed=51, causal=True)
    p2 = fi.make_problem([300, 129, 64], [300, 500, 64], hq=8, hkv=2, dk=128, seed=52, causal=True)
    t, t2 = to_device(p), to_device(p2)
    o_ref, l_ref = host(*run_gpu(p2, t2))
    out = torch.empty((p.total_q, p.hq, p.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.hq, p.total_q), dtype=torch.float32, device="cuda")
    plan = fa.FwdPlan(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                      max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, softmax_scale=p.softmax_scale, causal=True,
                      num_splits=0)
    run_gpu(p, t, out=out, lse=lse)       # warm up (module load, attributes) outside the capture
    plan.run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for use_plan in (False, True):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            if use_plan:
                plan.run(stream=s)
            else:
                run_gpu(p, t, out=out, lse=lse, stream=s)
        for name in ("q", "k", "v"):
            t[name].copy_(t2[name])
        out.zero_()
        plan.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        o, l = host(out, lse) if not use_plan else host(plan.out, plan.lse)
        assert np.array_equal(o, o_ref) and np.array_equal(l, l_ref)
        for name in ("q", "k", "v"):
            t[name].copy_(to_device(p)[name])


# ---------------------------------------------------------- deferred row max --

def _escalating_scores(p, boosts, kv_dtype="bf16"):
    """Key tile t of every sequence gets its scores raised by boosts[t] (scaled
    log2 units, approximately): K rows of tile t are offset along q's mean
    direction (bf16), or their per-token scales multiplied (e4m3)."""
    rng = np.random.default_rng(7)
    q = fi.bf16_to_f32(p.q).copy()
    q[:] = 0.5 + 0.05 * rng.standard_normal(q.shape).astype(np.float32)
    p = p.replace(q=fi.bf16_bits(q))
    lens = np.diff(p.cu_seqlens_k)
    if kv_dtype == "bf16":
        k = fi.bf16_to_f32(p.k).copy()
        for b, L in enumerate(lens):
            for t, boost in enumerate(boosts):
                lo, hi = t * 128, min((t + 1) * 128, L)
                if lo >= hi:
                    break
                # q.k ~ 0.5 * sum(k); raise each score by boost/(scale*log2e)
                shift = boost / (p.softmax_scale * 1.4426950408889634) / (0.5 * p.dk)
                k[p.cu_seqlens_k[b] + lo:p.cu_seqlens_k[b] + hi] += shift
        return p.replace(k=fi.bf16_bits(k))
    ks = p.k_scale.copy()
    for b, L in enumerate(lens):
        for t, boost in enumerate(boosts):
            lo, hi = t * 128, min((t + 1) * 128, L)
            if lo >= hi:
                break
            for key in range(lo, hi):
                page = p.block_table[b, key // p.page_size]
                ks[page, key % p.page_size] *= boost
    return p.replace(k_scale=ks)


@pytest.mark.parametrize("variant", ["onepass_d128", "twohalf_d128", "onepass_d192", "e4m3_d128", "plain_d128"])
def test_deferred_max_large_and_overflowing_tiles(monkeypatch, variant):
    """Scores that jump by ~46 log2 units after the first key tile (P values
    near 2^46 through the fast path) and by ~140 later (the 2^64 guard fires,
    the row max is taken and P redone) match the oracle.  The deferred max
    runs with a score mod: ALiBi with slope 0 gives plain attention through
    that path; `plain_d128` checks the max-first path on the same scores."""
    if variant == "twohalf_d128":
        monkeypatch.setenv("FA_GB300_PREFILL_VARIANT", "1")
    mod = dict(mod="none") if variant == "plain_d128" else dict(mod="alibi", alibi_slope=0.0)
    if variant == "e4m3_d128":
        p = fi.make_problem([300, 200], [700, 450], hq=2, dk=128, seed=61, kv_dtype="e4m3", page_size=64, **mod)
        # e4m3 K becomes f16 RN(e4m3 * k_scale): its 2^-12 relative rounding
        # puts an absolute error proportional to |q.k| on each score, so this
        # case stays at moderate scores (P up to ~2^20 on the fast path).
        p = _escalating_scores(p, [1.0, 6.0, 1.0, 6.0, 1.0, 1.0], kv_dtype="e4m3")
    else:
        dk = 192 if variant == "onepass_d192" else 128
        p = fi.make_problem([300, 200], [700, 450], hq=2, dk=dk, dv=128, seed=61, **mod)
        p = _escalating_scores(p, [0.0, 46.0, 10.0, 140.0, 20.0, 0.0])
    check(p)


@pytest.mark.parametrize("page_size", [16, 1024])
@pytest.mark.parametrize("case", ["d192_bf16", "d64_bf16", "decode_splits"])
def test_extreme_page_sizes_other_paths(page_size, case):
    """The smallest and largest page sizes (16: eight TMA boxes per 128-key
    tile, issued by the producer warp's lanes in parallel; 1024: a tile inside
    one page) on the chunked-ring kernel (Dk 192), the Dk 64 ping-pong kernel
    and the split-KV decode."""
    if case == "d192_bf16":
        p = fi.make_problem([300, 129, 1], [700, 129, 300], hq=4, hkv=2, dk=192, dv=128, seed=81,
                            page_size=page_size, spare_pages=3, causal=True)
        check(p)
    elif case == "d64_bf16":
        p = fi.make_problem([200, 3], [260, 500], hq=8, hkv=1, dk=64, seed=82, page_size=page_size,
                            spare_pages=3, causal=True, window=90)
        check(p)
    else:
        p = fi.make_problem([1] * 5, [1, 64, 65, 700, 2100], hq=8, hkv=2, dk=128, seed=83, page_size=page_size,
                            spare_pages=4)
        check(p, num_splits=3)


"""GPU parity of the e4m3 KV path (per-token scales, Q/K 192 with V/O 128,
paged and packed) against the fp64 oracle, plus the >4 GiB page-offset run."""
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


def test_config4_paged_fp8_every_row():
    """Config 4 (16 sequences of U{1..4096} tokens, H 16, e4m3 K/V with
    per-token scales, Q/K 192, V/O 128, page 64, causal), every (token,
    head) row against the oracle."""
    p = fi.config4()
    o, l = host(*run_gpu(p))
    ro, rl = oracle.forward(p)
    compare(o, l, ro, rl)


FP8_EDGE = [
    dict(lens_q=[300, 129, 1], lens_k=[700, 129, 300], hq=4, hkv=2, dk=192, dv=128, page_size=1024, causal=True),
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, dk=128, page_size=512, spare_pages=2),
    dict(lens_q=[300, 129, 1], lens_k=[300, 400, 77], hq=4, hkv=4, dk=192, dv=128, page_size=64, causal=True),
    dict(lens_q=[300, 129], lens_k=[300, 400], hq=4, hkv=2, dk=128, page_size=16, spare_pages=4),
    dict(lens_q=[200, 64, 3], lens_k=[260, 64, 500], hq=8, hkv=1, dk=64, page_size=32, causal=True, window=90),
    dict(lens_q=[257, 33], lens_k=[600, 33], hq=4, hkv=2, dk=192, dv=128),                       # packed e4m3
    dict(lens_q=[130, 260], lens_k=[130, 260], hq=4, dk=128, page_size=128, mod="alibi"),
    dict(lens_q=[130, 70], lens_k=[300, 70], hq=4, dk=128, page_size=64, mod="softcap", softcap=5.0),
    dict(lens_q=[0, 5, 0], lens_k=[7, 0, 0], hq=2, dk=64, page_size=16),                            # empty rows
    dict(lens_q=[200, 330], lens_k=[200, 330], hq=4, dk=128, page_size=64, block_mask_density=0.5),
]


@pytest.mark.parametrize("case", range(len(FP8_EDGE)))
def test_fp8_edge_cases(case):
    kw = dict(FP8_EDGE[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    check(fi.make_problem(lens_q, lens_k, seed=200 + case, kv_dtype="e4m3", **kw))


def test_fp8_single_key_all_bytes_bit_exact():
    """V holds every finite e4m3 byte, scales 1, one visible key per row:
    out must equal the decoded byte exactly (exact e4m3 -> bf16 conversion)."""
    p = fi.make_problem([64, 64], [64, 64], hq=4, hkv=2, dk=128, dv=128, seed=9, kv_dtype="e4m3",
                        page_size=16, causal=True, window=1)
    finite = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], dtype=np.uint8)
    v = p.v.copy()
    n = v.shape[0] * v.shape[1] * v.shape[2]
    v.reshape(n, -1)[:] = np.resize(finite, (n, v.shape[-1]))
    p = p.replace(v=v, v_scale=np.where(np.isnan(p.v_scale), np.nan, np.float32(1.0)).astype(np.float32))
    o, _ = run_gpu(p)
    torch.cuda.synchronize()
    got = o.view(torch.int16).cpu().numpy().view(np.uint16)
    ro, _ = oracle.forward(p)
    assert np.array_equal(got, fi.bf16_bits(ro.astype(np.float32)))


def test_fp8_matches_bf16_kernel_on_exact_values():
    """With unit scales, the e4m3 values are exact bf16 values: the e4m3 kernel
    and the bf16 kernel see the same S and V and must agree to rounding."""
    p8 = fi.make_problem([300, 90], [300, 500], hq=4, hkv=2, dk=128, seed=12, kv_dtype="e4m3",
                         page_size=64, causal=True, softmax_scale=0.0005)
    ones = lambda a: np.where(np.isnan(a), np.nan, np.float32(1.0)).astype(np.float32)
    p8 = p8.replace(k_scale=ones(p8.k_scale), v_scale=ones(p8.v_scale))
    kd = torch.from_numpy(p8.k.copy()).view(torch.float8_e4m3fn).float()
    vd = torch.from_numpy(p8.v.copy()).view(torch.float8_e4m3fn).float()
    pb = p8.replace(kv_dtype="bf16", k=fi.bf16_bits(torch.nan_to_num(kd).numpy()),
                    v=fi.bf16_bits(torch.nan_to_num(vd).numpy()), k_scale=None, v_scale=None)
    o8, l8 = host(*run_gpu(p8))
    ob, lb = host(*run_gpu(pb))
    ro, rl = oracle.forward(p8)
    scale = max(1.0, float(np.abs(ro).max()) / 4)      # |v| reaches 448 here
    assert np.max(np.abs(o8 - ob)) <= 2e-2 * scale
    fin = np.isfinite(lb)
    assert np.max(np.abs(l8[fin] - lb[fin])) <= 1e-4


def test_fp8_page_offsets_above_4gib():
    """524289 pages of (page 64, Hkv 1, Q/K 192, V/O 128) e4m3: page 524288 starts
    at byte 2**32 of V (and past it in K); two sequences read it."""
    geo = fi.big_pool_geometry()
    need = geo["cache_bytes"] + geo["num_pages"] * 64 * 4 * 2
    free, _ = torch.cuda.mem_get_info()
    if free < need + (2 << 30):
        pytest.skip(f"needs {need / 2**30:.1f} GiB + 2 GiB free, have {free / 2**30:.1f} GiB")
    p, pbt, n_pages = fi.config4_big()
    ro, rl = oracle.forward(p)
    t = to_device(p)
    # the same pages placed at the top of a 524289-page pool
    kbig = torch.zeros((n_pages, 64, 1, 192), dtype=torch.uint8, device="cuda")
    vbig = torch.zeros((n_pages, 64, 1, 128), dtype=torch.uint8, device="cuda")
    ksb = torch.zeros((n_pages, 64, 1), dtype=torch.float32, device="cuda")
    vsb = torch.zeros((n_pages, 64, 1), dtype=torch.float32, device="cuda")
    loc = torch.from_numpy(p.block_table[p.block_table >= 0].astype(np.int64)).cuda()
    phy = torch.from_numpy(pbt[pbt >= 0].astype(np.int64)).cuda()
    kbig[phy] = t["k"].view(torch.uint8)[loc]
    vbig[phy] = t["v"].view(torch.uint8)[loc]
    ksb[phy] = t["k_scale"][loc]
    vsb[phy] = t["v_scale"][loc]
    big = dict(t)
    big.update(k=kbig.view(torch.float8_e4m3fn), v=vbig.view(torch.float8_e4m3fn), k_scale=ksb, v_scale=vsb,
               bt=torch.from_numpy(pbt).cuda())
    assert int(pbt.max()) * 128 * 64 >= 2 ** 32
    o_big, l_big = host(*run_gpu(p, big))
    o_low, l_low = host(*run_gpu(p, t))
    compare(o_big, l_big, ro, rl)
    assert np.array_equal(o_big, o_low) and np.array_equal(l_big, l_low)
    del kbig, vbig, ksb, vsb
    torch.cuda.empty_cache()

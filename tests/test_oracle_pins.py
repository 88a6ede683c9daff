"""Pins of the fp64 oracle against things other than itself.

Each test fixes the oracle to a closed form, a brute-force enumeration, a
library routine (torch's fp64 scaled_dot_product_attention / logsumexp /
float8 decode), or an invariant that a plausible mistake (a dropped term, a
wrong sign or index, a transposed operand, a wrong head map) would break.
No GPU is used.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers ----

def kv_tokens_f64(p, which):
    """Per-sequence dequantised K or V as float64 [T_k, Hkv, D] (packed order).

    Test-side gather through the block table; scales applied with torch.
    """
    pool = p.k if which == "k" else p.v
    sc = p.k_scale if which == "k" else p.v_scale
    if p.kv_dtype == "bf16":
        vals = fi.bf16_to_f32(pool).astype(np.float64)
    else:
        vals = torch.from_numpy(pool.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        vals = vals * sc.astype(np.float64)[..., None]
    if not p.paged:
        return vals
    rows = []
    for b in range(p.num_seqs):
        j = np.arange(int(p.seqlens_k[b]))
        rows.append(vals[p.block_table[b, j // p.page_size], j % p.page_size])
    d = vals.shape[-1]
    return np.concatenate(rows) if rows else np.zeros((0, p.hkv, d))


def brute_mask(p, b, h, sq, sk):
    """The allowed set by nested loops over the reading of the masks."""
    m = np.zeros((sq, sk), dtype=bool)
    for i in range(sq):
        ip = i + sk - sq
        for j in range(sk):
            ok = True
            if p.causal and j > ip:
                ok = False
            if p.window > 0:
                if p.causal and ip - j >= p.window:
                    ok = False
                if not p.causal and abs(ip - j) >= p.window:
                    ok = False
            if p.block_mask is not None and not p.block_mask[b * p.hq + h, i // 128, j // 128]:
                ok = False
            m[i, j] = ok
    return m


def apply_ops(x, ops):
    """A prologue op chain applied to a widened numpy array, op after op."""
    for name, c in ops or ():
        x = {"mul": lambda a: a * c, "add": lambda a: a + c, "sub": lambda a: a - c,
             "div": lambda a: a / c}[name](x)
    return x


def sdpa_reference(p, bias_fn=None, maps=None):
    """torch fp64 SDPA per sequence (GQA by repeat_interleave) and logsumexp.
    ``maps``: prologue op chains {"q": [...], "k": [...], "v": [...]}
    applied to the widened tensors first."""
    if p.q_dtype == "e4m3":
        q = torch.from_numpy(p.q.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        q = fi.bf16_to_f32(p.q).astype(np.float64)
    k = kv_tokens_f64(p, "k")
    v = kv_tokens_f64(p, "v")
    if maps is not None:
        q, k, v = apply_ops(q, maps.get("q")), apply_ops(k, maps.get("k")), apply_ops(v, maps.get("v"))
    g = p.hq // p.hkv
    outs = np.zeros((p.total_q, p.hq, p.dv))
    lses = np.zeros((p.hq, p.total_q))
    for b in range(p.num_seqs):
        q0, q1 = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        k0, k1 = int(p.cu_seqlens_k[b]), int(p.cu_seqlens_k[b + 1])
        sq, sk = q1 - q0, k1 - k0
        if sq == 0:
            continue
        qt = torch.from_numpy(q[q0:q1]).permute(1, 0, 2)                      # [Hq, Sq, Dk]
        kt = torch.from_numpy(k[k0:k1]).permute(1, 0, 2).repeat_interleave(g, 0)
        vt = torch.from_numpy(v[k0:k1]).permute(1, 0, 2).repeat_interleave(g, 0)
        allow = torch.from_numpy(np.stack([brute_mask(p, b, h, sq, sk) for h in range(p.hq)]))
        bias = torch.zeros((p.hq, sq, sk), dtype=torch.float64)
        if bias_fn is not None:
            bias = bias + bias_fn(sq, sk)
        full = torch.where(allow, bias, torch.tensor(-math.inf, dtype=torch.float64))
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=full, scale=p.softmax_scale)
        scores = torch.einsum("hid,hjd->hij", qt, kt) * p.softmax_scale + full
        lse = torch.logsumexp(scores, dim=-1)
        empty = ~allow.any(-1)
        o = torch.where(empty[..., None], torch.zeros_like(o), o)
        outs[q0:q1] = o.permute(1, 0, 2).numpy()
        lses[:, q0:q1] = lse.numpy()
    return outs, lses


def assert_close(a, b, tol=1e-11):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    inf_a, inf_b = np.isneginf(a), np.isneginf(b)
    assert np.array_equal(inf_a, inf_b)
    assert not np.isnan(a).any() and not np.isnan(b).any()
    fa, fb = a[~inf_a], b[~inf_b]
    if fa.size:
        assert np.max(np.abs(fa - fb)) <= tol, np.max(np.abs(fa - fb))


# ------------------------------------------------------- scalar decoders ----

def test_e4m3_decode_ocp_points():
    """OCP E4M3 table points: max normal, min normal, min subnormal, one, NaN."""
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0xB8) == -1.0
    assert oracle.e4m3_decode(0x77) == 240.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    z = oracle.e4m3_decode(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


def test_e4m3_decode_all_bytes_match_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for b in range(256):
        mine, lib = oracle.e4m3_decode(b), float(ref[b])
        assert (math.isnan(mine) and math.isnan(lib)) or mine == lib, b


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 16, size=2000).astype(np.uint16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits, lib):
        m = oracle.bf16_decode(int(b))
        assert (math.isnan(m) and math.isnan(r)) or m == r


# ------------------------------------------------------------ closed forms --

def _identical_keys(p):
    """Overwrite every key of a sequence/head with that sequence's first key."""
    k = p.k.copy()
    for b in range(p.num_seqs):
        lo, hi = int(p.cu_seqlens_k[b]), int(p.cu_seqlens_k[b + 1])
        if hi > lo:
            k[lo:hi] = k[lo]
    return p.replace(k=k)


@pytest.mark.parametrize("mod", ["none", "softcap"])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5), (False, 7)])
def test_identical_keys_give_mean_and_log_count(mod, causal, window):
    """All allowed keys equal => out = mean of allowed V, LSE = s + ln|A|."""
    p = fi.make_problem([9, 0, 13, 4], [9, 3, 20, 11], hq=4, hkv=2, dk=16, dv=8, seed=1,
                        causal=causal, window=window, mod=mod, softcap=3.0)
    p = _identical_keys(p)
    out, lse = oracle.forward(p)
    q = fi.bf16_to_f32(p.q).astype(np.float64)
    k = fi.bf16_to_f32(p.k).astype(np.float64)
    v = fi.bf16_to_f32(p.v).astype(np.float64)
    for b in range(p.num_seqs):
        q0, q1 = p.cu_seqlens_q[b], p.cu_seqlens_q[b + 1]
        k0 = p.cu_seqlens_k[b]
        sq, sk = q1 - q0, p.cu_seqlens_k[b + 1] - k0
        for h in range(p.hq):
            hk = h // 2
            allow = brute_mask(p, b, h, sq, sk)
            for i in range(sq):
                n = allow[i].sum()
                t = q0 + i
                if n == 0:
                    assert lse[h, t] == -np.inf and np.all(out[t, h] == 0)
                    continue
                s = p.softmax_scale * float(q[t, h] @ k[k0, hk])
                if mod == "softcap":
                    s = 3.0 * math.tanh(s / 3.0)
                js = np.nonzero(allow[i])[0]
                mean = v[k0 + js, hk].mean(axis=0)
                assert abs(lse[h, t] - (s + math.log(n))) < 1e-12
                assert np.max(np.abs(out[t, h] - mean)) < 1e-12


def test_single_key_returns_that_value_row():
    """Sk = 1: out = v exactly, LSE = s (bit-exact in fp64)."""
    p = fi.make_problem([1, 1, 1], [1, 1, 1], hq=4, hkv=4, dk=32, seed=2)
    out, lse = oracle.forward(p)
    q = fi.bf16_to_f32(p.q).astype(np.float64)
    k = fi.bf16_to_f32(p.k).astype(np.float64)
    v = fi.bf16_to_f32(p.v).astype(np.float64)
    assert np.array_equal(out, v)
    s = np.einsum("thd,thd->ht", q, k) * p.softmax_scale
    assert np.max(np.abs(lse - s)) < 1e-13


def test_causal_window_one_picks_the_diagonal_key():
    """Causal with W=1 leaves only j = i' (paged, shuffled): out = v[i']."""
    p = fi.make_problem([5, 17], [9, 40], hq=2, hkv=1, dk=16, dv=16, seed=4, causal=True,
                        window=1, page_size=16, spare_pages=3)
    out, _ = oracle.forward(p)
    v = kv_tokens_f64(p, "v")
    for b in range(2):
        sq, sk = int(p.seqlens_q[b]), int(p.seqlens_k[b])
        for i in range(sq):
            t = p.cu_seqlens_q[b] + i
            for h in range(2):
                assert np.array_equal(out[t, h], v[p.cu_seqlens_k[b] + i + sk - sq, 0])


def test_zero_length_sequences():
    """Sq = 0 contributes no rows; Sk = 0 with Sq > 0 gives out 0 and LSE -inf."""
    p = fi.make_problem([0, 3, 0, 2], [5, 0, 0, 4], hq=2, dk=16, seed=5)
    out, lse = oracle.forward(p)
    assert out.shape == (5, 2, 16) and lse.shape == (2, 5)
    assert np.all(out[0:3] == 0) and np.all(np.isneginf(lse[:, 0:3]))
    assert np.all(np.isfinite(lse[:, 3:5]))


def test_softcap_two_key_closed_form():
    """q = c*e0, k1 = e0, k2 = 0: s1 = scale*c, s2 = 0, capped on the scaled score."""
    p = fi.make_problem([1], [2], hq=1, dk=16, dv=4, seed=6, mod="softcap", softcap=2.0,
                        softmax_scale=0.5)
    q = np.zeros((1, 1, 16), np.float32)
    q[0, 0, 0] = 6.0
    k = np.zeros((2, 1, 16), np.float32)
    k[0, 0, 0] = 1.0
    p = p.replace(q=fi.bf16_bits(q), k=fi.bf16_bits(k))
    out, lse = oracle.forward(p)
    v = fi.bf16_to_f32(p.v).astype(np.float64)[:, 0]
    a = 2.0 * math.tanh(0.5 * 6.0 / 2.0)
    w1, w2 = math.exp(a), 1.0
    assert abs(lse[0, 0] - math.log(w1 + w2)) < 1e-13
    assert np.max(np.abs(out[0, 0] - (w1 * v[0] + w2 * v[1]) / (w1 + w2))) < 1e-13


# --------------------------------------------------------- brute force masks --

@pytest.mark.parametrize("causal,window,density", [
    (False, 0, None), (True, 0, None), (True, 3, None), (False, 4, None),
    (False, 0, 0.5), (True, 0, 0.6), (True, 200, 0.5)])
def test_effective_mask_equals_brute_force(causal, window, density):
    """Identical keys and one-hot V (V[j] = e_j) expose the allowed set as the
    support of each output row; it must equal the brute-force enumeration."""
    lens_q, lens_k = [1, 130, 7, 0, 129], [1, 300, 260, 5, 129]
    p = fi.make_problem(lens_q, lens_k, hq=2, hkv=1, dk=8, dv=300, seed=7, causal=causal,
                        window=window, block_mask_density=density)
    p = _identical_keys(p)
    v = np.zeros((p.total_k, 1, 300), np.float32)
    for b in range(p.num_seqs):
        for j in range(int(p.seqlens_k[b])):
            v[p.cu_seqlens_k[b] + j, 0, j] = 1.0
    p = p.replace(v=fi.bf16_bits(v))
    out, lse = oracle.forward(p)
    for b in range(p.num_seqs):
        sq, sk = int(p.seqlens_q[b]), int(p.seqlens_k[b])
        for h in range(p.hq):
            allow = brute_mask(p, b, h, sq, sk)
            got = out[p.cu_seqlens_q[b]:p.cu_seqlens_q[b] + sq, h, :sk] > 0
            assert np.array_equal(got, allow)
            n = allow.sum(1)
            cnt = out[p.cu_seqlens_q[b]:p.cu_seqlens_q[b] + sq, h].sum(1)
            assert np.allclose(cnt[n > 0], 1.0, atol=1e-12)


# ------------------------------------------------------- library routines --

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hkv", [4, 2, 1])
def test_matches_torch_sdpa(causal, hkv):
    p = fi.make_problem([33, 0, 70, 128], [33, 4, 90, 128], hq=4, hkv=hkv, dk=32, dv=16,
                        seed=8, causal=causal)
    out, lse = oracle.forward(p)
    ro, rl = sdpa_reference(p)
    assert_close(out, ro, 1e-12)
    assert_close(lse, rl, 1e-12)


def test_alibi_matches_sdpa_additive_bias():
    p = fi.make_problem([40, 64], [70, 64], hq=2, dk=16, seed=9, mod="alibi",
                        alibi_slope=0.0625, causal=False)

    def bias(sq, sk):
        i = torch.arange(sq, dtype=torch.float64)[:, None] + (sk - sq)
        j = torch.arange(sk, dtype=torch.float64)[None, :]
        return -0.0625 * (i - j).abs()

    out, lse = oracle.forward(p)
    ro, rl = sdpa_reference(p, bias)
    assert_close(out, ro, 1e-12)
    assert_close(lse, rl, 1e-12)


def test_block_mask_matches_sdpa_boolean_mask():
    p = fi.make_problem([300, 129], [260, 400], hq=2, hkv=1, dk=16, seed=10,
                        block_mask_density=0.5)
    out, lse = oracle.forward(p)
    ro, rl = sdpa_reference(p)
    assert_close(out, ro, 1e-12)
    assert_close(lse, rl, 1e-12)


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 150), (False, 200)])
def test_alibi_gqa_window_block_mask_together_match_sdpa(causal, window):
    """Every mask and the ALiBi bias at once, with GQA and Sq != Sk, against
    torch SDPA with the brute-force mask and the bias written out."""
    slope = 0.03
    p = fi.make_problem([300, 129, 0], [420, 129, 50], hq=4, hkv=2, dk=16, seed=31, causal=causal,
                        window=window, mod="alibi", alibi_slope=slope, block_mask_density=0.6,
                        page_size=16, spare_pages=3)

    def bias(sq, sk):
        i = torch.arange(sq, dtype=torch.float64)[:, None] + (sk - sq)
        j = torch.arange(sk, dtype=torch.float64)[None, :]
        return -slope * (i - j).abs()

    out, lse = oracle.forward(p)
    ro, rl = sdpa_reference(p, bias)
    assert_close(out, ro, 1e-12)
    assert_close(lse, rl, 1e-12)


def test_softcap_with_masks_matches_explicit_scores():
    """The soft-cap under causal, window and block masks against scores formed
    one by one (cap * tanh(scale * q.k / cap), then the masks) and a plain
    softmax: the cap applies to the scaled score, before masking."""
    cap = 2.5
    p = fi.make_problem([200, 7], [260, 7], hq=2, hkv=1, dk=16, seed=32, causal=True, window=120,
                        mod="softcap", softcap=cap, block_mask_density=0.7)
    out, lse = oracle.forward(p)
    q = fi.bf16_to_f32(p.q).astype(np.float64)
    k = kv_tokens_f64(p, "k")
    v = kv_tokens_f64(p, "v")
    for b in range(p.num_seqs):
        q0, q1 = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        k0, k1 = int(p.cu_seqlens_k[b]), int(p.cu_seqlens_k[b + 1])
        sq, sk = q1 - q0, k1 - k0
        for h in range(p.hq):
            allow = brute_mask(p, b, h, sq, sk)
            s = cap * np.tanh(p.softmax_scale * (q[q0:q1, h] @ k[k0:k1, 0].T) / cap)
            for i in range(sq):
                a = allow[i]
                if not a.any():
                    assert np.isneginf(lse[h, q0 + i]) and not out[q0 + i, h].any()
                    continue
                m = s[i, a].max()
                w = np.exp(s[i, a] - m)
                np.testing.assert_allclose(out[q0 + i, h], (w @ v[k0:k1, 0][a]) / w.sum(), atol=1e-12)
                np.testing.assert_allclose(lse[h, q0 + i], m + np.log(w.sum()), atol=1e-12)


def test_block_causal_mask_equals_causal_on_block_level():
    """BlockMask.causal with Sq = Sk multiples of 128 keeps exactly the blocks kb <= qb."""
    p = fi.make_problem([256, 384], hq=2, dk=16, seed=11)
    bm = fi.block_causal_mask(4, 3, 3)
    out, lse = oracle.forward(p.replace(block_mask=bm))
    for b in range(2):
        sq = int(p.seqlens_q[b])
        for h in range(2):
            allow = brute_mask(p.replace(block_mask=bm), b, h, sq, sq)
            blk = np.kron(np.tril(np.ones((sq // 128, sq // 128), bool)), np.ones((128, 128), bool))
            assert np.array_equal(allow, blk)
    ro, rl = sdpa_reference(p.replace(block_mask=bm))
    assert_close(lse, rl, 1e-12)


# ------------------------------------------------------- special cases ------

def test_softcap_huge_and_alibi_zero_reduce_to_plain():
    base = fi.make_problem([50, 9], [70, 9], hq=2, dk=32, seed=12, causal=True)
    o0, l0 = oracle.forward(base)
    o1, l1 = oracle.forward(base.replace(mod_kind=fi.MOD_SOFTCAP, softcap=1e30))
    o2, l2 = oracle.forward(base.replace(mod_kind=fi.MOD_ALIBI, alibi_slope=0.0))
    o3, l3 = oracle.forward(base.replace(block_mask=np.ones((4, 1, 1), np.uint8)))
    for o, l in ((o1, l1), (o2, l2), (o3, l3)):
        assert_close(o, o0, 1e-12)
        assert_close(l, l0, 1e-12)


# ------------------------------------------------------- invariants ---------

@pytest.mark.parametrize("page_size", [1, 2, 16])
def test_paged_equals_packed_bit_identical(page_size):
    """Same K/V placed in shuffled pages (with NaN-poisoned spare slots and -1
    block-table padding) gives bit-identical fp64 results."""
    kw = dict(hq=4, hkv=2, dk=32, dv=16, seed=13, causal=True)
    packed = fi.make_problem([20, 37, 1], [50, 37, 70], **kw)
    paged = fi.make_problem([20, 37, 1], [50, 37, 70], page_size=page_size, spare_pages=5,
                            max_pages=(70 + page_size - 1) // page_size + 2, **kw)
    assert np.array_equal(kv_tokens_f64(paged, "k"), kv_tokens_f64(packed, "k"))
    o1, l1 = oracle.forward(packed)
    o2, l2 = oracle.forward(paged)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert not np.isnan(o2).any()


def test_e4m3_with_scales_equals_dequantised_f64():
    """e4m3 bytes x per-token scales (decoded by torch) fed as plain doubles
    give the same result: pins the decode and where each scale applies."""
    p = fi.make_problem([30, 64], [45, 64], hq=4, hkv=2, dk=48, dv=32, seed=14,
                        page_size=16, kv_dtype="e4m3", spare_pages=2, causal=True)
    kd = torch.from_numpy(p.k.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vd = torch.from_numpy(p.v.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    kd = kd * p.k_scale.astype(np.float64)[..., None]
    vd = vd * p.v_scale.astype(np.float64)[..., None]
    o1, l1 = oracle.forward(p)
    o2, l2 = oracle.forward(p, k_f64=np.nan_to_num(kd), v_f64=np.nan_to_num(vd))
    assert_close(o1, o2, 1e-13)
    assert_close(l1, l2, 1e-13)
    # Swapping the two scales must change the answer.
    o3, _ = oracle.forward(p.replace(k_scale=p.v_scale, v_scale=p.k_scale))
    assert np.max(np.abs(o3 - o1)) > 1e-3


def test_gqa_equals_repeated_kv_heads():
    """Hq=6, Hkv=2 with contiguous groups equals Hq=Hkv=6 with each kv head repeated."""
    p = fi.make_problem([25, 40], [31, 40], hq=6, hkv=2, dk=16, seed=15, causal=True)
    rep = p.replace(k=np.repeat(p.k, 3, axis=1), v=np.repeat(p.v, 3, axis=1), hkv=6)
    o1, l1 = oracle.forward(p)
    o2, l2 = oracle.forward(rep)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_combine_of_disjoint_key_ranges_equals_full(splits):
    p = fi.make_problem([3, 1, 6], [100, 37, 64], hq=4, hkv=2, dk=16, seed=16, causal=True,
                        page_size=16, spare_pages=2)
    full_o, full_l = oracle.forward(p)
    edges = np.linspace(0, 100, splits + 1).astype(int)
    parts_o, parts_l = [], []
    for s in range(splits):
        o, l = oracle.forward(p, kv_range=(edges[s], edges[s + 1]))
        parts_o.append(o.reshape(-1, p.dv))
        parts_l.append(l.T.reshape(-1))
    o, l = oracle.combine(np.stack(parts_o), np.stack(parts_l))
    assert_close(o.reshape(full_o.shape), full_o, 1e-12)
    assert_close(l.reshape(p.total_q, p.hq).T, full_l, 1e-12)


def test_combine_all_empty_gives_zero_and_neg_inf():
    o, l = oracle.combine(np.ones((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_unit_subset_matches_full_run():
    p = fi.make_problem([70, 5], [70, 300], hq=4, hkv=1, dk=32, seed=17, causal=True)
    full_o, full_l = oracle.forward(p)
    units = np.array([[0, 0], [69, 3], [70, 1], [74, 2]], np.int64)
    o, l = oracle.forward(p, units=units)
    for r, (t, h) in enumerate(units):
        assert np.array_equal(o[r], full_o[t, h]) and l[r] == full_l[h, t]


# ------------------------------------------------------- golden fixture ----

def test_big_pool_geometry_matches_the_page():
    g = json.load(open(os.path.join(GOLDEN, "big_pool_geometry.json")))
    mine = fi.big_pool_geometry(g["page_size"], g["qk_head_dim"], g["v_head_dim"], g["kv_heads"])
    assert min(mine["key_page_bytes"], mine["value_page_bytes"]) == g["min_page_bytes"]
    assert mine["high_page"] == g["high_page"]
    assert mine["num_pages"] == g["num_pages"]
    assert mine["cache_bytes"] == g["cache_bytes"]
    assert mine["key_page_bytes"] + mine["value_page_bytes"] == g["cache_bytes_per_page"]
    assert mine["high_page"] * mine["key_page_bytes"] >= 2 ** 32
    assert mine["high_page"] * mine["value_page_bytes"] >= 2 ** 32


# --------------------------------------------------------------- int8 KV --

def test_i8_decode_all_bytes_are_twos_complement():
    """Every stored byte decodes to the int8 value numpy assigns it."""
    ref = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    for b in range(256):
        assert oracle.i8_decode(b) == ref[b], b


def test_int8_encoder_bounds():
    """The generator's per-token int8 codes stay in [-127, 127], hit 127 in
    magnitude on every non-zero row, and round to nearest (|x - q*s| <= s/2)."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((50, 3, 40)).astype(np.float32)
    x[7, 1] = 0.0
    q, s = fi.int8_quantize_per_token(x)
    assert q.dtype == np.int8 and q.min() >= -127 and q.max() <= 127
    nz = s > 0
    assert np.all(np.abs(q).max(axis=-1)[nz] == 127) and not nz[7, 1] and np.all(q[7, 1] == 0)
    err = np.abs(x - q.astype(np.float32) * s[..., None])
    assert np.all(err <= s[..., None] * 0.5000001)


def test_int8_with_scales_matches_torch_sdpa_on_dequantised_values():
    """int8 K/V with per-token scales against torch's scaled-dot-product
    attention and logsumexp on the dequantised doubles (an implementation that
    shares nothing with the oracle): pins the decode and where each scale
    applies; swapping the two scales must change the answer."""
    p = fi.make_problem([37, 64], [45, 64], hq=4, hkv=2, dk=48, dv=32, seed=22,
                        page_size=16, kv_dtype="int8", spare_pages=2)
    o1, l1 = oracle.forward(p)
    for b in range(p.num_seqs):
        q0, q1 = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        sk = int(p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b])
        keys = np.arange(sk)
        pages = p.block_table[b, keys // p.page_size]
        slots = keys % p.page_size
        k = p.k[pages, slots].astype(np.float64) * p.k_scale[pages, slots].astype(np.float64)[..., None]
        v = p.v[pages, slots].astype(np.float64) * p.v_scale[pages, slots].astype(np.float64)[..., None]
        q = fi.bf16_to_f32(p.q[q0:q1]).astype(np.float64)
        kk = torch.from_numpy(np.repeat(k, 2, axis=1)).permute(1, 0, 2)     # [Hq, sk, dk]
        vv = torch.from_numpy(np.repeat(v, 2, axis=1)).permute(1, 0, 2)
        qq = torch.from_numpy(q).permute(1, 0, 2)
        s = torch.matmul(qq, kk.transpose(1, 2)) * p.softmax_scale
        ref_o = torch.softmax(s, dim=-1) @ vv
        ref_l = torch.logsumexp(s, dim=-1)
        assert_close(o1[q0:q1], ref_o.permute(1, 0, 2).numpy(), 1e-12)
        assert_close(l1[:, q0:q1], ref_l.numpy(), 1e-12)
    o3, _ = oracle.forward(p.replace(k_scale=p.v_scale, v_scale=p.k_scale))
    assert np.max(np.abs(o3 - o1)) > 1e-3


@pytest.mark.parametrize("dk,dv", [(32, 16), (192, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_e4m3_q_matches_torch_sdpa(causal, dk, dv):
    """e4m3 Q bytes (decoded by torch) with paged e4m3 K/V against torch's
    fp64 SDPA: pins the Q decode and the Q byte layout, also at the Q/K 192,
    V/O 128 geometry."""
    p = fi.make_problem([37, 0, 64], [45, 3, 64], hq=4, hkv=2, dk=dk, dv=dv, seed=23,
                        page_size=16, kv_dtype="e4m3", spare_pages=2, causal=causal,
                        q_dtype="e4m3")
    assert p.q.dtype == np.uint8 and p.q.shape == (101, 4, dk)
    out, lse = oracle.forward(p)
    ro, rl = sdpa_reference(p)
    assert_close(out, ro, 1e-12)
    assert_close(lse, rl, 1e-12)


def test_e4m3_q_scale_is_folded_into_softmax_scale():
    """The per-tensor Q scale (max|Q|/448) reaches the scores only through
    softmax_scale: the e4m3-Q problem must agree with the bf16-Q problem of the
    same seed to within e4m3's rounding (3 mantissa bits), and must not once the
    fold is undone."""
    kw = dict(hq=2, hkv=1, dk=64, dv=64, seed=24, causal=True)
    pb = fi.make_problem([96, 40], [128, 40], **kw)
    pe = fi.make_problem([96, 40], [128, 40], q_dtype="e4m3", **kw)
    qb = fi.bf16_to_f32(pb.q)
    qe = torch.from_numpy(pe.q.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    qs = pe.softmax_scale / pb.softmax_scale
    assert qs == pytest.approx(np.abs(qb).max() / 448.0, rel=1e-2)
    assert np.abs(qe).max() <= 448.0
    # every decoded Q element times the scale is within e4m3's half-ulp of Q
    err = np.abs(qe * qs - qb)
    assert np.all(err <= np.maximum(np.abs(qb) * 2.0 ** -4, 2.0 ** -10 * qs) + 1e-2 * np.abs(qb))
    ob, lb = oracle.forward(pb)
    oe, le = oracle.forward(pe)
    assert np.max(np.abs(oe - ob)) < 0.1 and np.max(np.abs(le - lb)) < 0.1
    ou, lu = oracle.forward(pe.replace(softmax_scale=pb.softmax_scale))
    assert np.max(np.abs(lu - lb)) > 1.0


# ---------------------------------------------------------------- prologue ----
# Op chains (Mul, Add, Sub, Div by scalars) applied in order to every element
# of Q, K and V as read (fkl_python PR #7, prologue-fusion commit).

PRO = {"q": [("mul", 0.75), ("add", 0.2)], "k": [("sub", 0.3), ("mul", -1.5), ("div", 1.25)],
       "v": [("add", -0.25), ("mul", 2.0)]}


@pytest.mark.parametrize("causal,paged", [(False, False), (True, False), (True, True)])
def test_prologue_matches_sdpa_on_transformed_inputs(causal, paged):
    p = fi.make_problem([33, 0, 70, 20], [33, 4, 90, 0], hq=4, hkv=2, dk=32, dv=16, seed=21, causal=causal,
                        page_size=16 if paged else 0, spare_pages=3).replace(prologue=PRO)
    out, lse = oracle.forward(p)
    ro, rl = sdpa_reference(p, maps=PRO)
    assert_close(out, ro, 1e-12)
    assert_close(lse, rl, 1e-12)


def test_prologue_ops_apply_in_order():
    """(x + 1) * 2 and x * 2 + 1 differ; x * 2 + 2 equals (x + 1) * 2."""
    base = fi.make_problem([40, 7], [50, 30], hq=2, dk=16, seed=25, causal=True)
    add_mul = oracle.forward(base.replace(prologue={"k": [("add", 1.0), ("mul", 2.0)]}))
    mul_add = oracle.forward(base.replace(prologue={"k": [("mul", 2.0), ("add", 1.0)]}))
    same = oracle.forward(base.replace(prologue={"k": [("mul", 2.0), ("add", 2.0)]}))
    assert np.max(np.abs(add_mul[1] - mul_add[1])[np.isfinite(add_mul[1])]) > 0.1
    assert_close(add_mul[0], same[0], 1e-12)
    assert_close(add_mul[1], same[1], 1e-12)
    sub_div = oracle.forward(base.replace(prologue={"v": [("sub", 0.5), ("div", 4.0)]}))
    mul_add_v = oracle.forward(base.replace(prologue={"v": [("mul", 0.25), ("add", -0.125)]}))
    assert_close(sub_div[0], mul_add_v[0], 1e-12)


def test_prologue_q_shift_adds_a_per_key_term():
    """Adding c to every element of q adds scale * c * sum_d k_j[d] to score
    j; with one visible key per row (causal, window 1) the output is that
    key's v exactly and the LSE is the shifted score."""
    base = fi.make_problem([20, 9], [20, 30], hq=2, dk=16, seed=26, causal=True, window=1)
    c = 0.6
    out0, lse0 = oracle.forward(base)
    out1, lse1 = oracle.forward(base.replace(prologue={"q": [("add", c)]}))
    assert_close(out1, out0, 0.0)
    k = kv_tokens_f64(base, "k")                                    # [T_k, Hkv, D]
    shift = np.zeros_like(lse0)
    for b in range(base.num_seqs):
        q0, q1 = int(base.cu_seqlens_q[b]), int(base.cu_seqlens_q[b + 1])
        k0, sk = int(base.cu_seqlens_k[b]), int(base.seqlens_k[b])
        sq = q1 - q0
        for i in range(sq):
            j = i + sk - sq                                         # the diagonal key
            for h in range(base.hq):
                shift[h, q0 + i] = base.softmax_scale * c * k[k0 + j, h // (base.hq // base.hkv)].sum()
    assert_close(lse1, lse0 + shift, 1e-11)


def test_prologue_k_shift_moves_only_the_lse():
    """Adding c to every key element adds scale * c * sum_d q_i[d] to every
    score of row i: the softmax is unchanged and the LSE moves by that much."""
    base = fi.make_problem([50, 9], [64, 30], hq=2, dk=16, seed=22, causal=True, mod="alibi", alibi_slope=0.1)
    c = 0.7
    out0, lse0 = oracle.forward(base)
    out1, lse1 = oracle.forward(base.replace(prologue={"k": [("add", c)]}))
    q = fi.bf16_to_f32(base.q).astype(np.float64)                  # [T, H, D]
    shift = base.softmax_scale * c * q.sum(-1).T                   # [H, T]
    assert_close(out1, out0, 1e-12)
    assert_close(lse1, lse0 + np.where(np.isneginf(lse0), 0.0, shift), 1e-11)


def test_prologue_v_map_acts_on_the_output():
    base = fi.make_problem([40, 5], [40, 0], hq=2, dk=16, seed=23, window=6)
    out0, lse0 = oracle.forward(base)
    out1, lse1 = oracle.forward(base.replace(prologue={"v": [("mul", -3.0), ("add", 0.5)]}))
    empty = np.isneginf(lse0).T[..., None]                         # [T, H, 1]
    assert_close(out1, np.where(empty, 0.0, -3.0 * out0 + 0.5), 1e-12)
    assert_close(lse1, lse0, 0.0)


def test_prologue_scales_equal_a_softmax_scale():
    base = fi.make_problem([30], [45], hq=2, dk=16, seed=24, mod="softcap", softcap=3.0)
    out0, lse0 = oracle.forward(base.replace(softmax_scale=base.softmax_scale * 0.5 * 3.0))
    out1, lse1 = oracle.forward(base.replace(prologue={"q": [("mul", 0.5)], "k": [("div", 1 / 3.0)]}))
    assert_close(out1, out0, 1e-12)
    assert_close(lse1, lse0, 1e-12)


def test_oracle_rejects_unknown_prologue_ops():
    base = fi.make_problem([3], [3], hq=1, dk=16, seed=27)
    with pytest.raises(ValueError):
        oracle.forward(base.replace(prologue={"q": [("pow", 2.0)]}))
    with pytest.raises(ValueError):
        oracle.forward(base.replace(prologue={"k": [("mul", 1.0)] * 9}))


def test_config5_runs_share_inputs_and_equal_config5():
    """The benchmark's shared-input config-5 runs are the config5(run)
    problems, field by field (checked at a small sequence length)."""
    import dataclasses
    runs = fi.config5_runs(seq=256, batch=2)
    for run, p in zip(fi.CONFIG5_RUNS, runs):
        ref = fi.config5(run, seq=256, batch=2)
        for f in dataclasses.fields(fi.Problem):
            a, b = getattr(p, f.name), getattr(ref, f.name)
            if isinstance(a, np.ndarray) or isinstance(b, np.ndarray):
                assert (a is None and b is None) or np.array_equal(a, b), (run, f.name)
            else:
                assert a == b, (run, f.name, a, b)

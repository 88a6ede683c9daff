"""Pins of the oracle's backward pass (gradients of sum(dO * out)) against
things other than itself, on the CPU.

* Central finite differences of the forward oracle (itself pinned in
  test_oracle_pins.py): the gradient of L = sum(dO * out) in q, k and v is
  checked entry by entry, including the soft-cap and ALiBi score mods, windows,
  GQA, Sq != Sk and a 128 x 128 block mask.
* torch autograd in float64 on an explicit masked softmax attention.
* Closed forms: with identical keys every row's scores are equal, so dQ = 0
  and dV_j is the mean of dO over the rows that see key j; a single key gives
  dQ = dK = 0 and dV = the sum of dO.
* GQA: a kv head's dK, dV equal the sums over its group of the repeated-heads
  problem.
"""
import numpy as np
import pytest
import torch

import fa_inputs as fi
import oracle


def _f64(p):
    q = fi.bf16_to_f32(p.q).astype(np.float64)
    k = fi.bf16_to_f32(p.k).astype(np.float64)
    v = fi.bf16_to_f32(p.v).astype(np.float64)
    return q, k, v


def _loss(p, dout, q, k, v):
    out, _ = oracle.forward(p, q_f64=q, k_f64=k, v_f64=v, nthreads=1)
    return float(np.sum(dout * out))


FD_CASES = [
    dict(lens_q=[3, 6], hq=2, dk=8, causal=True),
    dict(lens_q=[4, 2], lens_k=[7, 5], hq=4, hkv=2, dk=8, causal=True),          # Sq < Sk, GQA
    dict(lens_q=[6], lens_k=[6], hq=2, dk=8, window=3),                          # non-causal window
    dict(lens_q=[5, 3], hq=2, dk=8, mod="softcap", softcap=0.7, causal=True),    # cap in the curved part
    dict(lens_q=[5], hq=2, dk=8, mod="alibi", alibi_slope=0.5),
    dict(lens_q=[4], lens_k=[2], hq=2, dk=8, causal=True),                       # Sq > Sk: masked rows
    dict(lens_q=[200, 140], lens_k=[260, 140], hq=2, dk=8, causal=True,          # 128 x 128 block mask
         block_mask_density=0.5),
]


@pytest.mark.parametrize("case", range(len(FD_CASES)))
def test_gradients_match_central_differences(case):
    kw = dict(FD_CASES[case])
    lens_q = kw.pop("lens_q")
    lens_k = kw.pop("lens_k", None)
    p = fi.make_problem(lens_q, lens_k, seed=500 + case, **kw)
    q, k, v = _f64(p)
    rng = np.random.default_rng(case)
    dout = rng.standard_normal((p.total_q, p.hq, p.dv))
    dq, dk, dv = oracle.backward(p, dout, q_f64=q, k_f64=k, v_f64=v, nthreads=2)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        flat = x.reshape(-1)
        picks = rng.choice(flat.size, size=min(40, flat.size), replace=False)
        for idx in picks:
            xp, xm = x.copy(), x.copy()
            xp.reshape(-1)[idx] += eps
            xm.reshape(-1)[idx] -= eps
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            fd = (_loss(p, dout, **args_p) - _loss(p, dout, **args_m)) / (2 * eps)
            an = g.reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, an)


def _mask(p, b, sq, sk):
    i = np.arange(sq)[:, None] + (sk - sq)
    j = np.arange(sk)[None, :]
    m = np.ones((sq, sk), dtype=bool)
    if p.causal:
        m &= j <= i
    if p.window > 0:
        m &= ((i - j) < p.window) if p.causal else (np.abs(i - j) < p.window)
    return m


@pytest.mark.parametrize("causal,window,hkv", [(True, 0, 4), (False, 0, 2), (True, 5, 1), (False, 4, 4)])
def test_matches_torch_autograd_f64(causal, window, hkv):
    p = fi.make_problem([7, 0, 12], [9, 3, 12], hq=4, hkv=hkv, dk=16, seed=77, causal=causal, window=window)
    q, k, v = _f64(p)
    rng = np.random.default_rng(3)
    dout = rng.standard_normal((p.total_q, p.hq, p.dv))
    dq, dk, dv = oracle.backward(p, dout, q_f64=q, k_f64=k, v_f64=v)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    g = p.hq // p.hkv
    loss = torch.zeros((), dtype=torch.float64)
    for b in range(p.num_seqs):
        q0, q1 = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        k0, k1 = int(p.cu_seqlens_k[b]), int(p.cu_seqlens_k[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        m = torch.from_numpy(_mask(p, b, q1 - q0, k1 - k0))
        for h in range(p.hq):
            s = p.softmax_scale * tq[q0:q1, h] @ tk[k0:k1, h // g].T
            s = s.masked_fill(~m, float("-inf"))
            pr = torch.softmax(s, dim=-1)
            pr = torch.nan_to_num(pr, nan=0.0)          # fully masked rows: no contribution
            out = pr @ tv[k0:k1, h // g]
            loss = loss + (torch.from_numpy(dout[q0:q1, h]) * out).sum()
    loss.backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12, rtol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_zero_dq_and_mean_dv(causal):
    p = fi.make_problem([6, 9], hq=2, dk=8, seed=9, causal=causal)
    q, k, v = _f64(p)
    k[:] = k[:1]                                   # one key vector everywhere
    rng = np.random.default_rng(1)
    dout = rng.standard_normal((p.total_q, p.hq, p.dv))
    dq, dk, dv = oracle.backward(p, dout, q_f64=q, k_f64=k, v_f64=v)
    assert np.abs(dq).max() < 1e-12
    ref = np.zeros_like(dv)
    for b in range(p.num_seqs):
        q0, sq = int(p.cu_seqlens_q[b]), int(p.seqlens_q[b])
        k0, sk = int(p.cu_seqlens_k[b]), int(p.seqlens_k[b])
        m = _mask(p, b, sq, sk)
        for i in range(sq):
            n = m[i].sum()
            for j in np.nonzero(m[i])[0]:
                ref[k0 + j] += dout[q0 + i] / n
    np.testing.assert_allclose(dv, ref, atol=1e-12)


def test_single_key_gives_zero_dq_dk_and_summed_dv():
    p = fi.make_problem([5, 3], [1, 1], hq=2, dk=8, seed=4)
    q, k, v = _f64(p)
    rng = np.random.default_rng(2)
    dout = rng.standard_normal((p.total_q, p.hq, p.dv))
    dq, dk, dv = oracle.backward(p, dout, q_f64=q, k_f64=k, v_f64=v)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    np.testing.assert_allclose(dv[0], dout[0:5].sum(axis=0), atol=1e-12)
    np.testing.assert_allclose(dv[1], dout[5:8].sum(axis=0), atol=1e-12)


def test_gqa_equals_summed_repeated_heads():
    p = fi.make_problem([10, 7], hq=4, hkv=2, dk=8, seed=12, causal=True)
    q, k, v = _f64(p)
    rng = np.random.default_rng(5)
    dout = rng.standard_normal((p.total_q, p.hq, p.dv))
    dq, dk, dv = oracle.backward(p, dout, q_f64=q, k_f64=k, v_f64=v)
    rep = p.replace(hkv=4)
    k4, v4 = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq4, dk4, dv4 = oracle.backward(rep, dout, q_f64=q, k_f64=k4, v_f64=v4)
    np.testing.assert_allclose(dq, dq4, atol=1e-13)
    np.testing.assert_allclose(dk, dk4.reshape(dk4.shape[0], 2, 2, -1).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, dv4.reshape(dv4.shape[0], 2, 2, -1).sum(axis=2), atol=1e-13)

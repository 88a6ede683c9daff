"""Shared helpers for the GPU parity tests: move a ``fa_inputs.Problem`` to
the device, run the CUDA library through its C ABI, and compare against the
fp64 oracle with the tolerances of the contract:

  * max |out_gpu - out_oracle| <= 1e-2 (bf16 output),
  * |lse_gpu - lse_oracle| <= 1e-3 absolute, -inf matched exactly,
  * rows with an empty key set exactly 0, and no NaN anywhere.
"""
import numpy as np
import torch

import fa_inputs as fi

OUT_TOL = 1e-2
LSE_TOL = 1e-3


def to_device(p, dev="cuda"):
    t = {}
    if p.q_dtype == "e4m3":
        t["q"] = torch.from_numpy(p.q.copy()).view(torch.float8_e4m3fn).to(dev)
    else:
        t["q"] = torch.from_numpy(p.q.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    if p.kv_dtype == "bf16":
        t["k"] = torch.from_numpy(p.k.view(np.int16).copy()).view(torch.bfloat16).to(dev)
        t["v"] = torch.from_numpy(p.v.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    else:
        kvt = torch.int8 if p.kv_dtype == "int8" else torch.float8_e4m3fn
        t["k"] = torch.from_numpy(p.k.copy()).view(kvt).to(dev)
        t["v"] = torch.from_numpy(p.v.copy()).view(kvt).to(dev)
        t["k_scale"] = torch.from_numpy(p.k_scale.copy()).to(dev)
        t["v_scale"] = torch.from_numpy(p.v_scale.copy()).to(dev)
    t["cu_q"] = torch.from_numpy(p.cu_seqlens_q.copy()).to(dev)
    t["cu_k"] = torch.from_numpy(p.cu_seqlens_k.copy()).to(dev)
    if p.block_table is not None:
        t["bt"] = torch.from_numpy(p.block_table.copy()).to(dev)
    if p.block_mask is not None:
        t["bm"] = torch.from_numpy(p.block_mask.copy()).to(dev)
    return t


def run_gpu(p, t=None, num_splits=0, out=None, lse=None, stream=None, workspace=None):
    import flashattention_forward_gb300 as fa
    if t is None:
        t = to_device(p)
    o, l = fa.fwd_varlen(
        t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"],
        max_seqlen_q=p.max_seqlen_q, max_seqlen_k=p.max_seqlen_k, total_k=p.total_k,
        block_table=t.get("bt"), page_size=p.page_size,
        k_scale=t.get("k_scale"), v_scale=t.get("v_scale"),
        softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
        score_mod=p.mod_kind, alibi_slope=p.alibi_slope, softcap=p.softcap,
        block_mask=t.get("bm"), num_splits=num_splits, out=out, lse=lse, stream=stream,
        workspace=workspace, prologue=p.prologue)
    return o, l


def host(o, l):
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64)


def compare(out_g, lse_g, out_o, lse_o, out_tol=OUT_TOL, lse_tol=LSE_TOL):
    """Element-wise comparison; returns (max out err, max lse err)."""
    assert out_g.shape == out_o.shape, (out_g.shape, out_o.shape)
    assert lse_g.shape == lse_o.shape, (lse_g.shape, lse_o.shape)
    assert not np.isnan(out_g).any(), "NaN in GPU output"
    assert not np.isnan(lse_g).any(), "NaN in GPU LSE"
    inf_o = np.isneginf(lse_o)
    assert np.array_equal(np.isneginf(lse_g), inf_o), "-inf LSE rows differ"
    # rows with no allowed key: out exactly zero
    empty = inf_o.T  # [T_q, Hq]
    assert np.all(out_g[empty] == 0.0), "masked rows are not exactly zero"
    eo = float(np.max(np.abs(out_g - out_o))) if out_g.size else 0.0
    fin = ~inf_o
    el = float(np.max(np.abs(lse_g[fin] - lse_o[fin]))) if fin.any() else 0.0
    assert eo <= out_tol, f"max |dout| = {eo} > {out_tol}"
    assert el <= lse_tol, f"max |dlse| = {el} > {lse_tol}"
    return eo, el


def sample_units(p, n, seed=0):
    """(token, head) rows to check: every head of every row at a 128-row tile
    boundary or a sequence end, plus ``n`` distinct seeded random rows
    elsewhere."""
    rng = np.random.default_rng(seed)
    units = set()
    for b in range(p.num_seqs):
        q0, sq = int(p.cu_seqlens_q[b]), int(p.seqlens_q[b])
        for i in list(range(0, sq, 128)) + list(range(127, sq, 128)) + [sq - 1]:
            if 0 <= i < sq:
                for h in range(p.hq):
                    units.add((q0 + i, h))
    boundary = len(units)
    tq = p.total_q
    n = min(n, tq * p.hq - boundary)
    while len(units) < boundary + n:
        units.add((int(rng.integers(tq)), int(rng.integers(p.hq))))
    return np.array(sorted(units), dtype=np.int64)


def compare_units(out_g, lse_g, units, out_o, lse_o, out_tol=OUT_TOL, lse_tol=LSE_TOL):
    og = out_g[units[:, 0], units[:, 1]]
    lg = lse_g[units[:, 1], units[:, 0]]
    assert not np.isnan(og).any() and not np.isnan(lg).any()
    inf_o = np.isneginf(lse_o)
    assert np.array_equal(np.isneginf(lg), inf_o)
    assert np.all(og[inf_o] == 0.0)
    eo = float(np.max(np.abs(og - out_o)))
    el = float(np.max(np.abs(lg[~inf_o] - lse_o[~inf_o]))) if (~inf_o).any() else 0.0
    assert eo <= out_tol, f"max |dout| = {eo}"
    assert el <= lse_tol, f"max |dlse| = {el}"
    return eo, el

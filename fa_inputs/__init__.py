"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the fp64 oracle (``oracle/``) and the CUDA library
(``flashattention_forward_gb300``).  It holds no step of the attention method:
it only draws random numbers, rounds them to the storage formats (bf16, OCP
e4m3 with a per-token scale), lays tokens out packed or in pages behind a
shuffled block table, and poisons every byte the method must never read.

Workload shapes follow the five synthetic configurations of the pages:

* dense causal B=2, H=4, S=128, D=64, scale 1/8 (RL-Kernel PR #237 "SM90 TMA +
  mma.sync FlashAttention", test plan; fkl_python PR #7, host-overhead commit,
  s64 d64 bh8 shape family);
* packed varlen prefill, 8 sequences of length U{0..2048}, H=16, D=128
  (RL-Kernel PR #237, summary: uneven lengths, zero-length sequences);
* paged decode, 64 sequences, Sq=1, Sk U{512..8192}, page 16, Hq=32, Hkv=8
  (FlyDSL PR #1066, PR description: paged KV, GQA, shuffled pages);
* paged e4m3 KV with per-token scale max|row|/448, Q/K D=192, V/O D=128,
  page 64 (FlyDSL PR #1066 overview; fkl_python PR #7, fp8 KV commit), plus
  the >4 GiB page pool of the FlyDSL PR #1066 review (COMMENT, prior items);
* flex prefill B=4, H=16, S=8192, D=128 with ALiBi 0.0625, soft-cap 20,
  sliding window 256 and a 50% random 128x128 block mask (fkl_python PR #7,
  flex commit).

Every array is numpy; bf16 values are carried as their uint16 bit patterns and
e4m3 values as uint8 bytes, so both sides consume identical bytes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)
E4M3_MAX = 448.0
MOD_NONE, MOD_ALIBI, MOD_SOFTCAP = 0, 1, 2
BLOCK = 128


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def e4m3_quantize_per_token(x: np.ndarray):
    """Per-token e4m3 encoding of the last axis: scale = max|row| / 448.

    Returns ``(bytes uint8 same shape, scale fp32 x.shape[:-1])``.  An all-zero
    row gets scale 0 and bytes 0.  This produces the cache; it is not a step of
    the forward pass.
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    y = x / safe[..., None]
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32))
    b = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    b[scale == 0] = 0
    return b, scale


def int8_quantize_per_token(x: np.ndarray):
    """Per-token symmetric int8 encoding of the last axis: scale = max|row| /
    127, value = round-to-nearest-even(x / scale) in [-127, 127].

    Returns ``(int8 same shape, scale fp32 x.shape[:-1])``.  An all-zero row
    gets scale 0 and bytes 0.  This produces the cache; it is not a step of
    the forward pass.
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    q = np.clip(np.rint(x / safe[..., None]), -127, 127).astype(np.int8)
    q[scale == 0] = 0
    return q, scale


def block_causal_mask(bh: int, nqb: int, nkb: int) -> np.ndarray:
    """Block-causal 128x128 mask: block (qb, kb) active iff kb <= qb."""
    qb = np.arange(nqb)[:, None]
    kb = np.arange(nkb)[None, :]
    m = (kb <= qb).astype(np.uint8)
    return np.broadcast_to(m, (bh, nqb, nkb)).copy()


@dataclasses.dataclass
class Problem:
    """One attention-forward problem in storage formats, plus its parameters."""

    name: str
    q: np.ndarray                      # uint16 bf16 bits [T_q, Hq, Dk]
    k: np.ndarray                      # packed [T_k, Hkv, Dk] or paged [N_pg, P_s, Hkv, Dk]
    v: np.ndarray                      # same with Dv
    kv_dtype: str                      # "bf16" (uint16 bits) or "e4m3" (uint8 bytes)
    cu_seqlens_q: np.ndarray           # int32 [B+1]
    cu_seqlens_k: np.ndarray           # int32 [B+1]
    hq: int
    hkv: int
    dk: int
    dv: int
    block_table: Optional[np.ndarray] = None   # int32 [B, max_pages]; None => packed K/V
    page_size: int = 0
    k_scale: Optional[np.ndarray] = None       # fp32 [N_pg, P_s, Hkv] (paged) or [T_k, Hkv]
    v_scale: Optional[np.ndarray] = None
    softmax_scale: float = 1.0
    causal: bool = False
    window: int = 0
    mod_kind: int = MOD_NONE
    alibi_slope: float = 0.0
    softcap: float = 0.0
    block_mask: Optional[np.ndarray] = None    # uint8 [B*Hq, nqb, nkb]
    q_dtype: str = "bf16"                      # "bf16" (uint16 bits) or "e4m3" (uint8 bytes; its
                                               # per-tensor scale is folded into softmax_scale)
    # prologue op chains on Q, K, V as read: {"q": [("mul", 0.5), ("add", 1.0)],
    # "k": [...], "v": [...]}, each op ("mul" | "add" | "sub" | "div", value)
    # applied in order to every element; None or missing keys = no ops
    prologue: Optional[dict] = None

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens_q.shape[0] - 1)

    @property
    def seqlens_q(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q.astype(np.int64))

    @property
    def seqlens_k(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_k.astype(np.int64))

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_seqlens_k[-1])

    @property
    def max_seqlen_q(self) -> int:
        return int(self.seqlens_q.max()) if self.num_seqs else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seqlens_k.max()) if self.num_seqs else 0

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    def replace(self, **kw) -> "Problem":
        return dataclasses.replace(self, **kw)


def _cu(lens: Sequence[int]) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)


def page_pool(seqlens_k: np.ndarray, page_size: int, rng: np.random.Generator,
              spare_pages: int = 0, max_pages: Optional[int] = None,
              first_page: int = 0, num_pages: Optional[int] = None):
    """Assign shuffled physical pages to every sequence.

    Returns ``(block_table int32 [B, max_pages], num_pages)``; entries past a
    sequence's last page are -1.  Pages are drawn from
    ``[first_page, first_page + needed + spare)`` by a seeded permutation.
    """
    need = [int(math.ceil(int(s) / page_size)) for s in seqlens_k]
    total = sum(need) + spare_pages
    if max_pages is None:
        max_pages = max(max(need) if need else 0, 1)
    perm = rng.permutation(total) + first_page
    if num_pages is None:
        num_pages = first_page + total
    bt = np.full((len(need), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


def scatter_pages(tokens: np.ndarray, cu_k: np.ndarray, block_table: np.ndarray,
                  num_pages: int, page_size: int, fill) -> np.ndarray:
    """Place packed per-token rows [T_k, ...] into a page pool [N_pg, P_s, ...]."""
    pool = np.full((num_pages, page_size) + tokens.shape[1:], fill, dtype=tokens.dtype)
    for b in range(block_table.shape[0]):
        lo, hi = int(cu_k[b]), int(cu_k[b + 1])
        j = np.arange(hi - lo)
        pages = block_table[b, j // page_size]
        pool[pages, j % page_size] = tokens[lo:hi]
    return pool


def vectorize_pages(k: np.ndarray, v: np.ndarray, x: int = 16):
    """The vectorized 5-D page layouts of a paged byte cache: K [N_pg, P_s,
    Hkv, Dk] -> [N_pg, Hkv, Dk/x, P_s, x] and V [N_pg, P_s, Hkv, Dv] ->
    [N_pg, Hkv, P_s/x, Dv, x] (x = 16 one-byte elements, 16 bytes).  The
    permutes (0, 3, 1, 2, 4) of K and (0, 2, 4, 1, 3) of V undo them (FlyDSL
    PR #1066, review).  A layout only: the same bytes, moved."""
    n, ps, hkv, dk = k.shape
    dv = v.shape[3]
    k5 = np.ascontiguousarray(k.reshape(n, ps, hkv, dk // x, x).transpose(0, 2, 3, 1, 4))
    v5 = np.ascontiguousarray(v.reshape(n, ps // x, x, hkv, dv).transpose(0, 3, 1, 4, 2))
    return k5, v5


def make_problem(seqlens_q: Sequence[int], seqlens_k: Optional[Sequence[int]] = None, *,
                 hq: int = 4, hkv: Optional[int] = None, dk: int = 64, dv: Optional[int] = None,
                 seed: int = 0, page_size: int = 0, kv_dtype: str = "bf16",
                 spare_pages: int = 0, max_pages: Optional[int] = None,
                 causal: bool = False, window: int = 0, mod: str = "none",
                 alibi_slope: float = 0.0625, softcap: float = 20.0,
                 block_mask_density: Optional[float] = None,
                 softmax_scale: Optional[float] = None, name: str = "custom",
                 q_std: float = 1.0, q_dtype: str = "bf16") -> Problem:
    """General seeded problem: N(0,1) Q/K/V rounded to bf16 (or e4m3 / int8 per token).

    Draw order (fixed): Q, K, V, page permutation, block mask.
    """
    hkv = hq if hkv is None else hkv
    dv = dk if dv is None else dv
    seqlens_q = [int(s) for s in seqlens_q]
    seqlens_k = list(seqlens_q) if seqlens_k is None else [int(s) for s in seqlens_k]
    rng = np.random.default_rng(seed)
    cu_q, cu_k = _cu(seqlens_q), _cu(seqlens_k)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    qf = rng.standard_normal((tq, hq, dk), dtype=np.float32) * np.float32(q_std)
    q = bf16_bits(qf)
    q_scale = 1.0
    if q_dtype == "e4m3":
        # one scale for the whole tensor: max|Q| / 448; the forward pass sees
        # it only through softmax_scale
        amax = float(np.abs(qf).max()) if qf.size else 0.0
        q_scale = amax / E4M3_MAX if amax > 0 else 1.0
        q = torch.from_numpy(np.ascontiguousarray(qf / np.float32(q_scale))).to(torch.float8_e4m3fn) \
            .view(torch.uint8).numpy().copy()
    elif q_dtype != "bf16":
        raise ValueError(q_dtype)
    kf = bf16_to_f32(bf16_bits(rng.standard_normal((tk, hkv, dk), dtype=np.float32)))
    vf = bf16_to_f32(bf16_bits(rng.standard_normal((tk, hkv, dv), dtype=np.float32)))
    k_scale = v_scale = None
    if kv_dtype == "bf16":
        k_tok, v_tok, fill = bf16_bits(kf), bf16_bits(vf), BF16_NAN
    elif kv_dtype == "e4m3":
        k_tok, k_scale = e4m3_quantize_per_token(kf)
        v_tok, v_scale = e4m3_quantize_per_token(vf)
        fill = E4M3_NAN
    elif kv_dtype == "int8":
        k_tok, k_scale = int8_quantize_per_token(kf)
        v_tok, v_scale = int8_quantize_per_token(vf)
        fill = np.int8(-128)          # never produced by the encoder: poisons unused slots
    else:
        raise ValueError(kv_dtype)
    block_table = None
    if page_size:
        block_table, n_pg = page_pool(np.asarray(seqlens_k), page_size, rng, spare_pages, max_pages)
        k = scatter_pages(k_tok, cu_k, block_table, n_pg, page_size, fill)
        v = scatter_pages(v_tok, cu_k, block_table, n_pg, page_size, fill)
        if kv_dtype in ("e4m3", "int8"):
            k_scale = scatter_pages(k_scale, cu_k, block_table, n_pg, page_size, np.float32(np.nan))
            v_scale = scatter_pages(v_scale, cu_k, block_table, n_pg, page_size, np.float32(np.nan))
    else:
        k, v = k_tok, v_tok
    bm = None
    if block_mask_density is not None:
        nqb = max(1, -(-max(seqlens_q + [1]) // BLOCK))
        nkb = max(1, -(-max(seqlens_k + [1]) // BLOCK))
        bm = (rng.random((len(seqlens_q) * hq, nqb, nkb)) < block_mask_density).astype(np.uint8)
    mk = {"none": MOD_NONE, "alibi": MOD_ALIBI, "softcap": MOD_SOFTCAP}[mod]
    return Problem(
        name=name, q=q, k=k, v=v, kv_dtype=kv_dtype, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
        hq=hq, hkv=hkv, dk=dk, dv=dv, block_table=block_table, page_size=page_size,
        k_scale=k_scale, v_scale=v_scale,
        softmax_scale=((1.0 / math.sqrt(dk)) if softmax_scale is None else float(softmax_scale)) * q_scale,
        causal=causal, window=window, mod_kind=mk,
        alibi_slope=alibi_slope if mk == MOD_ALIBI else 0.0,
        softcap=softcap if mk == MOD_SOFTCAP else 0.0, block_mask=bm, q_dtype=q_dtype)


# --------------------------------------------------------------------------
# The five workload configurations.
# --------------------------------------------------------------------------

def config1() -> Problem:
    """Dense bf16 causal: B=2, H=4, Sq=Sk=128, D=64, seed 0, scale 1/8."""
    return make_problem([128, 128], hq=4, dk=64, seed=0, causal=True,
                        softmax_scale=0.125, name="dense_causal_b2_h4_s128_d64")


def config2_lengths(seed: int = 0) -> list:
    """8 lengths U{0..2048}; one forced to 0 and one to a non-multiple of 128."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(0, 2049, size=8)]
    lens[0] = 0
    if not any(l % 128 for l in lens[1:]):
        lens[1] = 1000
    return lens


def config2(causal: bool = True, seed: int = 0) -> Problem:
    """Packed varlen bf16 prefill: 8 seqs, U{0..2048}, H=16, D=128."""
    lens = config2_lengths(seed)
    return make_problem(lens, hq=16, dk=128, seed=seed + 1, causal=causal,
                        name="varlen_prefill_8seq_h16_d128" + ("_causal" if causal else ""))


def config3(seed: int = 0) -> Problem:
    """Paged bf16 decode with GQA: 64 seqs, Sq=1, Sk U{512..8192}, page 16, Hq=32, Hkv=8."""
    rng = np.random.default_rng(seed)
    lens_k = [int(x) for x in rng.integers(512, 8193, size=64)]
    return make_problem([1] * 64, lens_k, hq=32, hkv=8, dk=128, seed=seed + 1, page_size=16,
                        spare_pages=64, max_pages=512, name="paged_decode_64seq_hq32_hkv8_p16")


def config4(seed: int = 0, causal: bool = True) -> Problem:
    """Paged e4m3 KV, Q/K D=192, V/O D=128, page 64, 16 seqs U{1..4096}, H=16, causal."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(1, 4097, size=16)]
    return make_problem(lens, hq=16, hkv=16, dk=192, dv=128, seed=seed + 1, page_size=64,
                        kv_dtype="e4m3", spare_pages=16, causal=causal,
                        name="paged_fp8_d192_v128_16seq_h16_p64")


# Page geometry of the >4 GiB pool: one kv head, page 64, K 192 B/token, V 128 B/token.
BIG_PAGE_SIZE, BIG_DK, BIG_DV, BIG_HKV = 64, 192, 128, 1


def big_pool_geometry(page_size: int = BIG_PAGE_SIZE, dk: int = BIG_DK, dv: int = BIG_DV,
                      hkv: int = BIG_HKV) -> dict:
    """Smallest pool whose highest page starts at or above 2**32 bytes in both K and V."""
    key_page_bytes = page_size * hkv * dk
    value_page_bytes = page_size * hkv * dv
    high_page = int(math.ceil(2 ** 32 / min(key_page_bytes, value_page_bytes)))
    num_pages = high_page + 1
    return dict(key_page_bytes=key_page_bytes, value_page_bytes=value_page_bytes,
                high_page=high_page, num_pages=num_pages,
                cache_bytes=num_pages * (key_page_bytes + value_page_bytes))


def config4_big(seed: int = 0, lens: Optional[Sequence[int]] = None):
    """The >4 GiB run: Hq=16, Hkv=1, e4m3, page 64, pages taken from the top of a
    524289-page pool; page ``high_page`` is used by two sequences.

    Returns ``(compact Problem, physical_block_table, num_pages)``: the compact
    problem stores only the pages in use (local ids), ``physical_block_table``
    maps the same entries to their ids in the full pool.
    """
    geo = big_pool_geometry()
    rng = np.random.default_rng(seed)
    if lens is None:
        lens = [int(x) for x in rng.integers(1, 1025, size=4)]
    p = make_problem(lens, hq=16, hkv=1, dk=BIG_DK, dv=BIG_DV, seed=seed + 1,
                     page_size=BIG_PAGE_SIZE, kv_dtype="e4m3", causal=True,
                     name="paged_fp8_over_4gib")
    bt = p.block_table
    # Local pages in order of first use (row-major over the block table), mapped
    # to physical pages counted down from the top of the pool: sequence 0's
    # first page lands on ``high_page``, the one page whose V offset is >= 2**32.
    order = []
    for x in bt.ravel():
        if x >= 0 and int(x) not in order:
            order.append(int(x))
    phys_of = {u: geo["high_page"] - i for i, u in enumerate(order)}
    pbt = np.full_like(bt, -1)
    for (b, j), x in np.ndenumerate(bt):
        if x >= 0:
            pbt[b, j] = phys_of[int(x)]
    # Sequence 1's last page is re-pointed at that same top page, so two
    # sequences read it.
    if len(lens) > 1:
        n1 = int(math.ceil(lens[1] / BIG_PAGE_SIZE))
        bt[1, n1 - 1] = order[0]
        pbt[1, n1 - 1] = geo["high_page"]
    return p, pbt, geo["num_pages"]


CONFIG5_RUNS = ("alibi_causal", "alibi", "softcap_causal", "softcap", "window_causal", "blocksparse")


def _config5_kw(run: str) -> dict:
    if run == "alibi_causal":
        return dict(mod="alibi", causal=True)
    if run == "alibi":
        return dict(mod="alibi")
    if run == "softcap_causal":
        return dict(mod="softcap", causal=True)
    if run == "softcap":
        return dict(mod="softcap")
    if run == "window_causal":
        return dict(window=256, causal=True)
    if run == "blocksparse":
        return dict(block_mask_density=0.5)
    raise ValueError(run)


def config5(run: str = "alibi_causal", seed: int = 0, seq: int = 8192, batch: int = 4) -> Problem:
    """Flex bf16 prefill: B=4, H=16, S=8192, D=128 with one score mod or mask per run."""
    return make_problem([seq] * batch, hq=16, dk=128, seed=seed, name=f"flex_{run}_b{batch}_h16_s{seq}_d128",
                        **_config5_kw(run))


def config5_runs(seed: int = 0, seq: int = 8192, batch: int = 4) -> list:
    """The six config-5 runs in CONFIG5_RUNS order, sharing one set of Q, K, V
    arrays: every run draws the same Q, K, V (same seed and shapes, drawn
    first), so each equals config5(run) field by field."""
    base = config5("blocksparse", seed, seq, batch)
    runs = []
    for run in CONFIG5_RUNS:
        if run == "blocksparse":
            runs.append(base)
            continue
        kw = _config5_kw(run)
        mk = {"none": MOD_NONE, "alibi": MOD_ALIBI, "softcap": MOD_SOFTCAP}[kw.get("mod", "none")]
        runs.append(base.replace(name=f"flex_{run}_b{batch}_h16_s{seq}_d128", block_mask=None,
                                 causal=kw.get("causal", False), window=kw.get("window", 0), mod_kind=mk,
                                 alibi_slope=0.0625 if mk == MOD_ALIBI else 0.0,
                                 softcap=20.0 if mk == MOD_SOFTCAP else 0.0))
    return runs


# --------------------------------------------------------------------------
# Algorithmic work, the denominators of TFLOP/s and GB/s.  Counting only:
# the number of (query row, key) pairs that the mask allows.
# --------------------------------------------------------------------------

def allowed_pairs(p: Problem) -> int:
    """Number of allowed (head, query, key) triples, by interval arithmetic."""
    total = 0
    sq, sk = p.seqlens_q, p.seqlens_k
    for b in range(p.num_seqs):
        Sq, Sk = int(sq[b]), int(sk[b])
        if Sq == 0 or Sk == 0:
            continue
        i = np.arange(Sq, dtype=np.int64)
        ip = i + Sk - Sq
        lo = np.zeros(Sq, dtype=np.int64)
        hi = np.full(Sq, Sk, dtype=np.int64)        # exclusive
        if p.causal:
            hi = np.minimum(hi, ip + 1)
        if p.window > 0:
            lo = np.maximum(lo, ip - p.window + 1)
            if not p.causal:
                hi = np.minimum(hi, ip + p.window)
        if p.block_mask is None:
            total += int(np.clip(hi - lo, 0, None).sum()) * p.hq
        else:
            nkb = p.block_mask.shape[2]
            for h in range(p.hq):
                m = p.block_mask[b * p.hq + h]
                for qb in range(-(-Sq // BLOCK)):
                    rows = slice(qb * BLOCK, min(Sq, (qb + 1) * BLOCK))
                    l, u = lo[rows], hi[rows]
                    for kb in range(min(nkb, -(-Sk // BLOCK))):
                        if not m[qb, kb]:
                            continue
                        a = np.maximum(l, kb * BLOCK)
                        z = np.minimum(u, min(Sk, (kb + 1) * BLOCK))
                        total += int(np.clip(z - a, 0, None).sum())
    return total


def prefill_flops(p: Problem) -> float:
    """2*Dk + 2*Dv flops per allowed (head, query, key) triple."""
    return float(allowed_pairs(p)) * (2 * p.dk + 2 * p.dv)


def decode_bytes(p: Problem) -> float:
    """Bytes the method must move: every key's K and V row (and scales), Q, O, LSE, page ids."""
    esize = 2 if p.kv_dtype == "bf16" else 1
    tok = float(p.seqlens_k.sum())
    kv = tok * p.hkv * (p.dk + p.dv) * esize
    if p.kv_dtype in ("e4m3", "int8"):
        kv += tok * p.hkv * 8           # one fp32 k and v scale per token and kv head
    qo = p.total_q * p.hq * (p.dk * 2 + p.dv * 2 + 4)
    pages = sum(int(math.ceil(s / p.page_size)) for s in p.seqlens_k) * 4 if p.paged else 0
    return kv + qo + pages

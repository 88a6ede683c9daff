"""fp64 CPU oracle for the attention forward and backward passes -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it shares no code with the CUDA library; the only module both
sides use is ``fa_inputs`` (seeded inputs, no attention arithmetic).

The arithmetic lives in ``fa_oracle.c`` (plain C, double precision); this file
builds it with gcc on first use and marshals numpy arrays through ctypes.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute-force enumeration and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libfa_oracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16, KV_E4M3, KV_F64, KV_I8 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into a shared library (plain gcc, no CUDA)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_MAX_OPS = 8
_OP_CODES = {"mul": 1, "add": 2, "sub": 3, "div": 4}


class _Chain(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("op", ctypes.c_int32 * _MAX_OPS), ("c", ctypes.c_double * _MAX_OPS)]


def _chain(ops) -> _Chain:
    """One tensor's prologue op chain, e.g. [("mul", 2.0), ("add", 1.0)], as
    the C struct; the oracle applies the ops one after the other."""
    ch = _Chain()
    ops = list(ops or ())
    if len(ops) > _MAX_OPS:
        raise ValueError(f"at most {_MAX_OPS} prologue ops per tensor")
    ch.n = len(ops)
    for i, (name, c) in enumerate(ops):
        if name not in _OP_CODES:
            raise ValueError(f"prologue op {name!r}: mul, add, sub or div")
        ch.op[i] = _OP_CODES[name]
        ch.c[i] = float(c)
    return ch


class _Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("kv_dtype", ctypes.c_int32),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64),
        ("cu_q", ctypes.c_void_p), ("cu_k", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
        ("causal", ctypes.c_int32), ("window", ctypes.c_int32), ("mod_kind", ctypes.c_int32),
        ("alibi_slope", ctypes.c_double), ("softcap", ctypes.c_double),
        ("block_mask", ctypes.c_void_p),
        ("n_qblk", ctypes.c_int32), ("n_kblk", ctypes.c_int32),
        ("blk_q", ctypes.c_int32), ("blk_k", ctypes.c_int32),
        ("kv_lo", ctypes.c_int64), ("kv_hi", ctypes.c_int64),
        ("q_dtype", ctypes.c_int32),
        ("pro_q", _Chain), ("pro_k", _Chain), ("pro_v", _Chain),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.fa_oracle_fwd.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            L.fa_oracle_fwd.restype = ctypes.c_int
            L.fa_oracle_combine.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_void_p]
            L.fa_oracle_combine.restype = None
            L.fa_oracle_bwd.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            L.fa_oracle_bwd.restype = ctypes.c_int
            L.fa_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.fa_oracle_e4m3_decode.restype = ctypes.c_double
            L.fa_oracle_i8_decode.argtypes = [ctypes.c_uint8]
            L.fa_oracle_i8_decode.restype = ctypes.c_double
            L.fa_oracle_bf16_decode.argtypes = [ctypes.c_uint16]
            L.fa_oracle_bf16_decode.restype = ctypes.c_double
            _lib = L
    return _lib


def e4m3_decode(byte: int) -> float:
    return lib().fa_oracle_e4m3_decode(int(byte) & 0xFF)


def i8_decode(byte: int) -> float:
    return lib().fa_oracle_i8_decode(int(byte) & 0xFF)


def bf16_decode(bits: int) -> float:
    return lib().fa_oracle_bf16_decode(int(bits) & 0xFFFF)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _problem(p, keep, kv_range=None, q_f64=None, k_f64=None, v_f64=None):
    """The C problem descriptor for a ``fa_inputs.Problem`` (arrays kept alive in ``keep``)."""
    def c(a, dt):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dt)
        keep.append(a)
        return a

    q_e4m3 = getattr(p, "q_dtype", "bf16") == "e4m3"
    if q_f64 is not None:
        q, qd = c(q_f64, np.float64), 2
    else:
        q, qd = c(p.q, np.uint8 if q_e4m3 else np.uint16), (1 if q_e4m3 else 0)
    if k_f64 is not None:
        kd, k, v, ks, vs = KV_F64, c(k_f64, np.float64), c(v_f64, np.float64), None, None
    elif p.kv_dtype == "bf16":
        kd, k, v, ks, vs = KV_BF16, c(p.k, np.uint16), c(p.v, np.uint16), None, None
    else:
        kd = KV_E4M3 if p.kv_dtype == "e4m3" else KV_I8
        k, v = c(p.k.view(np.uint8), np.uint8), c(p.v.view(np.uint8), np.uint8)
        ks, vs = c(p.k_scale, np.float32), c(p.v_scale, np.float32)
    bt = c(p.block_table, np.int32)
    cq, ck = c(p.cu_seqlens_q, np.int32), c(p.cu_seqlens_k, np.int32)
    bm = c(p.block_mask, np.uint8)
    prob = _Problem(
        q=_ptr(q), k=_ptr(k), v=_ptr(v), kv_dtype=kd,
        block_table=_ptr(bt), bt_stride=(bt.shape[1] if bt is not None else 0),
        cu_q=_ptr(cq), cu_k=_ptr(ck), num_seqs=p.num_seqs,
        k_scale=_ptr(ks), v_scale=_ptr(vs),
        hq=p.hq, hkv=p.hkv, dk=p.dk, dv=p.dv, page_size=p.page_size,
        softmax_scale=p.softmax_scale, causal=int(p.causal), window=int(p.window),
        mod_kind=int(p.mod_kind), alibi_slope=float(p.alibi_slope), softcap=float(p.softcap),
        block_mask=_ptr(bm),
        n_qblk=(bm.shape[1] if bm is not None else 0), n_kblk=(bm.shape[2] if bm is not None else 0),
        blk_q=128, blk_k=128,
        kv_lo=(kv_range[0] if kv_range else 0), kv_hi=(kv_range[1] if kv_range else -1),
        q_dtype=qd)
    pro = getattr(p, "prologue", None) or {}
    prob.pro_q, prob.pro_k, prob.pro_v = _chain(pro.get("q")), _chain(pro.get("k")), _chain(pro.get("v"))
    return prob, c


def forward(p, units: Optional[np.ndarray] = None, nthreads: Optional[int] = None,
            kv_range: Optional[tuple] = None, k_f64: Optional[np.ndarray] = None,
            v_f64: Optional[np.ndarray] = None, q_f64: Optional[np.ndarray] = None):
    """Run the oracle on a ``fa_inputs.Problem``.

    units   : None for all rows, else int64 array [n, 2] of (query token, head).
    kv_range: optional (lo, hi) restriction of sequence-local key indices.
    q_f64, k_f64/v_f64 : optional double Q, K/V with the problem's layout,
                  replacing the stored values (no scales applied).
    Returns (out, lse): out float64 [T_q, Hq, Dv] and lse float64 [Hq, T_q] for
    all rows, or out [n, Dv] and lse [n] for a unit list.
    """
    keep = []
    prob, c = _problem(p, keep, kv_range, q_f64, k_f64, v_f64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    if units is None:
        n = p.total_q * p.hq
        u = None
    else:
        u = c(units, np.int64).reshape(-1, 2)
        n = u.shape[0]
    out = np.zeros((max(n, 1), p.dv), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    rc = lib().fa_oracle_fwd(ctypes.byref(prob), _ptr(u), n, out.ctypes.data, lse.ctypes.data,
                             int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    out, lse = out[:n], lse[:n]
    if units is None:
        return out.reshape(p.total_q, p.hq, p.dv), lse.reshape(p.total_q, p.hq).T.copy()
    return out, lse


def combine(o_part: np.ndarray, lse_part: np.ndarray):
    """Merge partials over disjoint key sets: o_part [S, n, Dv], lse_part [S, n]."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    s, n, dv = o_part.shape
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    lib().fa_oracle_combine(o_part.ctypes.data, lse_part.ctypes.data, s, n, dv,
                            out.ctypes.data, lse.ctypes.data)
    return out, lse


def backward(p, dout: np.ndarray, nthreads: Optional[int] = None, q_f64: Optional[np.ndarray] = None,
             k_f64: Optional[np.ndarray] = None, v_f64: Optional[np.ndarray] = None):
    """Gradients of sum(dout * out) with respect to q, k and v (packed K/V).

    dout: float64 [T_q, Hq, Dv].  Returns (dq [T_q, Hq, Dk], dk [T_k, Hkv, Dk],
    dv [T_k, Hkv, Dv]) in float64.
    """
    keep = []
    prob, _ = _problem(p, keep, None, q_f64, k_f64, v_f64)
    d = np.ascontiguousarray(dout, dtype=np.float64).reshape(p.total_q, p.hq, p.dv)
    dq = np.zeros((max(p.total_q, 1), p.hq, p.dk))
    dk = np.zeros((max(p.total_k, 1), p.hkv, p.dk))
    dv = np.zeros((max(p.total_k, 1), p.hkv, p.dv))
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib().fa_oracle_bwd(ctypes.byref(prob), d.ctypes.data, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                             int(nthreads))
    if rc != 0:
        raise ValueError("oracle backward rejected the problem")
    return dq[:p.total_q], dk[:p.total_k], dv[:p.total_k]

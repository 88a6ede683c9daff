"""GB300 (sm_103a) FlashAttention forward -- thin Python binding of the C ABI.

Every step of the forward pass runs in the CUDA library ``_build/libfa_gb300.so``
(see ``include/fa_gb300.h``).  This module only marshals torch tensors into
``fa_tensor_t`` descriptors, allocates outputs/workspace with torch on the
current stream, and raises on any non-OK status.  There is no fallback: if the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_OVERFLOW, FA_ERR_CUDA = 0, 1, 2, 3, 4
FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_BOUNDS = 5, 6
FA_BF16, FA_E4M3, FA_F32, FA_I32, FA_U8, FA_I8 = 0, 1, 2, 3, 4, 5
MOD_NONE, MOD_ALIBI, MOD_SOFTCAP = 0, 1, 2

EXPORTED = ("fa_fwd_varlen", "fa_fwd_workspace_bytes", "fa_fwd_default_splits", "fa_combine",
            "fa_last_error", "fa_get_device_error", "fa_version", "fa_fwd_varlen_noalloc",
            "fa_fwd_plan_create", "fa_fwd_plan_launch", "fa_fwd_plan_destroy", "fa_bwd_varlen",
            "fa_bwd_workspace_bytes")
NOALLOC_SCRATCH_BYTES = 32 << 20


class FaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"fa status {status}: {msg}")
        self.status = status


class Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


class ScoreMod(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("alibi_slope", ctypes.c_float), ("softcap", ctypes.c_float)]


class BlockMask(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("n_qblk", ctypes.c_int32), ("n_kblk", ctypes.c_int32),
                ("blk_q", ctypes.c_int32), ("blk_k", ctypes.c_int32)]


PROLOGUE_MAX_OPS = 8
FA_OP_MUL, FA_OP_ADD, FA_OP_SUB, FA_OP_DIV = 1, 2, 3, 4
_OPS = {"mul": FA_OP_MUL, "add": FA_OP_ADD, "sub": FA_OP_SUB, "div": FA_OP_DIV}


class PrologueOp(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("value", ctypes.c_float)]


class Prologue(ctypes.Structure):
    _fields_ = [("n_q", ctypes.c_int32), ("n_k", ctypes.c_int32), ("n_v", ctypes.c_int32),
                ("q", PrologueOp * PROLOGUE_MAX_OPS), ("k", PrologueOp * PROLOGUE_MAX_OPS),
                ("v", PrologueOp * PROLOGUE_MAX_OPS)]


def make_prologue(prologue) -> Optional[Prologue]:
    """The C ``fa_prologue_t`` for ``prologue``: None, a Prologue, or a dict
    mapping "q", "k", "v" to op chains -- lists of ("mul" | "add" | "sub" |
    "div", value), applied in order to each element as it is read.  The ops
    are copied as given; the library composes and folds them."""
    if prologue is None or isinstance(prologue, Prologue):
        return prologue
    pro = Prologue()
    for name in ("q", "k", "v"):
        ops = list(prologue.get(name, ()))
        if len(ops) > PROLOGUE_MAX_OPS:
            raise ValueError(f"at most {PROLOGUE_MAX_OPS} prologue ops per tensor")
        arr = getattr(pro, name)
        for i, (op, value) in enumerate(ops):
            if op not in _OPS:
                raise ValueError(f"prologue op {op!r}: mul, add, sub or div")
            arr[i].op = _OPS[op]
            arr[i].value = float(value)
        setattr(pro, "n_" + name, len(ops))
    return pro


class Launch(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
                ("max_seqlen_k", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("total_q", ctypes.c_int64), ("total_k", ctypes.c_int64),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("flags", ctypes.c_int32)]


# fa_launch_t.flags: P * V on e4m3 operands (opt-in precision mode, e4m3 q
# with e4m3 caches; see FA_FLAG_PV_E4M3 in fa_gb300.h)
FLAG_PV_E4M3 = 1


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m flashattention_forward_gb300.build` "
                    "(there is no fallback implementation)")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER
            L.fa_fwd_varlen.argtypes = [P(Tensor)] * 8 + [P(Tensor), P(Tensor), ctypes.c_float, ctypes.c_int32,
                                                         ctypes.c_int32, P(ScoreMod), P(BlockMask), P(Prologue),
                                                         ctypes.c_int32, P(Launch), ctypes.c_void_p]
            L.fa_fwd_varlen.restype = ctypes.c_int
            L.fa_fwd_workspace_bytes.argtypes = [P(Launch), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 P(Prologue)]
            L.fa_fwd_workspace_bytes.restype = ctypes.c_size_t
            L.fa_fwd_default_splits.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
            L.fa_fwd_default_splits.restype = ctypes.c_int32
            L.fa_combine.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p]
            L.fa_combine.restype = ctypes.c_int
            L.fa_last_error.restype = ctypes.c_char_p
            L.fa_get_device_error.argtypes = [ctypes.c_void_p, P(ctypes.c_int32)]
            L.fa_get_device_error.restype = ctypes.c_int
            L.fa_version.restype = ctypes.c_char_p
            L.fa_fwd_varlen_noalloc.argtypes = L.fa_fwd_varlen.argtypes
            L.fa_fwd_varlen_noalloc.restype = ctypes.c_int
            L.fa_fwd_plan_create.argtypes = L.fa_fwd_varlen.argtypes[:-1] + [P(ctypes.c_void_p)]
            L.fa_fwd_plan_create.restype = ctypes.c_int
            L.fa_fwd_plan_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            L.fa_fwd_plan_launch.restype = ctypes.c_int
            L.fa_fwd_plan_destroy.argtypes = [ctypes.c_void_p]
            L.fa_fwd_plan_destroy.restype = None
            L.fa_bwd_varlen.argtypes = [P(Tensor)] * 11 + [ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                                                          P(ScoreMod), P(BlockMask), P(Launch), ctypes.c_void_p]
            L.fa_bwd_varlen.restype = ctypes.c_int
            L.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32]
            L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
            _lib = L
    return _lib


def _check(status: int):
    if status != FA_OK:
        raise FaError(status, lib().fa_last_error().decode())


_DT = {torch.bfloat16: FA_BF16, torch.float32: FA_F32, torch.int32: FA_I32, torch.uint8: FA_U8, torch.int8: FA_I8}
if hasattr(torch, "float8_e4m3fn"):
    _DT[torch.float8_e4m3fn] = FA_E4M3


def _kv_dtype(k_cache: torch.Tensor) -> int:
    """bf16, int8 (per-token scaled) or e4m3 (float8_e4m3fn or raw uint8 bytes)."""
    if k_cache.dtype == torch.bfloat16:
        return FA_BF16
    if k_cache.dtype == torch.int8:
        return FA_I8
    return FA_E4M3


def _cache_dims(k_cache: torch.Tensor, v_cache: torch.Tensor):
    """(Hkv, Dv) of packed [T_k, Hkv, D] or paged [N_pg, P_s, Hkv, D] caches,
    or of the vectorized 5-D pages K [N_pg, Hkv, Dk/16, P_s, 16] and
    V [N_pg, Hkv, P_s/16, Dv, 16]."""
    if k_cache.dim() == 5:
        return k_cache.shape[1], v_cache.shape[3]
    return k_cache.shape[-2], v_cache.shape[-1]


def as_tensor(t: Optional[torch.Tensor], fa_dtype: Optional[int] = None) -> Optional[Tensor]:
    """Describe a torch tensor (device pointer, shape, element strides)."""
    if t is None:
        return None
    d = Tensor()
    d.data = t.data_ptr() if t.numel() else 0
    d.dtype = _DT[t.dtype] if fa_dtype is None else fa_dtype
    n = t.dim()
    d.ndim = n
    d.shape[:n] = t.shape
    d.stride[:n] = t.stride()
    return d


def _ref(x):
    return None if x is None else ctypes.byref(x)


def _block_mask(block_mask: Optional[torch.Tensor]):
    """A uint8 [B*Hq, n_qblk, n_kblk] tensor of 128 x 128 blocks as the C struct (None passes NULL)."""
    if block_mask is None:
        return None
    return BlockMask(data=block_mask.data_ptr(), n_qblk=block_mask.shape[1], n_kblk=block_mask.shape[2],
                     blk_q=128, blk_k=128)


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def default_splits(num_seqs, max_seqlen_q, max_seqlen_k, hq, hkv, page_size=0, total_k=0) -> int:
    return int(lib().fa_fwd_default_splits(num_seqs, max_seqlen_q, max_seqlen_k, int(total_k), hq, hkv, page_size))


def workspace_bytes(launch: "Launch", hq: int, hkv: int, dv: int, prologue=None) -> int:
    """Workspace bytes of a forward call (split-KV partials, a Q add's per-key
    terms, the V-scale maxima of the e4m3 P * V mode)."""
    return int(lib().fa_fwd_workspace_bytes(ctypes.byref(launch), hq, hkv, dv, _ref(make_prologue(prologue))))


def fwd_varlen(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, *,
               max_seqlen_q: int, max_seqlen_k: int, total_k: Optional[int] = None,
               block_table: Optional[torch.Tensor] = None, page_size: int = 0,
               k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
               softmax_scale: Optional[float] = None, causal: bool = False, window: int = 0,
               score_mod: int = MOD_NONE, alibi_slope: float = 0.0, softcap: float = 0.0,
               block_mask: Optional[torch.Tensor] = None, num_splits: Optional[int] = None,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               return_lse: bool = True, workspace: Optional[torch.Tensor] = None, stream=None, prologue=None,
               pv_e4m3: bool = False):
    """Attention forward over packed varlen Q and packed or paged K/V.

    q [T_q, Hq, Dk] bf16, or float8_e4m3fn with e4m3 caches at Dk 128 or 192
    and Dv 128 (QK then runs on the e4m3 bytes; fold a per-tensor Q scale into
    ``softmax_scale``); k_cache/v_cache packed [T_k, Hkv, D] or paged
    [N_pg, P_s, Hkv, D] (bf16, or e4m3 as float8_e4m3fn/uint8, or int8, with
    k_scale/v_scale), or -- e4m3 and int8 pages of >= 16 keys -- the
    vectorized 5-D pages K [N_pg, Hkv, Dk/16, P_s, 16], V [N_pg, Hkv, P_s/16,
    Dv, 16] (scales stay [N_pg, P_s, Hkv]); cu_seqlens int32 [B+1].  ``max_seqlen_q/k`` are host ints (no
    device read-back).  Returns ``(out [T_q, Hq, Dv] bf16, lse [Hq, T_q] fp32
    or None)``.  ``num_splits=None`` picks the library's default (split-KV for
    decode shapes); 0 forces the single-pass kernel.  ``prologue``: op chains
    on the Q/K/V reads, {"q": [("mul", c), ("add", d), ...], "k": ..., "v": ...}
    (see make_prologue and fa_prologue_t).  ``pv_e4m3``: the opt-in precision
    mode FA_FLAG_PV_E4M3 (P * V on e4m3 operands; e4m3 q with e4m3 caches).
    """
    L = lib()
    B = cu_seqlens_q.shape[0] - 1
    Tq, Hq, Dk = q.shape
    Hkv, Dv = _cache_dims(k_cache, v_cache)
    kv_dt = _kv_dtype(k_cache)
    if out is None:
        out = torch.empty((Tq, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dk)
    if total_k is None:
        total_k = k_cache.shape[0] if block_table is None else 0
    if num_splits is None:
        num_splits = default_splits(B, max_seqlen_q, max_seqlen_k, Hq, Hkv, page_size, total_k)
        if q.dtype != torch.bfloat16 or Dk != Dv:
            num_splits = 0
    launch = Launch(num_seqs=B, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                    num_splits=num_splits, total_q=Tq, total_k=total_k,
                    flags=FLAG_PV_E4M3 if pv_e4m3 else 0)
    pro = make_prologue(prologue)
    need = workspace_bytes(launch, Hq, Hkv, Dv, pro)
    if need:
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        launch.workspace = workspace.data_ptr()
        launch.workspace_bytes = workspace.numel()
    sm = ScoreMod(kind=score_mod, alibi_slope=alibi_slope, softcap=softcap)
    bm = _block_mask(block_mask)
    args = [as_tensor(q), as_tensor(k_cache, kv_dt), as_tensor(v_cache, kv_dt), as_tensor(block_table),
            as_tensor(cu_seqlens_q), as_tensor(cu_seqlens_k), as_tensor(k_scale), as_tensor(v_scale),
            as_tensor(out), as_tensor(lse)]
    st = L.fa_fwd_varlen(*[_ref(a) for a in args], float(softmax_scale), int(bool(causal)), int(window),
                         ctypes.byref(sm), _ref(bm), _ref(pro), int(page_size), ctypes.byref(launch),
                         ctypes.c_void_p(_stream_ptr(stream)))
    _check(st)
    return out, lse


def fwd_varlen_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, out: torch.Tensor,
                       lse: Optional[torch.Tensor], *, max_seqlen_q: int, max_seqlen_k: int,
                       total_k: Optional[int] = None, block_table: Optional[torch.Tensor] = None,
                       page_size: int = 0, k_scale: Optional[torch.Tensor] = None,
                       v_scale: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                       causal: bool = False, window: int = 0, score_mod: int = MOD_NONE,
                       alibi_slope: float = 0.0, softcap: float = 0.0,
                       block_mask: Optional[torch.Tensor] = None, num_splits: int = 0, stream=None,
                       prologue=None):
    """Split-KV decode through ``fa_fwd_varlen_noalloc``, for callers that cannot
    allocate device memory when they run attention: the split partials (and a
    Q add's per-key terms) go to the library's static scratch of
    NOALLOC_SCRATCH_BYTES.  Takes the arguments of fwd_varlen, including byte
    caches with their scales, score mods, block masks and prologues; ``out``
    (and ``lse`` if wanted) are caller-provided and this wrapper allocates
    nothing.  ``num_splits=0`` uses the library default."""
    L = lib()
    B = cu_seqlens_q.shape[0] - 1
    Tq, Hq, Dk = q.shape
    kv_dt = _kv_dtype(k_cache)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dk)
    if total_k is None:
        total_k = k_cache.shape[0] if block_table is None else 0
    launch = Launch(num_seqs=B, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                    num_splits=num_splits, total_q=Tq, total_k=total_k)
    args = [as_tensor(q), as_tensor(k_cache, kv_dt), as_tensor(v_cache, kv_dt), as_tensor(block_table),
            as_tensor(cu_seqlens_q), as_tensor(cu_seqlens_k), as_tensor(k_scale), as_tensor(v_scale),
            as_tensor(out), as_tensor(lse)]
    sm = ScoreMod(kind=score_mod, alibi_slope=alibi_slope, softcap=softcap)
    _check(L.fa_fwd_varlen_noalloc(*[_ref(a) for a in args], float(softmax_scale), int(bool(causal)),
                                   int(window), ctypes.byref(sm), _ref(_block_mask(block_mask)),
                                   _ref(make_prologue(prologue)), int(page_size), ctypes.byref(launch),
                                   ctypes.c_void_p(_stream_ptr(stream))))
    return out, lse


class FwdPlan:
    """A prepared fwd_varlen call through ``fa_fwd_plan_create``: validation,
    tensor maps and kernel parameters are built once, and run() only enqueues
    the kernels (``fa_fwd_plan_launch``) -- for repeated calls on the same
    buffers (serving loops, benchmarks) where the per-call host work would
    dominate small problems.  Takes the arguments of fwd_varlen; the tensors
    must stay alive, unmoved and of the same shape while the plan is used."""

    def __init__(self, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, **kw):
        L = lib()
        self._keep = [q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k] + [v for v in kw.values()
                                                                           if isinstance(v, torch.Tensor)]
        B = cu_seqlens_q.shape[0] - 1
        Tq, Hq, Dk = q.shape
        Hkv, Dv = _cache_dims(k_cache, v_cache)
        kv_dt = _kv_dtype(k_cache)
        self.out = kw.get("out")
        if self.out is None:
            self.out = torch.empty((Tq, Hq, Dv), dtype=torch.bfloat16, device=q.device)
        self.lse = kw.get("lse")
        if self.lse is None and kw.get("return_lse", True):
            self.lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
        scale = kw.get("softmax_scale")
        if scale is None:
            scale = 1.0 / math.sqrt(Dk)
        block_table = kw.get("block_table")
        total_k = kw.get("total_k")
        if total_k is None:
            total_k = k_cache.shape[0] if block_table is None else 0
        page_size = kw.get("page_size", 0)
        score_mod = kw.get("score_mod", MOD_NONE)
        block_mask = kw.get("block_mask")
        num_splits = kw.get("num_splits")
        if num_splits is None:
            num_splits = default_splits(B, kw["max_seqlen_q"], kw["max_seqlen_k"], Hq, Hkv, page_size, total_k)
            if q.dtype != torch.bfloat16 or Dk != Dv:
                num_splits = 0
        self.launch = Launch(num_seqs=B, max_seqlen_q=kw["max_seqlen_q"], max_seqlen_k=kw["max_seqlen_k"],
                             num_splits=num_splits, total_q=Tq, total_k=total_k,
                             flags=FLAG_PV_E4M3 if kw.get("pv_e4m3") else 0)
        ws = kw.get("workspace")
        pro = make_prologue(kw.get("prologue"))
        need = workspace_bytes(self.launch, Hq, Hkv, Dv, pro)
        if need:
            if ws is None or ws.numel() < need:
                ws = torch.empty(need, dtype=torch.uint8, device=q.device)
            self.launch.workspace = ws.data_ptr()
            self.launch.workspace_bytes = ws.numel()
        self._ws = ws
        sm = ScoreMod(kind=score_mod, alibi_slope=kw.get("alibi_slope", 0.0), softcap=kw.get("softcap", 0.0))
        bm = _block_mask(block_mask)
        descs = [as_tensor(q), as_tensor(k_cache, kv_dt), as_tensor(v_cache, kv_dt), as_tensor(block_table),
                 as_tensor(cu_seqlens_q), as_tensor(cu_seqlens_k), as_tensor(kw.get("k_scale")),
                 as_tensor(kw.get("v_scale")), as_tensor(self.out), as_tensor(self.lse)]
        handle = ctypes.c_void_p(0)
        _check(L.fa_fwd_plan_create(*[_ref(a) for a in descs], ctypes.c_float(scale),
                                    ctypes.c_int32(int(bool(kw.get("causal", False)))),
                                    ctypes.c_int32(int(kw.get("window", 0))), ctypes.byref(sm), _ref(bm),
                                    _ref(pro), ctypes.c_int32(int(page_size)), ctypes.byref(self.launch),
                                    ctypes.byref(handle)))
        self._plan = handle
        self._launch_fn = L.fa_fwd_plan_launch
        self._destroy_fn = L.fa_fwd_plan_destroy

    def run(self, stream=None):
        st = self._launch_fn(self._plan, ctypes.c_void_p(_stream_ptr(stream)))
        if st != FA_OK:
            _check(st)
        return self.out, self.lse

    def __del__(self):
        plan = getattr(self, "_plan", None)
        if plan is not None and plan.value:
            self._destroy_fn(plan)
            self._plan = None


def combine(o_part: torch.Tensor, lse_part: torch.Tensor, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, stream=None):
    """Merge split partials: o_part fp32 [S, n, Hq, Dv], lse_part fp32 [S, Hq, n]."""
    S, n, Hq, Dv = o_part.shape
    if out is None:
        out = torch.empty((n, Hq, Dv), dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty((Hq, n), dtype=torch.float32, device=o_part.device)
    o_part = o_part.contiguous()
    lse_part = lse_part.contiguous()
    _check(lib().fa_combine(o_part.data_ptr(), lse_part.data_ptr(), S, n, Hq, Dv, out.data_ptr(),
                            lse.data_ptr(), ctypes.c_void_p(_stream_ptr(stream))))
    return out, lse


def device_error(stream=None) -> int:
    """Synchronise and return (then clear) the device error word."""
    code = ctypes.c_int32(0)
    _check(lib().fa_get_device_error(ctypes.c_void_p(_stream_ptr(stream)), ctypes.byref(code)))
    return int(code.value)


def version() -> str:
    return lib().fa_version().decode()


def bwd_workspace_bytes(total_q: int, hq: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(int(total_q), int(hq)))


def bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, dout: torch.Tensor,
               lse: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, *,
               max_seqlen_q: int, max_seqlen_k: int, softmax_scale: Optional[float] = None,
               causal: bool = False, window: int = 0, score_mod: int = MOD_NONE,
               alibi_slope: float = 0.0, softcap: float = 0.0, block_mask: Optional[torch.Tensor] = None,
               dq: Optional[torch.Tensor] = None,
               dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward pass through ``fa_bwd_varlen``: returns (dq, dk, dv), bf16 with
    the shapes of q, k, v.  ``lse`` is the forward's fp32 [Hq, T_q] LSE for the
    same inputs, masks and score mod; K/V packed [T_k, Hkv, D]; D = 64 or 128."""
    L = lib()
    B = cu_seqlens_q.shape[0] - 1
    Tq, Hq, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_bytes(Tq, Hq)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    launch = Launch(num_seqs=B, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, num_splits=0,
                    total_q=Tq, total_k=k.shape[0])
    if need:
        launch.workspace = workspace.data_ptr()
        launch.workspace_bytes = workspace.numel()
    args = [as_tensor(x) for x in (q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, dq, dk, dv)]
    sm = ScoreMod(kind=score_mod, alibi_slope=alibi_slope, softcap=softcap)
    bm = _block_mask(block_mask)
    _check(L.fa_bwd_varlen(*[_ref(a) for a in args], ctypes.c_float(softmax_scale), int(bool(causal)),
                           int(window), ctypes.byref(sm), _ref(bm), ctypes.byref(launch),
                           ctypes.c_void_p(_stream_ptr(stream))))
    return dq, dk, dv

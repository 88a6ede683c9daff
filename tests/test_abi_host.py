"""Host-only checks of the C-ABI library: it loads, exports every entry point
that include/fa_gb300.h declares, and rejects malformed calls with a status
code before touching the GPU (validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

import flashattention_forward_gb300 as fa
from flashattention_forward_gb300 import build as fa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa_gb300.h")


@pytest.fixture(scope="module")
def L():
    fa_build.build()
    return fa.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_are_exported(L):
    syms = declared_symbols()
    assert "fa_fwd_varlen" in syms and "fa_combine" in syms
    for s in syms:
        assert hasattr(L, s), s
    assert set(syms) <= set(fa.EXPORTED) | set(syms)


def test_only_the_header_entry_points_are_exported(L):
    """Kernels, templates and helpers have hidden visibility: the dynamic
    symbol table's functions are exactly the declared entry points."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", fa_build.LIB], capture_output=True, text=True, check=True)
    funcs = sorted(ln.split()[-1] for ln in out.stdout.splitlines() if len(ln.split()) == 3 and ln.split()[1] == "T")
    assert funcs == declared_symbols()


def _header_prototypes():
    """{function name: parameter count} of the header's declarations."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(fa_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = " ".join(m.group(2).split())
        protos[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_binding_argtypes_match_header_prototypes(L):
    """The ctypes argument lists have as many entries as the C prototypes
    (guards the binding against a drifted signature)."""
    protos = _header_prototypes()
    assert set(fa.EXPORTED) <= set(protos), set(fa.EXPORTED) - set(protos)
    for name in fa.EXPORTED:
        argtypes = getattr(L, name).argtypes
        if argtypes is None:                       # no-argument functions keep ctypes' default
            assert protos[name] == 0, name
            continue
        assert len(argtypes) == protos[name], (name, len(argtypes), protos[name])


def test_version_and_last_error(L):
    assert "sm_103a" in fa.version()
    assert isinstance(L.fa_last_error(), bytes)


def _launch(num_seqs, total_q, num_splits, max_seqlen_k=0):
    return fa.Launch(num_seqs=num_seqs, max_seqlen_q=1, max_seqlen_k=max_seqlen_k, num_splits=num_splits,
                     total_q=total_q, total_k=0)


def test_workspace_bytes_and_default_splits(L):
    assert fa.workspace_bytes(_launch(4, 0, 4), 8, 8, 128) == 0
    assert fa.workspace_bytes(_launch(4, 10, 0), 8, 8, 128) == 0
    assert fa.workspace_bytes(_launch(4, 10, 1), 8, 8, 128) == 0          # one split writes out directly
    n = fa.workspace_bytes(_launch(64, 64, 16), 32, 8, 128)
    assert n == 16 * 64 * 32 * 128 * 4 + 16 * 32 * 64 * 4 and n % 256 == 0
    assert L.fa_fwd_workspace_bytes(None, 8, 8, 128, None) == 0
    s = fa.default_splits(64, 1, 8192, 32, 8, 16, 64 * 4400)   # decode shape
    assert 2 <= s <= 8
    assert fa.default_splits(64, 1, 8192, 32, 8, 16, 0) >= 1      # total unknown
    assert fa.default_splits(8, 2048, 2048, 16, 16, 0) == 0       # prefill shape
    assert fa.default_splits(64, 8, 8192, 32, 8, 16) == 0         # 8 * 4 rows > 16


def _t(data, dtype, shape, stride=None):
    t = fa.Tensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    if stride is None:
        stride, s = [], 1
        for x in reversed(shape):
            stride.insert(0, s)
            s *= x
    for i, (a, b) in enumerate(zip(shape, stride)):
        t.shape[i] = a
        t.stride[i] = b
    return t


FAKE = 1 << 20  # never dereferenced: validation fails first


def _call(L, **over):
    T, H, D = 256, 4, 64
    args = dict(
        q=_t(FAKE, fa.FA_BF16, [T, H, D]), k=_t(FAKE * 2, fa.FA_BF16, [T, H, D]),
        v=_t(FAKE * 3, fa.FA_BF16, [T, H, D]), bt=None,
        cq=_t(FAKE * 4, fa.FA_I32, [3]), ck=_t(FAKE * 5, fa.FA_I32, [3]), ks=None, vs=None,
        out=_t(FAKE * 6, fa.FA_BF16, [T, H, D]), lse=_t(FAKE * 7, fa.FA_F32, [H, T]),
        scale=0.125, causal=1, window=0, mod=None, bm=None, pro=None, page=0,
        launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, num_splits=0, total_q=T, total_k=T))
    args.update(over)
    r = lambda x: None if x is None else ctypes.byref(x)
    st = L.fa_fwd_varlen(r(args["q"]), r(args["k"]), r(args["v"]), r(args["bt"]), r(args["cq"]), r(args["ck"]),
                         r(args["ks"]), r(args["vs"]), r(args["out"]), r(args["lse"]), args["scale"],
                         args["causal"], args["window"], r(args["mod"]), r(args["bm"]), r(args["pro"]),
                         args["page"], r(args["launch"]), None)
    return st, L.fa_last_error().decode()


def _raw_prologue(n_q=0, n_v=0, q_op=1):
    pro = fa.Prologue()
    pro.n_q, pro.n_v = n_q, n_v
    pro.q[0].op, pro.q[0].value = q_op, 1.0
    return pro


def test_workspace_bytes_counts_a_q_add(L):
    """A Q add needs fp32 [num_seqs, Hkv, ceil(max_seqlen_k / 128) * 128] of
    per-key terms after the split partials; a K add or a Q add on keys
    multiplied by 0 needs nothing."""
    lau = _launch(3, 10, 0, max_seqlen_k=300)
    assert fa.workspace_bytes(lau, 8, 2, 128, {"k": [("add", 1.0)]}) == 0
    assert fa.workspace_bytes(lau, 8, 2, 128, {"q": [("add", 1.0)], "k": [("mul", 0.0)]}) == 0
    assert fa.workspace_bytes(lau, 8, 2, 128, {"q": [("add", 1.0)]}) == 3 * 2 * 384 * 4
    lau2 = _launch(3, 10, 4, max_seqlen_k=300)
    split = fa.workspace_bytes(lau2, 8, 2, 128)
    assert split > 0 and split % 256 == 0
    assert fa.workspace_bytes(lau2, 8, 2, 128, {"q": [("sub", 2.0), ("mul", 3.0)]}) == split + 3 * 2 * 384 * 4


def test_make_prologue_only_copies_the_ops():
    pro = fa.make_prologue({"q": [("mul", 2.0), ("add", 1.0)], "v": [("sub", 0.5), ("div", 4.0)]})
    assert (pro.n_q, pro.n_k, pro.n_v) == (2, 0, 2)
    assert [(pro.q[i].op, pro.q[i].value) for i in range(2)] == [(fa.FA_OP_MUL, 2.0), (fa.FA_OP_ADD, 1.0)]
    assert [(pro.v[i].op, pro.v[i].value) for i in range(2)] == [(fa.FA_OP_SUB, 0.5), (fa.FA_OP_DIV, 4.0)]
    with pytest.raises(ValueError):
        fa.make_prologue({"q": [("pow", 2.0)]})
    with pytest.raises(ValueError):
        fa.make_prologue({"k": [("mul", 1.0)] * 9})


@pytest.mark.parametrize("over,status,words", [
    (dict(q=_t(FAKE, fa.FA_F32, [256, 4, 64])), fa.FA_ERR_INVALID_ARG, "dtype"),
    (dict(q=_t(FAKE, fa.FA_BF16, [256, 4, 96]), k=_t(FAKE * 2, fa.FA_BF16, [256, 4, 96]),
          v=_t(FAKE * 3, fa.FA_BF16, [256, 4, 96]), out=_t(FAKE * 6, fa.FA_BF16, [256, 4, 96])),
     fa.FA_ERR_UNSUPPORTED, "not compiled"),
    (dict(k=_t(FAKE * 2, fa.FA_BF16, [256, 3, 64]), v=_t(FAKE * 3, fa.FA_BF16, [256, 3, 64])),
     fa.FA_ERR_INVALID_ARG, "multiple of Hkv"),
    (dict(cq=_t(FAKE * 4, fa.FA_I32, [4])), fa.FA_ERR_INVALID_ARG, "num_seqs+1"),
    (dict(out=_t(FAKE * 6, fa.FA_BF16, [256, 4, 64], [512, 64, 1])), fa.FA_ERR_INVALID_ARG, "contiguous"),
    (dict(lse=_t(FAKE * 7, fa.FA_F32, [256, 4])), fa.FA_ERR_INVALID_ARG, "lse must be"),
    (dict(lse=_t(FAKE * 6, fa.FA_F32, [4, 256])), fa.FA_ERR_INVALID_ARG, "alias"),
    (dict(q=_t(FAKE, fa.FA_BF16, [256, 4, 64], [256, 64, 2])), fa.FA_ERR_INVALID_ARG, "contiguous last dim"),
    (dict(launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=100, total_k=256)),
     fa.FA_ERR_INVALID_ARG, "total_q"),
    (dict(ks=_t(FAKE * 8, fa.FA_F32, [256, 4])), fa.FA_ERR_INVALID_ARG, "only valid with an e4m3"),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG, "finite"),
    (dict(mod=fa.ScoreMod(kind=2, softcap=0.0)), fa.FA_ERR_INVALID_ARG, "softcap"),
    (dict(mod=fa.ScoreMod(kind=7)), fa.FA_ERR_INVALID_ARG, "kind"),
    (dict(bm=fa.BlockMask(data=FAKE * 9, n_qblk=1, n_kblk=1, blk_q=64, blk_k=64)), fa.FA_ERR_UNSUPPORTED, "128x128"),
    (dict(pro=fa.make_prologue({"q": [("mul", float("nan"))]})), fa.FA_ERR_INVALID_ARG, "finite"),
    (dict(pro=fa.make_prologue({"k": [("div", 0.0)]})), fa.FA_ERR_INVALID_ARG, "divides by 0"),
    (dict(pro=_raw_prologue(n_v=9)), fa.FA_ERR_INVALID_ARG, "ops"),
    (dict(pro=_raw_prologue(n_q=1, q_op=7)), fa.FA_ERR_INVALID_ARG, "FA_OP_MUL"),
    (dict(pro=fa.make_prologue({"q": [("mul", 3e38)], "k": [("mul", 3e38)]})), fa.FA_ERR_INVALID_ARG, "overflow"),
    (dict(pro=fa.make_prologue({"q": [("add", 0.5)]})), fa.FA_ERR_INVALID_ARG, "workspace"),
    (dict(bm=fa.BlockMask(data=FAKE * 9, n_qblk=0, n_kblk=1, blk_q=128, blk_k=128)), fa.FA_ERR_INVALID_ARG, "cover"),
    (dict(launch=None), fa.FA_ERR_INVALID_ARG, "launch"),
])
def test_validation_rejects_before_launch(L, over, status, words):
    st, msg = _call(L, **over)
    assert st == status, msg
    assert words in msg, msg


def test_paged_validation(L):
    bt = _t(FAKE * 10, fa.FA_I32, [2, 8])
    k = _t(FAKE * 2, fa.FA_BF16, [32, 16, 4, 64])
    v = _t(FAKE * 3, fa.FA_BF16, [32, 16, 4, 64])
    st, msg = _call(L, bt=bt, k=k, v=v, page=24)
    assert st == fa.FA_ERR_UNSUPPORTED and "page_size" in msg
    st, msg = _call(L, bt=bt, k=k, v=v, page=2048)
    assert st == fa.FA_ERR_UNSUPPORTED and "1 to 1024" in msg
    st, msg = _call(L, bt=bt, k=k, v=v, page=8)         # a valid size, but not the cache's
    assert st == fa.FA_ERR_INVALID_ARG and "page_size" in msg
    st, msg = _call(L, bt=bt, k=k, v=v, page=32)
    assert st == fa.FA_ERR_INVALID_ARG and "page_size" in msg
    st, msg = _call(L, bt=_t(FAKE * 10, fa.FA_I32, [3, 8]), k=k, v=v, page=16)
    assert st == fa.FA_ERR_INVALID_ARG and "block_table" in msg
    st, msg = _call(L, bt=_t(FAKE * 10, fa.FA_I32, [2, 4]), k=k, v=v, page=16)
    assert st == fa.FA_ERR_INVALID_ARG and "capacity" in msg


@pytest.mark.parametrize("dt", [fa.FA_E4M3, fa.FA_I8])
def test_byte_caches_need_scales(L, dt):
    k = _t(FAKE * 2, dt, [256, 4, 64])
    v = _t(FAKE * 3, dt, [256, 4, 64])
    st, msg = _call(L, k=k, v=v)
    assert st == fa.FA_ERR_INVALID_ARG and "scale" in msg
    st, msg = _call(L, k=_t(FAKE * 2, fa.FA_U8, [256, 4, 64]), v=_t(FAKE * 3, fa.FA_U8, [256, 4, 64]))
    assert st == fa.FA_ERR_INVALID_ARG and "int8" in msg


def test_e4m3_q_limits(L):
    """e4m3 Q runs only with e4m3 K/V at (Dk, Dv) = (128, 128) or (192, 128) and
    without split-KV."""
    T, H = 256, 4
    q8 = _t(FAKE, fa.FA_E4M3, [T, H, 128])
    k8 = _t(FAKE * 2, fa.FA_E4M3, [T, H, 128])
    v8 = _t(FAKE * 3, fa.FA_E4M3, [T, H, 128])
    ks = _t(FAKE * 8, fa.FA_F32, [T, H])
    vs = _t(FAKE * 9, fa.FA_F32, [T, H])
    out = _t(FAKE * 6, fa.FA_BF16, [T, H, 128])
    st, msg = _call(L, q=q8, k=_t(FAKE * 2, fa.FA_BF16, [T, H, 128]), v=_t(FAKE * 3, fa.FA_BF16, [T, H, 128]),
                    out=out)
    assert st == fa.FA_ERR_UNSUPPORTED and "e4m3 k_cache" in msg
    st, msg = _call(L, q=_t(FAKE, fa.FA_E4M3, [T, H, 64]), k=_t(FAKE * 2, fa.FA_E4M3, [T, H, 64]),
                    v=_t(FAKE * 3, fa.FA_E4M3, [T, H, 64]), ks=ks, vs=vs)
    assert st == fa.FA_ERR_UNSUPPORTED and "(192, 128)" in msg
    st, msg = _call(L, q=q8, k=k8, v=v8, ks=ks, vs=vs, out=out,
                    launch=fa.Launch(num_seqs=2, max_seqlen_q=1, max_seqlen_k=128, num_splits=4,
                                     total_q=T, total_k=T))
    assert st == fa.FA_ERR_UNSUPPORTED and "split-KV" in msg
    # pages of < 16 keys are gathered row by row, which e4m3 Q does not have
    st, msg = _call(L, q=q8, k=_t(FAKE * 2, fa.FA_E4M3, [64, 8, H, 128]), v=_t(FAKE * 3, fa.FA_E4M3, [64, 8, H, 128]),
                    ks=_t(FAKE * 8, fa.FA_F32, [64, 8, H]), vs=_t(FAKE * 9, fa.FA_F32, [64, 8, H]), out=out,
                    bt=_t(FAKE * 10, fa.FA_I32, [2, 32]), page=8)
    assert st == fa.FA_ERR_UNSUPPORTED and "at least 16 keys" in msg
    # a row stride of 8 one-byte elements is not a multiple of 16 bytes
    st, msg = _call(L, q=_t(FAKE, fa.FA_E4M3, [T, H, 128], [H * 136, 136, 1]), k=k8, v=v8, ks=ks, vs=vs, out=out)
    assert st == fa.FA_ERR_INVALID_ARG and "16 bytes" in msg
    st, msg = _call(L, q=_t(FAKE, fa.FA_U8, [T, H, 128]), k=k8, v=v8, ks=ks, vs=vs, out=out)
    assert st == fa.FA_ERR_INVALID_ARG and "q dtype" in msg


def test_overflow_guard(L):
    big = (1 << 31)
    st, msg = _call(L, q=_t(FAKE, fa.FA_BF16, [big, 4, 64]), out=_t(FAKE * 6, fa.FA_BF16, [big, 4, 64]),
                    lse=None, launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=big,
                                               total_k=256))
    assert st == fa.FA_ERR_OVERFLOW, msg


def test_split_limits(L):
    st, msg = _call(L, launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, num_splits=4,
                                        total_q=256, total_k=256))
    assert st == fa.FA_ERR_UNSUPPORTED and "split-KV" in msg


def test_combine_validation(L):
    assert L.fa_combine(FAKE, FAKE, 0, 4, 4, 128, FAKE, None, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_combine(FAKE, FAKE, 2, 4, 4, 96, FAKE, None, None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_combine(FAKE, FAKE, 2, 0, 4, 128, FAKE, None, None) == fa.FA_OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        fa.lib()


def test_plan_create_validates_like_the_call(L):
    """fa_fwd_plan_create rejects what fa_fwd_varlen rejects, with the same
    message, and leaves the plan handle NULL; launch/destroy of NULL."""
    T, H, D = 256, 4, 64
    q = _t(FAKE, fa.FA_F32, [T, H, D])
    k, v = _t(FAKE * 2, fa.FA_BF16, [T, H, D]), _t(FAKE * 3, fa.FA_BF16, [T, H, D])
    cq, ck = _t(FAKE * 4, fa.FA_I32, [3]), _t(FAKE * 5, fa.FA_I32, [3])
    out, lse = _t(FAKE * 6, fa.FA_BF16, [T, H, D]), _t(FAKE * 7, fa.FA_F32, [H, T])
    launch = fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, num_splits=0, total_q=T, total_k=T)
    handle = ctypes.c_void_p(12345)
    r = ctypes.byref
    st = L.fa_fwd_plan_create(r(q), r(k), r(v), None, r(cq), r(ck), None, None, r(out), r(lse), 0.125, 1, 0,
                              None, None, None, 0, r(launch), r(handle))
    assert st == fa.FA_ERR_INVALID_ARG and "dtype" in L.fa_last_error().decode()
    assert not handle.value
    st = L.fa_fwd_plan_create(r(q), r(k), r(v), None, r(cq), r(ck), None, None, r(out), r(lse), 0.125, 1, 0,
                              None, None, None, 0, r(launch), None)
    assert st == fa.FA_ERR_INVALID_ARG and "plan" in L.fa_last_error().decode()
    assert L.fa_fwd_plan_launch(None, None) == fa.FA_ERR_INVALID_ARG
    L.fa_fwd_plan_destroy(None)


def _bcall(L, **over):
    T, H, D = 256, 4, 64
    ws = 1 << 30
    args = dict(
        q=_t(FAKE, fa.FA_BF16, [T, H, D]), k=_t(FAKE * 2, fa.FA_BF16, [T, H, D]),
        v=_t(FAKE * 3, fa.FA_BF16, [T, H, D]), out=_t(FAKE * 4, fa.FA_BF16, [T, H, D]),
        dout=_t(FAKE * 5, fa.FA_BF16, [T, H, D]), lse=_t(FAKE * 6, fa.FA_F32, [H, T]),
        cq=_t(FAKE * 7, fa.FA_I32, [3]), ck=_t(FAKE * 8, fa.FA_I32, [3]),
        dq=_t(FAKE * 9, fa.FA_BF16, [T, H, D]), dk=_t(FAKE * 10, fa.FA_BF16, [T, H, D]),
        dv=_t(FAKE * 11, fa.FA_BF16, [T, H, D]), scale=0.125, causal=1, window=0, mod=None, bm=None,
        launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, num_splits=0, total_q=T, total_k=T,
                         workspace=ws, workspace_bytes=fa.bwd_workspace_bytes(T, H)))
    args.update(over)
    r = lambda x: None if x is None else ctypes.byref(x)
    st = L.fa_bwd_varlen(*[r(args[n]) for n in ("q", "k", "v", "out", "dout", "lse", "cq", "ck", "dq", "dk", "dv")],
                         args["scale"], args["causal"], args["window"], r(args["mod"]), r(args["bm"]),
                         r(args["launch"]), None)
    return st, L.fa_last_error().decode()


def test_bwd_workspace_bytes(L):
    assert fa.bwd_workspace_bytes(0, 4) == 0
    n = fa.bwd_workspace_bytes(1000, 16)
    assert n >= 1000 * 16 * 4 and n % 256 == 0


@pytest.mark.parametrize("over,status,words", [
    (dict(q=_t(FAKE, fa.FA_BF16, [256, 4, 96])), fa.FA_ERR_UNSUPPORTED, "Dk = Dv in {64, 128}"),
    (dict(k=_t(FAKE * 2, fa.FA_BF16, [256, 3, 64]), v=_t(FAKE * 3, fa.FA_BF16, [256, 3, 64]),
          dk=_t(FAKE * 10, fa.FA_BF16, [256, 3, 64]), dv=_t(FAKE * 11, fa.FA_BF16, [256, 3, 64])),
     fa.FA_ERR_INVALID_ARG, "multiple of Hkv"),
    (dict(k=_t(FAKE * 2, fa.FA_BF16, [16, 16, 4, 64])), fa.FA_ERR_INVALID_ARG, "packed"),
    (dict(dout=_t(FAKE * 5, fa.FA_BF16, [255, 4, 64])), fa.FA_ERR_INVALID_ARG, "dout has shape"),
    (dict(dq=_t(FAKE * 9, fa.FA_BF16, [256, 4, 64], [256, 64, 2])), fa.FA_ERR_INVALID_ARG, "contiguous"),
    (dict(lse=_t(FAKE * 6, fa.FA_F32, [256, 4])), fa.FA_ERR_INVALID_ARG, "lse must be"),
    (dict(dk=_t(FAKE * 2, fa.FA_BF16, [256, 4, 64])), fa.FA_ERR_INVALID_ARG, "overlap"),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG, "softmax_scale"),
    (dict(mod=fa.ScoreMod(kind=2, softcap=-1.0)), fa.FA_ERR_INVALID_ARG, "softcap"),
    (dict(mod=fa.ScoreMod(kind=1, alibi_slope=float("inf"))), fa.FA_ERR_INVALID_ARG, "alibi_slope"),
    (dict(mod=fa.ScoreMod(kind=3)), fa.FA_ERR_INVALID_ARG, "kind"),
    (dict(bm=fa.BlockMask(data=FAKE * 12, n_qblk=1, n_kblk=0, blk_q=128, blk_k=128)), fa.FA_ERR_INVALID_ARG,
     "does not cover"),
    (dict(bm=fa.BlockMask(data=FAKE * 12, n_qblk=2, n_kblk=2, blk_q=64, blk_k=64)), fa.FA_ERR_UNSUPPORTED, "128x128"),
    (dict(launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=256, total_k=256)),
     fa.FA_ERR_INVALID_ARG, "workspace"),
    (dict(launch=fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=256, total_k=256,
                           workspace=(1 << 30) + 8, workspace_bytes=1 << 20)),
     fa.FA_ERR_INVALID_ARG, "256-byte aligned"),
    (dict(cq=_t(FAKE * 7, fa.FA_I32, [4])), fa.FA_ERR_INVALID_ARG, "num_seqs + 1"),
    (dict(launch=None), fa.FA_ERR_INVALID_ARG, "launch"),
])
def test_bwd_validation_rejects_before_launch(L, over, status, words):
    st, msg = _bcall(L, **over)
    assert st == status, msg
    assert words in msg, msg


def test_vec5_limits(L):
    """The vectorized 5-D pages are accepted for e4m3 and int8 caches with
    pages of >= 16 keys and bf16 q; other combinations fail before launch."""
    T, H = 256, 4
    q = _t(FAKE, fa.FA_BF16, [T, H, 128])
    out = _t(FAKE * 6, fa.FA_BF16, [T, H, 128])
    bt = _t(FAKE * 10, fa.FA_I32, [2, 8])
    ks = _t(FAKE * 8, fa.FA_F32, [32, 16, H])
    vs = _t(FAKE * 9, fa.FA_F32, [32, 16, H])
    k5 = _t(FAKE * 2, fa.FA_E4M3, [32, H, 8, 16, 16])
    v5 = _t(FAKE * 3, fa.FA_E4M3, [32, H, 1, 128, 16])
    lau = fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=T, total_k=0)
    st, msg = _call(L, q=q, k=_t(FAKE * 2, fa.FA_BF16, [32, H, 16, 16, 8]), v=_t(FAKE * 3, fa.FA_BF16, [32, H, 2, 128, 8]),
                    bt=bt, page=16, out=out, launch=lau)
    assert st == fa.FA_ERR_UNSUPPORTED and "5-D" in msg
    st, msg = _call(L, q=q, k=k5, v=_t(FAKE * 3, fa.FA_E4M3, [32, H, 2, 128, 16]), ks=ks, vs=vs, bt=bt, page=16,
                    out=out, launch=lau)
    assert st == fa.FA_ERR_INVALID_ARG and "disagree" in msg
    st, msg = _call(L, q=_t(FAKE, fa.FA_E4M3, [T, H, 128]), k=k5, v=v5, ks=ks, vs=vs, bt=bt, page=16, out=out,
                    launch=lau)
    assert st == fa.FA_ERR_UNSUPPORTED and "token-major" in msg
    st, msg = _call(L, q=q, k=k5, v=v5, ks=_t(FAKE * 8, fa.FA_F32, [32, H, 16]), vs=vs, bt=bt, page=16, out=out,
                    launch=lau)
    assert st == fa.FA_ERR_INVALID_ARG and "[N_pg, P_s, Hkv]" in msg
    # prologue adds that need key sums or the row term under the cap
    st, msg = _call(L, q=q, k=k5, v=v5, ks=ks, vs=vs, bt=bt, page=16, out=out, launch=lau,
                    pro=fa.make_prologue({"q": [("add", 0.5)]}))
    assert st == fa.FA_ERR_UNSUPPORTED and "token-major" in msg
    cap = fa.ScoreMod(kind=fa.MOD_SOFTCAP, alibi_slope=0.0, softcap=20.0)
    st, msg = _call(L, q=q, k=k5, v=v5, ks=ks, vs=vs, bt=bt, page=16, out=out, launch=lau, mod=cap,
                    pro=fa.make_prologue({"k": [("add", 0.5)]}))
    assert st == fa.FA_ERR_UNSUPPORTED and "5-D" in msg


def test_vectorize_pages_inverts_with_the_pages_permutes():
    """fa_inputs.vectorize_pages builds the 5-D K [N_pg, Hkv, Dk/16, P_s, 16]
    and V [N_pg, Hkv, P_s/16, Dv, 16]; the permutes (0, 3, 1, 2, 4) and
    (0, 2, 4, 1, 3) (FlyDSL PR #1066, review) give the token-major pages back."""
    import numpy as np
    import fa_inputs as fi
    p = fi.make_problem([40, 70], [100, 70], hq=4, hkv=2, dk=192, dv=128, seed=3, page_size=32, kv_dtype="e4m3",
                        spare_pages=2)
    k5, v5 = fi.vectorize_pages(p.k, p.v)
    assert k5.shape == (p.k.shape[0], 2, 12, 32, 16) and v5.shape == (p.v.shape[0], 2, 2, 128, 16)
    assert np.array_equal(k5.transpose(0, 3, 1, 2, 4).reshape(p.k.shape), p.k)
    assert np.array_equal(v5.transpose(0, 2, 4, 1, 3).reshape(p.v.shape), p.v)
    # element (page, slot, head, d) of K sits at [page, head, d // 16, slot, d % 16]
    assert k5[3, 1, 5, 7, 9] == p.k[3, 7, 1, 5 * 16 + 9]
    assert v5[2, 0, 1, 100, 3] == p.v[2, 16 + 3, 0, 100]


def test_pv_e4m3_flag_limits(L):
    """FA_FLAG_PV_E4M3 takes e4m3 q with e4m3 caches; other flag bits are
    rejected; the workspace gains one fp32 per (sequence, kv head)."""
    T, H = 256, 4
    bt = _t(FAKE * 10, fa.FA_I32, [2, 8])
    ks = _t(FAKE * 8, fa.FA_F32, [32, 16, H])
    vs = _t(FAKE * 9, fa.FA_F32, [32, 16, H])
    k8 = _t(FAKE * 2, fa.FA_E4M3, [32, 16, H, 128])
    v8 = _t(FAKE * 3, fa.FA_E4M3, [32, 16, H, 128])
    out = _t(FAKE * 6, fa.FA_BF16, [T, H, 128])
    lau = fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=T, total_k=0, flags=fa.FLAG_PV_E4M3)
    st, msg = _call(L, q=_t(FAKE, fa.FA_BF16, [T, H, 128]), k=k8, v=v8, ks=ks, vs=vs, bt=bt, page=16, out=out,
                    launch=lau)
    assert st == fa.FA_ERR_UNSUPPORTED and "FA_FLAG_PV_E4M3" in msg
    bad = fa.Launch(num_seqs=2, max_seqlen_q=128, max_seqlen_k=128, total_q=T, total_k=0, flags=6)
    st, msg = _call(L, q=_t(FAKE, fa.FA_E4M3, [T, H, 128]), k=k8, v=v8, ks=ks, vs=vs, bt=bt, page=16, out=out,
                    launch=bad)
    assert st == fa.FA_ERR_INVALID_ARG and "flags" in msg
    plain = fa.Launch(num_seqs=3, max_seqlen_q=10, max_seqlen_k=300, total_q=10, total_k=0)
    flagged = fa.Launch(num_seqs=3, max_seqlen_q=10, max_seqlen_k=300, total_q=10, total_k=0, flags=fa.FLAG_PV_E4M3)
    assert fa.workspace_bytes(flagged, 8, 2, 128) - fa.workspace_bytes(plain, 8, 2, 128) == 256
    st, msg = _call(L, q=_t(FAKE, fa.FA_E4M3, [T, H, 128]), k=k8, v=v8, ks=ks, vs=vs, bt=bt, page=16, out=out,
                    launch=lau)
    assert st == fa.FA_ERR_INVALID_ARG and "workspace" in msg

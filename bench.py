"""Benchmark of the attention forward pass on one GB300 (replicas for N > 1).

Headline workload: config 5, the flex bf16 prefill at B=4, H=16, S=8192,
D=128 (N(0,1) inputs, seed 0).  One step runs its six variants once each over
inputs already resident in HBM: ALiBi (slope 0.0625) causal and non-causal,
soft-cap 20 causal and non-causal, sliding window 256 causal, and a seeded
50% random 128x128 block mask.  The metric is algorithmic TFLOP/s: 2*Dk +
2*Dv flops per (head, query, key) pair the mask allows.  L2 is flushed (a
256 MiB write) before every launch, outside the timed events.

Other workloads are reported under ``workloads`` (full figures) and
``summary`` (compact, last in the line): the packed varlen prefill of config
2, the dense causal latency case, the paged split-KV decodes (KV-cache GB/s),
the paged e4m3 prefill of config 4, and the backward pass.  ``--impl
reference`` times the fp64 CPU oracle instead (bounded row samples of the
same six runs, on the host cores).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import fa_inputs as fi  # noqa: E402

METRIC = "attn fwd TFLOP/s (prefill) & KV-cache GB/s (decode), % of GB300 roofline"
# sources of the headline kernel (fa_prefill2_kernel): `traffic` is reported only
# while profiles/traffic.json was captured from these exact files
KERNEL_SOURCES = ["flashattention_forward_gb300/csrc/fa_prefill.cuh", "flashattention_forward_gb300/csrc/fa_prefill2.cuh",
                  "flashattention_forward_gb300/csrc/sm103_ptx.cuh",
                  "flashattention_forward_gb300/csrc/fa_gather.cuh"]


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle sampling; only samples whose timestamps fall
    inside the marked timed window are summarised."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.samples = []
        self.proc = None
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "10"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.5)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        import datetime
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            self.samples.append((ts, parts[1:]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def __exit__(self, *a):
        time.sleep(0.05)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sel = self.samples
        if self.window:
            t0, t1 = self.window
            sel = [s for s in self.samples if t0 - 0.01 <= s[0] <= t1 + 0.01]
        sel = [s[1] for s in sel]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(s[0]) for s in sel if num(s[0])]
        mx = [float(s[1]) for s in sel if num(s[1])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in sel for i in range(4) if s[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel)}


def dev_tensors(p, dev):
    if p.q_dtype == "e4m3":
        t = {"q": torch.from_numpy(p.q.copy()).view(torch.float8_e4m3fn).to(dev)}
    else:
        t = {"q": torch.from_numpy(p.q.view(np.int16).copy()).view(torch.bfloat16).to(dev)}
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


def prefill_bytes(p):
    """Algorithmic bytes of one prefill launch: Q, K, V read once, O and LSE written once."""
    esize = 2 if p.kv_dtype == "bf16" else 1
    kv_tok = float(p.seqlens_k.sum())
    qo = p.total_q * p.hq * (p.dk * 2 + p.dv * 2 + 4)
    kv = kv_tok * p.hkv * (p.dk + p.dv) * esize + (kv_tok * p.hkv * 8 if p.kv_dtype == "e4m3" else 0)
    return qo + kv


def make_call(p, t, num_splits=0, pv_e4m3=False):
    import flashattention_forward_gb300 as fa
    dev = t["q"].device
    out = torch.empty((p.total_q, p.hq, p.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.hq, p.total_q), dtype=torch.float32, device=dev)
    ws = None
    if num_splits is None:
        num_splits = fa.default_splits(p.num_seqs, p.max_seqlen_q, p.max_seqlen_k, p.hq, p.hkv, p.page_size,
                                       p.total_k)
    launch = fa.Launch(num_seqs=p.num_seqs, max_seqlen_q=p.max_seqlen_q, max_seqlen_k=p.max_seqlen_k,
                       num_splits=num_splits, total_q=p.total_q, total_k=p.total_k,
                       flags=fa.FLAG_PV_E4M3 if pv_e4m3 else 0)
    need = fa.workspace_bytes(launch, p.hq, p.hkv, p.dv, p.prologue)
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)

    plan = fa.FwdPlan(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                      max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, block_table=t.get("bt"),
                      page_size=p.page_size, k_scale=t.get("k_scale"), v_scale=t.get("v_scale"),
                      softmax_scale=p.softmax_scale, causal=p.causal, window=p.window, score_mod=p.mod_kind,
                      alibi_slope=p.alibi_slope, softcap=p.softcap, block_mask=t.get("bm"),
                      num_splits=num_splits, out=out, lse=lse, workspace=ws, pv_e4m3=pv_e4m3)

    def call():
        return plan.run()
    launches = 1 + (1 if num_splits > 1 else 0)
    return call, launches, out, lse


def make_bwd_call(p, t):
    """A backward call (fa_bwd_varlen) on preallocated buffers: out and LSE from
    one forward call, a seeded N(0,1) dout."""
    import flashattention_forward_gb300 as fa
    dev = t["q"].device
    out, lse = fa.fwd_varlen(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max_seqlen_q=p.max_seqlen_q,
                             max_seqlen_k=p.max_seqlen_k, total_k=p.total_k, softmax_scale=p.softmax_scale,
                             causal=p.causal, window=p.window, num_splits=0, score_mod=p.mod_kind,
                             alibi_slope=p.alibi_slope, softcap=p.softcap, block_mask=t.get("bm"))
    g = torch.Generator(device="cpu").manual_seed(17)
    dout = torch.randn(out.shape, generator=g).to(torch.bfloat16).to(dev)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    ws = torch.empty(max(fa.bwd_workspace_bytes(p.total_q, p.hq), 256), dtype=torch.uint8, device=dev)

    def call():
        return fa.bwd_varlen(t["q"], t["k"], t["v"], out, dout, lse, t["cu_q"], t["cu_k"],
                             max_seqlen_q=p.max_seqlen_q, max_seqlen_k=p.max_seqlen_k,
                             softmax_scale=p.softmax_scale, causal=p.causal, window=p.window,
                             score_mod=p.mod_kind, alibi_slope=p.alibi_slope, softcap=p.softcap,
                             block_mask=t.get("bm"), dq=dq, dk=dk, dv=dv, workspace=ws)
    return call


class Flusher:
    def __init__(self, dev):
        self.buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.fill_(1)


def time_calls(calls, warmup, steps, flush):
    """Per-step CUDA-event time of running every call once (L2 flushed between steps)."""
    for _ in range(warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for c in calls:
            c()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    return times


def time_each(calls, warmup, steps, flush):
    """Per-call CUDA-event times (one list per call)."""
    res = [[] for _ in calls]
    for _ in range(warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    for _ in range(steps):
        for i, c in enumerate(calls):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            c()
            e.record()
            e.synchronize()
            res[i].append(s.elapsed_time(e))
    return res


def e2e_measure(p, steps, dev):
    """Same metric through the public API with HOST inputs: pinned H2D copies of
    every input, the forward pass, and D2H of out + LSE, all inside the events."""
    import flashattention_forward_gb300 as fa
    hq = {k: v.cpu().pin_memory() for k, v in dev_tensors(p, "cpu").items()}
    dd = {k: torch.empty_like(v, device=dev) for k, v in hq.items()}
    out_h = torch.empty((p.total_q, p.hq, p.dv), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((p.hq, p.total_q), dtype=torch.float32).pin_memory()
    call, _, out, lse = make_call(p, dd, num_splits=0)
    h2d = sum(v.numel() * v.element_size() for v in hq.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    ts = []
    for i in range(steps + 2):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for k in hq:
            dd[k].copy_(hq[k], non_blocking=True)
        call()
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        e.record()
        e.synchronize()
        if i >= 2:
            ts.append(s.elapsed_time(e))
    return statistics.mean(ts), h2d, d2h


def e2e_pipelined(problems, steps, dev):
    """The same end-to-end step (pinned H2D of every input, the forward calls,
    D2H of out + LSE for every problem) run as a serving loop would: two device
    buffer sets, so that step i+1's H2D (copy stream) overlaps step i's
    forward passes (compute stream) and its D2H (return stream).  Every step
    still moves all of its inputs and results; returns ms per step over the
    whole loop (first H2D to last D2H)."""
    sets = []
    for p in problems:
        hq = {k: v.cpu().pin_memory() for k, v in dev_tensors(p, "cpu").items()}
        bufs = []
        for _ in range(2):
            dd = {k: torch.empty_like(v, device=dev) for k, v in hq.items()}
            call, _, out, lse = make_call(p, dd, num_splits=0)
            out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
            bufs.append((dd, call, out, lse, out_h, lse_h))
        sets.append((hq, bufs))
    s_copy, s_comp, s_back = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def loop(n):
        ev_comp, ev_back = [], []
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_copy)
        for i in range(n):
            b = i % 2
            h2d = torch.cuda.Event()
            with torch.cuda.stream(s_copy):
                if i >= 2:
                    s_copy.wait_event(ev_comp[i - 2])      # step i-2 no longer reads buffer set b
                for hq, bufs in sets:
                    for k, v in hq.items():
                        bufs[b][0][k].copy_(v, non_blocking=True)
                h2d.record(s_copy)
            ec = torch.cuda.Event()
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(h2d)
                if i >= 2:
                    s_comp.wait_event(ev_back[i - 2])      # step i-2's results are home
                for hq, bufs in sets:
                    bufs[b][1]()
                ec.record(s_comp)
            ev_comp.append(ec)
            eb = torch.cuda.Event()
            with torch.cuda.stream(s_back):
                s_back.wait_event(ec)
                for hq, bufs in sets:
                    _, _, out, lse, out_h, lse_h = bufs[b]
                    out_h.copy_(out, non_blocking=True)
                    lse_h.copy_(lse, non_blocking=True)
                eb.record(s_back)
            ev_back.append(eb)
        end.record(s_back)
        end.synchronize()
        return start.elapsed_time(end) / n

    loop(3)
    return loop(steps)


def row_flops(p, units):
    """Algorithmic flops of (token, head) rows: allowed keys * (2 Dk + 2 Dv),
    with the causal, window and block masks counted exactly."""
    sk, sq = p.seqlens_k, p.seqlens_q
    seq_of = np.searchsorted(p.cu_seqlens_q[1:], units[:, 0], side="right")
    total = 0
    for (t, h), b in zip(units, seq_of):
        i = int(t - p.cu_seqlens_q[b])
        ip = i + int(sk[b]) - int(sq[b])
        lo, hi = 0, int(sk[b])
        if p.causal:
            hi = min(hi, ip + 1)
        if p.window > 0:
            lo = max(lo, ip - p.window + 1)
            if not p.causal:
                hi = min(hi, ip + p.window)
        if hi <= lo:
            continue
        if p.block_mask is None:
            total += hi - lo
        else:
            m = p.block_mask[b * p.hq + int(h), i // fi.BLOCK]
            for kb in range(lo // fi.BLOCK, (hi - 1) // fi.BLOCK + 1):
                if kb < m.shape[0] and m[kb]:
                    total += min(hi, (kb + 1) * fi.BLOCK) - max(lo, kb * fi.BLOCK)
    return float(total) * (2 * p.dk + 2 * p.dv)


def cpu_oracle_sample(p, seconds_target=2.0, seed=0, n0=256):
    """Time the oracle on a seeded row sample of about ``seconds_target``
    seconds; return (flop/s, rows, threads, secs, flops)."""
    import oracle
    rng = np.random.default_rng(seed)
    n_all = p.total_q * p.hq
    threads = os.cpu_count() or 1
    n = max(16, n0)
    while True:
        idx = rng.choice(n_all, size=min(n, n_all), replace=False)
        units = np.stack([idx // p.hq, idx % p.hq], -1).astype(np.int64)
        t0 = time.time()
        oracle.forward(p, units=units, nthreads=threads)
        dt = time.time() - t0
        if dt > 0.5 * seconds_target or n >= n_all:
            break
        n = int(n * min(8.0, max(2.0, seconds_target / max(dt, 1e-3))))
    flops = row_flops(p, units)
    return flops / dt, len(units), threads, dt, flops


def measure_fp8_peak(dev, n=8192, reps=10):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput (torch._scaled_mm, cuBLASLt),
    best of `reps`, TFLOP/s: the denominator for contractions that run at the
    e4m3 rate.  None if this torch has no _scaled_mm."""
    if not hasattr(torch, "_scaled_mm"):
        return None
    a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device=dev)
    for _ in range(3):
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    best = float("inf")
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e))
    del a, b
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def max_over_ranks(ms, dist=None, device="cpu"):
    """The slowest rank's step time: every replica's work counts only once all
    ranks have finished it."""
    if dist is None:
        return ms
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_rate(flops_per_step, world, ms):
    """Whole-job TFLOP/s: `world` replicas each did `flops_per_step` in `ms`."""
    return flops_per_step * world / (ms * 1e-3) / 1e12


HEADLINE = ("flex_prefill_b4_h16_s8192_d128_bf16: 6 runs (ALiBi 0.0625 causal and non-causal, soft-cap 20 "
            "causal and non-causal, sliding window 256 causal, 50% random 128x128 block mask)")


def headline_problems():
    """The six config-5 runs (one shared set of Q, K, V; only the mods and
    masks differ)."""
    return fi.config5_runs()


def headline_calls(probs, t, dev):
    calls, outs = [], []
    for p in probs:
        tp = dict(t)
        if p.block_mask is not None:
            tp["bm"] = torch.from_numpy(p.block_mask.copy()).to(dev)
        call, n, out, lse = make_call(p, tp, num_splits=0)
        assert n == 1
        calls.append(call)
        outs.append((out, lse))
    return calls, outs


def e2e_headline(probs, steps, dev):
    """The headline step end to end through the public API with HOST inputs:
    every step copies the batch (Q, K, V, cu_seqlens, block mask) from pinned
    host memory, runs the six calls and copies every output and LSE back.
    Pipelined as a serving loop: two device buffer sets, step i+1's H2D (copy
    stream) overlaps step i's calls (compute stream) and D2H (return stream).
    Returns (ms per step pipelined, ms per step serial, H2D bytes, D2H bytes)."""
    host_in = {k: v.cpu().pin_memory() for k, v in dev_tensors(probs[0], "cpu").items()}
    bm_p = next(p for p in probs if p.block_mask is not None)
    host_in["bm"] = torch.from_numpy(bm_p.block_mask.copy()).pin_memory()
    sets = []
    for _ in range(2):
        dd = {k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
        calls = []
        for p in probs:
            tp = {k: v for k, v in dd.items() if k != "bm"}
            if p.block_mask is not None:
                tp["bm"] = dd["bm"]
            call, _, out, lse = make_call(p, tp, num_splits=0)
            calls.append((call, out, lse, torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                          torch.empty(lse.shape, dtype=lse.dtype).pin_memory()))
        sets.append((dd, calls))
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(c[3].numel() * c[3].element_size() + c[4].numel() * c[4].element_size() for c in sets[0][1])
    s_copy, s_comp, s_back = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def loop(n):
        ev_comp, ev_back = [], []
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_copy)
        for i in range(n):
            dd, calls = sets[i % 2]
            h2d_ev = torch.cuda.Event()
            with torch.cuda.stream(s_copy):
                if i >= 2:
                    s_copy.wait_event(ev_comp[i - 2])      # step i-2 no longer reads this buffer set
                for k, v in host_in.items():
                    dd[k].copy_(v, non_blocking=True)
                h2d_ev.record(s_copy)
            ec = torch.cuda.Event()
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(h2d_ev)
                if i >= 2:
                    s_comp.wait_event(ev_back[i - 2])      # step i-2's results are home
                for c in calls:
                    c[0]()
                ec.record(s_comp)
            ev_comp.append(ec)
            eb = torch.cuda.Event()
            with torch.cuda.stream(s_back):
                s_back.wait_event(ec)
                for _, out, lse, out_h, lse_h in calls:
                    out_h.copy_(out, non_blocking=True)
                    lse_h.copy_(lse, non_blocking=True)
                eb.record(s_back)
            ev_back.append(eb)
        end.record(s_back)
        end.synchronize()
        return start.elapsed_time(end) / n

    def serial(n):
        dd, calls = sets[0]
        ts = []
        for i in range(n + 1):
            s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_ev.record()
            for k, v in host_in.items():
                dd[k].copy_(v, non_blocking=True)
            for c in calls:
                c[0]()
            for _, out, lse, out_h, lse_h in calls:
                out_h.copy_(out, non_blocking=True)
                lse_h.copy_(lse, non_blocking=True)
            e_ev.record()
            e_ev.synchronize()
            if i:
                ts.append(s_ev.elapsed_time(e_ev))
        return statistics.mean(ts)

    loop(3)
    # the overlap of the three streams varies from loop to loop: the median
    # of three timed loops
    piped = statistics.median([loop(steps) for _ in range(3)])
    return piped, serial(max(2, steps // 2)), h2d, d2h


def reference_arm(args, warmup, probs, flops_runs, workload):
    """The fp64 CPU oracle as the reference arm: each step times a seeded row
    sample of every run of the headline step, sized so that the whole run
    (warm-up included) takes about a minute of host time."""
    per_step = min(12.0, max(0.3, 60.0 / (args.steps + warmup)))
    per_run = per_step / len(probs)
    n_cal = [256] * len(probs)
    for w in range(warmup):
        for j, p in enumerate(probs):
            n_cal[j] = cpu_oracle_sample(p, per_run, seed=1000 + 10 * w + j, n0=n_cal[j])[1]
    rates, t_steps, rows, threads = [], [], 0, os.cpu_count() or 1
    for k in range(args.steps):
        flops = secs = 0.0
        for j, p in enumerate(probs):
            r = cpu_oracle_sample(p, per_run, seed=10 * k + j, n0=n_cal[j])
            n_cal[j], threads = r[1], r[2]
            flops += r[4]
            secs += r[3]
            rows += r[1]
        rates.append(flops / secs / 1e12)
        t_steps.append(secs * 1e3)
    val = statistics.mean(rates)
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": warmup, "ms_per_step": statistics.mean(t_steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"per step, a seeded sample of (token, head) rows of each of the six runs "
                                       f"(about {per_run:.2f} s of fp64 C each, {threads} threads); "
                                       f"{rows} rows over the {args.steps} timed steps"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--profile", default=None,
                    help="run only `warmup + steps` launches of one workload (for ncu captures): "
                         "varlen_causal, varlen_noncausal, decode, dense, flex_<run>, ...")
    args = ap.parse_args()
    if args.profile:
        return profile_only(args.profile, args.warmup, args.steps)
    warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    probs = headline_problems()
    flops_runs = [fi.prefill_flops(p) for p in probs]
    flops_step = sum(flops_runs)
    workload = {"workload": HEADLINE, "runs": list(fi.CONFIG5_RUNS), "batch": 4, "seq_len": 8192, "hq": 16,
                "hkv": 16, "d": 128, "gflop_per_step": flops_step / 1e9,
                "l2": "flushed before every launch (256 MiB write)"}

    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, warmup, probs, flops_runs, workload)
        if dist:
            dist.destroy_process_group()
        return

    import flashattention_forward_gb300 as fa
    from flashattention_forward_gb300 import build as fa_build
    if rank == 0 or world == 1:
        fa_build.build()
    if dist:
        dist.barrier()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.lib()
    flush = Flusher(dev)
    pk = peaks()

    # ------------------------------------------------------- headline step --
    t = dev_tensors(probs[0], dev)
    t.pop("bm", None)
    calls, _ = headline_calls(probs, t, dev)
    for _ in range(warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.time()
        each = time_each(calls, 0, args.steps, flush)
        clk.mark(t0, time.time())
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    step_ms = [sum(x) for x in zip(*each)]
    ms = max_over_ranks(statistics.mean(step_ms), dist, dev)
    value = whole_job_rate(flops_step, world, ms)
    runs = {}
    for j, (run, p) in enumerate(zip(fi.CONFIG5_RUNS, probs)):
        mj = statistics.mean(each[j])
        tf = flops_runs[j] / (mj * 1e-3) / 1e12
        ent = {"ms": mj, "tflops": tf, "frac_bf16": tf / pk["bf16"], "gflop": flops_runs[j] / 1e9}
        if run == "window_causal":
            gbs = prefill_bytes(p) / (mj * 1e-3) / 1e9
            ent.update({"GB/s": gbs, "frac_hbm": gbs / pk["hbm"], "algorithmic_bytes": prefill_bytes(p)})
        runs[run] = ent
    # dominant launch: the run with the largest share of the step
    jd = max(range(len(probs)), key=lambda j: statistics.mean(each[j]))
    pd, run_d = probs[jd], fi.CONFIG5_RUNS[jd]
    ms_d = statistics.mean(each[jd])
    ach = flops_runs[jd] / (ms_d * 1e-3) / 1e12
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath))
        if tj.get("kernel_hash") == kernel_hash() and tj.get("workload") == "flex_" + run_d:
            traffic = tj.get("dram_bytes_per_launch")
    mod_name = {0: "none", 1: "alibi", 2: "softcap"}[pd.mod_kind]
    roofline = {"bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16"], "traffic": traffic, "algorithmic_bytes": prefill_bytes(pd),
                "kernel": f"fa_prefill2_kernel<128,128,packed,{mod_name}>, config-5 run '{run_d}' "
                          f"({'one query tile per CTA, two CTAs per SM' if pd.mod_kind == 2 or pd.window > 0 or (pd.mod_kind == 1 and pd.causal) or pd.block_mask is not None else 'two query tiles per CTA'}, as the library picks)",
                "share_of_step": ms_d / statistics.mean(step_ms),
                "peak_source": f"{pk['src']} bf16 burst (cuBLAS 8192^3)"}
    extra, summary, e2e, cpu = {}, {}, None, None
    if rank == 0:
        piped, serial, h2d, d2h = e2e_headline(probs, max(4, args.steps // 2), dev)
        e2e = {"value": flops_step / (piped * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": piped,
               "schedule": "two buffer sets: step i+1's pinned H2D overlaps step i's six calls and D2H",
               "serial": {"value": flops_step / (serial * 1e-3) / 1e12, "ms_per_step": serial,
                          "schedule": "H2D, six calls, D2H in sequence on one stream"}}
        torch.cuda.empty_cache()
        if not args.quick:
            extra = other_workloads(dev, warmup, max(5, args.steps // 2), flush, pk)
        if world == 1:
            flops = secs = 0.0
            rows = threads = 0
            for j, p in enumerate(probs):
                r = cpu_oracle_sample(p, 2.0, seed=j)
                flops += r[4]
                secs += r[3]
                rows += r[1]
                threads = r[2]
            cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"{rows} seeded (token, head) rows across the six runs (about 2 s each), "
                             f"{secs:.1f} s of fp64 C with {threads} threads"}
        summary = compact_summary(runs, extra, pk)
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": len(calls) * args.steps, "clocks": clk.summary(),
                "pct_of_peak": 100.0 * value / world / pk["bf16"], "kernel_hash": kernel_hash(),
                "runs": runs, "workloads": extra, "summary": summary}
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def compact_summary(runs, extra, pk):
    """Short per-workload figures (ms, TFLOP/s or GB/s, fraction of the
    roofline) placed last in the printed line."""
    r3 = lambda x: round(float(x), 3)
    out = {"c5": {k: [r3(v["ms"]), r3(v["tflops"]), r3(v.get("frac_hbm", v["frac_bf16"]))] for k, v in runs.items()}}
    key = {"varlen_prefill_8seq_h16_d128_causal": "c2_causal", "varlen_prefill_8seq_h16_d128_noncausal": "c2",
           "paged_decode_64seq_hq32_hkv8_p16": "c3", "paged_decode_e4m3_64seq_hq32_hkv8_p16": "c3_e4m3",
           "paged_decode_int8_64seq_hq32_hkv8_p16": "c3_int8", "paged_fp8_d192_v128_16seq_h16_p64_causal": "c4",
           "paged_fp8kv_qe4m3_d128_16seq_h16_p64_causal": "c4_q8_d128",
           "paged_fp8kv_qe4m3_d192_v128_16seq_h16_p64_causal": "c4_q8",
           "paged_fp8kv_qe4m3_pv8_d192_v128_16seq_h16_p64_causal": "c4_q8_pv8",
           "paged_fp8_d192_v128_16seq_h16_p64_causal_vec5": "c4_vec5",
           "paged_decode_e4m3_64seq_hq32_hkv8_p16_vec5": "c3_e4m3_vec5",
           "bwd_4x4096_h16_d128_noncausal": "bwd_4x4096"}
    for name, short in key.items():
        v = extra.get(name)
        if not v:
            continue
        if "GB/s" in v:
            out[short] = [r3(v["ms"]), r3(v["GB/s"]), r3(v["frac_hbm"])]
        else:
            out[short] = [r3(v["ms"]), r3(v["tflops"]), r3(v.get("frac_bf16", v.get("frac_fp8", 0.0)))]
    d = extra.get("dense_causal_b2_h4_s128_d64")
    if d:
        out["c1_us"] = [r3(d["device_us_per_launch"]), r3(d["wall_us_per_call"])]
    out["fields"] = ("c5 and prefill: [ms, TFLOP/s, frac of bf16 peak (c4_q8_pv8: of the e4m3 peak)]; "
                     "decode and window: [ms, GB/s, frac of HBM]")
    return out


def other_workloads(dev, warmup, steps, flush, pk):
    import flashattention_forward_gb300 as fa
    res = {}
    # config 2: packed varlen bf16 prefill, 8 seqs U{0..2048}, H 16, D 128
    for causal in (True, False):
        p = fi.config2(causal=causal)
        t = dev_tensors(p, dev)
        call, _, _, _ = make_call(p, t, num_splits=0)
        ms = statistics.mean(time_calls([call], warmup, steps, flush))
        fl = fi.prefill_flops(p)
        res["varlen_prefill_8seq_h16_d128_" + ("causal" if causal else "noncausal")] = {
            "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
            "gflop": fl / 1e9, "seqlens": [int(x) for x in p.seqlens_q]}
        del t
    # dense causal latency case (launch-latency bound): wall and device time
    p = fi.config1()
    t = dev_tensors(p, dev)
    call, _, _, _ = make_call(p, t)
    times = time_calls([call], warmup, steps, lambda: None)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for _ in range(200):
        call()
    torch.cuda.synchronize()
    wall_us = (time.perf_counter() - w0) / 200 * 1e6
    # device time per launch: events around 200 back-to-back launches
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record()
    for _ in range(200):
        call()
    e_ev.record()
    e_ev.synchronize()
    dev_us = s_ev.elapsed_time(e_ev) / 200 * 1e3
    res["dense_causal_b2_h4_s128_d64"] = {"device_us_per_launch": dev_us, "wall_us_per_call": wall_us,
                                          "single_call_event_us": 1e3 * statistics.median(times),
                                          "tflops": fi.prefill_flops(p) / (dev_us * 1e-6) / 1e12}
    # paged split-KV decode: KV-cache GB/s
    p = fi.config3()
    t = dev_tensors(p, dev)
    call, n, _, _ = make_call(p, t, num_splits=None)
    times = time_calls([call], warmup, steps, flush)
    ms = statistics.mean(times)
    gbs = fi.decode_bytes(p) / (ms * 1e-3) / 1e9
    res["paged_decode_64seq_hq32_hkv8_p16"] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / pk["hbm"],
                                               "num_splits": fa.default_splits(p.num_seqs, 1, p.max_seqlen_k, 32, 8, 16, p.total_k),
                                               "bytes": fi.decode_bytes(p)}
    # the same decode with a soft-cap of 50 (Gemma-style) and with ALiBi
    for run, kw in (("softcap50", dict(mod="softcap", softcap=50.0)), ("alibi", dict(mod="alibi"))):
        pm = fi.make_problem([1] * 64, [int(x) for x in p.seqlens_k], hq=32, hkv=8, dk=128, seed=1, page_size=16,
                             spare_pages=64, max_pages=512, name="paged_decode_" + run, **kw)
        t = dev_tensors(pm, dev)
        call, n, _, _ = make_call(pm, t, num_splits=None)
        ms = statistics.mean(time_calls([call], warmup, steps, flush))
        gbs = fi.decode_bytes(pm) / (ms * 1e-3) / 1e9
        res[f"paged_decode_64seq_hq32_hkv8_p16_{run}"] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / pk["hbm"],
                                                          "bytes": fi.decode_bytes(pm)}
        del t, pm
    # the same decode one key per page (rows gathered by cp.async)
    p1 = fi.make_problem([1] * 64, [int(x) for x in p.seqlens_k], hq=32, hkv=8, dk=128, seed=1, page_size=1,
                         spare_pages=64, max_pages=8192, name="paged_decode_p1")
    t = dev_tensors(p1, dev)
    call, n, _, _ = make_call(p1, t, num_splits=None)
    ms = statistics.mean(time_calls([call], warmup, steps, flush))
    gbs = fi.decode_bytes(p1) / (ms * 1e-3) / 1e9
    res["paged_decode_64seq_hq32_hkv8_p1"] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / pk["hbm"],
                                              "bytes": fi.decode_bytes(p1)}
    del t, p1
    # the same decode geometry on byte caches (e4m3, int8; per-token scales)
    for kvd in ("e4m3", "int8"):
        rng = np.random.default_rng(0)
        lens_k = [int(x) for x in rng.integers(512, 8193, size=64)]
        p = fi.make_problem([1] * 64, lens_k, hq=32, hkv=8, dk=128, seed=1, page_size=16, spare_pages=64,
                            max_pages=512, kv_dtype=kvd, name=f"paged_decode_{kvd}")
        t = dev_tensors(p, dev)
        call, n, _, _ = make_call(p, t, num_splits=None)
        ms = statistics.mean(time_calls([call], warmup, steps, flush))
        gbs = fi.decode_bytes(p) / (ms * 1e-3) / 1e9
        res[f"paged_decode_{kvd}_64seq_hq32_hkv8_p16"] = {
            "ms": ms, "GB/s": gbs, "frac_hbm": gbs / pk["hbm"], "bytes": fi.decode_bytes(p),
            "num_splits": fa.default_splits(p.num_seqs, 1, p.max_seqlen_k, 32, 8, 16, p.total_k)}
        # the same cache in the vectorized 5-D pages
        k5, v5 = fi.vectorize_pages(p.k.view(np.uint8), p.v.view(np.uint8))
        kvt = torch.int8 if kvd == "int8" else torch.float8_e4m3fn
        t["k"] = torch.from_numpy(k5).view(kvt).to(dev)
        t["v"] = torch.from_numpy(v5).view(kvt).to(dev)
        call, n, _, _ = make_call(p, t, num_splits=None)
        ms = statistics.mean(time_calls([call], warmup, steps, flush))
        gbs = fi.decode_bytes(p) / (ms * 1e-3) / 1e9
        res[f"paged_decode_{kvd}_64seq_hq32_hkv8_p16_vec5"] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / pk["hbm"],
                                                               "bytes": fi.decode_bytes(p)}
        del t
    # paged e4m3 KV, Q/K 192, V/O 128, page 64, 16 seqs U{1..4096}, causal
    p = fi.config4()
    t = dev_tensors(p, dev)
    call, _, _, _ = make_call(p, t, num_splits=0)
    times = time_calls([call], warmup, steps, flush)
    ms = statistics.mean(times)
    fl = fi.prefill_flops(p)
    res["paged_fp8_d192_v128_16seq_h16_p64_causal"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                                        "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
                                                        "gflop": fl / 1e9}
    del t
    # the same tokens in the vectorized 5-D pages (K [N_pg, Hkv, Dk/16, P_s,
    # 16], V [N_pg, Hkv, P_s/16, Dv, 16]; bit-identical results)
    k5, v5 = fi.vectorize_pages(p.k.view(np.uint8), p.v.view(np.uint8))
    t5 = dev_tensors(p, dev)
    t5["k"] = torch.from_numpy(k5).view(torch.float8_e4m3fn).to(dev)
    t5["v"] = torch.from_numpy(v5).view(torch.float8_e4m3fn).to(dev)
    call, _, _, _ = make_call(p, t5, num_splits=0)
    ms = statistics.mean(time_calls([call], warmup, steps, flush))
    res["paged_fp8_d192_v128_16seq_h16_p64_causal_vec5"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                                            "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
                                                            "gflop": fl / 1e9}
    del t5
    # the same tokens one key per page (rows gathered by cp.async, no TMA boxes)
    lens4 = [int(x) for x in np.diff(p.cu_seqlens_q)]
    p1 = fi.make_problem(lens4, hq=16, hkv=16, dk=192, dv=128, seed=1, page_size=1, spare_pages=16,
                         kv_dtype="e4m3", causal=True, name="config4_page1")
    t = dev_tensors(p1, dev)
    call, _, _, _ = make_call(p1, t, num_splits=0)
    ms = statistics.mean(time_calls([call], warmup, steps, flush))
    res["paged_fp8_d192_v128_16seq_h16_p1_causal"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                                       "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
                                                       "gflop": fl / 1e9}
    del t, p1
    # the same geometry with an int8 cache (per-token scales)
    p = fi.make_problem([int(x) for x in np.diff(p.cu_seqlens_q)], hq=16, hkv=16, dk=192, dv=128, seed=1,
                        page_size=64, kv_dtype="int8", causal=True, name="config4_int8")
    t = dev_tensors(p, dev)
    call, _, _, _ = make_call(p, t, num_splits=0)
    ms = statistics.mean(time_calls([call], warmup, steps, flush))
    fl = fi.prefill_flops(p)
    res["paged_int8_d192_v128_16seq_h16_p64_causal"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                                        "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
                                                        "gflop": fl / 1e9}
    del t
    # config 4 with e4m3 Q (QK on the e4m3 bytes by kind::f8f6f4, PV kind::f16):
    # besides the bf16 peak, the fraction of the peak of the mix the kernel
    # runs -- QK's 2 Dk flops per pair at the e4m3 rate, PV's 2 Dv at the
    # 16-bit rate
    fp8_peak = measure_fp8_peak(dev)
    lens4 = [int(x) for x in np.diff(fi.config4().cu_seqlens_q)]
    p = fi.make_problem(lens4, hq=16, hkv=16, dk=192, dv=128, seed=1, page_size=64, kv_dtype="e4m3",
                        q_dtype="e4m3", spare_pages=16, causal=True, name="config4_e4m3q")
    t = dev_tensors(p, dev)
    call, _, _, _ = make_call(p, t, num_splits=0)
    ms = statistics.mean(time_calls([call], warmup, steps, flush))
    fl = fi.prefill_flops(p)
    pairs = fl / (2 * p.dk + 2 * p.dv)
    t_peak = pairs * 2 * p.dk / (fp8_peak * 1e12) + pairs * 2 * p.dv / (pk["bf16"] * 1e12)
    res["paged_fp8kv_qe4m3_d192_v128_16seq_h16_p64_causal"] = {
        "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
        "frac_of_mixed_peak": t_peak / (ms * 1e-3), "fp8_peak_tflops": fp8_peak, "gflop": fl / 1e9}
    # the same with the opt-in e4m3 P * V (both contractions kind::f8f6f4):
    # against the measured e4m3 peak
    call, _, _, _ = make_call(p, t, num_splits=0, pv_e4m3=True)
    ms = statistics.mean(time_calls([call], warmup, steps, flush))
    res["paged_fp8kv_qe4m3_pv8_d192_v128_16seq_h16_p64_causal"] = {
        "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_fp8": fl / (ms * 1e-3) / 1e12 / fp8_peak,
        "fp8_peak_tflops": fp8_peak, "gflop": fl / 1e9, "mode": "FA_FLAG_PV_E4M3 (opt-in precision)"}
    del t
    # the same lengths at Dk = Dv = 128 with e4m3 K/V: bf16 Q (f16 QK) and
    # e4m3 Q (QK on the e4m3 bytes)
    for qd in ("bf16", "e4m3"):
        p = fi.make_problem([int(x) for x in np.diff(p.cu_seqlens_q)], hq=16, hkv=16, dk=128, dv=128, seed=1,
                            page_size=64, kv_dtype="e4m3", q_dtype=qd, causal=True, name="config4_d128_" + qd)
        t = dev_tensors(p, dev)
        call, _, _, _ = make_call(p, t, num_splits=0)
        ms = statistics.mean(time_calls([call], warmup, steps, flush))
        fl = fi.prefill_flops(p)
        res[f"paged_fp8kv_q{qd}_d128_16seq_h16_p64_causal"] = {
            "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
            "gflop": fl / 1e9}
        del t
    # backward (fa_bwd_varlen: Delta, dK/dV, dQ kernels): config-2 lengths and
    # 4 x 4096; algorithmic flops = 2.5 x the forward's (S, dP, dV, dK, dQ)
    for name, p in (("bwd_varlen_8seq_h16_d128_causal", fi.config2(causal=True)),
                    ("bwd_varlen_8seq_h16_d128_noncausal", fi.config2(causal=False)),
                    ("bwd_4x4096_h16_d128_causal", fi.make_problem([4096] * 4, hq=16, dk=128, seed=3, causal=True)),
                    ("bwd_4x4096_h16_d128_noncausal", fi.make_problem([4096] * 4, hq=16, dk=128, seed=3)),
                    ("bwd_4x4096_h16_d128_blocksparse50", fi.make_problem([4096] * 4, hq=16, dk=128, seed=3,
                                                                           block_mask_density=0.5))):
        t = dev_tensors(p, dev)
        call = make_bwd_call(p, t)
        ms = statistics.mean(time_calls([call], warmup, steps, flush))
        fl = 2.5 * fi.prefill_flops(p)
        res[name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_bf16": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
                     "gflop": fl / 1e9}
        del t
    return res


def profile_only(name, warmup, steps):
    """Launch one workload warmup + steps times, nothing else (for ncu)."""
    import flashattention_forward_gb300 as fa
    from flashattention_forward_gb300 import build as fa_build
    fa_build.build()
    dev = torch.device("cuda", 0)
    if name == "varlen_causal":
        p, splits = fi.config2(causal=True), 0
    elif name == "varlen_noncausal":
        p, splits = fi.config2(causal=False), 0
    elif name == "decode":
        p, splits = fi.config3(), None
    elif name == "dense":
        p, splits = fi.config1(), 0
    elif name == "long_noncausal":
        p, splits = fi.make_problem([8192] * 4, hq=16, dk=128, name="long_noncausal"), 0
    elif name == "fp8":
        p, splits = fi.config4(), 0
    elif name in ("e4m3q_d192", "e4m3q_pv8_d192"):
        lens = [int(x) for x in np.diff(fi.config4().cu_seqlens_q)]
        p = fi.make_problem(lens, hq=16, hkv=16, dk=192, dv=128, seed=1, page_size=64, kv_dtype="e4m3",
                            q_dtype="e4m3", spare_pages=16, causal=True, name=name)
        splits = 0
    elif name in ("fp8kv_d128", "e4m3q_d128"):
        lens = [int(x) for x in np.diff(fi.config4().cu_seqlens_q)]
        p = fi.make_problem(lens, hq=16, hkv=16, dk=128, dv=128, seed=1, page_size=64, kv_dtype="e4m3",
                            q_dtype="e4m3" if name == "e4m3q_d128" else "bf16", causal=True, name=name)
        splits = 0
    elif name == "long_e4m3q":
        p, splits = fi.make_problem([4096] * 4, hq=16, dk=128, dv=128, kv_dtype="e4m3", q_dtype="e4m3",
                                    name="long_e4m3q"), 0
    elif name.startswith("flex_"):
        p, splits = fi.config5(name[5:]), 0
    elif name in ("decode_e4m3", "decode_int8"):
        rng = np.random.default_rng(0)
        lens_k = [int(x) for x in rng.integers(512, 8193, size=64)]
        p = fi.make_problem([1] * 64, lens_k, hq=32, hkv=8, dk=128, seed=1, page_size=16, spare_pages=64,
                            max_pages=512, kv_dtype=name[7:], name=name)
        splits = None
    elif name == "decode_p1":
        rng = np.random.default_rng(0)
        lens_k = [int(x) for x in rng.integers(512, 8193, size=64)]
        p = fi.make_problem([1] * 64, lens_k, hq=32, hkv=8, dk=128, seed=1, page_size=1, spare_pages=64,
                            max_pages=8192, name=name)
        splits = None
    elif name == "prefill_p1":
        p, splits = fi.make_problem([4096] * 4, hq=16, dk=128, seed=3, page_size=1, causal=True, name=name), 0
    elif name in ("bwd_varlen_noncausal", "bwd_long_causal", "bwd_mid_noncausal"):
        p = {"bwd_varlen_noncausal": lambda: fi.config2(causal=False),
             "bwd_long_causal": lambda: fi.make_problem([4096] * 4, hq=16, dk=128, seed=3, causal=True),
             "bwd_mid_noncausal": lambda: fi.make_problem([2048] * 4, hq=16, dk=128, seed=3)}[name]()
        splits = "bwd"
    else:
        raise SystemExit(f"unknown workload {name}")
    t = dev_tensors(p, dev)
    if splits == "bwd":
        call = make_bwd_call(p, t)
    else:
        call, _, _, _ = make_call(p, t, num_splits=splits, pv_e4m3=(name == "e4m3q_pv8_d192"))
    for _ in range(warmup + steps):
        call()
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    print(f"profile workload {name}: {warmup + steps} calls done")


if __name__ == "__main__":
    main()

"""Benchmark of the score -> select -> compact path (plus decode attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline (one JSON line on rank 0): KV tokens/s scored + selected + compacted
for one Llama-3-8B-shaped layer cache (U=1, 32 q / 8 kv heads, d=128,
T=32768, bf16, observation window 64, global top-k across heads at keep
ratio 0.10, 4 sinks + 64 recent always kept).  A step is one pass of
kvc_score_attn -> kvc_select_compact (the selection and the compaction in
one call, outputs identical to kvc_select -> kvc_compact, which is timed
too: step_three_calls_us) over that cache; inputs are resident in HBM; L2
is flushed between steps, outside the step's CUDA events (a 256 MiB
read + write, then a 256 MiB read that writes the flush's own dirty lines
back before the step).
The same JSON line also reports:

* roofline: the dominant kernel (tensor-core scoring) against the measured
  HBM copy bandwidth, and its tensor-pipe rate;
* decode: split-K varlen decode attention with append on the batch-64
  compressed-cache workload (per-head lengths ~ U[0.1,0.3]*32768), HBM GB/s;
* fidelity: rel-L2 output error and KL of one decode step over the
  compressed cache against the full cache;
* e2e: the same metric through the C ABI with the step's inputs copied from
  pinned host memory and the compacted cache copied back, every step;
* cpu_baseline: the CPU oracle on a bounded token-prefix sample.

Multi-GPU (torchrun): every rank runs its own copy of the workload (units
are independent: no data-path collective), value = all ranks' tokens / the
slowest rank's time ("scaling": "weak").

--impl reference times the CPU oracle (the only reference implementation
of this path) on the host cores, on a token-prefix sample of the same
workload, and prints the same metric with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_compression_attention_b300 import inputs  # noqa: E402

METRIC = "KV tokens/s scored+selected+compacted"
WORKLOAD = "c2_llama32k"
DECODE_WORKLOAD = "c5_decode"
# passes of the window-against-keys contraction the attention-mass scorer issues
SCORE_PASSES = 2


def profiled_traffic(kernel_src, summary):
    """DRAM bytes per launch of a kernel from a committed ncu summary, or
    None when the kernel's source changed since the counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", summary)) as f:
            rec = json.load(f)
        with open(os.path.join(ROOT, "kv_cache_compression_attention_b300", "csrc", kernel_src),
                  "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") != digest:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        self.first = ""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        # nvidia-smi takes a moment to start: the timed work begins only once
        # its first sample is in (waiting 10 s at most)
        import select
        ready, _, _ = select.select([self.proc.stdout], [], [], 10.0)
        if ready:
            self.first = self.proc.stdout.readline()
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                rest, _ = self.proc.communicate(timeout=5)
                self.out = self.first + (rest or "")
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        mhz, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": mx or None, "samples": len(mhz), "reasons": sorted(reasons)}


# ------------------------------------------------------------- workloads
class LayerWorkload:
    """Device buffers of one score -> select -> compact pass (two calls, or one for
    the selection and the compaction together)."""

    def __init__(self, B, w, device):
        self.B, self.w = B, w
        self.q = inputs.window_queries(w, device)
        self.k, self.v = inputs.keys_values(w, self.q, device)
        n = w.U * w.Hkv
        self.n = n
        self.scores = torch.empty((w.U, w.Hkv, w.T), device=device)
        self.score_ws = torch.empty(B.lib().kvc_score_attn_workspace(
            w.U, w.Hq, w.Hkv, w.T, w.W, w.d, B.KVC_BF16 if w.dtype == "bf16" else B.KVC_F32),
            dtype=torch.uint8, device=device)
        self.sc_ws = torch.empty(B.lib().kvc_select_compact_workspace(w.U, w.Hkv, w.T,
                                                                      B.MODES["global"]),
                                 dtype=torch.uint8, device=device)
        self.kept = torch.empty((n, w.T), dtype=torch.int32, device=device)
        self.counts = torch.empty(n, dtype=torch.int32, device=device)
        self.offs = torch.empty(n + 1, dtype=torch.int64, device=device)
        cap = math.floor(w.keep_ratio * w.Hkv * w.T) * w.U + n * w.slack + n * (w.n_sink + w.n_recent)
        self.kc = torch.empty((cap, w.d), dtype=self.k.dtype, device=device)
        self.vc = torch.empty_like(self.kc)
        self.start = torch.empty(n, dtype=torch.int64, device=device)
        self.len = torch.empty(n, dtype=torch.int32, device=device)

    def score(self, aggregation="sum"):
        self.B.kvc_score_attn(self.q, self.k, self.scores, self.w.scale, workspace=self.score_ws,
                              aggregation=aggregation)

    def select(self):
        w = self.w
        self.B.kvc_select(self.scores, "global", self.kept, self.counts, self.offs,
                          keep_ratio=w.keep_ratio, n_sink=w.n_sink, n_recent=w.n_recent)

    def compact(self):
        self.B.kvc_compact(self.k, self.v, self.kept, self.counts, self.offs, self.kc, self.vc,
                           self.start, self.len, slack=self.w.slack)

    def select_compact(self, v=None):
        w = self.w
        self.B.kvc_select_compact(self.scores, "global", self.k, self.v if v is None else v,
                                  self.kept, self.counts,
                                  self.offs, self.kc, self.vc, self.start, self.len,
                                  keep_ratio=w.keep_ratio, n_sink=w.n_sink, n_recent=w.n_recent,
                                  slack=w.slack, workspace=self.sc_ws)


RAMP_STEPS = 200      # untimed steps (~30 ms of GPU time) before a layer bench's warm-up


_CLEAN = {}


def flush_l2(buf):
    """Evict everything from L2 between timed steps.  A 256 MiB read + write
    (larger than the 126 MB L2) leaves L2 full of dirty lines of `buf`; a
    256 MiB read of a second buffer then writes those back here, so that the
    next step's timed region does not pay the flush's write-backs (≈ 126 MB
    of DRAM writes: 5.2 against 5.65 TB/s on the 940 MB linear scorer).
    Either way no input of the step is left in L2.

    Last, the stream is held for 10^6 GPU cycles (≈ 0.5 ms, a bounded spin)
    so that the host has queued the whole step before the GPU reaches it:
    the step's CUDA events then time its kernels, not the Python launch path
    (which, on a busy host, fell behind the five-launch VECTOR step)."""
    buf.add_(1)
    c = _CLEAN.get(buf.device)
    if c is None:
        c = _CLEAN[buf.device] = (torch.zeros_like(buf), torch.empty(1, device=buf.device))
    torch.sum(c[0], dim=0, keepdim=True, out=c[1])
    torch.cuda._sleep(1_000_000)


def bench_layer(B, w, steps, warmup, device):
    """`warmup` untimed steps, then `steps` timed steps: each one score ->
    select + compact (kvc_select_compact, one call) with CUDA events around
    the launches only (the L2 flush before it stays outside).  Nothing is
    recorded between the kernels, so each may start while its predecessor
    drains (programmatic dependent launch).  The same steps with kvc_select
    and kvc_compact as two calls are timed next, then runs with events
    between the calls give the per-stage split (they serialise the stages)."""
    L = LayerWorkload(B, w, device)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=device)
    s = torch.cuda.current_stream()

    def timed(calls):
        for _ in range(warmup):
            flush_l2(flush)
            for f in calls:
                f()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush_l2(flush)
            ev[i][0].record(s)
            for f in calls:
                f()
            ev[i][1].record(s)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in ev]

    def staged(calls):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
              for _ in range(steps)]
        for i in range(steps):
            flush_l2(flush)
            ev[i][0].record(s)
            for x, f in enumerate(calls):
                f()
                ev[i][x + 1].record(s)
        torch.cuda.synchronize()
        return [[e[x].elapsed_time(e[x + 1]) for e in ev] for x in range(len(calls))]

    # clock ramp: the GPU's clocks climb during the first tens of ms of load;
    # untimed steps before the warm-up keep that out of the timed region
    for _ in range(RAMP_STEPS):
        flush_l2(flush)
        L.score(); L.select_compact()
    t_step = timed([L.score, L.select_compact])
    t_step3 = timed([L.score, L.select, L.compact])
    t_score, t_sel, t_comp = staged([L.score, L.select, L.compact])
    _, t_selcomp = staged([L.score, L.select_compact])
    kept_rows = int(L.offs[-1].item())
    return L, dict(score_ms=t_score, select_ms=t_sel, compact_ms=t_comp, step_ms=t_step,
                   step_three_calls_ms=t_step3, select_compact_ms=t_selcomp,
                   kept_rows=kept_rows)


def bench_score_max(L, steps, warmup):
    """The scoring kernel with max aggregation over the window rows (KVzip's
    score) on the same layer: mean CUDA-event time per launch, L2 flushed
    before each."""
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=L.k.device)
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        flush_l2(flush)
        L.score("max")
    ts = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s); L.score("max"); e1.record(s)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ts)


def bench_kvzip_plus(B, L, steps, warmup):
    """The KVzip+ score ([KVzap] §2.1) on the same layer: value norms on warp
    MMAs, then the SIMT column pass; mean CUDA-event time per call, L2 flushed
    before each."""
    w = L.w
    gram, hnorm = inputs.kvzip_plus_weights(w, L.k.device)
    ws = torch.empty(B.lib().kvc_score_kvzip_plus_workspace(w.U, w.Hq, w.Hkv, w.T, w.W),
                     dtype=torch.uint8, device=L.k.device)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=L.k.device)
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        B.kvc_score_kvzip_plus(L.q, L.k, L.v, gram, hnorm, L.scores, w.scale, workspace=ws)
    ts = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        B.kvc_score_kvzip_plus(L.q, L.k, L.v, gram, hnorm, L.scores, w.scale, workspace=ws)
        e1.record(s)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ts)


def bench_e2e(B, L, steps, warmup):
    """Same pass through the C ABI with host buffers: every step copies
    q_win and K from pinned host memory (the scorer reads all of K), runs
    score -> select + compact with V left in pinned host memory (the
    compaction reads only the kept V rows across the bus), and copies the
    compacted cache + offsets back.  Steps alternate between two streams,
    each with its own device buffers, so one step's transfers overlap the
    other's kernels (the bus, not the kernels, sets the pace)."""
    w = L.w
    hq = L.q.cpu().pin_memory()
    hk = L.k.cpu().pin_memory()
    hv = L.v.cpu().pin_memory()
    rows = int(L.offs[-1].item()) + L.n * w.slack
    pipes = []
    for Lp in (L, LayerWorkload(B, w, L.k.device)):
        okc = torch.empty((rows, w.d), dtype=L.k.dtype).pin_memory()
        pipes.append((Lp, torch.cuda.Stream(device=L.k.device), okc,
                      torch.empty_like(okc).pin_memory(),
                      torch.empty(L.n + 1, dtype=torch.int64).pin_memory()))
    s = torch.cuda.current_stream()

    def step(i):
        Lp, st, okc, ovc, oofs = pipes[i % 2]
        with torch.cuda.stream(st):
            Lp.q.copy_(hq, non_blocking=True)
            Lp.k.copy_(hk, non_blocking=True)
            Lp.score(); Lp.select_compact(v=hv)
            oofs.copy_(Lp.offs, non_blocking=True)
            okc.copy_(Lp.kc[:rows], non_blocking=True)
            ovc.copy_(Lp.vc[:rows], non_blocking=True)

    def run(n):
        start = torch.cuda.Event()
        start.record(s)
        for _, st, *_ in pipes:
            st.wait_event(start)
        for i in range(n):
            step(i)
        for _, st, *_ in pipes:
            done = torch.cuda.Event()
            done.record(st)
            s.wait_event(done)

    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    run(steps)
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # bytes across the bus to the device: the copies of q_win and K, and the
    # kept V rows the compaction reads from host memory
    kept_rows = int(L.offs[-1].item())
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk)) + kept_rows * w.d * hv.element_size()
    d2h = sum(t.numel() * t.element_size() for t in pipes[0][2:])
    return ms, h2d, d2h


def build_decode_caches(B, w, device):
    """The batch-64 decode workload's caches: full 32k caches (K, V with the
    sinks and needles of the generator) and the compressed caches cut from
    them by this library's own path -- window scores (W = 64), a per-head
    top-k at budgets floor(U[0.1, 0.3] * T) that keeps 4 sinks and the 64
    most recent tokens, and a compaction with 256 slack rows per head for the
    appends.  Also a second compressed cache at the same budgets whose kept
    tokens are chosen by random scores (random eviction), and the full cache
    laid out as a pool with the same slack (every token kept)."""
    q_win = inputs.window_queries(w, device)
    k, v = inputs.keys_values(w, q_win, device)
    n = w.U * w.Hkv
    budgets = inputs.head_budgets(w, device)
    scores = torch.empty((w.U, w.Hkv, w.T), device=device)
    B.kvc_score_attn(q_win, k, scores, w.scale)
    del q_win
    kept = torch.empty((n, w.T), dtype=torch.int32, device=device)
    counts = torch.empty(n, dtype=torch.int32, device=device)
    offs = torch.empty(n + 1, dtype=torch.int64, device=device)

    def cut(sc):
        B.kvc_select(sc, "per_head", kept, counts, offs, head_budget=budgets, n_sink=w.n_sink,
                     n_recent=w.n_recent)
        rows = int(offs[-1].item()) + n * w.slack
        kc = torch.empty((rows, w.d), dtype=k.dtype, device=device)
        vc = torch.empty_like(kc)
        st = torch.empty(n, dtype=torch.int64, device=device)
        ln = torch.empty(n, dtype=torch.int32, device=device)
        B.kvc_compact(k, v, kept, counts, offs, kc, vc, st, ln, slack=w.slack)
        return kc, vc, st, ln

    comp = cut(scores)
    rand = cut(inputs.random_scores((w.U, w.Hkv, w.T), device, seed=505))
    allk = torch.arange(w.T, dtype=torch.int32, device=device).repeat(n, 1)
    allc = torch.full((n,), w.T, dtype=torch.int32, device=device)
    allo = torch.arange(n + 1, device=device, dtype=torch.int64) * w.T
    kf = torch.empty((n * (w.T + w.slack), w.d), dtype=k.dtype, device=device)
    vf = torch.empty_like(kf)
    sf = torch.empty(n, dtype=torch.int64, device=device)
    lf = torch.empty(n, dtype=torch.int32, device=device)
    B.kvc_compact(k, v, allk, allc, allo, kf, vf, sf, lf, slack=w.slack)
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    del k, v, kept, scores, allk
    torch.cuda.empty_cache()
    return comp, rand, (kf, vf, sf, lf)


def _quantiles(x):
    x = x.flatten().float()
    q = torch.quantile(x, torch.tensor([0.5, 0.99], device=x.device))
    return {"mean": float(x.mean()), "p50": float(q[0]), "p99": float(q[1]),
            "max": float(x.max())}


def bench_decode(B, steps, warmup, device):
    """Decode over the compressed caches of the batch-64 workload: `steps`
    timed steps (256, the workload's count), each appending one token per
    head, then the same steps over the full caches for the fidelity of every
    step (rel-L2 output error and KL against full-cache attention)."""
    w = inputs.WORKLOADS[DECODE_WORKLOAD]
    assert steps <= w.slack, "every step appends one row per head into the slack"
    (kc, vc, start, length), rnd, full = build_decode_caches(B, w, device)
    n = w.U * w.Hkv
    len0 = length.clone()
    lens = len0.cpu()
    # the split-K grid is sized by max_len: the compressed caches' own bound,
    # and the full length for the full caches
    max_len = int(lens.max()) + max(steps, warmup) + 1
    max_len_full = w.T + max(steps, warmup) + 1
    ws = torch.empty(B.kvc_decode_workspace(w.U, w.Hq, w.Hkv, w.d, max_len_full),
                     dtype=torch.uint8, device=device)
    steps_in = [inputs.decode_step_inputs(w, i, device) for i in range(max(steps, warmup))]
    out = torch.empty((w.U, w.Hq, w.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.U, w.Hq), device=device)
    s = torch.cuda.current_stream()
    rows0 = int(lens.sum())

    def run(kc_, vc_, st_, ln_, i, o=out, l=lse, ml=max_len):
        q, kn, vn = steps_in[i]
        B.kvc_decode_attn(q, kc_, vc_, st_, ln_, o, l, k_new=kn, v_new=vn, max_len=ml,
                          scale=w.scale, workspace=ws)

    for i in range(warmup):
        run(kc, vc, start, length, i)
    length.copy_(len0)                      # the timed steps append into the same slack rows
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(steps):
        run(kc, vc, start, length, i)
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # rows attended per step: the cached rows (read from HBM) + the appended one
    mean_rows = rows0 + n * (steps - 1) / 2.0
    row_bytes = w.d * 2
    bytes_step = 2 * mean_rows * row_bytes            # K and V rows streamed once
    out_d = dict(workload=DECODE_WORKLOAD, steps=steps, us_per_step=ms * 1e3,
                 kv_rows_per_step=mean_rows + n, bytes_per_step=bytes_step,
                 kv_tokens_per_s=(mean_rows + n) / (ms * 1e-3),
                 gbs=bytes_step / (ms * 1e-3) / 1e9, launches_per_step=2, rows_at_start=rows0,
                 cache="cut from full 32k caches: window scores, per-head top-k at "
                       "floor(U[0.1,0.3]*T) with 4 sinks + 64 recent kept")
    # fidelity of every step against full-cache attention ([Sculpt] §4: KL);
    # the random-eviction cache at the same budgets is the comparison point
    kf, vf, sf, lf = full
    lf0 = lf.clone()
    rk, rv, rs, rl = rnd
    rl0 = rl.clone()
    of = torch.empty_like(out); lfu = torch.empty_like(lse)
    orr = torch.empty_like(out); lrr = torch.empty_like(lse)
    rel = torch.empty((steps, w.U * w.Hq), device=device); kl = torch.empty_like(rel)
    rrel = torch.empty_like(rel); rkl = torch.empty_like(rel)
    length.copy_(len0); lf.copy_(lf0); rl.copy_(rl0)
    for i in range(steps):
        run(kc, vc, start, length, i)
        run(kf, vf, sf, lf, i, of, lfu, max_len_full)
        run(rk, rv, rs, rl, i, orr, lrr)
        B.kvc_fidelity(out, of, lse, lfu, rel[i], kl[i])
        B.kvc_fidelity(orr, of, lrr, lfu, rrel[i], rkl[i])
    torch.cuda.synchronize()
    assert B.kvc_device_status() == 0
    out_d["fidelity"] = {
        "steps": steps, "pairs_per_step": w.U * w.Hq,
        "rel_err": _quantiles(rel), "kl": _quantiles(kl),
        "random_eviction": {"rel_err": _quantiles(rrel), "kl": _quantiles(rkl)},
        "kl_step0_mean": float(kl[0].mean()), "kl_last_step_mean": float(kl[-1].mean())}
    del kf, vf, rk, rv, full, rnd
    torch.cuda.empty_cache()
    # the same steps over the group-quantised pool ([KVTC] §2B groups of 32 with a
    # scale and an offset): the compressed pool quantised once before timing
    rows_pool = kc.shape[0]
    kq = torch.empty((rows_pool, w.d), dtype=torch.uint8, device=device)
    vq = torch.empty_like(kq)
    kp = torch.empty((rows_pool, w.d // 32, 2), dtype=torch.float16, device=device)
    vp = torch.empty_like(kp)
    B.kvc_quantize_rows(kc, kq, kp)
    B.kvc_quantize_rows(vc, vq, vp)

    def run8(i):
        q, kn, vn = steps_in[i]
        B.kvc_decode_attn_q8(q, kq, kp, vq, vp, start, length, out, lse, k_new=kn, v_new=vn,
                             max_len=max_len, scale=w.scale, workspace=ws)

    length.copy_(len0)
    for i in range(warmup):
        run8(i)
    length.copy_(len0)
    torch.cuda.synchronize()
    e0.record(s)
    for i in range(steps):
        run8(i)
    e1.record(s)
    torch.cuda.synchronize()
    ms8 = e0.elapsed_time(e1) / steps
    bytes8 = 2 * mean_rows * (w.d + (w.d // 32) * 4)  # codes + (scale, offset) pairs
    out_d["q8"] = dict(us_per_step=ms8 * 1e3, bytes_per_step=bytes8,
                       kv_tokens_per_s=(mean_rows + n) / (ms8 * 1e-3),
                       gbs=bytes8 / (ms8 * 1e-3) / 1e9, launches_per_step=2)
    del kq, vq, kp, vp
    # the same steps with decode-time threshold pruning ([KVzap] §2.3): the new
    # token is scored by the linear surrogate, attended and appended, then the
    # token leaving the 128-token window stays iff its score >= tau (the
    # window kept as a ring of row indices: a drop moves one row).  The
    # surrogate's synthetic scores of the cached rows are ~ N(0, 1).
    window, n_sink, tau, Dh = 128, 4, 0.5, 4096
    # pruning moves rows: the warm-up runs on a copy, the timed steps on the
    # pool as compacted (warm-up + timed appends together could exceed the slack)
    kc3, vc3, start3 = kc.clone(), vc.clone(), start
    length3 = len0.clone()
    rscore = inputs.row_scores(kc3.shape[0], device, seed=61)
    weight, bias = inputs.decode_surrogate(w, Dh, device)
    hid = [inputs.decode_hidden(w, Dh, i, device) for i in range(max(steps, warmup))]
    s_new = torch.empty((w.U, w.Hkv, 1), device=device)

    ring = torch.empty((n, window), dtype=torch.int32, device=device)
    B.kvc_prune_ring_init(length3, window, w.T, ring)

    def pruned_step(i):
        q, kn, vn = steps_in[i]
        B.kvc_score_linear(hid[i], weight, bias, s_new)
        B.kvc_decode_attn(q, kc3, vc3, start3, length3, out, lse, k_new=kn, v_new=vn,
                          max_len=max_len, scale=w.scale, workspace=ws)
        B.kvc_decode_prune_ring([kc3, vc3], rscore, start3, length3, ring, w.T + i,
                                s_new.view(-1), tau, window, n_sink)

    for i in range(warmup):
        pruned_step(i)
    # stage times from 4 extra warm-up steps with events between the kernels
    # (serialised), still on the copy
    hid_x = [inputs.decode_hidden(w, Dh, 10000 + i, device) for i in range(4)]
    in_x = [inputs.decode_step_inputs(w, 10000 + i, device) for i in range(4)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(4)]
    assert warmup + 4 <= w.slack
    for i in range(4):
        q, kn, vn = in_x[i]
        ev[i][0].record(s)
        B.kvc_score_linear(hid_x[i], weight, bias, s_new)
        ev[i][1].record(s)
        B.kvc_decode_attn(q, kc3, vc3, start3, length3, out, lse, k_new=kn, v_new=vn,
                          max_len=max_len, scale=w.scale, workspace=ws)
        ev[i][2].record(s)
        B.kvc_decode_prune_ring([kc3, vc3], rscore, start3, length3, ring, w.T + warmup + i,
                                s_new.view(-1), tau, window, n_sink)
        ev[i][3].record(s)
    torch.cuda.synchronize()
    kc3, vc3 = kc, vc
    length3.copy_(len0)
    rscore = inputs.row_scores(kc3.shape[0], device, seed=61)
    B.kvc_prune_ring_init(length3, window, w.T, ring)
    torch.cuda.synchronize()
    rows_p0 = int(length3.sum().item())
    e0.record(s)
    for i in range(steps):
        pruned_step(i)
    e1.record(s)
    torch.cuda.synchronize()
    msp = e0.elapsed_time(e1) / steps
    rows_p1 = int(length3.sum().item())
    t_lin = statistics.mean(e[0].elapsed_time(e[1]) for e in ev[1:]) * 1e3
    t_prune = statistics.mean(e[2].elapsed_time(e[3]) for e in ev[1:]) * 1e3
    mean_rows_p = (rows_p0 + rows_p1) / 2.0
    out_d["pruned"] = dict(us_per_step=msp * 1e3, window=window, n_sink=n_sink, tau=tau,
                           surrogate_hidden=Dh, rows_at_timed_start=rows_p0,
                           rows_at_timed_end=rows_p1,
                           dropped_fraction=1.0 - (rows_p1 - rows_p0) / (n * steps),
                           kv_tokens_per_s=(mean_rows_p + n) / (msp * 1e-3),
                           overhead_us=(msp - ms) * 1e3, launches_per_step=4,
                           window_layout="ring of row indices (one row moved per drop)",
                           stage_linear_us=t_lin, stage_prune_us=t_prune)
    del kc, vc, kc3, vc3, ws
    torch.cuda.empty_cache()
    return out_d


def bench_decode_q8_small(B, units, steps, warmup, device):
    """A cut of the decode workload for profiling: `units` sequences of
    N(0, 1) rows at the workload's per-head lengths, quantised with
    kvc_quantize_rows, then `steps` timed kvc_decode_attn_q8 calls without
    appends (the same cache every call)."""
    import dataclasses
    w = dataclasses.replace(inputs.WORKLOADS[DECODE_WORKLOAD], U=units)
    lens = inputs.head_budgets(w, "cpu")
    kc, vc, start, length = inputs.compressed_pool(w, lens, device)
    kq = torch.empty(kc.shape, dtype=torch.uint8, device=device)
    vq = torch.empty_like(kq)
    kp = torch.empty((kc.shape[0], w.d // 32, 2), dtype=torch.float16, device=device)
    vp = torch.empty_like(kp)
    B.kvc_quantize_rows(kc, kq, kp)
    B.kvc_quantize_rows(vc, vq, vp)
    del kc, vc
    max_len = int(lens.max()) + 8
    ws = torch.empty(B.kvc_decode_workspace(w.U, w.Hq, w.Hkv, w.d, max_len), dtype=torch.uint8,
                     device=device)
    q, _, _ = inputs.decode_step_inputs(w, 0, device)
    out = torch.empty_like(q)
    lse = torch.empty((w.U, w.Hq), device=device)

    def run():
        B.kvc_decode_attn_q8(q, kq, kp, vq, vp, start, length, out, lse, max_len=max_len,
                             scale=w.scale, workspace=ws)

    for _ in range(warmup):
        run()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        run()
    e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / max(steps, 1) * 1e3
    rows = int(lens.sum())
    nbytes = 2 * rows * (w.d + (w.d // 32) * 4)
    return {"workload": f"{w.name} cut to U={units}", "rows": rows, "bytes": nbytes,
            "us_per_step": us, "gbs": nbytes / (us * 1e-6) / 1e9}


def bench_vector(B, w, steps, warmup, device):
    """VECTOR three-way routing on the 32k layer (p_c = 0.9, p_a = 0.05): score ->
    pool select (1 - p_c + p_a, global top-k) -> reconstruction-error keys ->
    select of the 2 p_a lowest-error tokens -> K-for-all / V-for-exact
    compaction, timed as one step (L2 flushed before each) and stage by stage;
    then decode steps over batch-64 VECTOR caches (two thirds of every pool
    approximated) against the plain decode of the same pool lengths."""
    p_c, p_a = 0.9, 0.05
    L = LayerWorkload(B, w, device)
    W = inputs.vector_predictor(w, device)
    v = inputs.vector_values(w, L.k, W, device)
    n = L.n
    nP = w.n_sink + w.n_recent
    ratio = (1.0 - p_c) + p_a
    Bpool = max(math.floor(ratio * w.Hkv * w.T), w.Hkv * nP)
    A = min(math.floor(2.0 * p_a * w.Hkv * w.T), Bpool - w.Hkv * nP)
    key = torch.empty((w.U, w.Hkv, w.T), device=device)
    apos = torch.empty((n, w.T), dtype=torch.int32, device=device)
    acnt = torch.empty(n, dtype=torch.int32, device=device)
    aoff = torch.empty(n + 1, dtype=torch.int64, device=device)
    kc = torch.empty((Bpool * w.U + n * w.slack, w.d), dtype=L.k.dtype, device=device)
    vc = torch.empty(((Bpool - A) * w.U + n * w.slack, w.d), dtype=L.k.dtype, device=device)
    ks = torch.empty(n, dtype=torch.int64, device=device)
    kl = torch.empty(n, dtype=torch.int32, device=device)
    vs = torch.empty(n, dtype=torch.int64, device=device)
    na = torch.empty(n, dtype=torch.int32, device=device)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=device)
    s = torch.cuda.current_stream()

    def stages():
        yield lambda: L.score()
        yield lambda: B.kvc_select(L.scores, "global", L.kept, L.counts, L.offs, keep_ratio=ratio,
                                   n_sink=w.n_sink, n_recent=w.n_recent)
        yield lambda: B.kvc_vector_residual(L.k, v, W, L.kept, L.counts, key, w.n_sink,
                                            w.n_recent)
        yield lambda: B.kvc_vector_select(key, L.counts, A, apos, acnt, aoff)
        yield lambda: B.kvc_vector_compact(L.k, v, L.kept, L.counts, L.offs, apos, acnt, aoff,
                                           kc, vc, ks, kl, vs, na, slack=w.slack)

    for _ in range(warmup):
        flush_l2(flush)
        for f in stages():
            f()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush)
        ev[i][0].record(s)
        for f in stages():
            f()
        ev[i][1].record(s)
    torch.cuda.synchronize()
    t_step = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush)
        evs[i][0].record(s)
        for x, f in enumerate(stages()):
            f()
            evs[i][x + 1].record(s)
    torch.cuda.synchronize()
    st = [statistics.mean(e[x].elapsed_time(e[x + 1]) for e in evs) * 1e3 for x in range(5)]
    pool_rows = int(L.offs[-1].item())
    eligible = pool_rows - n * nP
    res_bytes = eligible * 2 * w.d * 2 + n * w.T * 4            # K and V rows read, keys written
    res_flops = eligible * 2.0 * w.d * w.d
    comp_bytes = pool_rows * (2 * w.d * 2 + 4) + (pool_rows - w.U * A) * 2 * w.d * 2
    out = dict(workload=w.name, p_c=p_c, p_a=p_a, pool_rows=pool_rows, approximated=w.U * A,
               step_us=t_step, kv_tokens_per_s=w.U * w.T / (t_step * 1e-6),
               stages_us=dict(score=st[0], select_pool=st[1], residual=st[2],
                              select_approx=st[3], compact=st[4]),
               residual_gbs=res_bytes / (st[2] * 1e-6) / 1e9,
               residual_tflops=res_flops / (st[2] * 1e-6) / 1e12,
               compact_gbs=comp_bytes / (st[4] * 1e-6) / 1e9,
               cache_rows_k=int(kl.sum()), cache_rows_v=int((kl - na).sum()))
    del L, v, kc, vc
    torch.cuda.empty_cache()
    # decode over batch-64 VECTOR caches
    wd = inputs.WORKLOADS[DECODE_WORKLOAD]
    lens = inputs.head_budgets(wd, "cpu")
    nap = (lens.to(torch.int64) * 2 // 3).to(torch.int32)
    dkc, dvc, dks, dkl, dvs, dna = inputs.vector_pool(wd, lens, nap, device)
    Wd = inputs.vector_predictor(wd, device)
    dsteps = max(16, steps)
    max_len = int(lens.max()) + dsteps + warmup + 1
    ws = torch.empty(B.kvc_decode_vector_workspace(wd.U, wd.Hq, wd.Hkv, wd.d, max_len),
                     dtype=torch.uint8, device=device)
    steps_in = [inputs.decode_step_inputs(wd, i, device) for i in range(dsteps + warmup)]
    o = torch.empty((wd.U, wd.Hq, wd.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((wd.U, wd.Hq), device=device)
    for i in range(warmup):
        q, kn, vn = steps_in[i]
        B.kvc_decode_attn_vector(q, dkc, dvc, dks, dkl, dvs, dna, Wd, o, lse, k_new=kn,
                                 v_new=vn, max_len=max_len, scale=wd.scale, workspace=ws)
    torch.cuda.synchronize()
    rows_k0 = int(dkl.sum())
    rows_a = int(dna.sum())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(warmup, warmup + dsteps):
        q, kn, vn = steps_in[i]
        B.kvc_decode_attn_vector(q, dkc, dvc, dks, dkl, dvs, dna, Wd, o, lse, k_new=kn,
                                 v_new=vn, max_len=max_len, scale=wd.scale, workspace=ws)
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / dsteps
    nh = wd.U * wd.Hkv
    mean_k = rows_k0 + nh * (dsteps - 1) / 2.0
    bytes_step = (mean_k + (mean_k - rows_a)) * wd.d * 2          # K rows + exact V rows
    out["decode"] = dict(workload=DECODE_WORKLOAD, approximated_fraction=rows_a / rows_k0,
                         us_per_step=ms * 1e3, bytes_per_step=bytes_step,
                         kv_tokens_per_s=(mean_k + nh) / (ms * 1e-3),
                         gbs=bytes_step / (ms * 1e-3) / 1e9, launches_per_step=2)
    return out


def compact_bytes(rows, d, elt):
    """Algorithmic bytes of one compaction: every kept K and V row read once
    and written once, plus its int32 source index."""
    return rows * (2 * 2 * d * elt + 4)


def bench_c4(B, steps, warmup, device):
    """Threshold pruning with the linear surrogate scorer on the 128k-token
    Qwen-shaped layer (28 q / 4 kv heads, hidden 3584): kvc_score_linear ->
    kvc_select (tau = 0.5, 4 sinks + 128 recent) -> kvc_compact, each stage
    timed with CUDA events; the 940 MB hidden-state read flushes L2 itself."""
    w = inputs.WORKLOADS["c4_qwen128k"]
    hidden, weight, bias = inputs.linear_scorer(w, device)
    k, v = inputs.keys_values(w, None, device)
    n = w.U * w.Hkv
    scores = torch.empty((w.U, w.Hkv, w.T), device=device)
    kept = torch.empty((n, w.T), dtype=torch.int32, device=device)
    counts = torch.empty(n, dtype=torch.int32, device=device)
    offs = torch.empty(n + 1, dtype=torch.int64, device=device)
    kc = torch.empty((n * w.T, w.d), dtype=k.dtype, device=device)
    vc = torch.empty_like(kc)
    start = torch.empty(n, dtype=torch.int64, device=device)
    length = torch.empty(n, dtype=torch.int32, device=device)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=device)
    s = torch.cuda.current_stream()

    def step(ev=None):
        flush_l2(flush)
        if ev: ev[0].record(s)
        B.kvc_score_linear(hidden, weight, bias, scores)
        if ev: ev[1].record(s)
        B.kvc_select(scores, "threshold", kept, counts, offs, tau=w.tau, n_sink=w.n_sink,
                     n_recent=w.n_recent)
        if ev: ev[2].record(s)
        B.kvc_compact(k, v, kept, counts, offs, kc, vc, start, length)
        if ev: ev[3].record(s)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize()
    t_score = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
    t_sel = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) * 1e3
    t_comp = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) * 1e3
    rows = int(offs[-1].item())
    score_bytes = hidden.numel() * 2 + weight.numel() * 2 + scores.numel() * 4
    comp_bytes = compact_bytes(rows, w.d, 2)
    out = dict(workload="c4_qwen128k", score_us=t_score, select_us=t_sel, compact_us=t_comp,
               kept_rows=rows, keep_fraction=rows / (n * w.T),
               score_linear_gbs=score_bytes / (t_score * 1e-6) / 1e9,
               score_linear_bytes=score_bytes,
               compact_gbs=comp_bytes / (t_comp * 1e-6) / 1e9, compact_bytes=comp_bytes,
               tokens_per_s=w.U * w.T / ((t_score + t_sel + t_comp) * 1e-6))
    # the two-layer surrogate ([KVzap] §2.2, width Dh / 8) on the same hidden states
    w1, b1, w2, b2 = inputs.mlp_scorer(w, device)
    mws = torch.empty(B.lib().kvc_score_mlp_workspace(w.Dh, w1.shape[1]), dtype=torch.uint8,
                      device=device)
    for _ in range(2):
        B.kvc_score_mlp(hidden, w1, b1, w2, b2, scores, workspace=mws)
    torch.cuda.synchronize()
    mev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in mev:
        flush_l2(flush)
        e[0].record(s)
        B.kvc_score_mlp(hidden, w1, b1, w2, b2, scores, workspace=mws)
        e[1].record(s)
    torch.cuda.synchronize()
    t_mlp = statistics.mean(e[0].elapsed_time(e[1]) for e in mev) * 1e3
    mlp_flops = 2.0 * w.U * w.T * w.Dh * w1.shape[1] + 2.0 * w.U * w.T * w1.shape[1] * w.Hkv
    out.update(score_mlp_us=t_mlp, score_mlp_tflops=mlp_flops / (t_mlp * 1e-6) / 1e12,
               score_mlp_width=int(w1.shape[1]))
    del hidden, k, v, kc, vc, kept, flush, mws
    torch.cuda.empty_cache()
    return out


def bench_c3(B, steps, warmup, device):
    """The 32-layer x batch-4 cache (U = 128 units, 8 kv heads, T = 16384):
    score (per-(layer, kv head) temperature) -> global top-k per unit at keep
    0.20 -> compact, each stage timed; 4.3 GB of K, so L2 holds none of it."""
    w = inputs.WORKLOADS["c3_32layer"]
    q = inputs.window_queries(w, device)
    k, v = inputs.keys_values(w, q, device)
    hs = inputs.head_scale(w, device)
    n = w.U * w.Hkv
    scores = torch.empty((w.U, w.Hkv, w.T), device=device)
    ws = torch.empty(B.lib().kvc_score_attn_workspace(w.U, w.Hq, w.Hkv, w.T, w.W, w.d, B.KVC_BF16),
                     dtype=torch.uint8, device=device)
    kept = torch.empty((n, w.T), dtype=torch.int32, device=device)
    counts = torch.empty(n, dtype=torch.int32, device=device)
    offs = torch.empty(n + 1, dtype=torch.int64, device=device)
    cap = w.U * math.floor(w.keep_ratio * w.Hkv * w.T) + n * (w.n_sink + w.n_recent)
    kc = torch.empty((cap, w.d), dtype=k.dtype, device=device)
    vc = torch.empty_like(kc)
    start = torch.empty(n, dtype=torch.int64, device=device)
    length = torch.empty(n, dtype=torch.int32, device=device)
    s = torch.cuda.current_stream()

    def step(ev=None):
        if ev: ev[0].record(s)
        B.kvc_score_attn(q, k, scores, w.scale, head_scale=hs, workspace=ws)
        if ev: ev[1].record(s)
        B.kvc_select(scores, "global", kept, counts, offs, keep_ratio=w.keep_ratio,
                     n_sink=w.n_sink, n_recent=w.n_recent)
        if ev: ev[2].record(s)
        B.kvc_compact(k, v, kept, counts, offs, kc, vc, start, length)
        if ev: ev[3].record(s)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize()
    t_score = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
    t_sel = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) * 1e3
    t_comp = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) * 1e3
    rows = int(offs[-1].item())
    per_head = counts.view(w.U, w.Hkv).float()
    score_bytes = k.numel() * 2 + q.numel() * 2 + scores.numel() * 4
    comp_bytes = compact_bytes(rows, w.d, 2)
    # one budget over every layer and kv head of a sequence (units are
    # batch-major, u = b * layers + layer, so the scores of a sequence are
    # one contiguous [layers * Hkv, T] pool): the streaming select
    nb = w.U // w.layers
    pooled = scores.view(nb, w.layers * w.Hkv, w.T)

    def cross():
        B.kvc_select(pooled, "global", kept, counts, offs, keep_ratio=w.keep_ratio,
                     n_sink=w.n_sink, n_recent=w.n_recent)
    for _ in range(warmup):
        cross()
    torch.cuda.synchronize()
    xe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in xe:
        e0.record(s); cross(); e1.record(s)
    torch.cuda.synchronize()
    t_cross = statistics.mean(e0.elapsed_time(e1) for e0, e1 in xe) * 1e3
    per_layer = counts.view(nb, w.layers, w.Hkv).sum(-1).float()
    out = dict(workload="c3_32layer", score_us=t_score, select_us=t_sel, compact_us=t_comp,
               kept_rows=rows,
               per_head_count_min=int(per_head.min()), per_head_count_max=int(per_head.max()),
               score_gbs=score_bytes / (t_score * 1e-6) / 1e9, score_bytes=score_bytes,
               compact_gbs=comp_bytes / (t_comp * 1e-6) / 1e9, compact_bytes=comp_bytes,
               tokens_per_s=w.U * w.T / ((t_score + t_sel + t_comp) * 1e-6),
               cross_layer_select_us=t_cross,
               cross_layer_keys_per_pool=w.layers * w.Hkv * w.T,
               cross_layer_per_layer_kept_min=int(per_layer.min()),
               cross_layer_per_layer_kept_max=int(per_layer.max()))
    del q, k, v, kc, vc, kept, scores, ws
    torch.cuda.empty_cache()
    return out


def fidelity_probe(B, L):
    """One decode step over the compacted cache and over the full cache, and
    the same step over a cache of the same size whose kept tokens are chosen
    by random scores (random eviction at the same keep ratio, the comparison
    point: a score that finds the attended tokens retains more of the probe's
    attention mass, i.e. a lower KL)."""
    w = L.w
    n = L.n
    dev = L.k.device
    g = torch.Generator(device=dev).manual_seed(2026)
    # the probe query is the last observation-window query of every q head
    q = L.q[:, :, -1, :].contiguous()
    kn = torch.randn((w.U, w.Hkv, w.d), generator=g, device=dev).to(L.k.dtype)
    vn = torch.randn((w.U, w.Hkv, w.d), generator=g, device=dev).to(L.k.dtype)
    allk = torch.arange(w.T, dtype=torch.int32, device=dev).repeat(n, 1).contiguous()
    allc = torch.full((n,), w.T, dtype=torch.int32, device=dev)
    allo = (torch.arange(n + 1, device=dev) * w.T).to(torch.int64)
    kf = torch.empty((n * (w.T + w.slack + 1), w.d), dtype=L.k.dtype, device=dev)
    vf = torch.empty_like(kf)
    sf = torch.empty(n, dtype=torch.int64, device=dev)
    lf = torch.empty(n, dtype=torch.int32, device=dev)
    B.kvc_compact(L.k, L.v, allk, allc, allo, kf, vf, sf, lf, slack=w.slack + 1)
    of = torch.empty_like(q)
    lfu = torch.empty((w.U, w.Hq), device=dev)
    B.kvc_decode_attn(q, kf, vf, sf, lf, of, lfu, k_new=kn, v_new=vn, max_len=w.T + 1,
                      scale=w.scale)
    res = {"workload": WORKLOAD, "keep_ratio": w.keep_ratio}
    for name, scores in (("score", None),
                         ("random_eviction", inputs.random_scores((w.U, w.Hkv, w.T), dev,
                                                                  seed=404))):
        if scores is None:
            L.score()
        else:
            L.scores.copy_(scores)
        L.select()
        # one slack row per head for the probe's appended token
        B.kvc_compact(L.k, L.v, L.kept, L.counts, L.offs, L.kc, L.vc, L.start, L.len, slack=1)
        oc = torch.empty_like(q)
        lc = torch.empty((w.U, w.Hq), device=dev)
        B.kvc_decode_attn(q, L.kc, L.vc, L.start, L.len, oc, lc, k_new=kn, v_new=vn,
                          max_len=w.T + 1, scale=w.scale)
        rel = torch.empty(w.U * w.Hq, device=dev); kl = torch.empty_like(rel)
        B.kvc_fidelity(oc, of, lc, lfu, rel, kl)
        torch.cuda.synchronize()
        d = {"rel_err_mean": float(rel.mean()), "rel_err_max": float(rel.max()),
             "kl_mean": float(kl.mean()), "kl_max": float(kl.max()),
             "retained_mass_mean": float(torch.exp(-kl).mean())}
        if scores is None:
            res.update(d)
        else:
            res[name] = d
    assert B.kvc_device_status() == 0
    del kf, vf
    return res


# ----------------------------------------------------------- CPU oracle
def oracle_sample_tokens(budget_s: float, steps: int):
    """Token-prefix length of the workload such that `steps` oracle passes
    take about budget_s seconds (cost is linear in T)."""
    from oracle import kvc_oracle as O
    w = inputs.WORKLOADS[WORKLOAD].with_(T=2048)
    t = time.perf_counter()
    _oracle_pass(O, w, *_oracle_inputs(w))
    per_token = (time.perf_counter() - t) / w.T
    T = int(budget_s / max(steps, 1) / per_token)
    return max(1024, min(32768, (T // 1024) * 1024))


def _oracle_inputs(w):
    q = inputs.window_queries(w, "cpu")
    k, v = inputs.keys_values(w, q, "cpu")
    return (q.to(torch.float64).numpy(), k.to(torch.float64).numpy(),
            k.view(torch.int16).numpy(), v.view(torch.int16).numpy())


def _oracle_pass(O, w, q, k64, kb, vb):
    s = O.score_attn(q, k64, w.scale).astype(np.float32)
    kept, counts, offs = O.select(s, "global", keep_ratio=w.keep_ratio, n_sink=w.n_sink,
                                  n_recent=w.n_recent)
    O.compact(kb, vb, kept, counts, offs, w.slack)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 1) for p in threadpool_info() if p.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(steps=1, budget_s=20.0):
    from oracle import kvc_oracle as O
    T = oracle_sample_tokens(budget_s, steps)
    w = inputs.WORKLOADS[WORKLOAD].with_(T=T)
    args = _oracle_inputs(w)
    t = time.perf_counter()
    for _ in range(steps):
        _oracle_pass(O, w, *args)
    dt = (time.perf_counter() - t) / steps
    return {"value": w.U * T / dt, "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"first {T} of 32768 tokens of the same layer (U=1, 8 kv heads, "
                      f"W=64, keep 0.10), {steps} pass(es), float64 numpy"}


# ------------------------------------------------------------------ main
def slowest_rank_ms(step_ms, world, device):
    """Per-step time of the job: the maximum over ranks (one all-reduce of the
    timing only; the data path has no collective)."""
    if world <= 1:
        return step_ms
    import torch.distributed as dist
    t = torch.tensor([step_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, step_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's step
    time (each rank holds its own copy of the workload: weak scaling)."""
    return world * tokens_per_rank / (step_ms * 1e-3)


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--units", type=int, default=16,
                    help="--only decode_q8: batch size of the decode workload's cut")
    ap.add_argument("--only", choices=["layer", "decode", "decode_q8", "c4", "c3", "vector"],
                    default=None,
                    help="profiling runs: time only one workload")
    args = ap.parse_args()
    world, rank, local = dist_setup(args.gpus)
    w = inputs.WORKLOADS[WORKLOAD]

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 150.0
        T = oracle_sample_tokens(budget, args.steps + args.warmup)
        ws = w.with_(T=T)
        from oracle import kvc_oracle as O
        a = _oracle_inputs(ws)
        for _ in range(args.warmup):
            _oracle_pass(O, ws, *a)
        t = time.perf_counter()
        for _ in range(args.steps):
            _oracle_pass(O, ws, *a)
        dt = (time.perf_counter() - t) / args.steps
        val = ws.U * T / dt
        sample = (f"first {T} of 32768 tokens of the same layer per step, float64 numpy oracle")
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "U": 1, "Hq": 32, "Hkv": 8, "d": 128, "T": T,
                       "W": 64, "keep_ratio": 0.1},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    from kv_cache_compression_attention_b300 import binding as B
    B.lib()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    hbm, bf16, src = peaks()

    if args.only == "decode":
        dec = bench_decode(B, args.steps, args.warmup, device)
        print(json.dumps({"decode": dec, "frac": dec["gbs"] / hbm}))
        return
    if args.only == "decode_q8":
        print(json.dumps(bench_decode_q8_small(B, args.units, args.steps, args.warmup, device)))
        return
    if args.only == "c4":
        print(json.dumps(bench_c4(B, args.steps, args.warmup, device)))
        return
    if args.only == "c3":
        print(json.dumps(bench_c3(B, args.steps, args.warmup, device)))
        return
    if args.only == "vector":
        vec = bench_vector(B, w, args.steps, args.warmup, device)
        vec["residual_frac"] = vec["residual_gbs"] / hbm
        vec["decode"]["frac"] = vec["decode"]["gbs"] / hbm
        print(json.dumps(vec))
        return

    # ---- timed region: exactly K steps of the layer pass
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        L, r = bench_layer(B, w, args.steps, args.warmup, device)
    torch.cuda.synchronize()
    step_ms = slowest_rank_ms(statistics.mean(r["step_ms"]), world, device)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    score_ms = statistics.mean(r["score_ms"])
    value = job_tokens_per_s(world, w.U * w.T, step_ms)
    if args.only == "layer":
        print(json.dumps({"value": value, "step_ms": step_ms, "score_ms": score_ms,
                          "select_ms": statistics.mean(r["select_ms"]),
                          "compact_ms": statistics.mean(r["compact_ms"]),
                          "select_compact_ms": statistics.mean(r["select_compact_ms"]),
                          "step_three_calls_ms": statistics.mean(r["step_three_calls_ms"])}))
        return

    # ---- sub-measurements (outside the headline timed region)
    e2e_ms, h2d, d2h = bench_e2e(B, L, max(6, args.steps // 2), 2)
    score_max_ms = bench_score_max(L, max(5, args.steps // 2), 3)
    kvzip_ms = bench_kvzip_plus(B, L, 3, 1)
    fid = fidelity_probe(B, L)
    del L
    torch.cuda.empty_cache()
    dec = bench_decode(B, inputs.WORKLOADS[DECODE_WORKLOAD].decode_steps, max(3, args.warmup),
                       device)
    dec["frac"] = dec["gbs"] / hbm
    dec["peak_gbs"] = hbm
    c4 = bench_c4(B, max(3, args.steps // 4), 3, device)
    c3 = bench_c3(B, 3, 3, device)
    vec = bench_vector(B, w, max(5, args.steps // 2), 3, device)
    comp_c2 = compact_bytes(r["kept_rows"], w.d, 2)
    comp_c2_us = statistics.mean(r["compact_ms"]) * 1e3

    score_bytes = (w.U * w.Hkv * w.T * w.d * 2 + w.U * w.Hq * w.W * w.d * 2 + w.U * w.Hkv * w.T * 4)
    score_flops = 2.0 * w.U * w.Hq * w.W * w.T * w.d
    # KVzip+: both scoring passes plus one d x d quadratic form per (query head, token)
    kvzip_flops = 2 * score_flops + 2.0 * w.U * w.Hq * w.T * w.d * w.d
    achieved = score_bytes / (score_ms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; Llama-3-8B-shaped layer cache at 32k tokens)",
        "config": {"workload": WORKLOAD, "U": w.U, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "T": w.T, "W": w.W, "keep_ratio": w.keep_ratio, "n_sink": w.n_sink,
                   "n_recent": w.n_recent,
                   "l2": "flushed between steps (256 MiB read + write, then a 256 MiB read)",
                   "clock_ramp_steps": RAMP_STEPS,
                   "parallelism": f"replicas x{world}"},
        # stage times from a separate run with events between the kernels
        "stages_us": {"score": score_ms * 1e3,
                      "select_compact": statistics.mean(r["select_compact_ms"]) * 1e3,
                      "select": statistics.mean(r["select_ms"]) * 1e3,
                      "compact": statistics.mean(r["compact_ms"]) * 1e3,
                      "kept_rows": r["kept_rows"]},
        # the same step with kvc_select and kvc_compact as two calls
        "step_three_calls_us": statistics.mean(r["step_three_calls_ms"]) * 1e3,
        "roofline": {"kernel": "score_tc_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": src,
                     "traffic": profiled_traffic("score_tc.cu", "score_tc_c2_llama32k_traffic.json"),
                     "algorithmic_bytes": score_bytes,
                     "tensor_tflops": score_flops / (score_ms * 1e-3) / 1e12,
                     "tensor_frac": score_flops / (score_ms * 1e-3) / 1e12 / bf16,
                     # the contraction the kernel issues: both of its passes
                     "tensor_tflops_issued": SCORE_PASSES * score_flops / (score_ms * 1e-3) / 1e12,
                     "tensor_frac_issued": SCORE_PASSES * score_flops / (score_ms * 1e-3) / 1e12 / bf16},
        "decode": dec,
        # the other workloads' whole-step throughput (score + select + compact)
        "tokens_per_s_c3_32layer": c3["tokens_per_s"],
        "tokens_per_s_c4_qwen128k": c4["tokens_per_s"],
        "c4_qwen128k": c4,
        "c3_32layer": c3,
        "vector": vec,
        "rooflines": [
            {"kernel": "score_tc_kernel", "workload": WORKLOAD, "bound": "hbm",
             "achieved_gbs": achieved, "frac": achieved / hbm},
            {"kernel": "score_tc_kernel (max aggregation)", "workload": WORKLOAD, "bound": "hbm",
             "time_us": score_max_ms * 1e3,
             "achieved_gbs": score_bytes / (score_max_ms * 1e-3) / 1e9,
             "frac": score_bytes / (score_max_ms * 1e-3) / 1e9 / hbm},
            {"kernel": "value_norm_kernel + score_tc_kernel<true, true> (KVzip+)",
             "workload": WORKLOAD, "bound": "tensor", "time_us": kvzip_ms * 1e3,
             "achieved_tflops": kvzip_flops / (kvzip_ms * 1e-3) / 1e12,
             "frac": kvzip_flops / (kvzip_ms * 1e-3) / 1e12 / bf16},
            {"kernel": "compact_kernel", "workload": WORKLOAD, "bound": "hbm",
             "achieved_gbs": comp_c2 / (comp_c2_us * 1e-6) / 1e9,
             "frac": comp_c2 / (comp_c2_us * 1e-6) / 1e9 / hbm},
            {"kernel": "linear_kernel", "workload": "c4_qwen128k", "bound": "hbm",
             "achieved_gbs": c4["score_linear_gbs"], "frac": c4["score_linear_gbs"] / hbm},
            {"kernel": "compact_kernel", "workload": "c4_qwen128k", "bound": "hbm",
             "achieved_gbs": c4["compact_gbs"], "frac": c4["compact_gbs"] / hbm},
            {"kernel": "w1_transpose_kernel + mlp_tc_kernel (two-layer surrogate, tcgen05)",
             "workload": "c4_qwen128k", "bound": "tensor", "time_us": c4["score_mlp_us"],
             "achieved_tflops": c4["score_mlp_tflops"], "frac": c4["score_mlp_tflops"] / bf16},
            {"kernel": "score_tc_kernel", "workload": "c3_32layer", "bound": "hbm",
             "achieved_gbs": c3["score_gbs"], "frac": c3["score_gbs"] / hbm},
            {"kernel": "compact_kernel", "workload": "c3_32layer", "bound": "hbm",
             "achieved_gbs": c3["compact_gbs"], "frac": c3["compact_gbs"] / hbm},
            {"kernel": "decode_partial_kernel+decode_combine_kernel", "workload": DECODE_WORKLOAD,
             "bound": "hbm", "achieved_gbs": dec["gbs"], "frac": dec["gbs"] / hbm},
            {"kernel": "decode_partial_q8_kernel+decode_combine_kernel (group-quantised pool)",
             "workload": DECODE_WORKLOAD, "bound": "hbm", "time_us": dec["q8"]["us_per_step"],
             "achieved_gbs": dec["q8"]["gbs"], "frac": dec["q8"]["gbs"] / hbm},
            {"kernel": "vector_residual_kernel", "workload": WORKLOAD + " (VECTOR p_c 0.9, p_a 0.05)",
             "bound": "hbm", "time_us": vec["stages_us"]["residual"],
             "achieved_gbs": vec["residual_gbs"], "frac": vec["residual_gbs"] / hbm,
             "tensor_tflops": vec["residual_tflops"]},
            {"kernel": "vector_compact_kernel", "workload": WORKLOAD + " (VECTOR)", "bound": "hbm",
             "time_us": vec["stages_us"]["compact"], "achieved_gbs": vec["compact_gbs"],
             "frac": vec["compact_gbs"] / hbm},
            {"kernel": "decode_partial_mma_kernel+decode_combine_vector_kernel (VECTOR cache)",
             "workload": DECODE_WORKLOAD, "bound": "hbm", "time_us": vec["decode"]["us_per_step"],
             "achieved_gbs": vec["decode"]["gbs"], "frac": vec["decode"]["gbs"] / hbm}],
        "fidelity": fid,
        "e2e": {"value": job_tokens_per_s(world, w.U * w.T, e2e_ms), "unit": "tokens/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "inputs": "q_win and K copied from pinned host memory each step; V read in "
                          "place from pinned host memory (only the kept rows cross the bus)"},
        # per step: score_tc_kernel, select_kernel (hand-off mode),
        # emit_compact_kernel
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

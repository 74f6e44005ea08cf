"""Benchmark: CSA decode queries/s at 1M-token context (and 128K), with the
dominant kernel's fraction of its roofline and the CPU oracle beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload W] [--quick]

One step = one pass of the decode hot path over one batch: one csa_layer call
(Lightning-Indexer scores -> top-k -> window-merged sparse attention) for the
B=4 sequences of the 1M-token workload (262144 compressed entries each, one
query at position 1048575), caches resident in HBM.  K steps are captured in
one CUDA graph and replayed once as the timed region; the device time is taken
with CUDA events on the launching stream.  Under torchrun every
rank runs its own replica (independent sequences: weak scaling, no data-path
collective); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import csa_synth as S  # noqa: E402

HEADLINE = "decode_1m"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM bytes (read + write) per launch of the indexer on the 1M decode
# workload, from an ncu capture (dram__bytes_read.sum + dram__bytes_write.sum)
# of this launch configuration; valid only for the source it was measured on.
TRAFFIC = {"indexer": {"src_sha": "0fd2e310cf61bfb5", "bytes": 273218816}}


def _src_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "long_context_sparse_23_b300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                smax = float(r[1])
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload

class DecodeStep:
    """Device buffers and the library call of one decode step: csa_layer with
    the compressed caches given (indexer scores -> top-k -> window-merged
    sparse attention, enqueued by one call)."""

    def __init__(self, name: str, device):
        import long_context_sparse_23_b300 as csa
        from long_context_sparse_23_b300 import _lib
        self.csa, self.L = csa, _lib.lib()
        self.wl = wl = S.WORKLOADS[name]
        self.inp = i = S.make_inputs(wl, device)
        B, Tq = i["q_pos"].shape
        self.B, self.Tq = B, Tq
        self.out = torch.empty(B, Tq, wl.H, wl.d, dtype=torch.bfloat16, device=device)
        self.args = csa.layer_args(B=B, Tq=Tq, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k,
                                   W=wl.W, T_raw=wl.raw_len, k_cmp=i["k_cmp"], v_cmp=i["v_cmp"],
                                   i_cmp=i["i_cmp"], k_win=i["k_raw"], v_win=i["v_raw"],
                                   raw_base=i["raw_base"], q=i["q"], q_idx=i["q_idx"], w=i["w"],
                                   q_pos=i["q_pos"], out=self.out)
        need = ctypes.c_size_t(0)
        assert self.L.csa_layer_workspace(ctypes.byref(self.args), ctypes.byref(need)) == 0
        self.ws = csa.Workspace(need.value, device)

    def step(self, st):
        r = self.L.csa_layer(ctypes.byref(self.args), self.ws.ptr, self.ws.nbytes, st)
        assert r == 0, r

    def kernels_per_step(self):
        """Our kernel launches in one csa_layer decode step.  Over 16384 entries
        (long rows): histogram zeroing, the indexer (which also accumulates the
        top-k histogram when Tq == 1, else a histogram kernel follows), then
        over 65536 entries the fused top-k + attention kernel; up to 32768
        entries the two-CTA-per-query top-k and the attention; in between the
        select and finish passes of the top-k and the attention.  Up to 16384
        entries: the indexer, the one-pass top-k and the attention.  The
        tensor-core decode attention (H = 64, d = 128) merges the key ranges of
        a query inside a cluster for up to eight ranges of five 128-slot tiles
        and adds a merge kernel beyond that."""
        wl = self.wl
        fused_hist = self.Tq == 1 and wl.H_I >= 16
        attention = 1
        if self.Tq < 16 and wl.H == 64 and wl.d == 128:
            tiles = -(-(wl.k + wl.W) // 128)
            attention += 1 if -(-tiles // 5) > 8 else 0
        if wl.N <= 16384:
            return 2 + attention
        n = 2 + (0 if fused_hist else 1)      # zeroing, indexer (+ histogram pass)
        if wl.N > 65536:
            return n + 1                      # fused tail
        return n + (1 if wl.N <= 32768 else 2) + attention  # top-k (one or two passes) + attention

    # algorithmic work of the indexer launch: every visible entry's d_I-wide bf16
    # key read once per sequence (the queries of a sequence share one pass over
    # the keys), one fp32 score written per (query, visible entry), and each
    # query's H_I x d_I bf16 indexer queries read once; 2 H_I d_I flops per
    # (query, visible entry)
    def indexer_work(self):
        wl = self.wl
        pos = self.inp["q_pos"].cpu().tolist()
        nv = [[min(wl.N, (int(t) + 1) // wl.m) for t in row] for row in pos]
        keys = sum(max(r) for r in nv) * wl.d_I * 2
        scores = sum(sum(r) for r in nv) * 4
        queries = self.B * self.Tq * wl.H_I * wl.d_I * 2
        flops = sum(sum(r) for r in nv) * 2 * wl.H_I * wl.d_I
        return keys + scores + queries, flops


def _step_bytes(self):
    """Algorithmic bytes of one decode step: the indexer's (keys, scores,
    queries), then per query the k kept compressed K/V rows and the W window
    rows (2 d bf16 each), its H x d query and its output."""
    wl = self.wl
    per_q = (wl.k + wl.W) * 2 * wl.d * 2 + 2 * wl.H * wl.d * 2
    return self.indexer_work()[0] + self.B * self.Tq * per_q


DecodeStep.step_bytes = _step_bytes


def graph_of(fn, st_torch, n=1, marks=None, L=None):
    """CUDA graph of ``n`` consecutive steps; with ``marks`` = (begin events,
    end events), step i records marks[0][i] / marks[1][i] around its indexer
    launch (csa_set_indexer_events), so the indexer is timed inside the graph."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st_torch):
        for i in range(n):
            if marks is not None:
                L.csa_set_indexer_events(marks[0][i].cuda_event, marks[1][i].cuda_event)
            fn(st_torch.cuda_stream)
        if marks is not None:
            L.csa_set_indexer_events(None, None)
    return g


def timing_events(n, stream):
    """n timing events, each recorded once so that its handle exists."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in ev:
        e.record(stream)
    stream.synchronize()
    return ev


def upload_graph(g, stream):
    """Upload an instantiated graph to the device without running it
    (cuGraphUpload), so that its first timed replay does not also upload it.
    Returns whether the upload was done."""
    try:
        from cuda.bindings import driver
        r = driver.cuGraphUpload(driver.CUgraphExec(g.raw_cuda_graph_exec()), driver.CUstream(stream.cuda_stream))
        stream.synchronize()
        return r[0] == driver.CUresult.CUDA_SUCCESS
    except Exception:  # noqa: BLE001 -- the first replay then uploads it, as before
        return False


def warm(g1, warmup, stream, min_warm_s=0.3):
    """``warmup`` replays of the one-step graph, then at least ``min_warm_s``
    seconds more of them (clocks and caches settle whatever ``warmup`` is)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g1.replay()
        stream.synchronize()
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < min_warm_s:
            for _ in range(20):
                g1.replay()
            stream.synchronize()


def time_steps(gk, steps, stream):
    """Device time of one replay of the ``steps``-step graph (CUDA events on
    the launching stream, synchronised on both sides): ms per step."""
    upload_graph(gk, stream)  # outside the timed region
    with torch.cuda.stream(stream):
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gk.replay()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) / steps


def layer_time(ds: DecodeStep, steps: int, warmup: int, stream):
    """Average device time of one csa_layer call between CUDA events recorded
    on the launching stream, from plain (non-graph) launches: each batch of
    calls is queued behind a GPU-side sleep, so the events time back-to-back
    kernels, not host launch latency."""
    st = stream.cuda_stream
    batch = 50
    tot, done = 0.0, 0
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            ds.step(st)
        while done < steps:
            nb = min(batch, steps - done)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
            torch.cuda._sleep(20_000_000)       # ~10 ms of GPU time to queue behind
            ev[0].record(stream)
            for i in range(nb):
                ds.step(st)
                ev[i + 1].record(stream)
            stream.synchronize()
            tot += sum(ev[i].elapsed_time(ev[i + 1]) for i in range(nb))
            done += nb
    return tot / steps


def e2e_decode(ds: DecodeStep, min_steps: int = 500, min_s: float = 1.0, warmup: int = 20, depth: int = 2):
    """Queries/s through csa_layer_host, the C-ABI call for callers whose step
    inputs and result live in host memory: every step copies its queries
    (q, q_idx) in from pinned host memory, runs the layer and copies its
    output back to pinned host memory, on one stream, inside the timed
    region.  ``depth`` steps are in flight, each on its own stream with its
    own device staging buffers, workspace and host output buffer, as a
    serving loop runs independent batches: the host waits for step s's output
    before it reuses step s's buffers for step s + depth.  Runs at least
    ``min_steps`` steps and at least ``min_s`` seconds.  Returns (ms per step,
    H2D bytes per step, D2H bytes per step, steps timed)."""
    csa, wl, i = ds.csa, ds.wl, ds.inp
    hq = i["q"].cpu().pin_memory()
    hqi = i["q_idx"].cpu().pin_memory()
    slots = []
    for _ in range(depth):
        dq, dqi = torch.empty_like(i["q"]), torch.empty_like(i["q_idx"])
        out = torch.empty_like(ds.out)
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        a = csa.layer_args(B=ds.B, Tq=ds.Tq, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k,
                           W=wl.W, T_raw=wl.raw_len, k_cmp=i["k_cmp"], v_cmp=i["v_cmp"], i_cmp=i["i_cmp"],
                           k_win=i["k_raw"], v_win=i["v_raw"], raw_base=i["raw_base"], q=dq, q_idx=dqi,
                           w=i["w"], q_pos=i["q_pos"], out=out)
        need = ctypes.c_size_t(0)
        ds.L.csa_layer_workspace(ctypes.byref(a), ctypes.byref(need))
        ws = csa.Workspace(need.value)
        st = torch.cuda.Stream()
        slots.append((ctypes.byref(a), a, hout, ws.ptr, ws.nbytes, st.cuda_stream, st, torch.cuda.Event(), dq, dqi,
                      out, ws))
    torch.cuda.synchronize()
    fn = ds.L.csa_layer_host
    hq_p, hqi_p = hq.data_ptr(), hqi.data_ptr()

    def run(n):
        for s in range(n):
            sl = slots[s % depth]
            if s >= depth:
                sl[7].synchronize()   # step s - depth's output is on the host
            r = fn(sl[0], hq_p, hqi_p, sl[2].data_ptr(), sl[3], sl[4], sl[5])
            if r:
                raise RuntimeError(f"csa_layer_host: {r}")
            sl[7].record(sl[6])
        for s in range(max(0, n - depth), n):
            slots[s % depth][7].synchronize()

    run(warmup)
    done, t = 0, 0.0
    while done < min_steps or t < min_s:
        t0 = time.perf_counter()
        run(250)
        t += time.perf_counter() - t0
        done += 250
    h2d = hq.numel() * 2 + hqi.numel() * 2
    d2h = slots[0][2].numel() * slots[0][2].element_size()
    for sl in slots:     # every slot's output equals the device-resident step's
        assert torch.equal(sl[2], ds.out.cpu()), "csa_layer_host output differs from csa_layer's"
    return t / done * 1e3, h2d, d2h, done


def host_call_us(ds: DecodeStep, stream, calls: int = 2000):
    """Host time of one csa_layer call (argument checks, tensor-map encoding
    and kernel launches; ctypes marshalling included): calls are made in
    bursts of 100, each timed with perf_counter without waiting for the GPU;
    the GPU is drained between bursts, outside the timing."""
    st = stream.cuda_stream
    tot = 0.0
    with torch.cuda.stream(stream):
        for _ in range(calls // 100):
            stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(100):
                ds.step(st)
            tot += time.perf_counter() - t0
        stream.synchronize()
    return tot / (calls // 100 * 100) * 1e6


def combine_over_ranks(ms: float, units_per_rank: int, world: int, device) -> tuple:
    """The step time of the slowest rank and the whole-job rate: every rank
    processes its own ``units_per_rank`` units per step (independent
    sequences, no data-path collective), so the job's rate is the units of all
    ranks over the slowest rank's time.  Returns (ms, units per second)."""
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.barrier()
        ms = float(t.item())
    return ms, units_per_rank * world / (ms * 1e-3)


# ---------------------------------------------------------------- CPU oracle

def oracle_rate(name: str, budget_s: float, steps: int = 0, warmup: int = 0):
    """The oracle on the host: queries/s on a bounded sample of the workload.

    One query of sequence 0: indexer scores over its most recent ``n`` visible
    entries, top-k of those scores, window-merged attention over the kept
    entries.  With steps = 0 every sample is a whole query (n = n_vis) and
    samples repeat until ``budget_s`` is spent; with steps = K each of the
    W + K samples is sized so that they fit the budget together, and the rate
    is scaled by n / n_vis (the indexer dominates the oracle's work).
    Input generation is outside the timed calls."""
    import numpy as np  # noqa: F401
    import oracle as O
    try:
        from threadpoolctl import threadpool_info
        threads = max([d.get("num_threads", 1) for d in threadpool_info()] + [1])
    except Exception:  # pragma: no cover
        threads = 1
    threads = max(threads, torch.get_num_threads())  # the generator / oracle's torch ops
    wl = S.WORKLOADS[name]
    t = wl.q_positions[0]
    n_vis = O.n_visible(t, wl.m, wl.N)
    c = S.make_inputs(wl.replace(B=1), "cpu", only={"q", "q_idx", "w", "q_pos", "k_raw", "v_raw"})
    q_bits, qi_bits = S.bf16_bits(c["q"]), S.bf16_bits(c["q_idx"])
    kr_bits, vr_bits = S.bf16_bits(c["k_raw"]), S.bf16_bits(c["v_raw"])
    w = c["w"].numpy()
    rows = torch.arange(0, n_vis, dtype=torch.int64)
    ki_bits = S.bf16_bits(S.rows_bf16(wl.seed, S.TID["i_cmp"], wl.N, wl.d_I, 0, rows))[None]
    kc_bits = S.bf16_bits(S.rows_bf16(wl.seed, S.TID["k_cmp"], wl.N, wl.d, 0, rows))[None]
    vc_bits = S.bf16_bits(S.rows_bf16(wl.seed, S.TID["v_cmp"], wl.N, wl.d, 0, rows))[None]
    base = [wl.raw_base]

    def sample(n):
        # the oracle's own batched calls: (2)+(3) over the newest n entries, then (4)
        t0 = time.perf_counter()
        lo = n_vis - n
        idx, _ = O.csa_index_topk(qi_bits, ki_bits[:, lo:], w, [[n * wl.m - 1]], wl.m, wl.k)
        O.csa_attend(q_bits, kc_bits[:, lo:], vc_bits[:, lo:], idx, kr_bits, vr_bits, base, [[t]],
                     wl.W, 1 / math.sqrt(wl.d))
        return time.perf_counter() - t0

    if steps <= 0:
        done, tot = 0, 0.0
        while done == 0 or tot < budget_s:
            tot += sample(n_vis)
            done += 1
        return done / tot, threads, (f"{done} whole queries of {name} (sequence 0, t={t}, "
                                     f"{n_vis} visible entries), inputs generated outside the timing; "
                                     f"host has {os.cpu_count()} logical CPUs"), 1e3 * tot / done
    probe = sample(min(n_vis, 16384))
    per_step = budget_s / (steps + warmup)
    n = int(min(n_vis, max(1024, min(n_vis, 16384) * per_step / max(probe, 1e-6))))
    for _ in range(warmup):
        sample(n)
    tot = sum(sample(n) for _ in range(steps))
    return steps * (n / n_vis) / tot, threads, (
        f"each timed step is 1 query of {name} (sequence 0) with its indexer over the most recent {n} of "
        f"{n_vis} visible entries, then top-k and attention; ms_per_step is that step's measured time, and "
        f"the rate is scaled by n/n_vis to whole queries"), 1e3 * tot / steps


# ---------------------------------------------------------------- other workloads

def time_calls(fn, stream, steps, warmup=3):
    """ms per call of ``fn(stream_handle)``: ``steps`` calls captured in one
    CUDA graph, replayed once between CUDA events (after warm-up replays)."""
    with torch.cuda.stream(stream):
        fn(stream.cuda_stream)
        stream.synchronize()
        g1 = graph_of(fn, stream)
        gk = graph_of(fn, stream, n=steps)
    warm(g1, warmup, stream, min_warm_s=0.1)
    return time_steps(gk, steps, stream)


def decode_also(name, dev, stream, steps):
    """Another decode workload: device time per csa_layer step (CUDA graph of
    ``steps`` calls), the indexer inside a second graph of the same steps
    (CUDA events around each indexer launch), the indexer's HBM and bf16
    tensor fractions and the step's fraction of its HBM floor."""
    ds = DecodeStep(name, dev)
    ev_b, ev_e = timing_events(steps, stream), timing_events(steps, stream)
    with torch.cuda.stream(stream):
        ds.step(stream.cuda_stream)
        stream.synchronize()
        g1 = graph_of(ds.step, stream)
        gk = graph_of(ds.step, stream, n=steps)
        gm = graph_of(ds.step, stream, n=steps, marks=(ev_b, ev_e), L=ds.L)
    assert ds.ws.check_error() == 0
    warm(g1, 10, stream)
    ms = time_steps(gk, steps, stream)
    time_steps(gm, steps, stream)
    ms_idx = sum(b.elapsed_time(e) for b, e in zip(ev_b, ev_e)) / steps
    peaks, _ = _peaks()
    ibytes, iflops = ds.indexer_work()
    sb = ds.step_bytes()
    return {"queries_per_s": ds.B * ds.Tq / (ms * 1e-3), "ms_per_step": ms, "B": ds.B, "Tq": ds.Tq,
            "indexer_ms": ms_idx, "indexer_bytes": ibytes, "indexer_flops": iflops,
            "indexer_frac_of_hbm": ibytes / (ms_idx * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "indexer_frac_of_bf16_peak": iflops / (ms_idx * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "step_bytes": sb, "step_floor_ms": sb / peaks["hbm_gbs"] / 1e6,
            "step_frac_of_hbm": sb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}


def _graph_ms(fn, stream, steps, marks=None, L=None):
    """ms per call of fn (a graph of ``steps`` calls, after warm-up)."""
    with torch.cuda.stream(stream):
        fn(stream.cuda_stream)
        stream.synchronize()
        g1 = graph_of(fn, stream)
        gk = graph_of(fn, stream, n=steps)
        gm = graph_of(fn, stream, n=steps, marks=marks, L=L) if marks is not None else None
    warm(g1, 10, stream, min_warm_s=0.1)
    ms = time_steps(gk, steps, stream)
    if gm is not None:
        time_steps(gm, steps, stream)
    return ms


def decode_1m_variants(dev, stream, steps):
    """The 1M decode step (B = 4) with the decode-time append of the block
    its position completes (t = 1048575: block 262143 is compressed from the
    window rows into all three caches before the indexer), and with E4M3
    indexer keys (quantised once, outside the timing; the step quantises its
    indexer queries)."""
    import long_context_sparse_23_b300 as csa
    out = {}
    ds = DecodeStep("decode_1m", dev)
    wl, i = ds.wl, ds.inp
    B = ds.B
    # append: raw indexer-key rows and gate logits of the window
    win = {n: S.normal_bf16(wl.seed, S.TID[n], (B, wl.raw_len, wl.d_I if n in ("i_raw", "g_i") else wl.d), dev,
                            offset=0)
           for n in ("i_raw", "g_k", "g_v", "g_i")}
    a = csa.layer_args(B=B, Tq=1, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=wl.W,
                       T_raw=wl.raw_len, k_cmp=i["k_cmp"], v_cmp=i["v_cmp"], i_cmp=i["i_cmp"], k_win=i["k_raw"],
                       v_win=i["v_raw"], raw_base=i["raw_base"], q=i["q"], q_idx=i["q_idx"], w=i["w"],
                       q_pos=i["q_pos"], out=ds.out, i_win=win["i_raw"], gk_win=win["g_k"], gv_win=win["g_v"],
                       gi_win=win["g_i"])
    need = ctypes.c_size_t(0)
    ds.L.csa_layer_workspace(ctypes.byref(a), ctypes.byref(need))
    ws = csa.Workspace(need.value, dev)

    def step_append(st):
        assert ds.L.csa_layer(ctypes.byref(a), ws.ptr, ws.nbytes, st) == 0

    ms = _graph_ms(step_append, stream, steps)
    assert ws.check_error() == 0
    out["decode_1m_append"] = {"ms_per_step": ms, "queries_per_s": B / (ms * 1e-3),
                               "appended": "block 262143 of K, V and the indexer keys, every step"}

    # FP8 indexer keys
    k8, ks = csa.csa_quantize_fp8(i["i_cmp"])
    a8 = csa.layer_args(B=B, Tq=1, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=wl.W,
                        T_raw=wl.raw_len, k_cmp=i["k_cmp"], v_cmp=i["v_cmp"], i_cmp=k8, k_win=i["k_raw"],
                        v_win=i["v_raw"], raw_base=i["raw_base"], q=i["q"], q_idx=i["q_idx"], w=i["w"],
                        q_pos=i["q_pos"], out=ds.out, i_scale=ks)
    ds.L.csa_layer_workspace(ctypes.byref(a8), ctypes.byref(need))
    ws8 = csa.Workspace(need.value, dev)

    def step_fp8(st):
        assert ds.L.csa_layer(ctypes.byref(a8), ws8.ptr, ws8.nbytes, st) == 0

    ev_b, ev_e = timing_events(steps, stream), timing_events(steps, stream)
    ms8 = _graph_ms(step_fp8, stream, steps, marks=(ev_b, ev_e), L=ds.L)
    assert ws8.check_error() == 0
    ms_idx = sum(b_.elapsed_time(e_) for b_, e_ in zip(ev_b, ev_e)) / steps
    peaks, _ = _peaks()
    n_vis = B * wl.N
    ibytes = n_vis * (wl.d_I + 4 + 4) + B * wl.H_I * (wl.d_I + 4)   # codes + key scale + score; query codes
    sb = ibytes + B * ((wl.k + wl.W) * 2 * wl.d * 2 + 2 * wl.H * wl.d * 2)
    out["decode_1m_fp8_indexer"] = {
        "ms_per_step": ms8, "queries_per_s": B / (ms8 * 1e-3), "indexer_ms": ms_idx, "indexer_bytes": ibytes,
        "indexer_frac_of_hbm": ibytes / (ms_idx * 1e-3) / 1e9 / peaks["hbm_gbs"], "step_bytes": sb,
        "step_frac_of_hbm": sb / (ms8 * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "keys": "E4M3 codes + one fp32 power-of-two scale per entry (132 B instead of 256 B)"}
    del ds
    return out


def hybrid_stack_1m(dev, stream, steps, n_pairs=7):
    """One decode step of the hybrid stack at 1M context, B = 4: two
    sliding-window layers, then n_pairs x (CSA, HCA) (CSA: 262144 entries at
    m = 4, top-1024; HCA: 8192 entries at m' = 128; window 128 everywhere),
    each layer with its own synthetic caches; one csa_stack_decode call."""
    import long_context_sparse_23_b300 as csa
    from long_context_sparse_23_b300 import _lib
    L = _lib.lib()
    wl = S.WORKLOADS["decode_1m"]
    B, H, d, W, T_raw = wl.B, wl.H, wl.d, wl.W, wl.raw_len
    t = wl.q_positions[0]
    q_pos = torch.full((B, 1), t, dtype=torch.int32, device=dev)
    raw_base = torch.full((B,), t + 1 - T_raw, dtype=torch.int32, device=dev)
    kinds = [_lib.CSA_STACK_SWA] * 2 + [_lib.CSA_STACK_CSA, _lib.CSA_STACK_HCA] * n_pairs
    layers = (_lib.csa_stack_layer * len(kinds))()
    keep = []
    N_h = (t + 1) // 128
    for li, kind in enumerate(kinds):
        sd = 100 + li
        kw = S.normal_bf16(sd, S.TID["k_raw"], (B, T_raw, d), dev)
        vw = S.normal_bf16(sd, S.TID["v_raw"], (B, T_raw, d), dev)
        keep += [kw, vw]
        if kind == _lib.CSA_STACK_CSA:
            kc = S.normal_bf16(sd, S.TID["k_cmp"], (B, wl.N, d), dev)
            vc = S.normal_bf16(sd, S.TID["v_cmp"], (B, wl.N, d), dev)
            ic = S.normal_bf16(sd, S.TID["i_cmp"], (B, wl.N, wl.d_I), dev)
            w = S.uniform_f32(sd, S.TID["w"], (wl.H_I,), dev)
            keep += [kc, vc, ic, w]
            a = csa.layer_args(B=B, Tq=1, N=wl.N, m=wl.m, H=H, d=d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=W,
                               T_raw=T_raw, k_cmp=kc, v_cmp=vc, i_cmp=ic, k_win=kw, v_win=vw, raw_base=raw_base,
                               w=w, q_pos=q_pos)
        elif kind == _lib.CSA_STACK_HCA:
            kc = S.normal_bf16(sd, S.TID["k_cmp"], (B, N_h, d), dev)
            vc = S.normal_bf16(sd, S.TID["v_cmp"], (B, N_h, d), dev)
            keep += [kc, vc]
            a = csa.layer_args(B=B, Tq=1, N=N_h, m=128, H=H, d=d, H_I=0, d_I=0, k=0, W=W, T_raw=T_raw, k_cmp=kc,
                               v_cmp=vc, k_win=kw, v_win=vw, raw_base=raw_base, q_pos=q_pos)
        else:
            a = csa.layer_args(B=B, Tq=1, N=0, m=1, H=H, d=d, H_I=0, d_I=0, k=0, W=W, T_raw=T_raw, k_win=kw,
                               v_win=vw, raw_base=raw_base, q_pos=q_pos)
        layers[li].kind = kind
        layers[li].a = a
    x = S.normal_bf16(99, S.TID["q"], (B, 1, H, d), dev)
    y = torch.empty_like(x)
    need = ctypes.c_size_t(0)
    assert L.csa_stack_workspace(layers, len(kinds), ctypes.byref(need)) == 0
    ws = csa.Workspace(need.value, dev)

    def step(st):
        assert L.csa_stack_decode(layers, len(kinds), x.data_ptr(), y.data_ptr(), 0, ws.ptr, ws.nbytes, st) == 0

    ms = _graph_ms(step, stream, steps)
    assert ws.check_error() == 0
    return {"layers": f"2 sliding-window + {n_pairs} x (CSA, HCA)", "ms_per_token_step": ms,
            "tokens_per_s": B / (ms * 1e-3), "B": B, "context": t + 1}


def prefill_8k(dev, stream, steps):
    """The whole layer over an 8192-token prefill (compress -> indexer ->
    top-k -> attention): tokens/s, and the indexer's bf16 tensor-core rate
    (timed inside the graph with csa_set_indexer_events)."""
    import long_context_sparse_23_b300 as csa
    from long_context_sparse_23_b300 import _lib
    L = _lib.lib()
    wl = S.WORKLOADS["prefill_8k"]
    i = S.make_inputs(wl, dev)
    B, T = wl.B, wl.T
    N = T // wl.m
    kc = torch.empty(B, N, wl.d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    ic = torch.empty(B, N, wl.d_I, dtype=torch.bfloat16, device=dev)
    out = torch.empty(B, T, wl.H, wl.d, dtype=torch.bfloat16, device=dev)
    a = csa.layer_args(B=B, Tq=T, N=N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=wl.W, T=T,
                       T_raw=T, x_k=i["k_raw"], x_v=i["v_raw"], x_i=i["i_raw"], g_k=i["g_k"], g_v=i["g_v"],
                       g_i=i["g_i"], k_cmp=kc, v_cmp=vc, i_cmp=ic, k_win=i["k_raw"], v_win=i["v_raw"],
                       raw_base=i["raw_base"], q=i["q"], q_idx=i["q_idx"], w=i["w"], q_pos=i["q_pos"], out=out)
    need = ctypes.c_size_t(0)
    L.csa_layer_workspace(ctypes.byref(a), ctypes.byref(need))
    ws = csa.Workspace(need.value, dev)

    def step(st):
        assert L.csa_layer(ctypes.byref(a), ws.ptr, ws.nbytes, st) == 0

    ms = time_calls(step, stream, steps)
    ev_b, ev_e = timing_events(steps, stream), timing_events(steps, stream)
    with torch.cuda.stream(stream):
        gk = graph_of(step, stream, n=steps, marks=(ev_b, ev_e), L=L)
        gk.replay()
        stream.synchronize()
    ms_idx = sum(b.elapsed_time(e) for b, e in zip(ev_b, ev_e)) / steps
    flops = sum(min(N, (t + 1) // wl.m) for t in range(T)) * wl.H_I * wl.d_I * 2
    peaks, _ = _peaks()
    tf = flops / (ms_idx * 1e-3) / 1e12

    # each step alone through its own public call (same buffers): compression
    # of the three streams, indexer + top-k, attention on the kept indices
    P = ctypes.c_void_p * 3
    xs = P(i["k_raw"].data_ptr(), i["v_raw"].data_ptr(), i["i_raw"].data_ptr())
    gs = P(i["g_k"].data_ptr(), i["g_v"].data_ptr(), i["g_i"].data_ptr())
    os_ = P(kc.data_ptr(), vc.data_ptr(), ic.data_ptr())
    Ds = (ctypes.c_int * 3)(wl.d, wl.d, wl.d_I)
    idx = torch.empty(B, T, wl.k, dtype=torch.int32, device=dev)
    need = ctypes.c_size_t(0)
    L.csa_index_topk_workspace(B, T, N, wl.H_I, wl.d_I, wl.k, ctypes.byref(need))
    ws_i = csa.Workspace(need.value, dev)
    L.csa_attend_workspace(B, T, wl.H, wl.d, wl.k, wl.W, ctypes.byref(need))
    ws_a = csa.Workspace(need.value, dev)

    def comp(st):
        assert L.csa_compress(3, xs, gs, os_, Ds, B, T, wl.m, 0, st) == 0

    def itk(st):
        assert L.csa_index_topk(i["q_idx"].data_ptr(), ic.data_ptr(), i["w"].data_ptr(), 0, i["q_pos"].data_ptr(), B,
                                T, N, wl.H_I, wl.d_I, wl.m, wl.k, idx.data_ptr(), None, ws_i.ptr, ws_i.nbytes,
                                st) == 0

    def att(st):
        assert L.csa_attend(i["q"].data_ptr(), kc.data_ptr(), vc.data_ptr(), idx.data_ptr(), i["k_raw"].data_ptr(),
                            i["v_raw"].data_ptr(), i["raw_base"].data_ptr(), i["q_pos"].data_ptr(), B, T, N, T,
                            wl.H, wl.d, wl.k, wl.W, 0.0, out.data_ptr(), 0, None, ws_a.ptr, ws_a.nbytes, st) == 0

    ms_c = time_calls(comp, stream, steps)
    ms_it = time_calls(itk, stream, steps)
    ms_a = time_calls(att, stream, steps)
    keys = sum(min(wl.k, min(N, (t + 1) // wl.m)) + min(wl.W, t + 1) for t in range(T)) * B
    att_flops = keys * 4 * wl.H * wl.d
    comp_bytes = B * T * (2 * wl.d + wl.d_I) * 2 * 2 + B * N * (2 * wl.d + wl.d_I) * 2
    return {"tokens_per_s": B * T / (ms * 1e-3), "ms_per_layer": ms, "indexer_ms": ms_idx,
            "indexer_tflops": tf, "indexer_flops": flops,
            "indexer_frac_of_bf16_peak": tf / peaks["bf16_tflops"], "bf16_peak_tflops": peaks["bf16_tflops"],
            "stages_ms": {"compress": ms_c, "index_topk": ms_it, "topk_after_indexer": ms_it - ms_idx,
                          "attention": ms_a},
            "compress_frac_of_hbm": comp_bytes / (ms_c * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "attention_flops": att_flops, "attention_kernel": "attend_kernel (mma.sync)",
            "attention_frac_of_bf16_peak": att_flops / (ms_a * 1e-3) / 1e12 / peaks["bf16_tflops"]}


def hca_decode_1m(dev, stream, steps):
    """HCA at 1M context, B = 8: compression of the raw K/V streams at m' = 128
    (GB/s) and the dense attention over the 8192 entries + window (queries/s)."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["hca_decode_1m"]
    i = S.make_inputs(wl, dev)
    B, T, m = wl.B, wl.T, wl.m
    outs = [torch.empty(B, T // m, wl.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    out = torch.empty(B, 1, wl.H, wl.d, dtype=torch.bfloat16, device=dev)
    ws = csa.Workspace(1 << 16, dev)

    def comp(st):
        csa.csa_compress([i["k_raw"], i["v_raw"]], [i["g_k"], i["g_v"]], m, outs=outs)

    def att(st):
        csa.hca_attend(i["q"], outs[0], outs[1], i["k_raw"], i["v_raw"], i["raw_base"], i["q_pos"], m, wl.W,
                       ws=ws)

    with torch.cuda.stream(stream):
        ms_c = time_calls(comp, stream, max(3, steps // 20))
        # the attention reads 34 MB of entries per call: consecutive calls take
        # their caches from a rotation of copies larger than L2 (126 MB), so
        # every call reads its keys and values from HBM
        sets = [outs] + [[o.clone() for o in outs] for _ in range(5)]
        turn = [0]

        def att_rot(st):
            kc, vc = sets[turn[0] % len(sets)]
            turn[0] += 1
            csa.hca_attend(i["q"], kc, vc, i["k_raw"], i["v_raw"], i["raw_base"], i["q_pos"], m, wl.W, ws=ws)

        ms_a = time_calls(att_rot, stream, steps)
    rd = 4 * B * T * wl.d * 2
    wr = 2 * B * (T // m) * wl.d * 2
    peaks, _ = _peaks()
    gbs = (rd + wr) / (ms_c * 1e-3) / 1e9
    # algorithmic bytes of the attention: every visible entry and window row,
    # K and V, once per query (the queries and outputs are 1/256 of that)
    keys = sum(min(wl.N, (t + 1) // m) + min(wl.W, t + 1) for t in wl.q_positions) * B
    att_bytes = keys * wl.d * 2 * 2
    att_gbs = att_bytes / (ms_a * 1e-3) / 1e9
    return {"compress_ms": ms_c, "compress_gbs": gbs, "compress_frac_of_hbm": gbs / peaks["hbm_gbs"],
            "raw_tokens_per_s": B * T / (ms_c * 1e-3), "attend_ms": ms_a, "queries_per_s": B / (ms_a * 1e-3),
            "attend_bytes": att_bytes, "attend_gbs": att_gbs, "attend_frac_of_hbm": att_gbs / peaks["hbm_gbs"],
            "attend_l2": "6 rotating copies of the entries (201 MB > L2)"}


def hca_attend_given(dev, stream, steps, warmup=3):
    """Only the HCA attention at 1M context (B = 8, 8192 entries given as
    synthetic caches, H = 64, d = 128, W = 128), six rotating copies of the
    caches (201 MB > L2): the small case used for kernel profiles."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["hca_decode_1m"]
    B, N, m = wl.B, wl.T // wl.m, wl.m
    q = S.normal_bf16(7, S.TID["q"], (B, 1, wl.H, wl.d), dev)
    kr = S.normal_bf16(7, S.TID["k_raw"], (B, 2 * wl.W, wl.d), dev)
    vr = S.normal_bf16(7, S.TID["v_raw"], (B, 2 * wl.W, wl.d), dev)
    t = wl.q_positions[0]
    q_pos = torch.full((B, 1), t, dtype=torch.int32, device=dev)
    raw_base = torch.full((B,), t + 1 - 2 * wl.W, dtype=torch.int32, device=dev)
    sets = [(S.normal_bf16(8 + r, S.TID["k_cmp"], (B, N, wl.d), dev), S.normal_bf16(8 + r, S.TID["v_cmp"], (B, N, wl.d), dev))
            for r in range(6)]
    ws = csa.Workspace(1 << 16, dev)
    turn = [0]

    def att(st):
        kc, vc = sets[turn[0] % len(sets)]
        turn[0] += 1
        csa.hca_attend(q, kc, vc, kr, vr, raw_base, q_pos, m, wl.W, ws=ws)

    ms = time_calls(att, stream, steps, warmup)
    assert ws.check_error() == 0
    return {"workload": "hca_attend_1m", "ms_per_call": ms, "queries_per_s": B / (ms * 1e-3), "steps": steps}


def workload_config(name: str) -> dict:
    wl = S.WORKLOADS[name]
    n_vis = sum(min(wl.N, (t + 1) // wl.m) for t in wl.q_positions) * wl.B
    return {"workload": name, "B": wl.B, "Tq": wl.Tq, "context": wl.T, "entries": wl.N, "m": wl.m, "H": wl.H,
            "d": wl.d, "H_I": wl.H_I, "d_I": wl.d_I, "k": wl.k, "W": wl.W,
            "l2": f"inputs exceed L2: {n_vis * wl.d_I * 2 / 1e6:.0f} MB of indexer keys streamed per step",
            "launch": "one CUDA graph of K unrolled csa_layer calls (caches resident, decode)"}


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["decode_1m", "decode_128k", "decode_1m_tail", "hca_attend_1m", "prefill_8k",
                             "decode_1m_variants", "hybrid_stack_1m"],
                    help="decode workload to time (the headline is decode_1m); with --quick also "
                         "hca_attend_1m (only the HCA attention over given caches), prefill_8k (the whole "
                         "layer over an 8192-token prefill), decode_1m_variants (the 1M step with the append "
                         "and with FP8 indexer keys) and hybrid_stack_1m (16 layers at 1M context)")
    ap.add_argument("--quick", action="store_true",
                    help="time the device step only: no stage breakdown, e2e, 128K line or CPU baseline "
                         "(the form used for kernel profiles)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload in ("hca_attend_1m", "prefill_8k", "decode_1m_variants", "hybrid_stack_1m"):
        if not args.quick or args.impl != "ours" or world != 1:
            raise SystemExit(f"{args.workload} is a profiling case: --quick, one GPU, --impl ours")
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        import __graft_entry__
        __graft_entry__.build()
        st = torch.cuda.Stream(device=dev)
        if args.workload == "hca_attend_1m":
            print(json.dumps(hca_attend_given(dev, st, args.steps, args.warmup)))
        elif args.workload == "decode_1m_variants":
            print(json.dumps(decode_1m_variants(dev, st, args.steps)))
        elif args.workload == "hybrid_stack_1m":
            print(json.dumps(hybrid_stack_1m(dev, st, args.steps)))
        else:
            print(json.dumps(prefill_8k(dev, st, args.steps)))
        return
    wl = S.WORKLOADS[args.workload]
    metric = (f"CSA decode queries/s @{'1M' if wl.T == 1 << 20 else '128K'} ctx (B={wl.B}, {wl.N} compressed "
              f"entries, top-{wl.k}, W={wl.W})")

    if args.impl == "reference":
        if rank != 0:
            return
        rate, threads, what, ms_step = oracle_rate(args.workload, budget_s=60.0, steps=args.steps,
                                                   warmup=args.warmup)
        line = {"impl": "reference", "metric": metric, "value": rate, "unit": "queries/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(args.workload),
                "cpu_baseline": {"value": rate, "unit": "queries/s", "cores": threads, "kind": "oracle", "sample": what},
                "e2e": {"value": rate, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()

    ds = DecodeStep(args.workload, dev)
    stream = torch.cuda.Stream(device=dev)
    K = args.steps
    ev_b, ev_e = timing_events(K, stream), timing_events(K, stream)
    with torch.cuda.stream(stream):
        ds.step(stream.cuda_stream)      # first calls outside capture (one-time set-up)
        stream.synchronize()
        g1 = graph_of(ds.step, stream)
        gk = graph_of(ds.step, stream, n=K)
        # the same K steps with CUDA events recorded around every indexer launch
        # (event nodes split the kernels' programmatic overlap, so this graph is
        # timed separately from the headline one)
        gm = graph_of(ds.step, stream, n=K, marks=(ev_b, ev_e), L=ds.L)
    assert ds.ws.check_error() == 0

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    warm(g1, args.warmup, stream)
    clk = ClockSampler(local)
    clk.start()
    ms = time_steps(gk, K, stream)
    clocks = clk.stop()
    ms_marked = time_steps(gm, K, stream)
    # the indexer's own launches inside the marked replay
    ms_idx = sum(b.elapsed_time(e) for b, e in zip(ev_b, ev_e)) / K
    if args.quick:
        stages = {"csa_layer_plain_launches": layer_time(ds, 50, 5, stream), "step_with_indexer_events": ms_marked}
        if rank == 0:
            print(json.dumps({"workload": args.workload, "ms_per_step": ms, "steps": K, "indexer_ms": ms_idx,
                              "stages_ms": stages, "queries_per_s": ds.B * ds.Tq * world / (ms * 1e-3),
                              "clocks": clocks}))
        return
    stages = {"csa_layer_plain_launches": layer_time(ds, max(20, min(args.steps, 400)), 5, stream),
              "step_with_indexer_events": ms_marked, "indexer_in_graph": ms_idx}
    host_us = host_call_us(ds, stream)
    torch.cuda.synchronize()
    ms, qps = combine_over_ranks(ms, ds.B * ds.Tq, world, dev)

    launches = args.steps * ds.kernels_per_step()
    e2e_ms, h2d, d2h, e2e_steps = e2e_decode(ds)
    _, e2e_qps = combine_over_ranks(e2e_ms, ds.B * ds.Tq, world, dev)

    peaks, src = _peaks()
    ibytes, _ = ds.indexer_work()
    achieved = ibytes / (ms_idx * 1e-3) / 1e9
    sha = _src_sha("indexer.cu", "common.cuh")
    traffic = TRAFFIC["indexer"]["bytes"] if TRAFFIC["indexer"]["src_sha"] == sha else None
    roof = {"kernel": "indexer_single_kernel (tcgen05)", "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic, "algorithmic_bytes": ibytes, "launch_us": round(ms_idx * 1e3, 2),
            "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback 6.4 TB/s"}
    step_bytes = ds.step_bytes()
    step_roof = {"bytes": step_bytes, "floor_us": round(step_bytes / peaks["hbm_gbs"] / 1e3, 2),
                 "frac": round(step_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}

    extra = {}
    del ds, g1, gk, gm
    torch.cuda.empty_cache()
    extra["decode_128k"] = decode_also("decode_128k", dev, stream, max(10, args.steps // 4))
    torch.cuda.empty_cache()
    extra["decode_1m_tail"] = decode_also("decode_1m_tail", dev, stream, max(10, args.steps // 8))
    torch.cuda.empty_cache()
    extra.update(decode_1m_variants(dev, stream, max(10, args.steps // 8)))
    torch.cuda.empty_cache()
    extra["hybrid_stack_1m"] = hybrid_stack_1m(dev, stream, max(5, args.steps // 50))
    torch.cuda.empty_cache()
    extra["prefill_8k"] = prefill_8k(dev, stream, max(5, args.steps // 100))
    torch.cuda.empty_cache()
    extra["hca_decode_1m"] = hca_decode_1m(dev, stream, max(10, args.steps // 10))
    torch.cuda.empty_cache()

    line = {"metric": metric, "value": qps, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args.workload),
            "clocks": clocks, "gpu_launches": launches, "roofline": roof,
            "e2e": {"value": e2e_qps, "unit": "queries/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": "csa_layer_host (pinned host q, q_idx in; out back to pinned host memory)",
                    "in_flight": 2, "steps_timed": e2e_steps, "ms_per_step": round(e2e_ms, 5)},
            "step_roofline": step_roof,
            "stages_ms": {k: round(v, 5) for k, v in stages.items()},
            "host_us_per_csa_layer_call": round(host_us, 2), "also": extra}
    if rank == 0:
        rate, threads, what, _ = oracle_rate(HEADLINE, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": rate, "unit": "queries/s", "cores": threads, "kind": "oracle", "sample": what}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

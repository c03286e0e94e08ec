"""Throughput of the attention hot path on one GB300 (or N, one process each).

A step is one forward plus one backward (preprocess, dK/dV pass, dQ pass) of
the key-padding-masked workload: fp16, B=8, H=8, Sq=Skv=2048, D=64, uniform
{0,1} key mask, dout ~ N(0,1).  The K timed steps are captured once as a CUDA
graph of the public API calls and replayed; `phase_ms` comes from a second,
directly launched pass with CUDA events between the calls.  FLOPs are counted as 4 B H Sq Skv D for the
forward and 2.5x that for the backward, so a step is 3.5 x 68.72 GFLOP.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Inputs are resident in HBM when the timed region
starts; four input sets (about 134 MB each, above the 129 MB L2) are rotated
so every step reads cold data.  The oracle (float64 NumPy) is timed on the
host cores on a bounded sample as the CPU baseline.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_attention_59_gb300 import dist as DIST  # noqa: E402
from exact_attention_59_gb300 import inputs as IN  # noqa: E402
from exact_attention_59_gb300 import workloads as W  # noqa: E402

WL = W.KEYPAD_FP16
DEC = W.CHECKERBOARD_DECODE_FP16
METRIC = "attention fwd+bwd TFLOP/s (fp16, B8 H8 S2048 D64, key-padding mask)"
UNIT = "TFLOP/s"


# DRAM bytes (read + write) of one bwd_dkdv_kernel launch at the bench workload, from
# `ncu --set full -k regex:bwd_dkdv -s 1 -c 1` of
# `python bench.py --mode profile --wl keypad --batch 8 --steps 2` (68.5 MB read,
# 9.5 MB written).  Set it back to None when the kernel changes until it is
# captured again.
DKDV_TRAFFIC_BYTES = 78.0e6

# Buffer sets of the end-to-end pipeline (device inputs and outputs, host
# outputs): step i's kernels wait for the download of step i - E2E_SETS.
E2E_SETS = 3


def counted_flops(w, backward=True):
    f = 4.0 * w.B * w.H * w.Sq * w.Skv * w.D * (0.5 if w.causal else 1.0)
    return f * (3.5 if backward else 1.0)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), d["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class Clocks:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=10):
        self.idx = gpu_index
        self.period_ms = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world):
    import exact_attention_59_gb300 as E
    from exact_attention_59_gb300 import build as BLD
    if rank == 0 or not os.path.exists(E.LIB_PATH):
        BLD.build()
    DIST.barrier()
    E.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = WL
    nsets = 4
    sets = []
    for i in range(nsets):
        c = IN.make_case(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, seed=IN.SEED + 1000 * rank + 17 * i,
                         with_key_mask=True)
        d = {k: v.to(dev) for k, v in c.items()}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
        d["dq"], d["dk"], d["dv"] = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]))
        sets.append(d)
    shape = E.make_shape(sets[0]["q"], sets[0]["k"])
    ws_f = E.workspace(E.OP_FWD, shape, dev)
    ws_b = E.workspace(E.OP_BWD, shape, dev)
    stream = torch.cuda.current_stream(dev)

    def step(d, ev=None):
        if ev is not None:
            ev[0].record(stream)
        E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], out=d["out"], lse=d["lse"], ws=ws_f)
        if ev is not None:
            ev[1].record(stream)
        E.attn_bwd_preprocess(d["q"], d["k"], d["out"], d["lse"], d["dout"], key_mask=d["key_mask"], ws=ws_b)
        if ev is not None:
            ev[2].record(stream)
        E.attn_bwd_dkdv(d["q"], d["k"], d["v"], d["dout"], d["dk"], d["dv"], key_mask=d["key_mask"], ws=ws_b)
        if ev is not None:
            ev[3].record(stream)
        E.attn_bwd_dq(d["q"], d["k"], d["v"], d["dout"], d["dq"], key_mask=d["key_mask"], ws=ws_b)
        if ev is not None:
            ev[4].record(stream)

    for i in range(args.warmup):
        step(sets[i % nsets])
    torch.cuda.synchronize()
    assert E.poll_status(ws_f) == 0 and E.poll_status(ws_b) == 0, "device-side timeout during warm-up"

    # The timed region replays a CUDA graph of the K steps: the same four launches
    # per step through the same API calls, captured once, so the host's launch
    # work (argument checks, tensor-map encoding, ctypes) stays off the timeline.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                step(sets[i % nsets])
    torch.cuda.synchronize()
    graph.replay()   # untimed: the first replay uploads the graph
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    DIST.barrier()
    torch.cuda.synchronize()
    # The clock sampler (every 10 ms) runs across the timed replay and the phase
    # pass that follows it (the same kernels launched directly), so its samples
    # see the GPU under this load even when the timed region itself is short.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    with Clocks(dev.index) as clk:
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        DIST.barrier()
        # per-kernel phase times: the same steps launched directly, CUDA events between the calls
        for i in range(args.steps):
            step(sets[i % nsets], evs[i])
        torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    ms = DIST.max_over_ranks(total_ms, device=dev) / args.steps   # the slowest rank sets the time
    assert E.poll_status(ws_f) == 0 and E.poll_status(ws_b) == 0, "device-side timeout in the timed region"
    ph = {n: [] for n in ("fwd", "pre", "dkdv", "dq")}
    for e in evs:
        for j, n in enumerate(ph):
            ph[n].append(e[j].elapsed_time(e[j + 1]))
    # each pass as a user issues it: K forwards back to back, then K backwards
    # (preprocess, dK/dV, dQ, overlapping under programmatic dependent launch),
    # events only around each run
    def fwd_only(d):
        E.attn_fwd(d["q"], d["k"], d["v"], key_mask=d["key_mask"], out=d["out"], lse=d["lse"], ws=ws_f)

    def bwd_only(d):
        E.attn_bwd_preprocess(d["q"], d["k"], d["out"], d["lse"], d["dout"], key_mask=d["key_mask"], ws=ws_b)
        E.attn_bwd_dkdv(d["q"], d["k"], d["v"], d["dout"], d["dk"], d["dv"], key_mask=d["key_mask"], ws=ws_b)
        E.attn_bwd_dq(d["q"], d["k"], d["v"], d["dout"], d["dq"], key_mask=d["key_mask"], ws=ws_b)

    chained = {}
    for name, fn in (("fwd", fwd_only), ("bwd", bwd_only)):
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        for i in range(args.steps):
            fn(sets[i % nsets])
        b_ev.record(stream)
        torch.cuda.synchronize()
        chained[name] = a_ev.elapsed_time(b_ev) / args.steps
    assert E.poll_status(ws_f) == 0 and E.poll_status(ws_b) == 0, "device-side timeout in the chained passes"

    # ---- decode (config: checkerboard fp16, q 8x8x1x64, K/V 8x8x2048x64), CUDA graph, rotating K/V
    dec = bench_decode(E, dev, args)

    # ---- end to end: pinned host buffers, copies inside the timed region; every
    # output comes back (and, as an extra figure, the run that reads back lse alone)
    e2e = bench_e2e(E, dev, args, w)
    e2e_lse = bench_e2e(E, dev, args, w, results=("lse",))

    # ---- the other named workloads, for context (outside the timed region)
    extras = None if args.no_extras else bench_extras(E, dev)

    res = {"ms": ms, "phases": {n: statistics.mean(v) for n, v in ph.items()}, "chained": chained,
           "clocks": clk.summary(),
           "decode": dec, "e2e": e2e, "e2e_lse": e2e_lse, "extras": extras}
    return res


def bench_decode(E, dev, args):
    w = DEC
    L2 = 129e6
    per = 2 * w.B * w.H * w.Skv * w.D * 2
    nsets = max(4, int(math.ceil(4 * L2 / per)))
    ks, vs = [], []
    q = IN.randn((w.B, w.H, 1, w.D), IN.SEED + 1, w.dtype).to(dev)
    for i in range(nsets):
        ks.append(IN.randn((w.B, w.H, w.Skv, w.D), IN.SEED + 3000 + i, w.dtype).to(dev))
        vs.append(IN.randn((w.B, w.H, w.Skv, w.D), IN.SEED + 5000 + i, w.dtype).to(dev))
    reps = nsets * 8

    def graph_us(call, ws):
        """Median time per call of `reps` calls captured in one CUDA graph, K/V rotating."""
        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(reps):
                    call(i)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) / reps)
        assert E.poll_status(ws) == 0
        return statistics.median(times) * 1e3

    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, 1), dtype=torch.float32, device=dev)
    ws = E.workspace(E.OP_DECODE, E.make_shape(q, ks[0]), dev)
    us = graph_us(lambda i: E.attn_decode(q, ks[i % nsets], vs[i % nsets], score_mod=w.score_mod, out=out, lse=lse,
                                          ws=ws), ws)
    res = {"workload": w.name, "us_per_call": us, "bytes_per_call": per + 2 * w.B * w.H * w.D * 2,
           "GB/s": (per + 2 * w.B * w.H * w.D * 2) / (us * 1e-6) / 1e9, "rotating_sets": nsets}
    # chunked decode: nq queries at the last nq positions of the same KV cache, causal
    # (speculative / chunked decoding); the K/V bytes bound it as for one query
    chunk = []
    for nq in (4, 16, 64):
        qc = IN.randn((w.B, w.H, nq, w.D), IN.SEED + 7 + nq, w.dtype).to(dev)
        oc = torch.empty_like(qc)
        lc = torch.empty((w.B, w.H, nq), dtype=torch.float32, device=dev)
        wsc = E.workspace(E.OP_DECODE_CHUNK, E.make_shape(qc, ks[0]), dev)
        usc = graph_us(lambda i: E.attn_decode_chunk(qc, ks[i % nsets], vs[i % nsets], w.Skv - nq, score_mod="causal",
                                                     out=oc, lse=lc, ws=wsc), wsc)
        byt = per + 2 * w.B * w.H * nq * w.D * 2
        chunk.append({"nq": nq, "us_per_call": usc, "GB/s": byt / (usc * 1e-6) / 1e9})
    res["chunk_causal_fp16_b8h8kv2048d64"] = chunk
    return res


E2E_ALL = ("out", "lse", "dq", "dk", "dv")


def bench_e2e(E, dev, args, w, results=E2E_ALL):
    """fwd+bwd through the public API with host buffers: every step copies its inputs
    (q, k, v, dout, key mask) from pinned host memory into the device and reads
    back the step's `results` (by default every output: out, lse, dq, dk, dv)
    into pinned host memory, inside the timed region.  Copies run on their own
    streams over E2E_SETS buffer sets, so step i+1's upload and step i-1's
    download overlap step i's kernels (as a training input pipeline would), and
    step i's kernels wait only for the download of step i - E2E_SETS."""
    hosts = []
    for j in range(2):
        c = IN.make_case(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, seed=IN.SEED + 7000 + j, with_key_mask=True)
        hosts.append({k: v.pin_memory() for k, v in c.items()})
    shapes = {"out": hosts[0]["q"].shape, "lse": hosts[0]["q"].shape[:3], "dq": hosts[0]["q"].shape,
              "dk": hosts[0]["k"].shape, "dv": hosts[0]["v"].shape}
    dts = {n: (torch.float32 if n == "lse" else hosts[0]["q"].dtype) for n in shapes}
    outs_h = [{n: torch.empty(shapes[n], dtype=dts[n]).pin_memory() for n in results} for _ in range(E2E_SETS)]
    ins_d = [{k: torch.empty_like(v, device=dev) for k, v in hosts[0].items()} for _ in range(E2E_SETS)]
    outs_d = [{"lse": torch.empty(hosts[0]["q"].shape[:3], dtype=torch.float32, device=dev),
               "out": torch.empty_like(hosts[0]["q"], device=dev), "dq": torch.empty_like(hosts[0]["q"], device=dev),
               "dk": torch.empty_like(hosts[0]["k"], device=dev), "dv": torch.empty_like(hosts[0]["v"], device=dev)}
              for _ in range(E2E_SETS)]
    shape = E.make_shape(ins_d[0]["q"], ins_d[0]["k"])
    ws_f = E.workspace(E.OP_FWD, shape, dev)
    ws_b = E.workspace(E.OP_BWD, shape, dev)
    s_up, s_cmp, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def compute(j):
        di, do = ins_d[j], outs_d[j]
        E.attn_fwd(di["q"], di["k"], di["v"], key_mask=di["key_mask"], out=do["out"], lse=do["lse"], ws=ws_f)
        E.attn_bwd(di["q"], di["k"], di["v"], do["out"], do["lse"], di["dout"], key_mask=di["key_mask"],
                   dq=do["dq"], dk=do["dk"], dv=do["dv"], ws=ws_b)
    # the kernels of one step on buffer set j, captured once as a CUDA graph
    # (the same API calls; the copies stay outside, on their own streams)
    with torch.cuda.stream(s_cmp):
        for j in range(E2E_SETS):
            compute(j)
    torch.cuda.synchronize()
    graphs = [torch.cuda.CUDAGraph() for _ in range(E2E_SETS)]
    for j in range(E2E_SETS):
        with torch.cuda.stream(s_cmp):
            with torch.cuda.graph(graphs[j], stream=s_cmp):
                compute(j)
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event()
    up_done, cmp_done, down_done = ([ev() for _ in range(E2E_SETS)] for _ in range(3))
    first = [True] * E2E_SETS

    def step(i):
        j = i % E2E_SETS
        di, do, hi, ho = ins_d[j], outs_d[j], hosts[i % 2], outs_h[j]
        with torch.cuda.stream(s_up):
            if not first[j]:
                s_up.wait_event(cmp_done[j])          # step i - E2E_SETS has finished reading these inputs
            for k in di:
                di[k].copy_(hi[k], non_blocking=True)
            up_done[j].record(s_up)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(up_done[j])
            if not first[j]:
                s_cmp.wait_event(down_done[j])        # step i - E2E_SETS's results have left these buffers
            graphs[j].replay()
            cmp_done[j].record(s_cmp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(cmp_done[j])
            for k in ho:
                ho[k].copy_(do[k], non_blocking=True)
            down_done[j].record(s_down)
        first[j] = False

    for i in range(2 * E2E_SETS):
        step(i)
    torch.cuda.synchronize()
    n = max(2 * E2E_SETS, min(args.steps, 40))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(n):
        step(i)
    s_down.wait_stream(s_up)
    s_down.wait_stream(s_cmp)
    b.record(s_down)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    assert E.poll_status(ws_f) == 0 and E.poll_status(ws_b) == 0
    h2d = sum(v.numel() * v.element_size() for v in hosts[0].values())
    d2h = sum(v.numel() * v.element_size() for v in outs_h[0].values())
    return {"ms": ms, "h2d": h2d, "d2h": d2h, "results": list(results),
            "pipeline": f"{E2E_SETS} buffer sets, copies on separate streams, kernels replayed as a CUDA graph; "
                        f"read back: {', '.join(results)}"}


def bench_extras(E, dev):
    """Context timings of the other named workloads (not part of `value`): forward and
    backward per call, CUDA events over repeated calls on two rotating input sets."""
    res = {}

    def timed(fn, n):
        fn(0)
        fn(1)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n):
            fn(i)
        b.record()
        torch.cuda.synchronize()
        # a wait that ran out inside the kernels would make this a time-out, not a timing
        code = E.poll_status_all(dev)
        assert code == E.ATTN_OK, f"device-side status {code} ({E.status_string(code)}) in a context timing"
        return a.elapsed_time(b) / n

    for w in (W.FLEX_CAUSAL_ALIBI_BF16, W.CHECKERBOARD_FP16):
        sets = []
        for i in range(2):
            c = IN.make_case(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, seed=IN.SEED + 9000 + i, dout=w.dout)
            d = {k: v.to(dev) for k, v in c.items() if v is not None}
            d["out"] = torch.empty_like(d["q"])
            d["lse"] = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
            d["dq"], d["dk"], d["dv"] = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
            sets.append(d)
        bm = E.create_block_mask(w.block_mask, 1, 1, w.Sq, w.Skv) if w.block_mask else None
        mod = w.score_mod

        def fwd(i, sets=sets, bm=bm, mod=mod):
            d = sets[i % 2]
            E.attn_fwd(d["q"], d["k"], d["v"], block_mask=bm, score_mod=mod, out=d["out"], lse=d["lse"])

        def bwd(i, sets=sets, bm=bm, mod=mod):
            d = sets[i % 2]
            E.attn_bwd(d["q"], d["k"], d["v"], d["out"], d["lse"], d["dout"], block_mask=bm, score_mod=mod,
                       dq=d["dq"], dk=d["dk"], dv=d["dv"])

        f_ms = timed(fwd, 50)
        b_ms = timed(bwd, 50)
        half = 0.5 if w.causal else 1.0
        f_fl = 4.0 * w.B * w.H * w.Sq * w.Skv * w.D * half
        res[w.name] = {"fwd_ms": f_ms, "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12, "bwd_ms": b_ms,
                       "bwd_tflops": 2.5 * f_fl / (b_ms * 1e-3) / 1e12}
    # dense (query, key) mask: a sliding window |q - k| < 256 shared by every head,
    # on the key-padding workload's shape (fp16, B8 H8 S2048 D64); tiles with no
    # kept pair are skipped, so the rate is quoted over kept pairs and visited tiles
    w = WL
    S, win = w.Sq, 256
    sets = []
    for i in range(2):
        c = IN.make_case(w.B, w.H, S, S, w.D, w.dtype, seed=IN.SEED + 9100 + i)
        d = {k: v.to(dev) for k, v in c.items() if v is not None}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
        d["dq"], d["dk"], d["dv"] = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
        sets.append(d)
    qi = torch.arange(S, device=dev)[:, None]
    mask = ((qi - torch.arange(S, device=dev)[None, :]).abs() < win).to(torch.uint8)[None, None]
    p_ms = timed(lambda i: E.pack_dense_mask(mask, w.B, w.H), 5)
    dm = E.pack_dense_mask(mask, w.B, w.H)

    def dfwd(i):
        d = sets[i % 2]
        E.attn_fwd(d["q"], d["k"], d["v"], dense_mask=dm, out=d["out"], lse=d["lse"])

    def dbwd(i):
        d = sets[i % 2]
        E.attn_bwd(d["q"], d["k"], d["v"], d["out"], d["lse"], d["dout"], dense_mask=dm, dq=d["dq"], dk=d["dk"],
                   dv=d["dv"])

    f_ms = timed(dfwd, 50)
    b_ms = timed(dbwd, 50)
    kept = int(mask.sum().item()) * w.B * w.H
    nt = -(-S // 128)
    vt = sum(1 for a in range(nt) for b in range(nt) if abs(a - b) * 128 < win + 127) * w.B * w.H
    f_kept = 4.0 * w.D * kept
    f_vis = 4.0 * w.D * vt * 128 * 128
    res[f"window{win}_dense_fp16_b8h8s2048d64"] = {
        "pack_ms": p_ms, "fwd_ms": f_ms, "bwd_ms": b_ms, "kept_pairs": kept, "visited_tiles": vt,
        "fwd_tflops_kept": f_kept / (f_ms * 1e-3) / 1e12, "fwd_tflops_visited": f_vis / (f_ms * 1e-3) / 1e12,
        "bwd_tflops_visited": 2.5 * f_vis / (b_ms * 1e-3) / 1e12}
    # a score_mod compiled at run time: a relative-position bias on the same shape
    try:
        um = E.compile_score_mod("0.05f * (float)(kv - q)", dtype=torch.float16)

        def ufwd(i):
            d = sets[i % 2]
            E.attn_fwd(d["q"], d["k"], d["v"], score_mod=um, out=d["out"], lse=d["lse"])

        def ubwd(i):
            d = sets[i % 2]
            E.attn_bwd(d["q"], d["k"], d["v"], d["out"], d["lse"], d["dout"], score_mod=um, dq=d["dq"], dk=d["dk"],
                       dv=d["dv"])
        f_ms, b_ms = timed(ufwd, 50), timed(ubwd, 50)
        f_fl = 4.0 * w.D * S * S * w.B * w.H
        res["user_relative_bias_fp16_b8h8s2048d64"] = {
            "expr": um.bias_expr, "fwd_ms": f_ms, "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12, "bwd_ms": b_ms,
            "bwd_tflops": 2.5 * f_fl / (b_ms * 1e-3) / 1e12}
    except Exception as e:   # noqa: BLE001 - context only: report, do not fail the bench
        res["user_relative_bias_fp16_b8h8s2048d64"] = {"error": str(e)[:300]}
    w = W.LONG_CAUSAL_BF16
    q = IN.randn((w.B, w.H, w.Sq, w.D), IN.SEED + 1, w.dtype).to(dev)
    k = IN.randn((w.B, w.H, w.Skv, w.D), IN.SEED, w.dtype).to(dev)
    v = IN.randn((w.B, w.H, w.Skv, w.D), IN.SEED + 2, w.dtype).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    bm = E.create_block_mask("causal", 1, 1, w.Sq, w.Skv)
    f_ms = timed(lambda i: E.attn_fwd(q, k, v, block_mask=bm, out=out, lse=lse), 3)
    f_fl = 4.0 * w.B * w.H * w.Sq * w.Skv * w.D * 0.5
    res[w.name] = {"fwd_ms": f_ms, "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12}
    return res


# ------------------------------------------------------------------ oracle (CPU) legs
def oracle_case():
    """The bench workload's inputs as float64 arrays, built once (outside any timing)."""
    import numpy as np  # noqa: F401
    w = WL
    c = IN.make_case(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, with_key_mask=True)
    q, k, v, do = (c[n].float().double().numpy() for n in ("q", "k", "v", "dout"))
    return {"q": q, "k": k, "v": v, "dout": do, "key_mask": c["key_mask"].numpy()}


def oracle_head(case, idx):
    """The oracle's forward and backward of head `idx` (b = idx // H, h = idx % H)."""
    import oracle.attention as OR
    b, h = divmod(idx % (WL.B * WL.H), WL.H)
    OR.attn_fwd(case["q"], case["k"], case["v"], key_mask=case["key_mask"], heads=[(b, h)])
    OR.attn_bwd(case["q"], case["k"], case["v"], case["dout"], key_mask=case["key_mask"], heads=[(b, h)])


def oracle_sample(case, seconds=12.0, max_heads=64):
    """Times the oracle's fwd+bwd on whole heads of the workload until `seconds` pass."""
    done, t0 = 0, time.perf_counter()
    while done < max_heads:
        oracle_head(case, done)
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * WL.Sq * WL.Skv * WL.D * done
    return flops / dt / 1e12, done, dt


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return None


def host_cores():
    """Threads the oracle's BLAS uses (its `cores`) and the host's CPU count, separately."""
    bt = blas_threads()
    return {"cores": bt if bt is not None else os.cpu_count(), "blas_threads": bt, "host_cpus": os.cpu_count()}


def cpu_baseline(seconds=12.0):
    case = oracle_case()
    v, heads, dt = oracle_sample(case, seconds)
    return {"value": v, "unit": UNIT, **host_cores(), "kind": "oracle",
            "sample": f"float64 NumPy fwd+bwd of {heads} of {WL.B * WL.H} (b,h) heads of the workload in {dt:.1f} s "
                      "(inputs built before the timing)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    case = oracle_case()   # inputs once, outside the timed steps
    for i in range(args.warmup):
        oracle_head(case, i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_head(case, i)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    val = 3.5 * 4.0 * WL.Sq * WL.Skv * WL.D / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": val, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WL.name, "B": WL.B, "H": WL.H, "Sq": WL.Sq, "Skv": WL.Skv, "D": WL.D,
                       "step": "oracle fwd+bwd of one (b, h) head per step (bounded sample)"},
            "cpu_baseline": {"value": val, "unit": UNIT, **host_cores(), "kind": "oracle",
                             "sample": "one (b, h) head of the workload per step, float64 NumPy, inputs built once "
                                       "before the timed steps"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """A few untimed fwd+bwd steps of the workload at batch `--batch`, for ncu captures."""
    import exact_attention_59_gb300 as E
    from exact_attention_59_gb300 import build as BLD
    BLD.build()
    E.load()
    dev = torch.device("cuda", 0)
    w = {"keypad": WL, "checkerboard": W.CHECKERBOARD_FP16, "causal_alibi": W.FLEX_CAUSAL_ALIBI_BF16}[args.wl]
    c = IN.make_case(args.batch, w.H, w.Sq, w.Skv, w.D, w.dtype, with_key_mask=w.key_mask, dout=w.dout)
    d = {k: v.to(dev) for k, v in c.items() if v is not None}
    km = d.get("key_mask")
    bm = E.create_block_mask(w.block_mask, 1, 1, w.Sq, w.Skv) if w.block_mask else None
    for _ in range(args.steps):
        out, lse = E.attn_fwd(d["q"], d["k"], d["v"], key_mask=km, block_mask=bm, score_mod=w.score_mod)
        E.attn_bwd(d["q"], d["k"], d["v"], out, lse, d["dout"], key_mask=km, block_mask=bm, score_mod=w.score_mod)
    if args.d512:
        S = args.d512
        q = IN.randn((1, 2, S, 512), IN.SEED + 1, "bf16").to(dev)
        k = IN.randn((1, 2, S, 512), IN.SEED, "bf16").to(dev)
        v = IN.randn((1, 2, S, 512), IN.SEED + 2, "bf16").to(dev)
        bm = E.create_block_mask("causal", 1, 1, S, S)
        for _ in range(args.steps):
            E.attn_fwd(q, k, v, block_mask=bm)
    if args.decode:
        dw = DEC
        q = IN.randn((args.batch, dw.H, 1, dw.D), IN.SEED + 1, dw.dtype).to(dev)
        k = IN.randn((args.batch, dw.H, dw.Skv, dw.D), IN.SEED, dw.dtype).to(dev)
        v = IN.randn((args.batch, dw.H, dw.Skv, dw.D), IN.SEED + 2, dw.dtype).to(dev)
        for _ in range(args.steps):
            E.attn_decode(q, k, v, score_mod=dw.score_mod)
    torch.cuda.synchronize()
    ws = E.workspace(E.OP_FWD, E.make_shape(d["q"], d["k"]), dev)
    assert E.poll_status(ws) == 0
    print(json.dumps({"mode": "profile", "batch": args.batch, "steps": args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads' context timings")
    ap.add_argument("--mode", choices=["bench", "profile"], default="bench",
                    help="profile: a few untimed steps at --batch, for ncu captures")
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--wl", choices=["keypad", "checkerboard", "causal_alibi"], default="keypad",
                    help="profile mode: the workload whose fwd+bwd runs (at --batch)")
    ap.add_argument("--decode", action="store_true", help="profile mode: also run decode at --batch")
    ap.add_argument("--d512", type=int, default=0,
                    help="profile mode: also run the causal 1 x 2 x S x S x 512 bf16 forward at this S")
    args = ap.parse_args()
    if args.mode == "profile":
        run_profile_case(args)
        return
    args.warmup = max(3, args.warmup)
    rank, world = DIST.world()
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        DIST.init("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        res = run_ours(args, rank, world)
        if rank != 0:
            return
        fl = counted_flops(WL)
        value = fl * world / (res["ms"] * 1e-3) / 1e12
        burst, sustained, hbm, src = peaks()
        ph = res["phases"]
        # dominant kernel: the longest phase
        dk_ms = ph["dkdv"]
        dkdv_flops = 8.0 * WL.B * WL.H * WL.Sq * WL.Skv * WL.D
        achieved = dkdv_flops / (dk_ms * 1e-3) / 1e12
        dec = res["decode"]
        e2e = res["e2e"]
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WL.name, "B": WL.B, "H": WL.H, "Sq": WL.Sq, "Skv": WL.Skv, "D": WL.D,
                       "key_mask": "uniform {0,1}", "l2": "4 rotating input sets of 134 MB (> 129 MB L2)",
                       "launch": "timed steps replayed as one CUDA graph of the API calls",
                       "parallelism": f"replicas x{world}"},
            "fwd_tflops": 4.0 * WL.B * WL.H * WL.Sq * WL.Skv * WL.D / (ph["fwd"] * 1e-3) / 1e12,
            "bwd_tflops": 10.0 * WL.B * WL.H * WL.Sq * WL.Skv * WL.D / ((ph["pre"] + ph["dkdv"] + ph["dq"]) * 1e-3)
            / 1e12,
            "phase_ms": ph,
            # each pass timed over K back-to-back calls (the backward's three launches
            # overlapping as in the step), events only around the run
            "chained": {"fwd_ms": res["chained"]["fwd"], "bwd_ms": res["chained"]["bwd"],
                        "fwd_tflops": 4.0 * WL.B * WL.H * WL.Sq * WL.Skv * WL.D / (res["chained"]["fwd"] * 1e-3)
                        / 1e12,
                        "bwd_tflops": 10.0 * WL.B * WL.H * WL.Sq * WL.Skv * WL.D / (res["chained"]["bwd"] * 1e-3)
                        / 1e12},
            "frac_of_peak": {"burst": value / burst, "sustained": value / sustained, "peak_source": src},
            "decode": {"workload": dec["workload"], "us_per_call": dec["us_per_call"], "GB/s": dec["GB/s"],
                       "frac_of_hbm": dec["GB/s"] / hbm,
                       "chunk_causal_fp16_b8h8kv2048d64": [dict(c, frac_of_hbm=c["GB/s"] / hbm)
                                                           for c in dec["chunk_causal_fp16_b8h8kv2048d64"]]},
            "roofline": {"kernel": "bwd_dkdv_kernel", "bound": "tensor", "achieved": achieved, "peak": burst,
                         "unit": "TFLOP/s", "frac": achieved / burst, "traffic": DKDV_TRAFFIC_BYTES,
                         "peak_kind": f"bf16 burst, {src} (the kernel is timed in a ms-scale region)",
                         "frac_of_sustained": achieved / sustained},
            "e2e": {"value": fl / (e2e["ms"] * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                    "d2h_bytes_per_step": e2e["d2h"], "pipeline": e2e["pipeline"]},
            "e2e_lse_only": {"value": fl / (res["e2e_lse"]["ms"] * 1e-3) / 1e12, "unit": UNIT,
                             "h2d_bytes_per_step": res["e2e_lse"]["h2d"],
                             "d2h_bytes_per_step": res["e2e_lse"]["d2h"],
                             "pipeline": res["e2e_lse"]["pipeline"]},
            # per step: forward (reads the byte key mask itself), preprocess (packs the
            # key mask for the backward), dK/dV, dQ
            "gpu_launches": 4 * args.steps,
            "clocks": res["clocks"],
        }
        if res["extras"] is not None:
            line["extras"] = res["extras"]
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark: mixed-format (FP8 / TQ3) paged decode attention on GB300.

One step = one decode step of the whole hot path over the workload's batch:
extend every request by one token (page-table bookkeeping), demote pages
that left the Recent window (FP8 -> TQ3 kernel), then for each of the 16
layers append the new K/V token (FP8 quantise kernel) and run mixed-format
decode attention (partial-attention kernel + LSE merge kernel).

value       = algorithmic KV bytes read by decode attention / timed seconds
              (inputs resident in HBM; the per-layer working set cycled over
              16 layers exceeds L2).
e2e         = the same metric with each step's q/k/v copied from pinned host
              memory and out/lse copied back inside the timed region.
roofline    = the partial-attention kernel alone, timed per launch with CUDA
              events on its stream, against the measured HBM copy bandwidth.
cpu_baseline = the CPU oracle (fp64 numpy) on a bounded sample, host cores.

Multi-GPU: every rank runs an independent replica of the batch (requests
are independent; no collective on the data path); value sums all ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s read & ctx-tokens/s per layer; fraction of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
ROW_BYTES = {"fp8": 2 * (256 + 2), "tq3": 2 * (96 + 2)}   # K+V bytes per token per kv head


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mkv", "reference"], default="mkv")
    ap.add_argument("--workload", default="cfg5",
                    help="cfg5 (16 x 131K tokens, the largest single-GPU workload) by default; cfg1..cfg4")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-full", action="store_true",
                    help="also time the oracle over a full layer-step (every request and kv head of layer 0); "
                         "minutes on the larger workloads, so off by default")
    ap.add_argument("--requests", default=None,
                    help="comma-separated request indices: run a reduced-size slice of the workload "
                         "(same shapes; e.g. for a profiler capture)")
    ap.add_argument("--graph", action="store_true",
                    help="run each step as one recorded CUDA graph over all layers (mkv_step_graph_*): a "
                         "separate line, on fixed input buffers filled by one copy per step")
    ap.add_argument("--nq", type=int, default=1,
                    help="query tokens per request and step (> 1: the multi-query path, a separate line)")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers
def make_workload(args):
    from mixed_format_paged_gb300 import workloads
    w = workloads.make(args.workload)
    if args.requests:
        w = w.subset([int(x) for x in args.requests.split(",")])
    return w


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def kernel_source_hash():
    """Hash of the decode kernel's source with comments and blank lines
    removed, so that a comment-only edit keeps committed counters valid."""
    import re
    h = hashlib.sha256()
    for f in ("mkv_kernels.cu", "mkv_internal.h"):
        with open(os.path.join(ROOT, "mixed_format_paged_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        lines = [ln.rstrip() for ln in src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload, alg_bytes_per_launch):
    """Per-launch DRAM bytes (read + write) of the partial-attention kernel
    from the committed ncu summary, only if it was taken on the current
    kernel source.  A capture of the full workload gives them directly; a
    capture of a reduced-size slice of the same shape gives DRAM bytes per
    algorithmic byte, scaled here by the launch's algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    if "dram_bytes_per_launch" in e:
        return e["dram_bytes_per_launch"]
    return e["dram_bytes_per_alg_byte"] * alg_bytes_per_launch


class ClockSampler:
    """nvidia-smi clock and throttle samples (every 10 ms, timestamped).  Start
    it before the warm-up; `stop(t0, t1)` keeps the samples taken inside the
    timed region [t0, t1] (host wall clock), padded by one sampling period."""

    PERIOD_S = 0.010

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                       "-lms", str(int(self.PERIOD_S * 1000)), "-i", str(gpu_index)],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self, t0: float, t1: float):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = []
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.f.name)
        pad = self.PERIOD_S
        inside = [r for r in rows if t0 - pad <= r[0] <= t1 + pad]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "window_ms": round((t1 - t0) * 1e3, 2), "period_ms": int(self.PERIOD_S * 1000)}


def job_totals(local_ms: float, local_bytes: float, world: int, device=None):
    """Whole-job figures over ranks: the slowest rank's time and the bytes of
    all ranks (each rank runs an independent replica)."""
    if world <= 1:
        return local_ms, local_bytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def kv_bytes_now(pool, P, L):
    """Algorithmic KV bytes one decode pass over every live sequence reads, all
    layers: every valid token once per kv head, K and V, at its tier's size."""
    st = pool.stats()
    tq3_tok = st.stale_pages * P
    fp8_tok = st.live_tokens - tq3_tok
    per_layer = pool.num_kv_heads * (fp8_tok * ROW_BYTES["fp8"] + tq3_tok * ROW_BYTES["tq3"])
    return L * per_layer, st.live_tokens


# ----------------------------------------------------------------- CPU oracle sample
def oracle_sample(w, pages_by_req, seconds: float):
    """Time the oracle's streaming decode over (request, kv head) samples until
    `seconds` have passed.  Returns (GB/s, bytes, seconds, description)."""
    import numpy as np
    from oracle.paged import TIER_STALE, decode_attention_streaming
    t0 = time.perf_counter()
    nbytes = 0
    done = []
    rng = np.random.default_rng(0)
    reqs = list(pages_by_req)
    i = 0
    while time.perf_counter() - t0 < seconds and i < 64:
        r = reqs[i % len(reqs)]
        kvh = int(rng.integers(0, w.Hkv))
        pages = pages_by_req[r]
        q = np.asarray(rng.standard_normal((w.Hq, w.D)))
        decode_attention_streaming(q, pages, w.P, w.Hkv, w.D, 99, kv_heads=[kvh])
        for t, _, n in pages:
            nbytes += n * (ROW_BYTES["tq3"] if t == TIER_STALE else ROW_BYTES["fp8"])
        done.append((r, kvh))
        i += 1
    dt = time.perf_counter() - t0
    desc = (f"oracle streaming decode (fp64 numpy) of {len(done)} (request, kv head) pairs of workload "
            f"{w.name}, layer 0, {sum(len(pages_by_req[r]) for r, _ in done)} pages")
    return nbytes / dt / 1e9, nbytes, dt, desc


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count()


def oracle_layer_step(w, pages_by_req, q):
    """Time the oracle's streaming decode over every (request, kv head) of one
    layer: one full layer-step.  q: [n, Hq, D] (the GPU step's query).
    Returns (GB/s, bytes, seconds)."""
    import numpy as np
    from oracle.paged import TIER_STALE, decode_attention_streaming
    t0 = time.perf_counter()
    nbytes = 0
    for r, pages in pages_by_req.items():
        decode_attention_streaming(np.asarray(q[r], dtype=np.float64), pages, w.P, w.Hkv, w.D, 99)
        for t, _, n in pages:
            nbytes += w.Hkv * n * (ROW_BYTES["tq3"] if t == TIER_STALE else ROW_BYTES["fp8"])
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, nbytes, dt


# ----------------------------------------------------------------- reference arm
def run_reference(args):
    """Time the CPU oracle, as it stands, on the same workload: each step is a
    bounded sample (one request's layer-0 pages, one kv head), its pages built
    by the oracle's own encoders from the workload's inputs."""
    import numpy as np
    import torch

    from mixed_format_paged_gb300 import workloads
    from oracle.paged import TIER_STALE, decode_attention_streaming, demote_page, encode_fp8_page
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = make_workload(args)
    r = 0
    K, V = w.prefill_kv(0, r, device="cpu")
    K = K.float().numpy()
    V = V.float().numpy()
    npg = w.npages(r)
    max_pages = 48
    pages = []
    for p in range(max(0, npg - max_pages), npg):
        nv = min(w.P, w.lengths[r] - p * w.P)
        pg = encode_fp8_page(K[p * w.P:p * w.P + nv], V[p * w.P:p * w.P + nv], w.P)
        t = w.tier(r, p)
        if t == TIER_STALE:
            pg = demote_page(pg, w.P, w.Hkv, w.D, 99)[0]
        pages.append((t, pg, nv))
    step_bytes = sum(n * (ROW_BYTES["tq3"] if t == TIER_STALE else ROW_BYTES["fp8"]) for t, _, n in pages)
    q = np.random.default_rng(0).standard_normal((w.Hq, w.D))
    for _ in range(args.warmup):
        decode_attention_streaming(q, pages, w.P, w.Hkv, w.D, 99, kv_heads=[0])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        decode_attention_streaming(q, pages, w.P, w.Hkv, w.D, 99, kv_heads=[0])
    dt = time.perf_counter() - t0
    gbs = step_bytes * args.steps / dt / 1e9
    sample = (f"oracle streaming decode of request 0, layer 0, kv head 0, last {len(pages)} pages "
              f"({step_bytes} KV bytes) of workload {w.name}, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "sample": sample},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm
def run_mkv(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from mixed_format_paged_gb300 import binding as B
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import Stepper, make_pool, prefill

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    w = make_workload(args)
    L, P = w.num_layers, w.P
    e2e_steps = 0 if args.no_e2e else args.steps
    total_steps = args.warmup + args.steps + e2e_steps
    pool = make_pool(w, device=dev, extra_steps=total_steps + 1, seed=99)
    prefill(pool, w, device=dev)
    torch.cuda.synchronize()
    stepper = Stepper(pool, w, device=dev)
    # per-step inputs, resident on the device before the timed region
    ins = []
    for s in range(args.warmup + args.steps):
        row = []
        for layer in range(L):
            k, v = w.step_kv(layer, s, device=dev)
            row.append((k, v, w.query(layer, s, device=dev)))
        ins.append(row)
    outs = [(torch.empty((w.n, w.Hq, w.D), device=dev), torch.empty((w.n, w.Hq), device=dev)) for _ in range(L)]
    demotes = [0]
    demote_events = []                # (start, stop) CUDA events of the timed region's demotions
    timing_demotes = [False]
    orig_demote = pool.demote

    def counting_demote(*a, **kw):
        demotes[0] += 1
        if not timing_demotes[0]:
            return orig_demote(*a, **kw)
        e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        e[0].record()
        r = orig_demote(*a, **kw)
        e[1].record()
        demote_events.append(e)
        return r
    pool.demote = counting_demote

    # The decode kernel is timed on the last layer of every timed step: events
    # recorded between it and the merge kernel stop the merge from launching
    # ahead of it (programmatic dependent launch), so timing all layers would
    # slow the step that `value` measures.  Every layer's decode has the same
    # shape, so the last layer's launches stand for all of them.
    TIMED_LAYER = L - 1

    graph = [None]
    if args.graph:
        # every step's inputs (all layers' q, k, v) packed in one device
        # buffer; the graph reads fixed views of `gbuf`, filled by one copy
        def nbytes(t):
            return t.numel() * t.element_size()
        seg = lambda nb: (nb + 255) // 256 * 256
        k0, v0, q0 = ins[0][0]
        lay = seg(nbytes(q0)) + seg(nbytes(k0)) + seg(nbytes(v0))
        packed = []
        for srow in ins:
            buf = torch.empty(L * lay, dtype=torch.uint8, device=dev)
            for layer, (k, v, q) in enumerate(srow):
                off = layer * lay
                for t in (q, k, v):
                    buf[off:off + nbytes(t)].copy_(t.contiguous().view(torch.uint8).reshape(-1))
                    off += seg(nbytes(t))
            packed.append(buf)
        gbuf = torch.empty(L * lay, dtype=torch.uint8, device=dev)
        gviews = []
        for layer in range(L):
            off = layer * lay
            gq = gbuf[off:off + nbytes(q0)].view(q0.dtype).view(q0.shape)
            off += seg(nbytes(q0))
            gk = gbuf[off:off + nbytes(k0)].view(k0.dtype).view(k0.shape)
            off += seg(nbytes(k0))
            gv = gbuf[off:off + nbytes(v0)].view(v0.dtype).view(v0.shape)
            gviews.append((gq, gk, gv))

    def step(s, ev_pair=None, bytes_acc=None):
        stepper.pre_step()
        if bytes_acc is not None:
            bytes_acc.append(kv_bytes_now(pool, P, L))
        if args.graph:
            gbuf.copy_(packed[s])
            if graph[0] is None:
                graph[0] = pool.step_graph(stepper.ids, [x[0] for x in gviews], [o for o, _ in outs],
                                           [l_ for _, l_ in outs], k=[x[1] for x in gviews], v=[x[2] for x in gviews])
            graph[0].launch()
            return
        for layer in range(L):
            k, v, q = ins[s][layer]
            if ev_pair is not None and layer == TIMED_LAYER:
                B.mkv_set_timing_events(pool.handle, *ev_pair)
            stepper.layer(layer, k, v, q, *outs[layer])

    # clocks are sampled from before the warm-up on; only samples inside the
    # timed region count (nvidia-smi takes a while to start)
    sampler = ClockSampler(local)
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    pool.check_device_errors()
    # ---------------- timed region (device-resident inputs)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:                  # torch creates the CUDA event on first record
        a.record()
        b.record()
    bytes_acc = []
    barrier()
    torch.cuda.synchronize()
    demotes[0] = 0
    timing_demotes[0] = True
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record()
    for i in range(args.steps):
        step(args.warmup + i, ev[i], bytes_acc)
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    timing_demotes[0] = False
    barrier()
    clocks = sampler.stop(t_wall0, t_wall1)
    demote_ms = [a.elapsed_time(b) for a, b in demote_events]
    pool.check_device_errors()
    ms = e0.elapsed_time(e1)
    timed_demotes = demotes[0]
    kv_total = sum(b for b, _ in bytes_acc)
    t_max, kv_job = job_totals(ms, kv_total, world, dev)
    ctx_total = sum(c for _, c in bytes_acc)
    kernel_bytes = [b / L for b, _ in bytes_acc]
    if args.graph:
        # no events can sit between the kernels of a graph: the whole step's
        # time per layer stands in for the decode kernel's (an upper bound)
        kernel_ms = [ms / args.steps / L] * args.steps
    else:
        kernel_ms = [a.elapsed_time(b) for a, b in ev]
    achieved = (sum(kernel_bytes) / len(kernel_bytes)) / (sum(kernel_ms) / len(kernel_ms) * 1e-3) / 1e9
    peak, peak_src = measured_peaks()
    # per layer and step: the decode kernel (with the fused append) and the merge
    gpu_launches = args.steps * L * 2 + timed_demotes
    # ---------------- e2e through host buffers
    e2e = None
    if e2e_steps:
        # Each step's inputs (q, k, v of every layer) sit in one pinned host
        # buffer and go to the device in one copy at the start of the step;
        # the step's result, the last layer's out and lse, comes back at its
        # end.  Segments are 256-byte aligned so that typed views of the byte
        # buffer are legal.
        elt = lambda dt: torch.tensor([], dtype=dt).element_size()
        qb = w.n * w.Hq * w.D * elt(w.q_dtype)
        kb = w.n * w.Hkv * w.D * elt(w.kv_dtype)
        seg = lambda nb: (nb + 255) // 256 * 256
        layer_bytes = seg(qb) + 2 * seg(kb)
        hbuf = [torch.empty(L * layer_bytes, dtype=torch.uint8).pin_memory() for _ in range(e2e_steps)]
        for s in range(e2e_steps):
            for layer in range(L):
                k, v = w.step_kv(layer, 10_000 + s)
                q = w.query(layer, 10_000 + s)
                off = layer * layer_bytes
                for t, nb in ((q, qb), (k, kb), (v, kb)):
                    hbuf[s][off:off + nb].copy_(t.contiguous().view(torch.uint8).reshape(-1))
                    off += seg(nb)
        # two device input buffers: step s + 1's copy (on a copy stream) runs
        # while step s computes, as a serving loop would stage its inputs
        dbufs = [torch.empty(L * layer_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        views = []
        for dbuf in dbufs:
            vb = []
            for layer in range(L):
                off = layer * layer_bytes
                dq = dbuf[off:off + qb].view(w.q_dtype).view(w.n, w.Hq, w.D)
                dk = dbuf[off + seg(qb):off + seg(qb) + kb].view(w.kv_dtype).view(w.n, w.Hkv, w.D)
                off2 = off + seg(qb) + seg(kb)
                dv = dbuf[off2:off2 + kb].view(w.kv_dtype).view(w.n, w.Hkv, w.D)
                vb.append((dq, dk, dv))
            views.append(vb)
        ho = torch.empty((w.n, w.Hq, w.D), dtype=torch.float32).pin_memory()
        hl = torch.empty((w.n, w.Hq), dtype=torch.float32).pin_memory()
        e2e_bytes = []
        comp = torch.cuda.current_stream()
        copy_stream = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]      # buffer i holds its step's inputs
        ev_free = [torch.cuda.Event() for _ in range(2)]    # buffer i's previous step is done with it
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(comp)

        def stage(s):
            i = s % 2
            copy_stream.wait_event(f0 if s < 2 else ev_free[i])
            with torch.cuda.stream(copy_stream):
                dbufs[i].copy_(hbuf[s], non_blocking=True)
            ev_in[i].record(copy_stream)

        stage(0)
        for s in range(e2e_steps):
            if s + 1 < e2e_steps:
                stage(s + 1)
            stepper.pre_step()
            e2e_bytes.append(kv_bytes_now(pool, P, L)[0])
            comp.wait_event(ev_in[s % 2])
            for layer in range(L):
                dq, dk, dv = views[s % 2][layer]
                o, l_ = stepper.layer(layer, dk, dv, dq, *outs[layer])
            ev_free[s % 2].record(comp)
            ho.copy_(o, non_blocking=True)
            hl.copy_(l_, non_blocking=True)
        f1.record(comp)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier()
        e2e_ms, e2e_job = job_totals(max(f0.elapsed_time(f1), wall * 1e3), sum(e2e_bytes), world, dev)
        h2d = L * (qb + 2 * kb)
        d2h = w.n * (w.Hq * w.D * 4 + w.Hq * 4)
        e2e = {"value": e2e_job / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / e2e_steps,
               "copies_per_step": "one host-to-device copy of every layer's q, k, v (on a copy stream, into "
                                  "one of two device buffers, overlapping the previous step); the last "
                                  "layer's out and lse back"}
    # ---------------- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pages_by_req = {}
        for r in range(min(w.n, 4)):
            pages_by_req[r] = []
            for p in range(pool.seq_info(r)[1]):
                b, t, nv = pool.export_page(0, r, p)
                pages_by_req[r].append((t, np.frombuffer(b, dtype=np.uint8).copy(), nv))
        gbs, nb, dt, desc = oracle_sample(w, pages_by_req, args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": desc,
               "seconds": dt}
        if args.cpu_full:
            for r in range(len(pages_by_req), w.n):
                pages_by_req[r] = []
                for p in range(pool.seq_info(r)[1]):
                    b, t, nv = pool.export_page(0, r, p)
                    pages_by_req[r].append((t, np.frombuffer(b, dtype=np.uint8).copy(), nv))
            qf = ins[args.warmup + args.steps - 1][0][2].float().cpu().numpy()
            fg, fb, fdt = oracle_layer_step(w, pages_by_req, qf)
            cpu["layer_step"] = {"value": fg, "unit": "GB/s", "seconds": fdt, "bytes": fb,
                                 "us_per_layer_step": fdt * 1e6, "cores": cpu_threads(),
                                 "sample": f"full layer-step: every request and kv head of layer 0 of {w.name}"}
        else:
            lb = sum(kernel_bytes) / len(kernel_bytes)
            cpu["layer_step_estimate"] = {
                "seconds": lb / (gbs * 1e9), "bytes": lb, "kind": "extrapolated, not timed",
                "how": "one full layer-step's algorithmic bytes at the sample's bytes per second "
                       "(--cpu-full times it whole)"}
    if rank != 0:
        return
    value = kv_job / (t_max * 1e-3) / 1e9
    per_layer_step_s = (t_max * 1e-3) / (args.steps * L)
    st = pool.stats()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16xf16->f32 (fp8/tq3 storage)", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "requests": w.n, "layers": L, "page_size": P,
                   "heads": f"{w.Hq}q/{w.Hkv}kv x {w.D}",
                   "context_tokens": int(ctx_total / max(1, len(bytes_acc))),
                   "l2": "inputs larger than L2: per-layer KV working set cycled over 16 layers",
                   "parallelism": f"replicas x{world}"},
        "path": "step graph (mkv_step_graph_launch, one launch per step)" if args.graph else
                "per-layer calls (mkv_append_decode)",
        "kv_gbs": value,
        "ctx_tokens_per_s_per_layer": world * (ctx_total / len(bytes_acc)) / per_layer_step_s,
        "us_per_layer_step": per_layer_step_s * 1e6,
        "frac_of_hbm_peak": value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": committed_traffic(w.name, sum(kernel_bytes) / len(kernel_bytes)),
                     "kernel": "mkv_decode_kernel (partial attention)",
                     "peak_source": peak_src, "launches": len(kernel_ms),
                     "timed_launches": ("whole step / layers (graph launches: no events between kernels)"
                                        if args.graph else
                                        f"layer {TIMED_LAYER} of each timed step (CUDA events on the call's stream)"),
                     "avg_launch_us": 1e3 * sum(kernel_ms) / len(kernel_ms)},
        "bytes_per_token_per_tier": {"fp8": 2064 * L, "tq3": 784 * L, "bf16": 4096 * L,
                                     "pool_kv_bytes_per_live_token": st.kv_bytes_per_live_token,
                                     "pages_reported_kib_per_token": 18.3},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clocks,
        "append": "fused into the decode kernel (one launch per layer appends the step's token and decodes)",
        "demote": {"calls": len(demote_ms), "ms_total": round(sum(demote_ms), 4),
                   "ms_per_step": round(sum(demote_ms) / args.steps, 4),
                   "share_of_step": round(sum(demote_ms) / ms, 4) if ms > 0 else None},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_multi(args):
    """Several query tokens per request and step (mkv_decode_attention_multi):
    each step appends nq tokens to every request (mkv_append_tokens) and runs
    the causal multi-query attention per layer.  No pages are demoted during
    the few timed steps (the Recent window grows by their tokens).  value =
    the unique KV bytes of the cache (each byte once per kv head and step) per
    second; the decode kernel reads each batch entry's prefix once (a pair of
    query tokens per entry for nq >= 2), about ceil(nq / 2) times those
    bytes, reported as kernel_read_bytes_per_launch."""
    import torch

    from mixed_format_paged_gb300 import binding as B
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import make_pool, prefill

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    w = make_workload(args)
    L, P, nq, n = w.num_layers, w.P, args.nq, w.n
    total_steps = args.warmup + args.steps
    pool = make_pool(w, device=dev, extra_steps=nq * (total_steps + 1), seed=99, max_batch=n * nq)
    prefill(pool, w, device=dev)
    ids = list(range(n))
    g = torch.Generator().manual_seed(7)
    ins = []
    for s in range(total_steps):
        row = []
        for layer in range(L):
            k = torch.randn(n * nq, w.Hkv, w.D, generator=g).to(w.kv_dtype).to(dev)
            v = torch.randn(n * nq, w.Hkv, w.D, generator=g).to(w.kv_dtype).to(dev)
            q = torch.randn(n, nq, w.Hq, w.D, generator=g).to(w.q_dtype).to(dev)
            row.append((k, v, q))
        ins.append(row)
    outs = [(torch.empty((n, nq, w.Hq, w.D), device=dev), torch.empty((n, nq, w.Hq), device=dev)) for _ in range(L)]
    TIMED_LAYER = L - 1

    def step(s, ev_pair=None, acc=None):
        pool.extend(ids, [nq] * n)
        if acc is not None:
            acc.append(kv_bytes_now(pool, P, L))
        for layer in range(L):
            k, v, q = ins[s][layer]
            pool.append(layer, ids, [nq] * n, k, v)
            if ev_pair is not None and layer == TIMED_LAYER:
                B.mkv_set_timing_events(pool.handle, *ev_pair)
            pool.decode_multi(layer, ids, q, *outs[layer])

    sampler = ClockSampler(0)
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    pool.check_device_errors()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record()
        b.record()
    acc = []
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record()
    for i in range(args.steps):
        step(args.warmup + i, ev[i], acc)
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    pool.check_device_errors()
    ms = e0.elapsed_time(e1)
    kv_total = sum(b for b, _ in acc)
    kernel_ms = [a.elapsed_time(b) for a, b in ev]
    unique = sum(b for b, _ in acc) / len(acc) / L
    avg_us = 1e3 * sum(kernel_ms) / len(kernel_ms)
    ctx = sum(c for _, c in acc) / len(acc)
    # the kernel reads each batch entry's prefix once: with nq >= 2 the query
    # tokens go in pairs and entry j reads up to query token min(2j + 1, nq - 1),
    # (nq - 1 - that) tokens fewer than the whole cache, all of them FP8 (the
    # newest pages)
    per_tok_fp8 = w.Hkv * ROW_BYTES["fp8"]
    last = [0] if nq == 1 else [min(2 * j + 1, nq - 1) for j in range((nq + 1) // 2)]
    read = sum(unique - per_tok_fp8 * n * (nq - 1 - i) for i in last)
    peak, peak_src = measured_peaks()
    line = {
        "metric": "multi-query decode-attn KV GB/s (unique cache bytes) and query tokens/s",
        "value": kv_total / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16xf16->f32 (fp8/tq3 storage)", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "nq": nq, "requests": n, "layers": L,
                   "context_tokens": int(ctx), "demotion": "none during the timed steps"},
        "query_tokens_per_s": n * nq * args.steps * L / (ms * 1e-3),
        "roofline": {"bound": "hbm", "kernel": "mkv_decode_kernel (partial attention)",
                     "unique_bytes_per_launch": unique, "kernel_read_bytes_per_launch": read,
                     "avg_launch_us": avg_us, "achieved_unique": unique / (avg_us * 1e-6) / 1e9,
                     "achieved_read": read / (avg_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac_read": read / (avg_us * 1e-6) / 1e9 / peak, "peak_source": peak_src},
        "gpu_launches": args.steps * L * 3, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.nq > 1:
        run_multi(args)
    else:
        run_mkv(args)


if __name__ == "__main__":
    main()

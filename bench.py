"""Benchmark of the AATC hot path on one B300 per rank.

One step = the workload's whole pass through the codec on synthetic data:
encode the full prefill (all KV heads, keys and values) into the packed
cache, then one decode step (encode the new token at position L, then decode
attention of every query head over the L+1 packed tokens).  Calibration is an
offline, once-per-layer step: it runs (and is timed) once before the loop.

Headline `value`: decode-attention packed-KV GB/s = (packed K + packed V
bytes + q bytes + output bytes) / decode time; `encode` reports prefill token
positions per second per layer.  Times come from CUDA events on the launching
stream around CUDA-graph replays (so the host launch path is not timed; the
`e2e` figure goes through the public API with host buffers instead).  The L2
(126 MB) is defeated by rotation: each call works on its own copy of the
packed cache, with enough copies that the working set is several L2 sizes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama_32k]
    python bench.py --impl reference     # the CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_attention_kv_b300 import synth  # noqa: E402

# decode call: one kernel when every (row, KV head group) has a single split
# (the call then needs no workspace), else split kernel + combine kernel
def _kernel_nodes(g):
    """Kernel nodes of a captured CUDA graph (kept with keep_graph=True), or None."""
    try:
        from cuda.bindings import runtime as rt
        graph = rt.cudaGraph_t(init_value=int(g.raw_cuda_graph()))
        err, _, n = rt.cudaGraphGetNodes(graph, 0)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        err, nodes, n = rt.cudaGraphGetNodes(graph, n)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        kinds = [rt.cudaGraphNodeGetType(nd)[1] for nd in nodes[:n]]
        return sum(1 for k_ in kinds if k_ == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel)
    except Exception:
        return None

L2_BYTES = 126 << 20
ENCODE_KERNELS_PER_CALL = 1


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# sources the decode kernels are built from: the kernels, the structures and
# constants they share with the host, and the record layout and read plan
DECODE_SOURCES = ("decode.cu", "internal.h", "plan.cu")


def decode_source_hash(root=None):
    """First 16 hex digits of the sha256 of the decode sources, concatenated."""
    import hashlib
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(root or ROOT, "quantized_attention_kv_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(algorithmic_bytes):
    """DRAM bytes per decode call from the committed ncu summary, if it was
    taken on the current decode sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
            rec = json.load(f)
        if rec.get("decode_sources_sha256_16") != decode_source_hash():
            return None
        return rec["dram_bytes_per_call"]
    except Exception:
        return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def run_ours(args, ws, rank, local):
    from quantized_attention_kv_b300 import aatc
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[args.workload]
    L = args.seq_len or wl.seq_len
    B, Hkv, Hq = wl.batch, wl.n_kv_heads, wl.n_q_heads
    bits = args.bits or wl.bits

    # inputs resident in HBM before anything is timed
    k_cal, v_cal, q_cal = synth.calib_inputs(wl, device=dev)
    kc, vc = synth.cache_inputs(wl, device=dev, seq_len=L)
    kn, vn = synth.cache_inputs(wl, layer=1, device=dev, seq_len=1)
    q = synth.query_inputs(wl, device=dev)
    stream = torch.cuda.current_stream(dev)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cal = aatc.calibrate(k_cal, v_cal, q_cal, bits, joint=args.joint)
    torch.cuda.synchronize()
    calib_ms = (time.perf_counter() - t0) * 1e3
    Wk, Wv = cal.W_k, cal.W_v
    packed_bytes = B * Hkv * (L + 1) * (Wk + Wv) * 4
    # L2 (126 MB) defeat: every call reads its own copy of the packed cache,
    # rotating over enough copies that the working set is several L2 sizes
    n_rot = int(min(64, max(3, -(-3 * L2_BYTES // packed_bytes))))
    if args.paged:
        # paged pools: each copy's rows on shuffled blocks of args.paged tokens
        bt = args.paged
        bpr = -(-(L + 1) // bt)
        gen = torch.Generator().manual_seed(1234)
        table = torch.randperm(B * bpr + 8, generator=gen)[:B * bpr].reshape(B, bpr).to(torch.int32).to(dev)
        kps = [aatc.alloc_pool(cal, B * bpr + 8, bt, device=dev, tensor="k") for _ in range(n_rot)]
        vps = [aatc.alloc_pool(cal, B * bpr + 8, bt, device=dev, tensor="v") for _ in range(n_rot)]
    else:
        kps = [aatc.alloc_cache(cal, B, L + 1, device=dev, tensor="k") for _ in range(n_rot)]
        vps = [aatc.alloc_cache(cal, B, L + 1, device=dev, tensor="v") for _ in range(n_rot)]

    def enc(k_, v_, kp, vp, start):
        if args.paged:
            aatc.encode_paged(cal, k_, v_, kp, vp, table, start_pos=start)
        else:
            aatc.encode(cal, k_, v_, kp, vp, start_pos=start)

    def dec(q_, kp, vp):
        if args.paged:
            aatc.decode_attention_paged(cal, q_, kp, vp, table, L + 1, out=out, workspace=wsb)
        else:
            aatc.decode_attention(cal, q_, kp, vp, L + 1, out=out, workspace=wsb)
    def fused(q_, kn_, vn_, kp, vp):
        """A serving step's append + decode: one fused call (the paged cache: the two calls)."""
        if args.paged:
            enc(kn_, vn_, kp, vp, L)
            dec(q_, kp, vp)
        else:
            aatc.append_decode_attention(cal, kn_, vn_, q_, kp, vp, L, out=out, workspace=wsb)
    out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
    wsb = aatc.new_append_workspace(cal, B, L, 1, device=dev)   # serves the decode-only calls too
    for kp, vp in zip(kps, vps):        # every copy holds a valid cache
        enc(kc, vc, kp, vp, 0)
        enc(kn, vn, kp, vp, L)
    torch.cuda.synchronize()

    q_bytes = q.numel() * q.element_size()
    out_bytes = out.numel() * 4
    decode_bytes = packed_bytes + q_bytes + out_bytes

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(c):
        """One step on cache copy c: prefill encode, then a serving step (append one token and decode)."""
        enc(kc, vc, kps[c], vps[c], 0)
        fused(q, kn, vn, kps[c], vps[c])

    # each step is captured once per cache copy into a CUDA graph, so the
    # timed region measures the device, not the Python launch path
    for c in range(n_rot):
        step(c)
    torch.cuda.synchronize()
    graphs = []
    for c in range(n_rot):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(c)
        graphs.append(g)
    g_dec = torch.cuda.CUDAGraph()          # decode alone, every copy once
    with torch.cuda.graph(g_dec):
        for c in range(n_rot):
            dec(q, kps[c], vps[c])
    g_app = torch.cuda.CUDAGraph()          # a serving step as two calls: append one token, then decode
    with torch.cuda.graph(g_app):
        for c in range(n_rot):
            enc(kn, vn, kps[c], vps[c], L)
            dec(q, kps[c], vps[c])
    g_fus = torch.cuda.CUDAGraph()          # a serving step as one call
    with torch.cuda.graph(g_fus):
        for c in range(n_rot):
            fused(q, kn, vn, kps[c], vps[c])
    # the kernels one timed step launches, counted in a capture of it
    g_cnt = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g_cnt):
        step(0)
    launches_per_step = _kernel_nodes(g_cnt)
    del g_cnt
    g_enc = torch.cuda.CUDAGraph()          # prefill encode alone, every copy once
    with torch.cuda.graph(g_enc):
        for c in range(n_rot):
            enc(kc, vc, kps[c], vps[c], 0)
    torch.cuda.synchronize()

    # End to end through the public API with host buffers, measured before the
    # clock sampler starts: while nvidia-smi samples, and for a while after it
    # stopped, each call's host path measured about six times as long (about 9
    # -> 60 us per launch on the B300 machine), an effect of the sampler, not of
    # the library.  H2D of the step's inputs (query, new key/value token),
    # append + decode, D2H of the output
    # the step's inputs (query, new key and value token) staged in one pinned
    # buffer and sent by one copy; the device copies are views of one buffer
    parts = [q, kn, vn]
    nbytes_in = [t.numel() * t.element_size() for t in parts]
    hbuf = torch.empty(sum(nbytes_in), dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(sum(nbytes_in), dtype=torch.uint8, device=dev)
    views_h, views_d, o = [], [], 0
    for t, nb in zip(parts, nbytes_in):
        views_h.append(hbuf[o:o + nb].view(t.dtype).view(t.shape))
        views_d.append(dbuf[o:o + nb].view(t.dtype).view(t.shape))
        o += nb
    for vh, t in zip(views_h, parts):
        vh.copy_(t.cpu())
    qd, knd, vnd = views_d
    outh = torch.empty(out.shape, dtype=torch.float32).pin_memory()

    def e2e_step(evs=None, c=0, host=None):
        kp, vp = kps[c % n_rot], vps[c % n_rot]
        if evs:
            evs[0].record(stream)
        t0 = time.perf_counter()
        dbuf.copy_(hbuf, non_blocking=True)
        t1 = time.perf_counter()
        fused(qd, knd, vnd, kp, vp)
        t2 = t3 = time.perf_counter()
        outh.copy_(out, non_blocking=True)
        t4 = time.perf_counter()
        if evs:
            evs[1].record(stream)
        if host is not None:
            host["h2d"] += t1 - t0
            host["append_decode"] += t3 - t1
            host["d2h"] += t4 - t3

    # warm-up, then at least 100 timed steps: the host path reaches a steady
    # state only after a few dozen calls
    for c in range(20):
        e2e_step(c=c)
    torch.cuda.synchronize()
    n_e2e = max(100, args.steps)
    e2e_evs = [[ev() for _ in range(2)] for _ in range(n_e2e)]
    host = {"h2d": 0.0, "append_decode": 0.0, "d2h": 0.0}
    w0 = time.perf_counter()
    for s in range(n_e2e):
        e2e_step(e2e_evs[s], c=s, host=host)
    torch.cuda.synchronize()
    e2e_wall_us = (time.perf_counter() - w0) / n_e2e * 1e6
    # host time of each call of the step, averaged over the timed loop; the
    # device keeps up when their sum is below the device time of a step
    host = {k_: round(v_ / n_e2e * 1e6, 2) for k_, v_ in host.items()}
    e2e_ms = sorted(e[0].elapsed_time(e[1]) for e in e2e_evs)
    e2e_step_s = _max_over_ranks(e2e_ms[len(e2e_ms) // 2] / 1e3, ws)   # median step
    for s_ in range(args.warmup):
        graphs[s_ % n_rot].replay()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    with ClockSampler(local) as clk:
        _barrier(ws)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        e0.record(stream)
        for s_ in range(args.steps):
            graphs[s_ % n_rot].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        _barrier(ws)
        wall = time.perf_counter() - w0
        step_ms_dev = e0.elapsed_time(e1) / args.steps
        # decode and encode alone (same rotation), for the per-kernel rates:
        # each replay of a graph (one call per cache copy) is timed on its own,
        # at least 200 calls in all; per-call times are replay time / copies
        reps = max(10, -(-200 // n_rot))

        def timed(g):
            g.replay()
            torch.cuda.synchronize()
            evs = [(ev(), ev()) for _ in range(reps)]
            for a_, b_ in evs:
                a_.record(stream)
                g.replay()
                b_.record(stream)
            torch.cuda.synchronize()
            return sorted(a_.elapsed_time(b_) / 1e3 / n_rot for a_, b_ in evs)

        # NVTX ranges name the calls for a profiler (ncu --nvtx --nvtx-include "decode_calls/")
        with torch.cuda.nvtx.range("decode_calls"):
            dec_t = timed(g_dec)
        with torch.cuda.nvtx.range("append_decode_calls"):
            app_t = timed(g_app)
        with torch.cuda.nvtx.range("fused_step_calls"):
            fus_t = timed(g_fus)
        with torch.cuda.nvtx.range("encode_calls"):
            enc_t = timed(g_enc)

    def pct(v, q):
        return v[min(len(v) - 1, int(round(q * (len(v) - 1))))]

    dec_call_s = _max_over_ranks(pct(dec_t, 0.5), ws)
    enc_call_s = _max_over_ranks(pct(enc_t, 0.5), ws)
    app_call_s = _max_over_ranks(pct(app_t, 0.5), ws)
    fus_call_s = _max_over_ranks(pct(fus_t, 0.5), ws)
    wall = _max_over_ranks(wall, ws)
    spread = {name: {"p10_us": round(pct(v, 0.1) * 1e6, 3), "median_us": round(pct(v, 0.5) * 1e6, 3),
                     "p90_us": round(pct(v, 0.9) * 1e6, 3), "calls": len(v) * n_rot, "replays": len(v)}
              for name, v in (("decode", dec_t), ("append_decode", app_t), ("append_decode_fused", fus_t),
                              ("encode", enc_t))}
    kp, vp = kps[0], vps[0]

    h2d = sum(nbytes_in)
    d2h = out_bytes

    peak, peak_kind = _peaks()
    value = decode_bytes * ws / dec_call_s / 1e9
    per_launch_s = dec_call_s
    achieved = decode_bytes / per_launch_s / 1e9
    res = {
        "metric": "decode-attn packed-KV GB/s (% of HBM peak) and encode tokens/s at 32k ctx",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_dev, 4),
        "wall_ms_per_step": round(wall / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded Gaussian KV shaped like the workload; no weights or datasets)",
        "config": {"workload": wl.name, "batch": B, "seq_len": L + 1, "n_q_heads": Hq, "n_kv_heads": Hkv,
                   "head_dim": 128, "bits_per_element": bits, "record_words": [Wk, Wv],
                   "allocation": "joint K/V split" if args.joint else "B bits per tensor",
                   "l2": "defeated by rotation: each call reads its own cache copy, %d copies = %.0f MB > 126 MB L2"
                         % (n_rot, n_rot * packed_bytes / 1e6),
                   "timing": "CUDA graphs of whole steps replayed K times; decode/encode rates: the median of "
                             "separately timed graph replays (one call per cache copy, >= 200 calls); CUDA events "
                             "on the launching stream",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "cache": ("paged, %d-token blocks, shuffled block table" % args.paged) if args.paged
                   else "contiguous"},
        "pct_of_hbm_peak": round(100 * value / ws / peak, 2),
        "encode": {"value": round(B * L * ws / enc_call_s, 1), "unit": "tokens/s",
                   "ms": round(enc_call_s * 1e3, 4),
                   "gb_s": round((B * Hkv * L * (2 * 128 * kc.element_size() + (Wk + Wv) * 4)) / enc_call_s / 1e9,
                                 2)},
        "decode_us": round(per_launch_s * 1e6, 3),
        "append_decode_us": round(app_call_s * 1e6, 3),
        "append_decode_fused_us": round(fus_call_s * 1e6, 3),
        "call_times": spread,
        "calibrate_ms": round(calib_ms, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic(decode_bytes),
                     "kernel": "decode_attention call (%s)" % ("k_decode_fast, one launch" if cal.decode_launches() == 1
                                                               else "query prep + splits + combine"),
                     "peak_kind": peak_kind},
        "e2e": {"value": round(decode_bytes * ws / e2e_step_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(e2e_step_s * 1e6, 2), "wall_us_per_step": round(e2e_wall_us, 2),
                "steps": n_e2e, "host_us_per_call": host,
                "what": "median over steps of the device time from before the H2D copy of the step's query "
                        "and new key/value token (one pinned buffer) to after the D2H copy of the output, "
                        "through the Python API (append_decode_attention: the new token encoded and the "
                        "decode attention, one call); calls are enqueued back "
                        "to back"},
        "gpu_launches": args.steps * (launches_per_step if launches_per_step is not None
                                      else ENCODE_KERNELS_PER_CALL + cal.decode_launches() + (1 if args.paged else 0)),
        "n_cache_copies": n_rot,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, L, bits)
    return res


def cpu_baseline(wl, L, bits, budget_s=20.0):
    """The fp64 oracle on the host cores: decode attention of ONE KV head (its
    G query heads) over the full context, from records the oracle encoded."""
    import numpy as np

    import oracle
    k_cal, v_cal, q_cal = synth.calib_inputs(wl, device="cpu")
    h = 0
    G = wl.group
    sub = lambda t: t[h:h + 1].double().numpy()  # noqa: E731
    cal = oracle.calibrate(sub(k_cal), sub(v_cal), q_cal[h * G:(h + 1) * G].double().numpy(), bits)
    kc, vc = synth.cache_inputs(synth.dataclasses.replace(wl, n_kv_heads=1, n_q_heads=G, batch=1),
                                device="cpu", seq_len=L)
    t0 = time.perf_counter()
    kp, _, _ = oracle.encode_cache(kc.double().numpy(), cal, "k")
    vp, _, _ = oracle.encode_cache(vc.double().numpy(), cal, "v")
    enc_s = time.perf_counter() - t0
    q = synth.query_inputs(wl, batch=1)[:, h * G:(h + 1) * G].double().numpy()
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.decode_attention(q, kp, vp, cal)
        n += 1
        if time.perf_counter() - t0 > min(budget_s, 5.0) or n >= 3:
            break
    dec_s = (time.perf_counter() - t0) / n
    W = cal["W"]
    nbytes = 2 * L * W * 4 + G * 128 * 2 + G * 128 * 4
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": round(nbytes / dec_s / 1e9, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "1 of %d KV heads (%d query heads) at %d tokens: decode %.3f s/call; encode %d tokens x K,V "
                      "%.2f s (%.0f tokens/s)" % (wl.n_kv_heads, G, L, dec_s, L, enc_s, L / enc_s),
            "encode_tokens_per_s": round(L / enc_s, 1)}


def run_reference(args, ws, rank):
    """Reference arm: the CPU oracle, as it stands, on a bounded sample of the
    same workload; each step decodes one KV head over the full context."""
    if rank != 0:
        return None
    wl = synth.WORKLOADS[args.workload]
    L = args.seq_len or wl.seq_len
    bits = args.bits or wl.bits
    base = cpu_baseline(wl, L, bits)
    import oracle  # noqa: F401
    return {
        "impl": "reference",
        "metric": "decode-attn packed-KV GB/s (% of HBM peak) and encode tokens/s at 32k ctx",
        "value": base["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "seq_len": L, "bits_per_element": bits},
        "cpu_baseline": {"kind": "oracle", "cores": base["cores"], "sample": base["sample"], "value": base["value"]},
        "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama_32k", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--seq-len", type=int, default=None)
    ap.add_argument("--bits", type=float, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--joint", action="store_true",
                    help="calibrate with the joint K/V budget split (attention-aware token weights)")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK_TOKENS",
                    help="run the step on paged pools with blocks of this many tokens (32 times a power of two)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, local = _dist()
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    else:
        from quantized_attention_kv_b300 import build
        if rank == 0:
            build.build()
        _barrier(ws)
        res = run_ours(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()

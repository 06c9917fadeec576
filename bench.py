"""Benchmark of the LazyAttention hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of the workload:
prefill of every request's query segment against its documents (TTFT), then
the configured number of decode steps (append + attention) for every request.
Inputs are synthetic (seeded), resident in HBM before the timed region; the L2
is flushed before every step; per-phase times come from CUDA events on the
launching stream.

Reported: value = decode KV-read throughput (logical K+V bytes of every
request's full context per decode step / decode time), plus prefill TFLOP/s
(QK^T and PV MMA FLOPs only), TTFT, roofline fractions, the in-run
materialising baseline (copy + eager RoPE into private pages, then the same
kernels without rotation), an end-to-end number through host buffers and the
fp64 oracle timed on a bounded sample on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "llama3_8b"
METRIC = "decode KV-read GB/s & prefill TFLOP/s (fraction of GB300 peak); TTFT ms"
UNIT = "GB/s"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# DRAM bytes (read + write) per launch from one ncu capture of this bench's own
# command on the named workload (summary: profiles/traffic_llama3_8b.md), keyed
# by a hash of the kernel sources the capture ran; reported only while the
# sources still hash the same, else null. "decode" = one lazyattn_decode call
# (append + attention kernels), "prefill" = the prefill kernel.
KERNEL_SOURCES = {
    "decode": ["k_decode_bf16.cu", "k_paging.cu", "internal.h", "tc_ptx.cuh"],
    "prefill": ["k_prefill_tc.cu", "internal.h", "tc_ptx.cuh"],
}
# RoPE variants the bench can time: the kernels' work does not depend on the
# values (only the position table and, for YaRN, the logit scale change).
ROPE_PRESETS = {
    "default": None,
    "linear": dict(kind="linear", factor=4.0),
    "ntk": dict(kind="ntk", factor=4.0),
    "yarn": dict(kind="yarn", factor=4.0, original_max_position=2048, low=1.0, high=32.0),
    "llama3": dict(kind="llama3", factor=8.0, original_max_position=8192, low=1.0, high=4.0),
}

NCU_TRAFFIC = {
    ("llama3_8b", "decode"): (69.25e6, "b19624a9cee07e87"),
    ("llama3_8b", "prefill"): (77.89e6, "0c435da0e4b12845"),
    ("few_shot_skewed", "decode"): (494.20e6, "b19624a9cee07e87"),
    ("few_shot_skewed", "prefill"): (599.04e6, "0c435da0e4b12845"),
}


def sources_sha(kind):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "position_agnostic_kv_lazyattn_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, kind):
    entry = NCU_TRAFFIC.get((workload, kind))
    if entry is None or entry[1] != sources_sha(kind):
        return None
    return entry[0]


def work_model(cfg):
    """Algorithmic bytes / FLOPs of one step of cfg (all requests)."""
    import workload
    Hkv, Hq, D = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim
    esz = 4 if cfg.dtype == "f32" else 2
    L0 = workload.request_context_lens(cfg)            # document tokens of each request
    Lq = cfg.q_len
    pairs = float(np.sum(Lq * L0 + Lq * (Lq + 1) // 2))   # visible (query, key) pairs per head, all requests
    prefill_flops = 4.0 * D * pairs * Hq
    dec_bytes = [2.0 * float(np.sum(L0 + Lq + t + 1)) * Hkv * D * esz for t in range(cfg.decode_steps)]
    return prefill_flops, dec_bytes


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"lazyattn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sms.append(float(parts[0]))
                    mx = float(parts[1])
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


def run_ours(args, rank, world):
    import torch
    import workload
    import workload.device as wdev
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = workload.CONFIGS[args.config]
    if args.requests:
        import dataclasses
        cfg = dataclasses.replace(cfg, n_requests=min(args.requests, cfg.n_requests))
    doc_local = args.keys == "doc_local" or args.pos == "alibi"   # no materialising baseline / no-RoPE leg
    env = wdev.setup(cfg, baseline=not args.no_extras and not doc_local, key_storage=args.keys,
                     position_encoding=args.pos, rope_scaling=ROPE_PRESETS[args.rope],
                     rope_interleaved=args.interleaved)
    R = cfg.n_requests
    b = env.batch
    stream = torch.cuda.current_stream()
    hbm_peak, tc_peak, tc_sust, peak_kind = peaks()
    prefill_flops, dec_bytes = work_model(cfg)

    # per-step inputs, resident in HBM
    dec_in = [wdev.decode_step_tensors(cfg, t, range(R)) for t in range(cfg.decode_steps)]
    out_p = torch.empty((max(b.total_q, 1), cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device=dev)
    out_d = torch.empty((R, cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device=dev)
    ws_bytes = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, b.c)
    ws = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device=dev)
    entries0 = b.entries.clone()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # > 129 MB L2

    # materialising baseline: private copies of every entry's page (position-free
    # pools only: doc-local keys are already rotated)
    if not args.no_extras and not doc_local:
        base_pages = env.pool.alloc_pages(len(b.entries_host))
        dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.array(base_pages, np.uint64)
        dst_dev = torch.from_numpy(dst.view(np.int64).copy()).to(dev)
        mb = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED, device=dev)
        mb_entries0 = mb.entries.clone()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # One CUDA graph per phase: the prefill launch, and the decode steps (append +
    # attention each). Replays remove host launch gaps from the timed region.
    def capture(fn):
        fn()                                    # eager run first (also a warm-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    def prefill_lazy():
        if b.total_q:
            L.lazyattn_prefill(env.pool.handle, b.c, env.q, out_p, None, 0, None)

    def decode_lazy():
        for t in range(cfg.decode_steps):
            q, k, v = dec_in[t]
            L.lazyattn_decode(env.pool.handle, b.c, q, k, v, out_d, ws, ws_bytes, None)

    def materialize_base():
        L.lazyattn_materialize(env.pool.handle, b.c, dst_dev, None)

    def prefill_base():
        if b.total_q:
            L.lazyattn_prefill(env.pool.handle, mb.c, env.q, out_p, None, 0, None)

    def decode_base():
        for t in range(cfg.decode_steps):
            q, k, v = dec_in[t]
            L.lazyattn_decode(env.pool.handle, mb.c, q, k, v, out_d, ws, ws_bytes, None)

    g_pre = capture(prefill_lazy)
    b.entries.copy_(entries0)
    g_dec = capture(decode_lazy)
    b.entries.copy_(entries0)

    def lazy_step(rec):
        b.entries.copy_(entries0)
        flush.zero_()
        e = [ev(), ev(), ev()]
        e[0].record(stream)
        g_pre.replay()
        e[1].record(stream)
        g_dec.replay()
        e[2].record(stream)
        rec.append(e)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        lazy_step([])
    barrier()
    rec = []
    with Clocks(dev.index) as clk:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            lazy_step(rec)
        barrier()
        wall = time.perf_counter() - t0
    status = env.pool.device_status()

    # warm-L2 numbers: the same replays without the flush (the timed value above is cold)
    wrec = []
    for it in range(min(max(args.steps, 3), 20) + 1):
        b.entries.copy_(entries0)
        e = [ev(), ev(), ev()]
        e[0].record(stream)
        g_pre.replay()
        e[1].record(stream)
        g_dec.replay()
        e[2].record(stream)
        if it >= 1:
            wrec.append(e)
    torch.cuda.synchronize()
    warm_pre = statistics.median(r[0].elapsed_time(r[1]) for r in wrec)
    warm_dec = statistics.median(r[1].elapsed_time(r[2]) for r in wrec)

    pre_ms = [r[0].elapsed_time(r[1]) for r in rec]
    dec_ms = [r[1].elapsed_time(r[2]) for r in rec]
    dec_call_ms = [d / max(cfg.decode_steps, 1) for d in dec_ms]
    step_ms = [p + d for p, d in zip(pre_ms, dec_ms)]
    dec_total_bytes = sum(dec_bytes)
    mean_dec_s = statistics.mean(dec_ms) / 1e3
    # end to end through host buffers (pinned), copies inside the timed region;
    # every rank runs it on its own GPU, like the timed steps
    e2e_s, e2e_info = None, None
    if cfg.decode_steps and not args.no_extras:
        # a step's q | k_new | v_new packed in one pinned buffer and sent with one copy;
        # the decode call takes device views into it (each part starts 16-byte aligned)
        sizes = [x.numel() for x in dec_in[0]]
        offs = [0, sizes[0], sizes[0] + sizes[1], sum(sizes)]
        host_in = []
        for t in range(cfg.decode_steps):
            buf = torch.empty(offs[3], dtype=dec_in[t][0].dtype).pin_memory()
            for i, x in enumerate(dec_in[t]):
                buf[offs[i]:offs[i + 1]].copy_(x.reshape(-1).cpu())
            host_in.append(buf)
        dbuf = torch.empty(offs[3], dtype=dec_in[0][0].dtype, device=dev)
        dq, dk, dv = (dbuf[offs[i]:offs[i + 1]].view(dec_in[0][i].shape) for i in range(3))
        host_out = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
        h2d = host_in[0].numel() * host_in[0].element_size()
        d2h = host_out.numel() * host_out.element_size()
        times = []
        for it in range(2):
            b.entries.copy_(entries0)
            flush.zero_()
            torch.cuda.synchronize()
            s0, s1 = ev(), ev()
            s0.record(stream)
            for t in range(cfg.decode_steps):
                dbuf.copy_(host_in[t], non_blocking=True)
                L.lazyattn_decode(env.pool.handle, b.c, dq, dk, dv, out_d, ws, ws_bytes, stream)
                host_out.copy_(out_d, non_blocking=True)
            s1.record(stream)
            torch.cuda.synchronize()
            times.append(s0.elapsed_time(s1) / 1e3)
        e2e_s = min(times)
        e2e_info = {"unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "note": "decode phase with, per step, one pinned H2D of the packed q/k_new/v_new and a D2H of "
                            "the output; every rank, slowest rank's time, bytes of all ranks"}

    local = {"step_ms": statistics.mean(step_ms), "dec_s": mean_dec_s, "pre_ms": statistics.mean(pre_ms),
             "wall": wall}
    if e2e_s is not None:
        local["e2e_s"] = e2e_s
    local = reduce_max_over_ranks(local, world)
    e2e = None
    if e2e_info is not None:
        e2e = dict(e2e_info, value=round(world * dec_total_bytes / local["e2e_s"] / 1e9, 1))
    if rank != 0:
        return None

    # baseline (same box, same inputs): materialise, prefill and decode on private rotated copies
    b_mat = b_pre = b_dec = None
    if not args.no_extras and not doc_local:
        b.entries.copy_(entries0)   # the tables as the lazy path's first step sees them
        g_bmat = capture(materialize_base)
        g_bpre = capture(prefill_base)
        mb.entries.copy_(mb_entries0)
        g_bdec = capture(decode_base)
        brec = []
        for it in range(max(2, min(args.steps, 20)) + 2):
            mb.entries.copy_(mb_entries0)
            flush.zero_()
            e = [ev() for _ in range(4)]
            e[0].record(stream)
            g_bmat.replay()
            e[1].record(stream)
            g_bpre.replay()
            e[2].record(stream)
            g_bdec.replay()
            e[3].record(stream)
            if it >= 2:
                brec.append(e)
        torch.cuda.synchronize()
        b_mat = statistics.mean(r[0].elapsed_time(r[1]) for r in brec)
        b_pre = statistics.mean(r[1].elapsed_time(r[2]) for r in brec)
        b_dec = statistics.mean(r[2].elapsed_time(r[3]) for r in brec)

    # No-RoPE comparison (the paper's Table 12 experiment): the same kernels on the
    # same shared pages with rotation switched off (the keys are treated as
    # already rotated: numerically meaningless, identical data movement), so the
    # ratio is the cost of rotating at run time.
    norope = None
    if not args.no_extras and not doc_local:
        nb = b.with_entries(b.entries_host, L.LAZYATTN_KEYS_PREROTATED, device=dev)
        nb_entries0 = nb.entries.clone()

        def prefill_plain():
            if nb.total_q:
                L.lazyattn_prefill(env.pool.handle, nb.c, env.q, out_p, None, 0, None)

        def decode_plain():
            for t in range(cfg.decode_steps):
                q, k, v = dec_in[t]
                L.lazyattn_decode(env.pool.handle, nb.c, q, k, v, out_d, ws, ws_bytes, None)

        g_npre = capture(prefill_plain)
        nb.entries.copy_(nb_entries0)
        g_ndec = capture(decode_plain)
        nrec = []
        for it in range(max(2, min(args.steps, 20)) + 2):
            nb.entries.copy_(nb_entries0)
            flush.zero_()
            e = [ev() for _ in range(3)]
            e[0].record(stream)
            g_npre.replay()
            e[1].record(stream)
            g_ndec.replay()
            e[2].record(stream)
            if it >= 2:
                nrec.append(e)
        torch.cuda.synchronize()
        n_pre = statistics.mean(r[0].elapsed_time(r[1]) for r in nrec)
        n_dec = statistics.mean(r[1].elapsed_time(r[2]) for r in nrec)
        norope = {"prefill_ms": round(n_pre, 4), "decode_ms": round(n_dec, 4),
                  "prefill_overhead": round(local["pre_ms"] / n_pre, 3) if cfg.q_len and n_pre else None,
                  "decode_overhead": round(local["dec_s"] * 1e3 / n_dec, 3) if cfg.decode_steps and n_dec else None,
                  "note": "same kernels and pages, rotation off; overhead = lazy time / no-RoPE time"}

    dec_gbs = world * dec_total_bytes / local["dec_s"] / 1e9 if cfg.decode_steps else 0.0
    pre_tflops = prefill_flops / (local["pre_ms"] / 1e3) / 1e12 if cfg.q_len else 0.0
    mean_call = statistics.mean(dec_call_ms) if dec_call_ms else 0.0
    per_call_bytes = dec_total_bytes / max(cfg.decode_steps, 1)
    achieved = per_call_bytes / (mean_call / 1e3) / 1e9 if mean_call else 0.0
    line = {
        "metric": METRIC, "value": round(dec_gbs, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(local["step_ms"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": cfg.name, "requests": R, "docs_per_request": cfg.docs_per_request,
                   "doc_len": (f"{cfg.doc_len_min}..{cfg.doc_len}" if cfg.doc_len_min else cfg.doc_len),
                   "pool_docs": cfg.n_docs, "q_heads": cfg.n_q_heads,
                   "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim, "query_len": cfg.q_len,
                   "decode_steps": cfg.decode_steps, "zipf_alpha": cfg.zipf_alpha, "seed": cfg.seed,
                   "l2": "flushed before every step (256 MB write)", "parallelism": f"replicas x{world}",
                   "keys": args.keys, "position_encoding": args.pos, "rope": args.rope,
                   "rope_interleaved": args.interleaved},
        "prefill_tflops": round(pre_tflops, 2), "ttft_ms": round(local["pre_ms"], 4),
        "decode_ms_per_token_step": round(mean_call, 4),
        "median_step_ms": round(statistics.median(step_ms), 4),
        "warm_l2": {"ttft_ms": round(warm_pre, 4),
                    "decode_gbs": round(dec_total_bytes / (warm_dec / 1e3) / 1e9, 1) if cfg.decode_steps and warm_dec else None,
                    "prefill_tflops": round(prefill_flops / (warm_pre / 1e3) / 1e12, 2) if cfg.q_len and warm_pre else None,
                    "note": "median of replays without the L2 flush"},
        "timing": "CUDA events around CUDA-graph replays (prefill graph; graph of all decode steps)",
        "frac_hbm_peak": round(dec_gbs / world / hbm_peak, 4),
        "frac_tensor_peak": round(pre_tflops / world / tc_peak, 4),
        "roofline": {"kernel": "lazyattn_decode (append + split-K attention)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": measured_traffic(cfg.name, "decode"),
                     "traffic_unit": "bytes per decode call (DRAM read + write, ncu)",
                     "algorithmic_bytes_per_call": round(per_call_bytes), "peak_kind": peak_kind},
        "prefill_roofline": {"kernel": "prefill_tc_kernel", "bound": "tensor", "achieved": round(pre_tflops, 2),
                             "peak": tc_peak, "unit": "TFLOP/s", "frac": round(pre_tflops / tc_peak, 4),
                             "traffic": measured_traffic(cfg.name, "prefill"),
                             "traffic_unit": "bytes per launch (DRAM read + write, ncu)", "peak_kind": peak_kind},
        "materialising_baseline": None if b_mat is None else {
            "materialise_ms": round(b_mat, 4), "ttft_ms": round(b_mat + b_pre, 4), "decode_ms": round(b_dec, 4),
            "decode_gbs": round(dec_total_bytes / (b_dec / 1e3) / 1e9, 1) if b_dec else None,
            "lazy_ttft_speedup": round((b_mat + b_pre) / local["pre_ms"], 3) if local["pre_ms"] else None,
            "lazy_decode_speedup": round(b_dec / (local["dec_s"] * 1e3), 3) if local["dec_s"] else None,
            "lazy_step_speedup": round((b_mat + b_pre + b_dec) / local["step_ms"], 3)},
        "norope": norope,
        "e2e": e2e,
        "gpu_launches": args.steps * ((1 if cfg.q_len else 0) + 2 * cfg.decode_steps),
        "wall_s_timed": round(local["wall"], 4),
        "device_status": status,
    }
    clocks = clk.summary()
    line["clocks"] = clocks
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, budget_s=args.cpu_budget)
    return line


def reduce_max_over_ranks(local: dict, world: int) -> dict:
    """Timing of a multi-rank run = the slowest rank (max over ranks)."""
    if world <= 1:
        return dict(local)
    import torch
    import torch.distributed as dist
    keys = sorted(local)
    # NCCL reduces device tensors only; gloo (CPU tests, the reference arm) host ones
    device = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(local[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(keys, t.cpu().tolist()))


def cpu_baseline(cfg, budget_s=15.0, n_steps=None):
    """The fp64 oracle, as it stands, on a bounded sample: decode steps of a few
    requests (every step attends over the request's full context)."""
    import oracle
    import workload
    docs = workload.request_docs(cfg)
    t0 = time.perf_counter()
    nbytes = 0.0
    esz = 4 if cfg.dtype == "f32" else 2
    done_req = 0
    steps = n_steps or min(cfg.decode_steps, 16) or 1
    for r in range(cfg.n_requests):
        ctx = [workload.doc_kv(cfg, int(d)) for d in docs[r]]
        if cfg.q_len:
            _, kq, vq = workload.query_segment(cfg, r)
        else:
            kq = np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
            vq = kq.copy()
        st = [tuple(a[0] for a in workload.decode_inputs(cfg, t, [r])) for t in range(steps)]
        ts = time.perf_counter()
        oracle.decode_request(ctx, kq, vq, st, cfg.rope_theta)
        L0 = sum(a[0].shape[0] for a in ctx)
        nbytes += sum(2.0 * (L0 + cfg.q_len + t + 1) * cfg.n_kv_heads * cfg.head_dim * esz
                      for t in range(steps))
        done_req += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": round(nbytes / el / 1e9, 4), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done_req} request(s) x {steps} decode step(s) of {cfg.name}, fp64 numpy, "
                      f"{el:.1f} s incl. input generation"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import workload
    cfg = workload.CONFIGS[args.config]
    for _ in range(args.warmup):
        cpu_baseline(cfg, budget_s=0.0, n_steps=1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(cfg, budget_s=0.0, n_steps=1))
    wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "kind": "oracle", "cores": os.cpu_count(),
                             "sample": vals[0]["sample"]},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the baseline and end-to-end legs")
    ap.add_argument("--requests", type=int, default=0, help="use only the first N requests (profiling captures)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--keys", default="position_free", choices=["position_free", "doc_local"],
                    help="key layout: stored without RoPE (default) or rotated at document-local positions")
    ap.add_argument("--pos", default="rope", choices=["rope", "alibi"],
                    help="position encoding: RoPE (default) or the ALiBi score bias")
    ap.add_argument("--rope", default="default", choices=list(ROPE_PRESETS),
                    help="RoPE variant of the position table (presets in ROPE_PRESETS)")
    ap.add_argument("--interleaved", action="store_true", help="interleaved RoPE pairs (2i, 2i+1)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist.init_process_group(backend)
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of the LazyAttention hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of the workload:
prefill of every request's query segment against its documents (TTFT), then
the configured number of decode calls (append + attention) for every request.
The default workload is the Llama-3-70B-shaped batch (64 requests x 32
documents of 1024 tokens from a 4000-document pool, 256-token query segment,
128 decode steps), the largest single-GPU one. Inputs are synthetic (seeded)
and resident in HBM before the timed region; the L2 is flushed before the
prefill and before every decode call, outside the timed events; each launch
(prefill; each decode call) is timed by CUDA events on the launching stream.

Reported: value = decode KV-read throughput (logical K+V bytes of every
request's full context per decode call / decode time), its fraction of the
measured HBM peak, and the DRAM-level fraction on the distinct tiles a call
reads; prefill TFLOP/s (QK^T and PV MMA FLOPs only) and TTFT; the in-run
materialising baseline (copy + eager RoPE into private pages, then the same
kernels without rotation) and the no-RoPE comparison; end-to-end numbers
through the C ABI with host buffers; the fp64 oracle timed on a bounded sample
on the host cores.

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

DEFAULT_CONFIG = "llama3_70b"
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
# command on the named workload (summary: profiles/traffic_llama3_70b.md), keyed
# by a hash of the kernel sources the capture ran; reported only while the
# sources still hash the same, else null. "decode" = one lazyattn_decode call
# through the batch's decode plan (append + document-major units + combine),
# "prefill" = the prefill kernel.
KERNEL_SOURCES = {
    "decode": ["k_decode_shared.cu", "decode_plan.cu", "k_paging.cu", "internal.h", "tc_ptx.cuh"],
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
    # decode call = decode_shared 4,638,851,242 + 71,246,848; combine 70,299,648 + 40,106;
    # append 297,984 (read + write bytes, mean of three calls); prefill 8,550,291,968 + 261,769,216
    ("llama3_70b", "decode"): (4780735829.0, "4f7db189cf4decee"),
    ("llama3_70b", "prefill"): (8812061184.0, "176d1c203b16d929"),
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


def unique_tiles_per_call(entries_host, offsets_host, steps):
    """Distinct (page, KV head) tiles each decode call reads, for every step t.

    Pages of non-writable entries (documents) are counted once however many
    requests or entries name them; a request's writable pages (its query
    segment and generated tokens) are private. Appends follow the library's
    rule: the first entry with free slots in the trailing run of writable
    entries. Returns a list of page counts (multiply by Hkv for tiles)."""
    e = np.asarray(entries_host, np.uint64)
    nvalid = ((e >> np.uint64(58)) & np.uint64(0x1F)).astype(np.int64)
    writable = (e >> np.uint64(63)).astype(bool)
    pages = (e & np.uint64(0xFFFFFFFF)).astype(np.int64)
    shared = len(set(pages[(~writable) & (nvalid > 0)].tolist()))
    tails = []   # per request: nvalid of its trailing writable run
    for r in range(len(offsets_host) - 1):
        a, b = int(offsets_host[r]), int(offsets_host[r + 1])
        i = b
        while i > a and writable[i - 1]:
            i -= 1
        tails.append(list(nvalid[i:b]))
    counts = []
    for _ in range(steps):
        n = shared
        for tail in tails:
            for j, v in enumerate(tail):
                if v < 16:
                    tail[j] = v + 1
                    break
            n += sum(1 for v in tail if v > 0)
        counts.append(n)
    return counts


def run_ours(args, rank, world):
    import dataclasses
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
        cfg = dataclasses.replace(cfg, n_requests=min(args.requests, cfg.n_requests))
    if args.decode_steps >= 0:
        cfg = dataclasses.replace(cfg, decode_steps=min(args.decode_steps, cfg.decode_steps))
    doc_local = args.keys == "doc_local" or args.pos == "alibi"   # no materialising baseline / no-RoPE leg
    extras = not args.no_extras and not doc_local
    env = wdev.setup(cfg, baseline=extras, key_storage=args.keys, all_docs=not args.used_docs,
                     position_encoding=args.pos, rope_scaling=ROPE_PRESETS[args.rope],
                     rope_interleaved=args.interleaved)
    R, T = cfg.n_requests, cfg.decode_steps
    b = env.batch
    stream = torch.cuda.current_stream()
    hbm_peak, tc_peak, tc_sust, peak_kind = peaks()
    prefill_flops, dec_bytes = work_model(cfg)
    esz = 4 if cfg.dtype == "f32" else 2
    tile_bytes = 2 * 16 * cfg.head_dim * esz * cfg.n_kv_heads          # K + V of one page, every KV head
    uniq_bytes = [n * tile_bytes for n in unique_tiles_per_call(b.entries_host, b.offsets_host, T)]

    # Document-major decode plan of the batch (host, once per table; every
    # decode call of the step reuses it): built and uploaded outside the timed region.
    use_plan = cfg.dtype == "bf16" and not args.no_plan
    plan_info = None
    if use_plan:
        tp = time.perf_counter()
        plan_info = b.plan_decode(env.pool)
        torch.cuda.synchronize()
        plan_info["build_upload_ms"] = round((time.perf_counter() - tp) * 1e3, 2)

    # per-step inputs, resident in HBM
    dec_in = [wdev.decode_step_tensors(cfg, t, range(R)) for t in range(T)]
    out_p = torch.empty((max(b.total_q, 1), cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device=dev)
    out_d = torch.empty((R, cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device=dev)
    ws_bytes = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, b.c)
    ws = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device=dev)
    entries0 = b.entries.clone()

    def ws_for(batch):
        """A workspace for decode calls on batch (its own plan may need more)."""
        n = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, batch.c)
        return (ws, ws_bytes) if n <= ws_bytes else (torch.zeros((n + 3) // 4, dtype=torch.int32, device=dev), n)

    pws = {}

    def pws_for(batch):
        """The prefill workspace of batch (room for the partials of a split prefill)."""
        n = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_PREFILL, batch.c)
        if n not in pws:
            pws[n] = torch.zeros((n + 3) // 4, dtype=torch.int32, device=dev)
        return pws[n], n
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # > 129 MB L2

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # One CUDA graph for the prefill launch and one per decode call (append +
    # attention): replays remove host launch gaps, and the L2 can be flushed
    # between any two calls outside the timed events.
    def capture(fn):
        fn()                                    # eager run first (also a warm-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    def prefill_fn(batch):
        w, wb = pws_for(batch)
        return lambda: L.lazyattn_prefill(env.pool.handle, batch.c, env.q, out_p, w, wb, None)

    def decode_fn(batch, t):
        q, k, v = dec_in[t]
        w, wb = ws_for(batch)
        return lambda: L.lazyattn_decode(env.pool.handle, batch.c, q, k, v, out_d, w, wb, None)

    def graphs(batch, reset):
        reset()
        g_pre = capture(prefill_fn(batch)) if b.total_q else None
        reset()
        g_dec = [capture(decode_fn(batch, t)) for t in range(T)]
        reset()
        return g_pre, g_dec

    def run_phases(g_pre, g_dec, reset, iters, cold=True, g_mat=None, rec=None):
        """iters passes of (materialise?) + prefill + every decode call, each
        timed by its own events; cold: the L2 is flushed before the prefill
        and before every decode call (outside the events). Returns a list of
        (materialise ms, prefill ms, [decode call ms])."""
        recs = []
        for _ in range(iters):
            reset()
            if cold:
                flush.zero_()
            em = None
            if g_mat is not None:
                em = (ev(), ev())
                em[0].record(stream)
                g_mat.replay()
                em[1].record(stream)
                if cold:
                    flush.zero_()
            ep = None
            if g_pre is not None:
                ep = (ev(), ev())
                ep[0].record(stream)
                g_pre.replay()
                ep[1].record(stream)
            ed = []
            for g in g_dec:
                if cold:
                    flush.zero_()
                a, z = ev(), ev()
                a.record(stream)
                g.replay()
                z.record(stream)
                ed.append((a, z))
            recs.append((em, ep, ed))
        if rec is not None:
            return recs
        torch.cuda.synchronize()
        return resolve(recs)

    def resolve(recs):
        return [(em[0].elapsed_time(em[1]) if em else 0.0, ep[0].elapsed_time(ep[1]) if ep else 0.0,
                 [a.elapsed_time(z) for a, z in ed]) for em, ep, ed in recs]

    def reset_lazy():
        b.entries.copy_(entries0)

    g_pre, g_dec = graphs(b, reset_lazy)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    run_phases(g_pre, g_dec, reset_lazy, args.warmup)
    barrier()
    with Clocks(dev.index) as clk:
        t0 = time.perf_counter()
        recs = run_phases(g_pre, g_dec, reset_lazy, args.steps, rec=True)
        barrier()
        wall = time.perf_counter() - t0
    timed = resolve(recs)
    status = env.pool.device_status()
    warm = run_phases(g_pre, g_dec, reset_lazy, min(max(args.steps, 3), 10), cold=False)

    pre_ms = [p for _, p, _ in timed]
    dec_ms = [sum(d) for _, _, d in timed]
    call_ms = [x for _, _, d in timed for x in d]
    step_ms = [p + d for p, d in zip(pre_ms, dec_ms)]
    dec_total_bytes = sum(dec_bytes)
    uniq_total_bytes = sum(uniq_bytes)
    mean_dec_s = statistics.mean(dec_ms) / 1e3

    # end to end through the C ABI with host buffers (pinned), every copy inside
    # the timed region: per decode call the H2D of its q | k_new | v_new (one
    # packed buffer) and the D2H of its output; TTFT: H2D of the query rows,
    # prefill, D2H of its output. L2 flushed before each timed call, as above.
    e2e_info, e2e_local = None, {}
    if not args.no_extras and (T or b.total_q):
        reps = max(args.e2e_reps, 1)
        info = {"unit": UNIT, "repeats": reps, "statistic": "median over repeats",
                "note": "through the C ABI with pinned host buffers: per decode call one H2D of the packed "
                        "q/k_new/v_new and a D2H of the output; L2 flushed before each call (outside the "
                        "events); every rank, slowest rank's median, bytes of all ranks"}
        h2d = d2h = 0
        if T:
            sizes = [x.numel() for x in dec_in[0]]
            offs = [0, sizes[0], sizes[0] + sizes[1], sum(sizes)]
            host_in = []
            for t in range(T):
                buf = torch.empty(offs[3], dtype=dec_in[t][0].dtype).pin_memory()
                for i, x in enumerate(dec_in[t]):
                    buf[offs[i]:offs[i + 1]].copy_(x.reshape(-1).cpu())
                host_in.append(buf)
            dbuf = torch.empty(offs[3], dtype=dec_in[0][0].dtype, device=dev)
            dq, dk, dv = (dbuf[offs[i]:offs[i + 1]].view(dec_in[0][i].shape) for i in range(3))
            host_out = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
            h2d = host_in[0].numel() * host_in[0].element_size()
            d2h = host_out.numel() * host_out.element_size()
            per_rep = []
            for _ in range(reps):
                reset_lazy()
                ed = []
                for t in range(T):
                    flush.zero_()
                    a, z = ev(), ev()
                    a.record(stream)
                    dbuf.copy_(host_in[t], non_blocking=True)
                    L.lazyattn_decode(env.pool.handle, b.c, dq, dk, dv, out_d, ws, ws_bytes, stream)
                    host_out.copy_(out_d, non_blocking=True)
                    z.record(stream)
                    ed.append((a, z))
                torch.cuda.synchronize()
                per_rep.append(sum(a.elapsed_time(z) for a, z in ed))
            e2e_local["e2e_dec_ms"] = statistics.median(per_rep)
        if b.total_q:
            q_host = env.q.cpu().pin_memory()
            o_host = torch.empty(out_p.shape, dtype=out_p.dtype).pin_memory()
            q_dev = torch.empty_like(env.q)
            pw, pwb = pws_for(b)
            per_rep = []
            for _ in range(reps):
                flush.zero_()
                a, z = ev(), ev()
                a.record(stream)
                q_dev.copy_(q_host, non_blocking=True)
                L.lazyattn_prefill(env.pool.handle, b.c, q_dev, out_p, pw, pwb, stream)
                o_host.copy_(out_p, non_blocking=True)
                z.record(stream)
                torch.cuda.synchronize()
                per_rep.append(a.elapsed_time(z))
            e2e_local["e2e_ttft_ms"] = statistics.median(per_rep)
            info["ttft_h2d_bytes"] = int(q_host.numel() * q_host.element_size())
            info["ttft_d2h_bytes"] = int(o_host.numel() * o_host.element_size())
        info["h2d_bytes_per_step"] = int(h2d)
        info["d2h_bytes_per_step"] = int(d2h)
        e2e_info = info

    local = {"step_ms": statistics.mean(step_ms), "dec_s": mean_dec_s, "pre_ms": statistics.mean(pre_ms),
             "wall": wall}
    local.update(e2e_local)
    local = reduce_max_over_ranks(local, world)
    e2e = None
    if e2e_info is not None:
        e2e = dict(e2e_info)
        if "e2e_dec_ms" in local:
            e2e["value"] = round(replica_throughput(dec_total_bytes, local["e2e_dec_ms"] / 1e3, world), 1)
            e2e["decode_ms"] = round(local["e2e_dec_ms"], 4)
        else:
            e2e["value"] = None
        if "e2e_ttft_ms" in local:
            e2e["ttft_e2e_ms"] = round(local["e2e_ttft_ms"], 4)
    if rank != 0:
        return None

    # Materialising baseline (same box, same inputs): private copies of every
    # entry's page, K rotated eagerly; then the same kernels without rotation.
    base = None
    if extras:
        base_pages = env.pool.alloc_pages(len(b.entries_host))
        dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.array(base_pages, np.uint64)
        dst_dev = torch.from_numpy(dst.view(np.int64).copy()).to(dev)
        mb = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED, device=dev)
        if use_plan:
            mb.plan_decode(env.pool)     # private pages: every run has one reader
        mb_entries0 = mb.entries.clone()

        def reset_base():
            b.entries.copy_(entries0)
            mb.entries.copy_(mb_entries0)

        reset_base()
        g_mat = capture(lambda: L.lazyattn_materialize(env.pool.handle, b.c, dst_dev, None))
        gb_pre, gb_dec = graphs(mb, reset_base)
        n_b = max(3, min(args.steps, 10))
        r_b = run_phases(gb_pre, gb_dec, reset_base, n_b + 1, g_mat=g_mat)[1:]
        base = (statistics.mean(x[0] for x in r_b), statistics.mean(x[1] for x in r_b),
                statistics.mean(sum(x[2]) for x in r_b))

    # No-RoPE comparison (the paper's Table 12 experiment): the same kernels on
    # the same shared pages with rotation switched off (keys treated as already
    # rotated: numerically meaningless, identical data movement), so the ratio
    # is the cost of rotating at run time. Timed like the lazy path.
    norope = None
    if extras:
        nb = b.with_entries(b.entries_host, L.LAZYATTN_KEYS_PREROTATED, device=dev)
        if use_plan:
            nb.plan_decode(env.pool)     # the same shared pages as the lazy path
        nb_entries0 = nb.entries.clone()

        def reset_nb():
            nb.entries.copy_(nb_entries0)

        gn_pre, gn_dec = graphs(nb, reset_nb)
        n_n = max(3, min(args.steps, 10))
        r_n = run_phases(gn_pre, gn_dec, reset_nb, n_n + 1)[1:]
        n_pre = statistics.mean(x[1] for x in r_n)
        n_dec = statistics.mean(sum(x[2]) for x in r_n)
        norope = {"prefill_ms": round(n_pre, 4), "decode_ms": round(n_dec, 4),
                  "prefill_overhead": round(local["pre_ms"] / n_pre, 3) if b.total_q and n_pre else None,
                  "decode_overhead": round(local["dec_s"] * 1e3 / n_dec, 3) if T and n_dec else None,
                  "note": "same kernels and pages, rotation off; overhead = lazy time / no-RoPE time"}

    dec_gbs = replica_throughput(dec_total_bytes, local["dec_s"], world) if T else 0.0
    pre_tflops = prefill_flops / (local["pre_ms"] / 1e3) / 1e12 if b.total_q else 0.0
    mean_call = statistics.mean(call_ms) if call_ms else 0.0
    per_call_bytes = dec_total_bytes / max(T, 1)
    per_call_uniq = uniq_total_bytes / max(T, 1)
    achieved = dec_total_bytes / local["dec_s"] / 1e9 if T else 0.0            # one GPU's decode calls
    achieved_dram = uniq_total_bytes / local["dec_s"] / 1e9 if T else 0.0
    warm_pre = statistics.median(p for _, p, _ in warm)
    warm_dec = statistics.median(sum(d) for _, _, d in warm)
    line = {
        "metric": METRIC, "value": round(dec_gbs, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(local["step_ms"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": cfg.name, "requests": R, "docs_per_request": cfg.docs_per_request,
                   "doc_len": (f"{cfg.doc_len_min}..{cfg.doc_len}" if cfg.doc_len_min else cfg.doc_len),
                   "pool_docs": cfg.n_docs if not args.used_docs else f"{cfg.n_docs} (only used ones stored)",
                   "q_heads": cfg.n_q_heads,
                   "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim, "query_len": cfg.q_len,
                   "decode_steps": T, "zipf_alpha": cfg.zipf_alpha, "seed": cfg.seed,
                   "l2": "flushed (256 MB write) before the prefill and before every decode call, "
                         "outside the timed events",
                   "parallelism": f"replicas x{world}",
                   "keys": args.keys, "position_encoding": args.pos, "rope": args.rope,
                   "rope_interleaved": args.interleaved},
        "prefill_tflops": round(pre_tflops, 2), "ttft_ms": round(local["pre_ms"], 4),
        "decode_ms_per_token_step": round(mean_call, 4),
        "decode_ms_per_step_all_calls": round(local["dec_s"] * 1e3, 4),
        "median_step_ms": round(statistics.median(step_ms), 4),
        "warm_l2": {"ttft_ms": round(warm_pre, 4),
                    "decode_gbs": round(dec_total_bytes / (warm_dec / 1e3) / 1e9, 1) if T and warm_dec else None,
                    "prefill_tflops": round(prefill_flops / (warm_pre / 1e3) / 1e12, 2) if b.total_q and warm_pre else None,
                    "note": "median of passes without any L2 flush"},
        "timing": "CUDA events on the launching stream around CUDA-graph replays: one graph for the prefill "
                  "launch, one per decode call (append + attention)",
        "frac_hbm_peak": round(achieved / hbm_peak, 4),
        "frac_tensor_peak": round(pre_tflops / world / tc_peak, 4),
        "decode_plan": plan_info,
        "roofline": {"kernel": ("lazyattn_decode with a decode plan (append + document-major units + combine)"
                                if use_plan else "lazyattn_decode (append + split-K attention)"), "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "frac_logical": round(achieved / hbm_peak, 4),
                     "achieved_dram": round(achieved_dram, 1),
                     "frac_dram": round(achieved_dram / hbm_peak, 4),
                     "traffic": measured_traffic(cfg.name, "decode"),
                     "traffic_unit": "bytes per decode call (DRAM read + write, ncu)",
                     "algorithmic_bytes_per_call": round(per_call_bytes),
                     "unique_bytes_per_call": round(per_call_uniq),
                     "note": "achieved/frac: logical K+V bytes of every request's context (the 2LD model) per "
                             "second of decode; achieved_dram/frac_dram: the distinct (page, KV head) tiles a "
                             "call reads (a document shared by several requests counted once) per second",
                     "peak_kind": peak_kind},
        "prefill_roofline": {"kernel": "prefill_tc_kernel", "bound": "tensor", "achieved": round(pre_tflops, 2),
                             "peak": tc_peak, "unit": "TFLOP/s", "frac": round(pre_tflops / tc_peak, 4),
                             "frac_sustained_peak": round(pre_tflops / tc_sust, 4),
                             "traffic": measured_traffic(cfg.name, "prefill"),
                             "traffic_unit": "bytes per launch (DRAM read + write, ncu)", "peak_kind": peak_kind},
        "materialising_baseline": None if base is None else {
            "materialise_ms": round(base[0], 4), "ttft_ms": round(base[0] + base[1], 4),
            "decode_ms": round(base[2], 4),
            "decode_gbs": round(dec_total_bytes / (base[2] / 1e3) / 1e9, 1) if base[2] else None,
            "lazy_ttft_speedup": round((base[0] + base[1]) / local["pre_ms"], 3) if local["pre_ms"] else None,
            "lazy_decode_speedup": round(base[2] / (local["dec_s"] * 1e3), 3) if local["dec_s"] else None,
            "lazy_step_speedup": round((base[0] + base[1] + base[2]) / local["step_ms"], 3)},
        "norope": norope,
        "e2e": e2e,
        "gpu_launches": args.steps * ((1 if b.total_q else 0) + (3 if use_plan else 2) * T),
        "wall_s_timed": round(local["wall"], 4),
        "device_status": status,
    }
    line["clocks"] = clk.summary()
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, budget_s=args.cpu_budget)
    return line


def replica_throughput(bytes_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job GB/s of N replicas (weak scaling): every rank runs the whole
    workload on its own GPU, so the job moves world x the bytes of one rank in
    the slowest rank's time (seconds_max, the max over ranks)."""
    return world * bytes_per_rank / seconds_max / 1e9


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


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _request_inputs(cfg, r, steps):
    import workload
    docs = workload.request_docs(cfg)
    ctx = [workload.doc_kv(cfg, int(d)) for d in docs[r]]
    if cfg.q_len:
        q, kq, vq = workload.query_segment(cfg, r)
    else:
        q = np.zeros((0, cfg.n_q_heads, cfg.head_dim), np.float32)
        kq = np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
        vq = kq.copy()
    st = [tuple(a[0] for a in workload.decode_inputs(cfg, t, [r])) for t in range(steps)]
    return ctx, q, kq, vq, st


def cpu_baseline(cfg, budget_s=15.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload, on
    the host cores: decode steps of whole requests (every step attends over
    the request's full context) for about half the budget, then whole
    requests' prefill for the other half. Input generation is not timed."""
    import oracle
    esz = 4 if cfg.dtype == "f32" else 2
    steps = min(cfg.decode_steps, 16)
    dec_bytes = dec_s = 0.0
    dec_req = 0
    pre_flops = pre_s = 0.0
    pre_req = 0
    for r in range(cfg.n_requests):
        if dec_s >= budget_s / 2 or not steps:
            break
        ctx, _, kq, vq, st = _request_inputs(cfg, r, steps)
        ts = time.perf_counter()
        oracle.decode_request(ctx, kq, vq, st, cfg.rope_theta)
        dec_s += time.perf_counter() - ts
        L0 = sum(a[0].shape[0] for a in ctx)
        dec_bytes += sum(2.0 * (L0 + cfg.q_len + t + 1) * cfg.n_kv_heads * cfg.head_dim * esz for t in range(steps))
        dec_req += 1
    for r in range(cfg.n_requests):
        if pre_s >= budget_s / 2 or not cfg.q_len:
            break
        ctx, q, kq, vq, _ = _request_inputs(cfg, r, 0)
        ts = time.perf_counter()
        oracle.prefill_request(ctx, q, kq, vq, cfg.rope_theta)
        pre_s += time.perf_counter() - ts
        L0 = sum(a[0].shape[0] for a in ctx)
        pre_flops += 4.0 * cfg.head_dim * (cfg.q_len * L0 + cfg.q_len * (cfg.q_len + 1) // 2) * cfg.n_q_heads
        pre_req += 1
    out = {"value": round(dec_bytes / dec_s / 1e9, 4) if dec_s else None, "unit": UNIT,
           "cores": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle",
           "threads": "numpy (fp64) with its BLAS thread pool on all host cores",
           "sample": f"decode: {dec_req} request(s) x {steps} step(s) of {cfg.name} ({dec_s:.1f} s of oracle time); "
                     f"prefill: {pre_req} request(s) ({pre_s:.1f} s); input generation not timed"}
    if pre_req:
        out["prefill"] = {"value": round(pre_flops / pre_s / 1e12, 6), "unit": "TFLOP/s",
                          "ms_per_request": round(pre_s / pre_req * 1e3, 1), "requests": pre_req}
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one decode step of one
    request of the workload (a bounded sample), timed on the host cores."""
    if rank != 0:
        return None
    import oracle
    import workload
    cfg = workload.CONFIGS[args.config]
    esz = 4 if cfg.dtype == "f32" else 2
    n_req = min(cfg.n_requests, 4)
    inputs = {r: _request_inputs(cfg, r, 1) for r in range(n_req)}   # not timed

    def one(i):
        ctx, _, kq, vq, st = inputs[i % n_req]
        ts = time.perf_counter()
        oracle.decode_request(ctx, kq, vq, st, cfg.rope_theta)
        el = time.perf_counter() - ts
        L0 = sum(a[0].shape[0] for a in ctx)
        return el, 2.0 * (L0 + cfg.q_len + 1) * cfg.n_kv_heads * cfg.head_dim * esz

    for i in range(args.warmup):
        one(i)
    res = [one(i) for i in range(args.steps)]
    el = sum(x[0] for x in res)
    v = sum(x[1] for x in res) / el / 1e9
    sample = (f"{args.steps} decode step(s), one request each (requests 0..{n_req - 1} in turn) of {cfg.name}, "
              "fp64 numpy; input generation not timed")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "kind": "oracle", "cores": os.cpu_count(),
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the baseline and end-to-end legs")
    ap.add_argument("--requests", type=int, default=0, help="use only the first N requests (profiling captures)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--decode-steps", type=int, default=-1,
                    help="use only the first N decode steps of the workload (profiling captures)")
    ap.add_argument("--used-docs", action="store_true",
                    help="store only the documents the requests use (profiling captures; launches are unchanged)")
    ap.add_argument("--e2e-reps", type=int, default=20, help="repetitions of each end-to-end leg (median)")
    ap.add_argument("--no-plan", action="store_true",
                    help="decode request by request (no document-major plan)")
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

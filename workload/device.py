"""Upload a synthetic workload into a lazyattn pool on the GPU.

Stores every pool document (pre-RoPE K/V) with lazyattn_store_doc, stores each
request's query-segment K/V in private writable pages, reserves writable pages
for generated tokens, and builds the block tables. Input plumbing only.
"""
from __future__ import annotations

import types
from typing import Optional, Sequence

import numpy as np
import torch

from . import Config, PAGE_SIZE, decode_inputs, doc_kv, doc_lengths, query_segment, request_docs, request_layout


def _generate_docs(cfg: Config, doc_ids: Sequence[int], window: int = 64):
    """(doc id, (k, v)) in the order of doc_ids. Documents are drawn by a pool of
    host threads (each from its own seeded stream, so the values do not depend
    on the threading), at most `window` ahead of the consumer to bound host
    memory; pages are still handed out in doc_ids order."""
    import concurrent.futures
    import os
    workers = max(1, min(16, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        pending = []
        it = iter(doc_ids)
        for d in it:
            pending.append((d, ex.submit(doc_kv, cfg, d)))
            if len(pending) >= window:
                break
        while pending:
            d, fut = pending.pop(0)
            nxt = next(it, None)
            if nxt is not None:
                pending.append((nxt, ex.submit(doc_kv, cfg, nxt)))
            yield d, fut.result()


def to_device(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
    return t if dtype == "f32" else t.to(torch.bfloat16)


def setup(cfg: Config, requests: Optional[Sequence[int]] = None, baseline: bool = False,
          extra_pages: int = 0, device="cuda", all_docs: bool = True, key_storage: str = "position_free",
          position_encoding: str = "rope", rope_scaling=None, rope_interleaved: bool = False):
    """Build pool + tables for `requests` (default: all) of cfg.

    all_docs=False stores only the documents those requests use (the pool is
    still sized for every document). baseline=True reserves room for the
    materialising baseline's private copies. key_storage selects the pool's key
    layout ("position_free" or "doc_local"); every stored run (a document, a
    query segment) is its own document, so its entries' delta is its start.
    position_encoding, rope_scaling and rope_interleaved pass through to the
    pool (see DevicePool).
    """
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment

    reqs = list(range(cfg.n_requests)) if requests is None else list(requests)
    docs = request_docs(cfg)
    R = len(reqs)
    lens = doc_lengths(cfg)
    dpages = -(-lens // PAGE_SIZE)
    per_req = cfg.q_pages + cfg.decode_pages
    base_pages = sum(int(dpages[docs[r]].sum()) + per_req for r in reqs) if baseline else 0
    num_pages = int(dpages.sum()) + R * per_req + base_pages + extra_pages
    pool = DevicePool(num_pages, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.dtype, cfg.rope_theta,
                      cfg.max_position, device, key_storage=key_storage, position_encoding=position_encoding,
                      rope_scaling=rope_scaling, rope_interleaved=rope_interleaved)
    doc_ids = list(range(cfg.n_docs)) if all_docs else sorted({int(d) for r in reqs for d in docs[r]})
    doc_pages = {}
    for d, (k, v) in _generate_docs(cfg, doc_ids):
        doc_pages[d] = pool.store_doc(to_device(k, cfg.dtype, device), to_device(v, cfg.dtype, device))
    segs, qs, q_starts = [], [], []
    for r in reqs:
        s = []
        starts = request_layout(cfg, r)
        for i, d in enumerate(docs[r]):
            s.append(Segment(doc_pages[int(d)], starts[i], int(lens[d]), False))
        ctx = starts[-1]
        if cfg.q_len:
            q, kq, vq = query_segment(cfg, r)
            qs.append(q)
            pages = pool.store_doc(to_device(kq, cfg.dtype, device), to_device(vq, cfg.dtype, device))
            s.append(Segment(pages, ctx, cfg.q_len, True))
            q_starts.append(ctx)
        if cfg.decode_pages:
            pages = pool.alloc_pages(cfg.decode_pages)
            s.append(Segment(pages, ctx + cfg.q_pages * PAGE_SIZE, 0, True))
        segs.append(s)
    q_lens = [cfg.q_len] * R if cfg.q_len else []
    batch = Batch(segs, q_lens, q_starts, device)
    batch.check(num_pages, cfg.max_position)   # every table in range, one token per logical position
    q = to_device(np.concatenate(qs), cfg.dtype, device) if qs else None
    torch.cuda.synchronize()
    return types.SimpleNamespace(cfg=cfg, pool=pool, batch=batch, q=q, requests=reqs, docs=docs,
                                 doc_pages=doc_pages, segments=segs)


def decode_step_tensors(cfg: Config, step: int, requests: Sequence[int], device="cuda"):
    q, k, v = decode_inputs(cfg, step, requests)
    return to_device(q, cfg.dtype, device), to_device(k, cfg.dtype, device), to_device(v, cfg.dtype, device)

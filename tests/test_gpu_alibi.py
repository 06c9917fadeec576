"""GPU parity of the ALiBi pool mode (§3.5 "Score-space positional methods":
the bias is added to the score from logical positions, so documents are
reused at any offset without copies) against the oracle's own ALiBi: prefill
of two requests sharing a document at different offsets, then decode steps,
for a power-of-two head count and one that is not (24 query heads).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workload
import workload.device  # noqa: F401
from tests.gpu_common import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


@pytest.mark.parametrize("hq,hkv", [(32, 8), (24, 6)])
def test_alibi_prefill_and_decode(L, hq, hkv):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    cfg = dataclasses.replace(workload.CONFIGS["llama3_8b"], n_q_heads=hq, n_kv_heads=hkv)
    spec = oracle.AlibiSpec()
    rng = np.random.default_rng(21)
    plan = [([4, 5, 4], 29), ([5, 6], 29)]
    ql, steps = 29, 3
    used = sorted({d for docs, _ in plan for d in docs})
    n_pages = len(used) * cfg.doc_pages + len(plan) * (-(-(ql + steps) // 16) + 1) + 4
    max_pos = max(len(docs) for docs, _ in plan) * cfg.doc_len + ql + steps + 16
    pool = DevicePool(n_pages, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.dtype, cfg.rope_theta, max_pos,
                      position_encoding="alibi")
    dev = lambda a: workload.device.to_device(a, cfg.dtype)   # noqa: E731
    rnd = lambda shape: workload.round_bf16(rng.standard_normal(shape).astype(np.float32))   # noqa: E731
    doc_pages = {d: pool.store_doc(dev(workload.doc_kv(cfg, d)[0]), dev(workload.doc_kv(cfg, d)[1])) for d in used}
    segs, qs, kqs, vqs, starts = [], [], [], [], []
    for docs, n in plan:
        s = [Segment(doc_pages[d], i * cfg.doc_len, cfg.doc_len) for i, d in enumerate(docs)]
        q, kq, vq = rnd((n, hq, cfg.head_dim)), rnd((n, hkv, cfg.head_dim)), rnd((n, hkv, cfg.head_dim))
        start = len(docs) * cfg.doc_len
        s.append(Segment(pool.store_doc(dev(kq), dev(vq)), start, n, True))
        segs.append(s)
        qs.append(q); kqs.append(kq); vqs.append(vq); starts.append(start)
    batch = Batch(segs, [ql] * len(plan), starts)

    out = torch.full((batch.total_q, hq, cfg.head_dim), float("nan"), dtype=pool.tdtype, device="cuda")
    L.lazyattn_prefill(pool.handle, batch.c, dev(np.concatenate(qs)), out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    for i, (docs, n) in enumerate(plan):
        ref = oracle.prefill_request([workload.doc_kv(cfg, d) for d in docs], qs[i], kqs[i], vqs[i], spec)
        compare(got[i * ql:(i + 1) * ql], ref, "bf16")

    ws_bytes = L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_DECODE, batch.c)
    ws = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device="cuda")
    step_in = [(rnd((len(plan), hq, cfg.head_dim)), rnd((len(plan), hkv, cfg.head_dim)),
                rnd((len(plan), hkv, cfg.head_dim))) for _ in range(steps)]
    outs = []
    for q, k, v in step_in:
        o = torch.empty((len(plan), hq, cfg.head_dim), dtype=pool.tdtype, device="cuda")
        L.lazyattn_decode(pool.handle, batch.c, dev(q), dev(k), dev(v), o, ws, ws_bytes)
        torch.cuda.synchronize()
        outs.append(o.float().cpu().numpy())
    for i, (docs, n) in enumerate(plan):
        ref = oracle.decode_request([workload.doc_kv(cfg, d) for d in docs], kqs[i], vqs[i],
                                    [(step_in[t][0][i], step_in[t][1][i], step_in[t][2][i]) for t in range(steps)],
                                    spec)
        for t in range(steps):
            compare(outs[t][i], ref[t], "bf16")
    assert pool.device_status() == 0

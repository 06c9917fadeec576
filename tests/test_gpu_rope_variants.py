"""GPU parity of the RoPE-family variants (§3.5 "RoPE-family variants": scaled
/ NTK and YaRN keep the score form; the kernels take the variant's position
table and logit scale) against the fp64 oracle's own restatement of each
variant: prefill of two requests that share a document at different offsets,
then two decode steps, for bf16 (both key layouts) and for the fp32 path.
"""
import numpy as np
import pytest
import torch

import oracle
import workload
import workload.device  # noqa: F401
from oracle import RopeSpec
from tests.gpu_common import compare

pytestmark = pytest.mark.gpu

VARIANTS = {
    "linear": dict(kind="linear", factor=4.0),
    "ntk": dict(kind="ntk", factor=8.0),
    "yarn": dict(kind="yarn", factor=8.0, original_max_position=256, low=1.0, high=32.0),
    "llama3": dict(kind="llama3", factor=8.0, original_max_position=512, low=1.0, high=4.0),
    "interleaved": dict(kind="default", factor=1.0, interleaved=True),
    "yarn+interleaved": dict(kind="yarn", factor=8.0, original_max_position=256, low=1.0, high=32.0,
                             interleaved=True),
}


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


def _spec(cfg, v):
    return RopeSpec(cfg.rope_theta, v["kind"], v["factor"], v.get("original_max_position", 0), v.get("low", 0.0),
                    v.get("high", 0.0), "interleaved" if v.get("interleaved") else "half")


@pytest.mark.parametrize("config,keys", [("llama3_8b", "position_free"), ("llama3_8b", "doc_local"),
                                         ("tiny_fp32", "position_free")])
@pytest.mark.parametrize("variant", list(VARIANTS))
def test_rope_variant_prefill_and_decode(L, config, keys, variant):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    cfg = workload.CONFIGS[config]
    v = VARIANTS[variant]
    if v.get("interleaved") and cfg.dtype != "bf16":
        pytest.skip("interleaved pairing is supported for bf16 pools")
    spec = _spec(cfg, v)
    rng = np.random.default_rng(11)
    plan = [([1, 2, 1], 21), ([2, 3], 21)]   # document 1 twice in one request; document 2 at two offsets
    ql, steps = 21, 2
    used = sorted({d for docs, _ in plan for d in docs})
    n_pages = len(used) * cfg.doc_pages + len(plan) * (-(-(ql + steps) // 16) + 1) + 4
    max_pos = max(len(docs) for docs, _ in plan) * cfg.doc_len + ql + steps + 16
    scaling = None if v["kind"] == "default" else {x: y for x, y in v.items() if x != "interleaved"}
    pool = DevicePool(n_pages, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.dtype, cfg.rope_theta, max_pos,
                      rope_scaling=scaling, rope_interleaved=bool(v.get("interleaved")), key_storage=keys)
    dev = lambda a: workload.device.to_device(a, cfg.dtype)   # noqa: E731
    rnd = lambda shape: workload.round_bf16(rng.standard_normal(shape).astype(np.float32)) \
        if cfg.dtype == "bf16" else rng.standard_normal(shape).astype(np.float32)   # noqa: E731
    doc_pages = {d: pool.store_doc(dev(workload.doc_kv(cfg, d)[0]), dev(workload.doc_kv(cfg, d)[1])) for d in used}
    segs, qs, kqs, vqs, starts = [], [], [], [], []
    for docs, n in plan:
        s = [Segment(doc_pages[d], i * cfg.doc_len, cfg.doc_len) for i, d in enumerate(docs)]
        q, kq, vq = rnd((n, cfg.n_q_heads, cfg.head_dim)), rnd((n, cfg.n_kv_heads, cfg.head_dim)), \
            rnd((n, cfg.n_kv_heads, cfg.head_dim))
        start = len(docs) * cfg.doc_len
        s.append(Segment(pool.store_doc(dev(kq), dev(vq)), start, n, True))
        segs.append(s)
        qs.append(q); kqs.append(kq); vqs.append(vq); starts.append(start)
    batch = Batch(segs, [ql] * len(plan), starts)

    out = torch.full((batch.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=pool.tdtype, device="cuda")
    L.lazyattn_prefill(pool.handle, batch.c, dev(np.concatenate(qs)), out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    for i, (docs, n) in enumerate(plan):
        ref = oracle.prefill_request([workload.doc_kv(cfg, d) for d in docs], qs[i], kqs[i], vqs[i], spec)
        compare(got[i * ql:(i + 1) * ql], ref, cfg.dtype)

    ws_bytes = L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_DECODE, batch.c)
    ws = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device="cuda")
    step_in = [(rnd((len(plan), cfg.n_q_heads, cfg.head_dim)), rnd((len(plan), cfg.n_kv_heads, cfg.head_dim)),
                rnd((len(plan), cfg.n_kv_heads, cfg.head_dim))) for _ in range(steps)]
    outs = []
    for q, k, vv in step_in:
        o = torch.empty((len(plan), cfg.n_q_heads, cfg.head_dim), dtype=pool.tdtype, device="cuda")
        L.lazyattn_decode(pool.handle, batch.c, dev(q), dev(k), dev(vv), o, ws, ws_bytes)
        torch.cuda.synchronize()
        outs.append(o.float().cpu().numpy())
    for i, (docs, n) in enumerate(plan):
        ref = oracle.decode_request([workload.doc_kv(cfg, d) for d in docs], kqs[i], vqs[i],
                                    [(step_in[t][0][i], step_in[t][1][i], step_in[t][2][i]) for t in range(steps)],
                                    spec)
        for t in range(steps):
            compare(outs[t][i], ref[t], cfg.dtype)
    assert pool.device_status() == 0

"""GPU parity of the tcgen05 prefill kernel against the fp64 oracle.

Covers the Llama-3-8B-shaped workload in full, the materialising baseline,
ragged query lengths (several 128-row tiles plus a ragged tail, a single-token
query), a request whose only keys are its own query segment, a document shared
by two requests at different offsets (zero copy: same physical pages), empty
entries inside a table, and the bigger workloads on sampled requests.
"""
import numpy as np
import pytest
import torch

import oracle
import workload
import workload.device  # noqa: F401
from tests.gpu_common import Reference, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


def _prefill(L, env, batch=None):
    b = batch or env.batch
    cfg = env.cfg
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_prefill_llama3_8b_all_requests(L):
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg)
    ref = Reference(cfg)
    got = _prefill(L, env).reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    errs = [compare(got[r], ref.prefill(r), "bf16") for r in range(cfg.n_requests)]
    print("prefill llama3_8b worst max-abs %.3e rel-L2 %.3e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_prefill_materialised_baseline(L):
    cfg = workload.CONFIGS["llama3_8b"]
    reqs = [1, 4, 9]
    env = workload.device.setup(cfg, requests=reqs, baseline=True, all_docs=False)
    ref = Reference(cfg)
    b = env.batch
    new_pages = env.pool.alloc_pages(len(b.entries_host))
    dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.array(new_pages, np.uint64)
    L.lazyattn_materialize(env.pool.handle, b.c, torch.from_numpy(dst.view(np.int64).copy()).cuda())
    mb = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED)
    got = _prefill(L, env, mb).reshape(len(reqs), cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    for i, r in enumerate(reqs):
        compare(got[i], ref.prefill(r), "bf16")
    assert env.pool.device_status() == 0


def _custom(L, cfg, plan, seed):
    """plan: list of (doc ids, q_len). Documents come from cfg's pool; the query
    segments are drawn here. Returns env-like namespace and oracle outputs."""
    import types
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    rng = np.random.default_rng(seed)
    used = sorted({d for docs, _ in plan for d in docs})
    n_pages = len(used) * cfg.doc_pages + sum(-(-q // 16) + 1 for _, q in plan) + 4
    max_pos = max(len(docs) * cfg.doc_len + q for docs, q in plan) + 16
    pool = DevicePool(n_pages, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.dtype, cfg.rope_theta, max_pos)
    dp = {}
    for d in used:
        k, v = workload.doc_kv(cfg, d)
        dp[d] = pool.store_doc(workload.device.to_device(k, cfg.dtype), workload.device.to_device(v, cfg.dtype))
    segs, qs, refs, starts = [], [], [], []
    for docs, ql in plan:
        s = [Segment(dp[d], i * cfg.doc_len, cfg.doc_len) for i, d in enumerate(docs)]
        # an empty entry inside the table must contribute nothing
        s.append(Segment(pool.alloc_pages(1), 0, 0))
        q = workload.round_bf16(rng.standard_normal((ql, cfg.n_q_heads, cfg.head_dim)).astype(np.float32))
        kq = workload.round_bf16(rng.standard_normal((ql, cfg.n_kv_heads, cfg.head_dim)).astype(np.float32))
        vq = workload.round_bf16(rng.standard_normal((ql, cfg.n_kv_heads, cfg.head_dim)).astype(np.float32))
        start = len(docs) * cfg.doc_len
        pages = pool.store_doc(workload.device.to_device(kq, cfg.dtype), workload.device.to_device(vq, cfg.dtype))
        s.append(Segment(pages, start, ql, True))
        segs.append(s)
        qs.append(q)
        starts.append(start)
        refs.append(oracle.prefill_request([workload.doc_kv(cfg, d) for d in docs], q, kq, vq, cfg.rope_theta))
    batch = Batch(segs, [ql for _, ql in plan], starts)
    env = types.SimpleNamespace(cfg=cfg, pool=pool, batch=batch,
                                q=workload.device.to_device(np.concatenate(qs), cfg.dtype), segments=segs)
    return env, refs


def test_prefill_ragged_tiles_and_edge_requests(L):
    cfg = workload.CONFIGS["llama3_8b"]
    plan = [([3, 7, 3], 37),        # several tiles of 32 tokens, ragged tail; doc 3 twice
            ([], 100),              # only its own query segment (causal within it)
            ([11], 1),              # a single query token
            ([0, 1, 2, 5, 6], 64)]
    env, refs = _custom(L, cfg, plan, 5)
    got = _prefill(L, env)
    off = 0
    for (docs, ql), ref in zip(plan, refs):
        compare(got[off:off + ql], ref, "bf16")
        off += ql
    assert env.pool.device_status() == 0


def test_prefill_shared_document_zero_copy(L):
    """(c) one physical copy of a document serves two requests at different
    offsets: both tables name the same pages, both outputs match the oracle."""
    cfg = workload.CONFIGS["llama3_8b"]
    plan = [([42, 17], 48), ([17, 42, 99], 48)]
    env, refs = _custom(L, cfg, plan, 6)
    p0 = env.segments[0][1].pages
    p1 = env.segments[1][0].pages
    assert list(p0) == list(p1)
    got = _prefill(L, env)
    compare(got[:48], refs[0], "bf16")
    compare(got[48:], refs[1], "bf16")


@pytest.mark.parametrize("name,sample", [("ttft_sweep_10", [0, 13, 31]), ("llama3_70b", [37])])
def test_prefill_large_configs_sampled(L, name, sample):
    """Full-size pools and tables; the oracle checks the sampled requests."""
    cfg = workload.CONFIGS[name]
    env = workload.device.setup(cfg, requests=sample, all_docs=False)
    ref = Reference(cfg)
    got = _prefill(L, env).reshape(len(sample), cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    for i, r in enumerate(sample):
        compare(got[i], ref.prefill(r), "bf16")
    assert env.pool.device_status() == 0

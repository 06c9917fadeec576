"""Document-major decode (a decode plan in the batch) against the fp64 oracle.

The plan groups the pages of a batch's tables into runs that several requests
read; decode then reads each run once per group of readers, rotates its keys
at run-local positions and each reader's q at m - delta. These tests run the
plan path on the workloads' own tables (shared Zipf documents, ragged few-shot
chunks that end in partial pages mid-table, the tail run filling up across
steps) and on the pool layouts (position-free, doc-local, ALiBi, the
materialising baseline's private pre-rotated pages), and check the host-side
rules of plans (which batches a plan fits).
"""
import numpy as np
import pytest
import torch

import workload
import workload.device  # noqa: F401
from tests.gpu_common import Reference, compare, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


@pytest.mark.parametrize("name,requests,steps,check", [
    ("llama3_8b", None, 32, range(16)),
    ("few_shot_skewed", None, 4, [0, 1, 2, 3, 64, 127]),
    ("few_shot_uniform", list(range(0, 128, 3)), 4, [0, 5, 10]),
])
def test_plan_decode_against_oracle(L, name, requests, steps, check):
    cfg = workload.CONFIGS[name]
    env = workload.device.setup(cfg, requests=requests, all_docs=False)
    entries0 = env.batch.entries.clone()
    stats = env.batch.plan_decode(env.pool)
    assert stats["pass_pages"] <= stats["logical_pages"]
    outs = run_decode(L, env, steps)
    assert env.pool.device_status() == 0
    ref = Reference(cfg)
    reqs = env.requests
    errs = []
    for i in check:
        want = ref.decode(reqs[i], steps)
        errs += [compare(outs[t][i], want[t], "bf16") for t in range(steps)]
    # the same table decoded request by request (no plan) agrees too
    env.batch.drop_plan()
    env.batch.entries.copy_(entries0)
    outs2 = run_decode(L, env, steps)
    for t in range(steps):
        compare(outs[t], outs2[t], "bf16")
    print("%s plan decode: %s; worst max-abs %.3e rel-L2 %.3e"
          % (name, stats, max(e[0] for e in errs), max(e[1] for e in errs)))


@pytest.mark.parametrize("keys,pos", [("doc_local", "rope"), ("position_free", "alibi")])
def test_plan_decode_layouts(L, keys, pos):
    import oracle
    cfg = workload.CONFIGS["llama3_8b"]
    reqs = [0, 2, 5, 7, 11]
    env = workload.device.setup(cfg, requests=reqs, all_docs=False, key_storage=keys, position_encoding=pos)
    env.batch.plan_decode(env.pool)
    steps = 6
    outs = run_decode(L, env, steps)
    assert env.pool.device_status() == 0
    ref = Reference(cfg)
    positional = oracle.AlibiSpec() if pos == "alibi" else cfg.rope_theta
    for i, r in enumerate(reqs):
        _, kq, vq = ref.qseg(r)
        st = [tuple(a[0] for a in workload.decode_inputs(cfg, t, [r])) for t in range(steps)]
        want = oracle.decode_request(ref.ctx(r), kq, vq, st, positional)
        for t in range(steps):
            compare(outs[t][i], want[t], "bf16")


def test_plan_decode_materialised_baseline(L):
    """The baseline's private pre-rotated copies through a plan: no run is
    shared, every run is read by one request, q is rotated at m."""
    cfg = workload.CONFIGS["llama3_8b"]
    reqs = [1, 4, 9]
    env = workload.device.setup(cfg, requests=reqs, all_docs=False, baseline=True)
    b = env.batch
    dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.array(env.pool.alloc_pages(len(b.entries_host)), np.uint64)
    L.lazyattn_materialize(env.pool.handle, b.c, torch.from_numpy(dst.view(np.int64).copy()).cuda())
    mb = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED)
    stats = mb.plan_decode(env.pool)
    assert stats["max_readers"] == 1
    steps = 5
    outs = run_decode(L, env, steps, batch=mb)
    assert env.pool.device_status() == 0
    ref = Reference(cfg)
    for i, r in enumerate(reqs):
        want = ref.decode(r, steps)
        for t in range(steps):
            compare(outs[t][i], want[t], "bf16")


def test_plan_shares_documents(L):
    """A document placed at two offsets in two requests (and twice in one) is
    one run with three readers; the batch decodes to the oracle's outputs."""
    import oracle
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    hq, hkv, D, theta = 32, 8, 128, 5.0e5
    rng = np.random.default_rng(71)
    rnd = lambda *s: workload.round_bf16(rng.standard_normal(s).astype(np.float32))  # noqa: E731
    pool = DevicePool(64, hq, hkv, D, "bf16", theta, 2048)
    dev = lambda a: workload.device.to_device(a, "bf16")  # noqa: E731
    A = (rnd(90, hkv, D), rnd(90, hkv, D))      # 6 pages, the last one partial
    B = (rnd(40, hkv, D), rnd(40, hkv, D))
    pa = pool.store_doc(dev(A[0]), dev(A[1]))
    pb = pool.store_doc(dev(B[0]), dev(B[1]))
    layouts = [[A, B], [B, A, A]]
    segs = []
    for docs in layouts:
        s, p = [], 0
        for d in docs:
            s.append(Segment(pa if d is A else pb, p, d[0].shape[0]))
            p += d[0].shape[0]
        s.append(Segment(pool.alloc_pages(1), p, 0, True))
        segs.append(s)
    batch = Batch(segs)
    stats = batch.plan_decode(pool)
    assert stats["runs"] == 2 + 2 and stats["max_readers"] == 3, stats
    nbytes = L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_DECODE, batch.c)
    ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device="cuda")
    ctx = [[*docs] for docs in layouts]
    news = [[], []]
    for t in range(3):
        q, k, v = rnd(2, hq, D), rnd(2, hkv, D), rnd(2, hkv, D)
        out = torch.empty((2, hq, D), dtype=torch.bfloat16, device="cuda")
        L.lazyattn_decode(pool.handle, batch.c, dev(q), dev(k), dev(v), out, ws, nbytes)
        torch.cuda.synchronize()
        for r in range(2):
            news[r].append((q[r], k[r], v[r]))
            empty = np.zeros((0, hkv, D), np.float32)
            want = oracle.decode_request(ctx[r], empty, empty, news[r], theta)[-1]
            compare(out[r].float().cpu().numpy(), want, "bf16")
    assert pool.device_status() == 0


def test_plan_rules(L):
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg, requests=[0, 1, 2], all_docs=False)
    other = workload.device.setup(cfg, requests=[0, 1], all_docs=False)
    env.batch.plan_decode(env.pool)
    # a plan built for 3 requests does not fit a batch of 2
    bad = L.make_batch(other.batch.num_requests, other.batch.max_entries, other.batch.entries,
                       other.batch.entry_offsets, decode_plan=env.batch.plan)
    assert L.lazyattn_workspace_size(other.pool.handle, L.LAZYATTN_OP_DECODE, bad) == 0
    # a plan that was never uploaded is refused
    plan = L.lazyattn_decode_plan_create(env.pool.handle, env.batch.entries_host, env.batch.offsets_host)
    nup = L.make_batch(env.batch.num_requests, env.batch.max_entries, env.batch.entries, env.batch.entry_offsets,
                       decode_plan=plan)
    assert L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, nup) == 0
    L.lazyattn_decode_plan_destroy(plan)
    # fp32 pools decode without plans
    tiny = workload.device.setup(workload.CONFIGS["tiny_fp32"], all_docs=False)
    with pytest.raises(L.LazyAttnError) as e:
        L.lazyattn_decode_plan_create(tiny.pool.handle, tiny.batch.entries_host, tiny.batch.offsets_host)
    assert e.value.code == L.LAZYATTN_EDTYPE
    # a table the host check rejects (a page past the pool) has no plan
    eh = env.batch.entries_host.copy()
    eh[3] = (eh[3] & ~np.uint64(0xFFFFFFFF)) | np.uint64(env.pool.num_pages + 5)
    with pytest.raises(L.LazyAttnError) as e:
        L.lazyattn_decode_plan_create(env.pool.handle, eh, env.batch.offsets_host)
    assert e.value.code == L.LAZYATTN_ERANGE

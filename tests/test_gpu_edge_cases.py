"""GPU edge cases of the hot path, each against the fp64 oracle or a closed form.

* A decode step whose request holds no key but its own new token: the softmax
  has one term, so the output is that token's v, bit for bit (every mode).
* Logical positions past two million (documents placed far into the context),
  for position-free and doc-local keys: the position table's rows there and
  the angle composition must still match the fp64 rotation.
* Prefill batches with requests of zero query rows next to ragged ones, an
  all-empty batch (nothing launched), and batches with no request or more
  requests than a grid dimension holds (rejected on the host).
* Query-head groups of 1 and 2 (every head its own KV head; pairs), which the
  bf16 kernels pack differently from the 4 and 8 of the model-shaped workloads.
"""
import numpy as np
import pytest
import torch

import oracle
import workload
import workload.device  # noqa: F401
from tests.gpu_common import compare

pytestmark = pytest.mark.gpu

D = 128
THETA = 5.0e5


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


def _rnd(rng, shape):
    return workload.round_bf16(rng.standard_normal(shape).astype(np.float32))


def _dev(a):
    return workload.device.to_device(a, "bf16")


def _decode(L, pool, batch, q, k, v):
    nbytes = L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_DECODE, batch.c)
    ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device="cuda")
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lazyattn_decode(pool.handle, batch.c, _dev(q), _dev(k), _dev(v), out, ws, nbytes)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("keys,pos", [("position_free", "rope"), ("doc_local", "rope"), ("position_free", "alibi")])
def test_decode_with_only_its_own_token(L, keys, pos):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    hq, hkv = 32, 8
    starts = [0, 17, 1000, 4093]
    pool = DevicePool(16, hq, hkv, D, "bf16", THETA, 4200, key_storage=keys, position_encoding=pos)
    segs = [[Segment(pool.alloc_pages(2), s, 0, True)] for s in starts]
    batch = Batch(segs)
    rng = np.random.default_rng(31)
    R = len(starts)
    steps = [(_rnd(rng, (R, hq, D)), _rnd(rng, (R, hkv, D)), _rnd(rng, (R, hkv, D))) for _ in range(3)]
    outs = [_decode(L, pool, batch, *st) for st in steps]
    # first step: one visible key, weight exactly 1
    got = outs[0].view(torch.int16).cpu().numpy()
    want = _dev(np.repeat(steps[0][2], hq // hkv, axis=1)).view(torch.int16).cpu().numpy()
    assert np.array_equal(got, want)
    # later steps against the oracle (both position encodings are shift invariant,
    # so the request's start does not enter)
    positional = oracle.AlibiSpec() if pos == "alibi" else THETA
    empty_k = np.zeros((0, hkv, D), np.float32)
    for r in range(R):
        ref = oracle.decode_request([], empty_k, empty_k, [(st[0][r], st[1][r], st[2][r]) for st in steps],
                                    positional)
        for t in (1, 2):
            compare(outs[t][r].float().cpu().numpy(), ref[t], "bf16")
    assert pool.device_status() == 0


@pytest.mark.parametrize("keys", ["position_free", "doc_local"])
def test_logical_positions_past_two_million(L, keys):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    hq, hkv, ql, n_steps = 32, 8, 29, 3
    base = (1 << 21) - 600                  # documents at [base, base + 2 * 256)
    doc_lens = [256, 200]
    max_pos = base + sum(doc_lens) + ql + n_steps + 64
    pool = DevicePool(64, hq, hkv, D, "bf16", THETA, max_pos, key_storage=keys)
    rng = np.random.default_rng(32)
    docs = [(_rnd(rng, (n, hkv, D)), _rnd(rng, (n, hkv, D))) for n in doc_lens]
    segs, p = [], base
    for k, v in docs:
        segs.append(Segment(pool.store_doc(_dev(k), _dev(v)), p, k.shape[0]))
        p += k.shape[0]
    q, kq, vq = _rnd(rng, (ql, hq, D)), _rnd(rng, (ql, hkv, D)), _rnd(rng, (ql, hkv, D))
    segs.append(Segment(pool.store_doc(_dev(kq), _dev(vq)), p, ql, True))
    segs.append(Segment(pool.alloc_pages(1), p + 32, 0, True))
    batch = Batch([segs], [ql], [p])
    out = torch.full((ql, hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lazyattn_prefill(pool.handle, batch.c, _dev(q), out)
    torch.cuda.synchronize()
    k_all = np.concatenate([d[0] for d in docs] + [kq])
    v_all = np.concatenate([d[1] for d in docs] + [vq])
    k_pos = np.arange(base, base + k_all.shape[0])
    ref = oracle.attention(q, k_all, v_all, np.arange(p, p + ql), k_pos, THETA)
    compare(out.float().cpu().numpy(), ref, "bf16")
    for t in range(n_steps):
        qd, kd, vd = _rnd(rng, (1, hq, D)), _rnd(rng, (1, hkv, D)), _rnd(rng, (1, hkv, D))
        o = _decode(L, pool, batch, qd, kd, vd)
        k_all = np.concatenate([k_all, kd])
        v_all = np.concatenate([v_all, vd])
        k_pos = np.arange(base, base + k_all.shape[0])
        ref = oracle.attention(qd, k_all, v_all, [k_pos[-1]], k_pos, THETA)
        compare(o.float().cpu().numpy(), ref, "bf16")
    assert pool.device_status() == 0


def test_prefill_zero_row_requests_and_empty_batches(L):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    hq, hkv = 32, 8
    cfg = workload.CONFIGS["llama3_8b"]
    rng = np.random.default_rng(33)
    q_lens = [5, 0, 7, 1, 0]
    pool = DevicePool(64, hq, hkv, D, "bf16", THETA, 4096)
    doc = workload.doc_kv(cfg, 3)
    doc_pages = pool.store_doc(_dev(doc[0]), _dev(doc[1]))
    segs, qs, refs, starts = [], [], [], []
    for i, n in enumerate(q_lens):
        s = [Segment(doc_pages, 0, cfg.doc_len)]
        q, kq, vq = _rnd(rng, (n, hq, D)), _rnd(rng, (max(n, 1), hkv, D)), _rnd(rng, (max(n, 1), hkv, D))
        s.append(Segment(pool.store_doc(_dev(kq), _dev(vq)), cfg.doc_len, n, True))
        segs.append(s)
        qs.append(q)
        starts.append(cfg.doc_len)
        refs.append(oracle.prefill_request([doc], q, kq[:n], vq[:n], THETA))
    batch = Batch(segs, q_lens, starts)
    assert batch.total_q == sum(q_lens)
    out = torch.full((batch.total_q, hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lazyattn_prefill(pool.handle, batch.c, _dev(np.concatenate(qs)), out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    off = 0
    for n, ref in zip(q_lens, refs):
        compare(got[off:off + n], ref, "bf16")
        off += n
    # every request with zero rows: nothing is launched, nothing written
    empty = Batch(segs[:2], [0, 0], starts[:2])
    sentinel = torch.full((4, hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lazyattn_prefill(pool.handle, empty.c, sentinel, sentinel)
    torch.cuda.synchronize()
    assert torch.isnan(sentinel.float()).all()
    # an empty request list is an invalid batch
    none = Batch([], [], [])
    with pytest.raises(L.LazyAttnError) as err:
        L.lazyattn_prefill(pool.handle, none.c, sentinel, sentinel)
    assert err.value.code == L.LAZYATTN_EINVAL
    # more requests than a grid dimension holds: rejected on the host, nothing read
    big = L.make_batch(65536, batch.max_entries, batch.entries, batch.entry_offsets, batch.q_offsets, batch.q_start,
                       1, 1, 0, batch.entry_delta)
    with pytest.raises(L.LazyAttnError) as err:
        L.lazyattn_prefill(pool.handle, big, sentinel, sentinel)
    assert err.value.code == L.LAZYATTN_EINVAL
    assert L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_DECODE, big) == 0
    assert pool.device_status() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8)])
def test_small_head_groups(L, hq, hkv):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    cfg = workload.CONFIGS["llama3_8b"]
    rng = np.random.default_rng(34)
    ql, n_steps = 37, 2
    pool = DevicePool(96, hq, hkv, D, "bf16", THETA, 4096)
    plan = [[4, 9], [9]]
    doc_kv = {d: workload.doc_kv(cfg, d) for d in (4, 9)}
    doc_pages = {d: pool.store_doc(_dev(k), _dev(v)) for d, (k, v) in doc_kv.items()}
    segs, qs, kqs, vqs, starts = [], [], [], [], []
    for docs in plan:
        s = [Segment(doc_pages[d], i * cfg.doc_len, cfg.doc_len) for i, d in enumerate(docs)]
        q, kq, vq = _rnd(rng, (ql, hq, D)), _rnd(rng, (ql, hkv, D)), _rnd(rng, (ql, hkv, D))
        start = len(docs) * cfg.doc_len
        s.append(Segment(pool.store_doc(_dev(kq), _dev(vq)), start, ql, True))
        segs.append(s)
        qs.append(q); kqs.append(kq); vqs.append(vq); starts.append(start)
    batch = Batch(segs, [ql] * len(plan), starts)
    out = torch.full((batch.total_q, hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lazyattn_prefill(pool.handle, batch.c, _dev(np.concatenate(qs)), out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    steps = [(_rnd(rng, (len(plan), hq, D)), _rnd(rng, (len(plan), hkv, D)), _rnd(rng, (len(plan), hkv, D)))
             for _ in range(n_steps)]
    outs = [_decode(L, pool, batch, *st).float().cpu().numpy() for st in steps]
    for i, docs in enumerate(plan):
        ctx = [doc_kv[d] for d in docs]
        compare(got[i * ql:(i + 1) * ql], oracle.prefill_request(ctx, qs[i], kqs[i], vqs[i], THETA), "bf16")
        ref = oracle.decode_request(ctx, kqs[i], vqs[i], [(st[0][i], st[1][i], st[2][i]) for st in steps], THETA)
        for t in range(n_steps):
            compare(outs[t][i], ref[t], "bf16")
    assert pool.device_status() == 0

"""Numerical edges of the bf16 kernels, against the fp64 oracle.

* A "needle" document late in the context whose keys score far above every
  earlier key (a large component at the lowest RoPE frequency, where the
  rotation is nearly the identity over the whole context, met by a large
  component of every query): each row's running maximum jumps by more than
  2^8 at a K tile after the first, so prefill must rescale the partial output
  it already holds in TMEM, and decode must rescale in its page loop and merge
  splits whose maxima differ by orders of magnitude. Both key layouts and the
  materialising baseline, query-head groups of 4 and 8, decode with and
  without a decode plan.
* The documented input range (lazyattn.h, "Input range"): keys and queries at
  the largest in-range rotate-half pair norms give finite outputs equal to the
  oracle's (the fp16 operands of QK^T would be infinite past fp16's maximum,
  and 0 * inf would poison the scores); a pair past the bound is reported as
  LAZYATTN_ERANGE by lazyattn_store_doc, the decode append, lazyattn_prefill
  and lazyattn_decode. fp32 pools have no such bound.
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
ERANGE = -3


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


def _dev(a, dtype="bf16"):
    return workload.device.to_device(a, dtype)


class Request:
    """One request built by hand: documents, a query segment, decode steps; run
    through the library on a pool of the given layout."""

    def __init__(self, L, hq, hkv, docs, q, kq, vq, steps, keys="position_free", dtype="bf16", theta=THETA):
        from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
        self.L, self.dtype = L, dtype
        n_ctx = sum(k.shape[0] for k, _ in docs) + q.shape[0]
        pages = sum(-(-k.shape[0] // 16) for k, _ in docs) + 2 * (-(-(q.shape[0] + len(steps)) // 16)) + 8
        self.pool = DevicePool(2 * pages, hq, hkv, D, dtype, theta, n_ctx + len(steps) + 16, key_storage=keys)
        self.store_status = []
        segs, p = [], 0
        for k, v in docs:
            segs.append(Segment(self.pool.store_doc(_dev(k, dtype), _dev(v, dtype)), p, k.shape[0]))
            self.store_status.append(self.pool.device_status())
            p += k.shape[0]
        lq = q.shape[0]
        segs.append(Segment(self.pool.store_doc(_dev(kq, dtype), _dev(vq, dtype)), p, lq, True))
        self.store_status.append(self.pool.device_status())
        tail = -(-lq // 16) * 16
        segs.append(Segment(self.pool.alloc_pages(-(-max(len(steps) - (tail - lq), 1) // 16)), p + tail, 0, True))
        self.segs, self.q_start, self.q, self.steps = segs, p, q, steps
        self.batch = Batch([segs], [lq], [p])

    def prefill(self, batch=None):
        L = self.L
        b = batch or self.batch
        out = torch.full(self.q.shape, float("nan"), dtype=self.pool.tdtype, device="cuda")
        L.lazyattn_prefill(self.pool.handle, b.c, _dev(self.q, self.dtype), out)
        torch.cuda.synchronize()
        return out.float().cpu().numpy(), self.pool.device_status()

    def decode(self, batch=None, plan=False):
        L = self.L
        b = batch or self.batch
        if plan:
            b.plan_decode(self.pool)
        nbytes = L.lazyattn_workspace_size(self.pool.handle, L.LAZYATTN_OP_DECODE, b.c)
        ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device="cuda")
        outs, status = [], []
        for qd, kd, vd in self.steps:
            out = torch.full((1,) + qd.shape, float("nan"), dtype=self.pool.tdtype, device="cuda")
            L.lazyattn_decode(self.pool.handle, b.c, _dev(qd[None], self.dtype), _dev(kd[None], self.dtype),
                              _dev(vd[None], self.dtype), out, ws, nbytes)
            torch.cuda.synchronize()
            outs.append(out[0].float().cpu().numpy())
            status.append(self.pool.device_status())
        return outs, status

    def materialised(self):
        """The materialising baseline's batch: private copies of every page with
        K rotated at its logical positions."""
        L = self.L
        eh = self.batch.entries_host
        dst = (eh & ~np.uint64(0xFFFFFFFF)) | np.array(self.pool.alloc_pages(len(eh)), np.uint64)
        L.lazyattn_materialize(self.pool.handle, self.batch.c,
                               torch.from_numpy(dst.view(np.int64).copy()).cuda())
        torch.cuda.synchronize()
        return self.batch.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED)


def _needle_inputs(hq, hkv, seed):
    """Six 256-token documents, the fifth a needle: every key has 16 in dim 63
    and 0 in dim 127 (the pair of the lowest frequency); queries (the 100-row
    segment and 12 decode steps) have 8 and 0 there."""
    rng = np.random.default_rng(seed)
    docs = []
    for j in range(6):
        k, v = _rnd(rng, (256, hkv, D)), _rnd(rng, (256, hkv, D))
        if j == 4:
            k[:, :, 63], k[:, :, 127] = 16.0, 0.0
        docs.append((k, v))
    lq = 100
    q, kq, vq = _rnd(rng, (lq, hq, D)), _rnd(rng, (lq, hkv, D)), _rnd(rng, (lq, hkv, D))
    q[:, :, 63], q[:, :, 127] = 8.0, 0.0
    steps = []
    for _ in range(12):
        qd = _rnd(rng, (hq, D))
        qd[:, 63], qd[:, 127] = 8.0, 0.0
        steps.append((qd, _rnd(rng, (hkv, D)), _rnd(rng, (hkv, D))))
    return docs, q, kq, vq, steps


def _score_jump_log2(docs, q, hq, hkv):
    """Smallest, over query rows and heads, of (largest needle score) minus
    (largest score of the tiles before the needle), in log2 units (test-side
    check that the inputs do force a late rescale)."""
    k_pre = np.concatenate([k for k, _ in docs[:4]])
    k_needle = docs[4][0]
    pos_q = np.arange(1536, 1536 + q.shape[0])
    qr = oracle.rope(q, pos_q[:, None], THETA)
    kr_pre = oracle.rope(k_pre, np.arange(1024)[:, None], THETA)
    kr_n = oracle.rope(k_needle, np.arange(1024, 1280)[:, None], THETA)
    g = hq // hkv
    jump = np.inf
    for h in range(hq):
        s_pre = qr[:, h] @ kr_pre[:, h // g].T
        s_n = qr[:, h] @ kr_n[:, h // g].T
        jump = min(jump, float(np.min(s_n.max(axis=1) - s_pre.max(axis=1))))
    return jump / np.sqrt(D) * np.log2(np.e)


@pytest.mark.parametrize("plan", [False, True])
@pytest.mark.parametrize("hq", [32, 64])
@pytest.mark.parametrize("keys", ["position_free", "doc_local", "materialised"])
def test_late_needle_forces_rescale(L, keys, hq, plan):
    hkv = 8
    docs, q, kq, vq, steps = _needle_inputs(hq, hkv, seed=40 + hq)
    assert _score_jump_log2(docs, q, hq, hkv) > 8.0
    req = Request(L, hq, hkv, docs, q, kq, vq, steps, keys="doc_local" if keys == "doc_local" else "position_free")
    assert req.store_status == [0] * len(req.store_status)
    batch = req.materialised() if keys == "materialised" else None
    got, st = req.prefill(batch)
    assert st == 0
    compare(got, oracle.prefill_request(docs, q, kq, vq, THETA), "bf16")
    outs, sts = req.decode(batch, plan=plan)
    assert sts == [0] * len(sts)
    want = oracle.decode_request(docs, kq, vq, steps, THETA)
    for o, w in zip(outs, want):
        compare(o, w, "bf16")


def _range_inputs(hkv, hq, seed, key_pair, q_pair):
    """Two documents with N(0,1) keys except: dims (10, 74) of token 5 of the
    first document hold key_pair (queries are 0 there), and dims (20, 84) of
    every query hold q_pair (keys are 0 there), so neither large pair moves a
    score; only an overflow in an operand would (0 * inf)."""
    rng = np.random.default_rng(seed)
    docs = []
    for j in range(2):
        k, v = _rnd(rng, (160, hkv, D)), _rnd(rng, (160, hkv, D))
        k[:, :, 20] = k[:, :, 84] = 0.0
        docs.append((k, v))
    docs[0][0][5, :, 10] = docs[0][0][5, :, 74] = key_pair
    lq = 40
    q, kq, vq = _rnd(rng, (lq, hq, D)), _rnd(rng, (lq, hkv, D)), _rnd(rng, (lq, hkv, D))
    kq[:, :, 20] = kq[:, :, 84] = 0.0
    q[:, :, 10] = q[:, :, 74] = 0.0
    q[:, :, 20] = q[:, :, 84] = q_pair
    steps = []
    for _ in range(3):
        qd, kd, vd = _rnd(rng, (hq, D)), _rnd(rng, (hkv, D)), _rnd(rng, (hkv, D))
        qd[:, 10] = qd[:, 74] = 0.0
        qd[:, 20] = qd[:, 84] = q_pair
        kd[:, 20] = kd[:, 84] = 0.0
        steps.append((qd, kd, vd))
    return docs, q, kq, vq, steps


# largest in-range pairs: 45824 * sqrt(2) = 64,805 <= 65,024 for keys;
# 360448 * sqrt(2) * log2(e) / sqrt(128) = 65,004 <= 65,024 for queries
IN_KEY, IN_Q = 45824.0, 360448.0
OUT_KEY, OUT_Q = 46080.0, 524288.0   # 65,166 and 94,551: past the bound


@pytest.mark.parametrize("keys", ["position_free", "doc_local", "materialised"])
def test_largest_in_range_pairs_stay_finite(L, keys):
    hq, hkv = 32, 8
    docs, q, kq, vq, steps = _range_inputs(hkv, hq, 50, IN_KEY, IN_Q)
    req = Request(L, hq, hkv, docs, q, kq, vq, steps, keys="doc_local" if keys == "doc_local" else "position_free")
    assert req.store_status == [0] * len(req.store_status)
    batch = req.materialised() if keys == "materialised" else None
    got, st = req.prefill(batch)
    assert st == 0
    compare(got, oracle.prefill_request(docs, q, kq, vq, THETA), "bf16")
    outs, sts = req.decode(batch)
    assert sts == [0] * len(sts)
    for o, w in zip(outs, oracle.decode_request(docs, kq, vq, steps, THETA)):
        compare(o, w, "bf16")


def test_out_of_range_key_is_reported_by_store(L):
    hq, hkv = 32, 8
    docs, q, kq, vq, steps = _range_inputs(hkv, hq, 51, OUT_KEY, 1.0)
    req = Request(L, hq, hkv, docs, q, kq, vq, steps)
    assert req.store_status[0] == ERANGE
    assert req.store_status[1:] == [0] * (len(req.store_status) - 1)


@pytest.mark.parametrize("keys", ["position_free", "doc_local"])
def test_out_of_range_key_is_reported_by_store_layouts(L, keys):
    hq, hkv = 32, 8
    rng = np.random.default_rng(52)
    from position_agnostic_kv_lazyattn_gb300 import DevicePool
    pool = DevicePool(8, hq, hkv, D, "bf16", THETA, 64, key_storage=keys)
    for pair, want in ((IN_KEY, 0), (OUT_KEY, ERANGE)):
        k, v = _rnd(rng, (20, hkv, D)), _rnd(rng, (20, hkv, D))
        k[17, 3, 5] = k[17, 3, 69] = pair
        pages = pool.store_doc(_dev(k), _dev(v))
        assert pool.device_status() == want
        pool.free_pages(pages)


def test_out_of_range_appended_key_is_reported(L):
    hq, hkv = 32, 8
    docs, q, kq, vq, steps = _range_inputs(hkv, hq, 53, 1.0, 1.0)
    steps[1][1][2, 7] = steps[1][1][2, 71] = OUT_KEY
    req = Request(L, hq, hkv, docs, q, kq, vq, steps)
    _, sts = req.decode()
    assert sts == [0, ERANGE, 0]


def test_out_of_range_query_is_reported(L):
    hq, hkv = 32, 8
    docs, q, kq, vq, steps = _range_inputs(hkv, hq, 54, 1.0, OUT_Q)
    req = Request(L, hq, hkv, docs, q, kq, vq, steps)
    _, st = req.prefill()
    assert st == ERANGE
    _, sts = req.decode()
    assert sts == [ERANGE] * len(sts)


def test_fp32_pool_has_no_fp16_bound(L):
    """fp32 pools compute in fp32 end to end: pairs far past the bf16 kernels'
    bound still match the oracle, and nothing is reported."""
    hq, hkv, d = 4, 2, 64
    rng = np.random.default_rng(55)
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    pool = DevicePool(16, hq, hkv, d, "f32", 1.0e4, 256)
    k, v = rng.standard_normal((40, hkv, d)).astype(np.float32), rng.standard_normal((40, hkv, d)).astype(np.float32)
    k[3, :, 1] = k[3, :, 33] = 1.0e6
    q = rng.standard_normal((8, hq, d)).astype(np.float32)
    q[:, :, 1] = q[:, :, 33] = 0.0
    q[:, :, 2] = q[:, :, 34] = 1.0e7
    k[:, :, 2] = k[:, :, 34] = 0.0
    kq, vq = np.zeros((8, hkv, d), np.float32), rng.standard_normal((8, hkv, d)).astype(np.float32)
    segs = [Segment(pool.store_doc(_dev(k, "f32"), _dev(v, "f32")), 0, 40),
            Segment(pool.store_doc(_dev(kq, "f32"), _dev(vq, "f32")), 40, 8, True)]
    batch = Batch([segs], [8], [40])
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    L.lazyattn_prefill(pool.handle, batch.c, _dev(q, "f32"), out)
    torch.cuda.synchronize()
    compare(out.cpu().numpy(), oracle.prefill_request([(k, v)], q, kq, vq, 1.0e4), "f32")
    assert pool.device_status() == 0

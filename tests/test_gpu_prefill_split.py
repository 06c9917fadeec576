"""Prefill with its KV tiles split over several CTAs, against the fp64 oracle.

When the caller passes a workspace of lazyattn_workspace_size(..., PREFILL)
bytes and the batch holds few CTAs' worth of long requests, the library splits
each (request, KV head, query pair)'s tiles into 2..4 shares, one CTA each,
and merges their partial outputs (reference maximum, sum, unnormalised O) in a
second kernel. These tests check:
* a long request next to a short one: the split count is set by the long one,
  so the short request's later shares hold no tile at all (its merge must
  skip them); the position table's 16-row view ends before the long request's
  last positions (max_position not a multiple of 16), so its last tiles copy
  their rows page by page;
* the same batch without a workspace, and with one too small for the partials
  (one CTA per item, no merge): the same outputs within the same bounds;
* the TTFT sweep's 20- and 40-document batches (where the split is chosen) in
  the launch configuration the benchmark times;
* every other instantiation of the split kernel: doc-local keys, ALiBi, the
  materialising baseline's pre-rotated pages, interleaved RoPE pairs (with
  position-free and doc-local keys).
"""
import numpy as np
import pytest
import torch

import oracle
import workload
import workload.device  # noqa: F401
from tests.gpu_common import Reference, compare

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


def _workspace(L, pool, batch, nbytes=None):
    n = L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_PREFILL, batch.c) if nbytes is None else nbytes
    return torch.zeros((n + 3) // 4, dtype=torch.int32, device="cuda"), n


def test_split_long_and_short_requests(L):
    from position_agnostic_kv_lazyattn_gb300 import Batch, DevicePool, Segment
    hq, hkv = 32, 8
    cfg = workload.CONFIGS["llama3_8b"]
    rng = np.random.default_rng(51)
    long_docs, q_lens = list(range(40)), [37, 5]
    max_pos = len(long_docs) * cfg.doc_len + q_lens[0] + 6     # 10283: not a multiple of 16
    assert max_pos % 16 != 0
    pool = DevicePool(900, hq, hkv, D, "bf16", THETA, max_pos)
    kv = {d: workload.doc_kv(cfg, d) for d in long_docs}
    pages = {d: pool.store_doc(_dev(k), _dev(v)) for d, (k, v) in kv.items()}
    plans = [long_docs, [7]]
    segs, qs, refs, starts = [], [], [], []
    for docs, n in zip(plans, q_lens):
        s = [Segment(pages[d], i * cfg.doc_len, cfg.doc_len) for i, d in enumerate(docs)]
        start = len(docs) * cfg.doc_len
        q, kq, vq = _rnd(rng, (n, hq, D)), _rnd(rng, (n, hkv, D)), _rnd(rng, (n, hkv, D))
        s.append(Segment(pool.store_doc(_dev(kq), _dev(vq)), start, n, True))
        segs.append(s)
        qs.append(q)
        starts.append(start)
        refs.append(oracle.prefill_request([kv[d] for d in docs], q, kq, vq, THETA))
    batch = Batch(segs, q_lens, starts)
    q_dev = _dev(np.concatenate(qs))
    nbytes = L.lazyattn_workspace_size(pool.handle, L.LAZYATTN_OP_PREFILL, batch.c)
    assert nbytes > 256, "a batch of two long-context items splits its tiles"
    outs = {}
    for mode, ws in (("split", _workspace(L, pool, batch)), ("none", (None, 0)),
                     ("small", _workspace(L, pool, batch, 256))):
        out = torch.full((batch.total_q, hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lazyattn_prefill(pool.handle, batch.c, q_dev, out, ws[0], ws[1])
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        off = 0
        for n, ref in zip(q_lens, refs):
            compare(got[off:off + n], ref, "bf16")
            off += n
        outs[mode] = got
    assert pool.device_status() == 0
    # without room for the partials the library runs one CTA per item: the
    # same launch as without a workspace
    assert np.array_equal(outs["none"], outs["small"])


@pytest.mark.parametrize("name", ["ttft_sweep_20", "ttft_sweep_40"])
def test_ttft_sweep_split(L, name):
    cfg = workload.CONFIGS[name]
    env = workload.device.setup(cfg, all_docs=False)
    b = env.batch
    ws, nbytes = _workspace(L, env.pool, b)
    assert nbytes > 256
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out, ws, nbytes)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    ref = Reference(cfg)
    errs = [compare(got[r], ref.prefill(r), "bf16") for r in (0, 13, 31)]
    print("%s split prefill worst max-abs %.3e rel-L2 %.3e" % (name, max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


@pytest.mark.parametrize("mode", ["doc_local", "alibi", "materialised", "interleaved", "doc_local+interleaved"])
def test_split_layouts(L, mode):
    """Every instantiation of the split kernel: two long requests of the
    40-document sweep (one wave of CTAs, so the tiles split four ways) in each
    pool layout and position encoding, against the oracle's attention for it."""
    cfg = workload.CONFIGS["ttft_sweep_40"]
    reqs = [0, 5]
    kw = {}
    if "doc_local" in mode:
        kw["key_storage"] = "doc_local"
    if mode == "alibi":
        kw["position_encoding"] = "alibi"
    if "interleaved" in mode:
        kw["rope_interleaved"] = True
    env = workload.device.setup(cfg, requests=reqs, all_docs=False, baseline=(mode == "materialised"), **kw)
    batch = env.batch
    if mode == "materialised":
        b = env.batch
        dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.array(env.pool.alloc_pages(len(b.entries_host)), np.uint64)
        L.lazyattn_materialize(env.pool.handle, b.c, torch.from_numpy(dst.view(np.int64).copy()).cuda())
        batch = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED)
    ws, nbytes = _workspace(L, env.pool, batch)
    assert nbytes > 256
    out = torch.full((batch.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, batch.c, env.q, out, ws, nbytes)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(len(reqs), cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    ref = Reference(cfg)
    if mode == "alibi":
        positional = oracle.AlibiSpec()
    elif "interleaved" in mode:
        positional = oracle.RopeSpec(cfg.rope_theta, "default", 1.0, 0, 0.0, 0.0, "interleaved")
    else:
        positional = cfg.rope_theta
    errs = []
    for i, r in enumerate(reqs):
        q, kq, vq = ref.qseg(r)
        errs.append(compare(got[i], oracle.prefill_request(ref.ctx(r), q, kq, vq, positional), "bf16"))
    print("%s split prefill worst max-abs %.3e rel-L2 %.3e" % (mode, max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0

"""GPU parity on the few-shot classification pattern (LazyAttention, App. C.7
"Beyond RAG: Few-Shot Classification"): exemplar chunks of 32..96 tokens recur
across prompts at different positions and in different orders, so block-table
entries start off page boundaries and documents end in partial pages in the
middle of a table; the query segment (48 tokens) ends in a partial page too.

Each case builds the whole 128-prompt batch (the launch the benchmark times),
runs prefill and the 4 decode steps, and checks sampled prompts against the
fp64 oracle: position-free keys with RoPE, the doc-local key layout (document
offsets that are not multiples of the page size), and the ALiBi bias. The
materialising baseline and the tiny fp32 variant of the pattern are checked too.
"""
import numpy as np
import pytest
import torch

import oracle
import workload
import workload.device  # noqa: F401
from tests.gpu_common import compare, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


def _sample(cfg):
    ctx = workload.request_context_lens(cfg)
    return sorted({0, 1, int(np.argmax(ctx)), int(np.argmin(ctx)), cfg.n_requests - 1})


def _refs(cfg, r, positional, steps):
    docs = workload.request_docs(cfg)[r]
    ctx = [workload.doc_kv(cfg, int(d)) for d in docs]
    q, kq, vq = workload.query_segment(cfg, r)
    pre = oracle.prefill_request(ctx, q, kq, vq, positional)
    st = [tuple(a[0] for a in workload.decode_inputs(cfg, t, [r])) for t in range(steps)]
    return pre, oracle.decode_request(ctx, kq, vq, st, positional)


def _prefill(L, env, batch=None):
    b = batch or env.batch
    cfg = env.cfg
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().reshape(len(env.requests), cfg.q_len, cfg.n_q_heads, cfg.head_dim)


@pytest.mark.parametrize("name", ["few_shot_skewed", "few_shot_uniform"])
@pytest.mark.parametrize("keys,pos", [("position_free", "rope"), ("doc_local", "rope"), ("position_free", "alibi")])
def test_few_shot_full_batch(L, name, keys, pos):
    cfg = workload.CONFIGS[name]
    env = workload.device.setup(cfg, key_storage=keys, position_encoding=pos)
    positional = oracle.AlibiSpec() if pos == "alibi" else cfg.rope_theta
    got = _prefill(L, env)
    outs = run_decode(L, env, cfg.decode_steps)
    errs = []
    for r in _sample(cfg):
        pre, dec = _refs(cfg, r, positional, cfg.decode_steps)
        errs.append(compare(got[r], pre, "bf16"))
        for t in range(cfg.decode_steps):
            errs.append(compare(outs[t][r], dec[t], "bf16"))
    print("%s %s/%s worst max-abs %.3e rel-L2 %.3e" % (name, keys, pos, max(e[0] for e in errs),
                                                       max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_few_shot_materialised_baseline(L):
    cfg = workload.CONFIGS["few_shot_skewed"]
    reqs = _sample(cfg)
    env = workload.device.setup(cfg, requests=reqs, baseline=True, all_docs=False)
    b = env.batch
    new_pages = env.pool.alloc_pages(len(b.entries_host))
    dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.array(new_pages, np.uint64)
    L.lazyattn_materialize(env.pool.handle, b.c, torch.from_numpy(dst.view(np.int64).copy()).cuda())
    mb = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED)
    got = _prefill(L, env, mb)
    outs = run_decode(L, env, cfg.decode_steps, batch=mb)
    for i, r in enumerate(reqs):
        pre, dec = _refs(cfg, r, cfg.rope_theta, cfg.decode_steps)
        compare(got[i], pre, "bf16")
        for t in range(cfg.decode_steps):
            compare(outs[t][i], dec[t], "bf16")
    assert env.pool.device_status() == 0


def test_tiny_ragged_fp32(L):
    cfg = workload.CONFIGS["tiny_ragged_fp32"]
    env = workload.device.setup(cfg)
    got = _prefill(L, env)
    outs = run_decode(L, env, cfg.decode_steps)
    for r in range(cfg.n_requests):
        pre, dec = _refs(cfg, r, cfg.rope_theta, cfg.decode_steps)
        compare(got[r], pre, "f32")
        for t in range(cfg.decode_steps):
            compare(outs[t][r], dec[t], "f32")
    assert env.pool.device_status() == 0

"""Full-batch launches of the large workloads, checked on sampled requests.

Every request of the workload is in the batch, so the kernels run in the same
launch configuration the benchmark times (grid, splits, tile counts); the fp64
oracle recomputes a few requests one by one:
* the decode-heavy RAG batch (128 requests x 20 documents of 512 tokens), three
  decode steps on the whole batch, three requests checked at every step;
* the 40-document TTFT sweep (32 requests x 40 documents of 1024 tokens plus a
  128-token query), prefill of the whole batch, two requests checked;
* the Llama-3-70B-shaped batch (64 requests x 32 documents of 1024 tokens plus a
  256-token query), prefill and two decode steps on the whole batch.
The pool holds the documents the batch uses (the benchmark stores every
document of the pool; the launches do not depend on the unused ones).
"""
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


def test_rag_decode_full_batch(L):
    cfg = workload.CONFIGS["rag_decode"]
    env = workload.device.setup(cfg, all_docs=False)
    steps, sample = 3, [0, 64, 127]
    outs = run_decode(L, env, steps)
    ref = Reference(cfg)
    errs = []
    for r in sample:
        want = ref.decode(r, steps)
        for t in range(steps):
            errs.append(compare(outs[t][r], want[t], "bf16"))
    print("rag_decode full batch worst max-abs %.3e rel-L2 %.3e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_ttft_sweep_40_full_batch(L):
    cfg = workload.CONFIGS["ttft_sweep_40"]
    env = workload.device.setup(cfg, all_docs=False)
    b = env.batch
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    ref = Reference(cfg)
    errs = [compare(got[r], ref.prefill(r), "bf16") for r in (0, 31)]
    print("ttft_sweep_40 full batch worst max-abs %.3e rel-L2 %.3e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_llama3_70b_full_batch(L):
    """64 requests x 32 documents of 1024 tokens plus a 256-token query (group of
    8 query heads per KV head): prefill of the whole batch, then two decode steps
    on it; one request checked in prefill, two at every decode step."""
    cfg = workload.CONFIGS["llama3_70b"]
    env = workload.device.setup(cfg, all_docs=False)
    b = env.batch
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    outs = run_decode(L, env, 2)
    ref = Reference(cfg)
    errs = [compare(got[5], ref.prefill(5), "bf16")]
    for r in (5, 63):
        want = ref.decode(r, 2)
        errs += [compare(outs[t][r], want[t], "bf16") for t in range(2)]
    print("llama3_70b full batch worst max-abs %.3e rel-L2 %.3e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0

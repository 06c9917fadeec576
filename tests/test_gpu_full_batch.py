"""Full-batch launches of the large workloads, checked on sampled requests.

Every request of the workload is in the batch, so the kernels run in the same
launch configuration the benchmark times (grid, splits, tile counts); the fp64
oracle recomputes a few requests one by one:
* the decode-heavy RAG batch (128 requests x 20 documents of 512 tokens), all
  256 decode steps on the whole batch, three requests checked at every step
  (16 generated pages each: every page rollover into a fresh reserved page);
  decoded request by request and again through the batch's decode plan;
* the TTFT sweep at 20 and 40 documents (32 requests x documents of 1024
  tokens plus a 128-token query), prefill of the whole batch, two requests
  checked;
* the Llama-3-70B-shaped batch (64 requests x 32 documents of 1024 tokens plus
  a 256-token query), prefill of the whole batch, then all 128 decode steps
  (both decode paths), two requests checked at every step.
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


def _decode_both(L, env, steps):
    """Every decode step on the whole batch twice: request by request, then
    (table reset) through the batch's document-major plan."""
    entries0 = env.batch.entries.clone()
    outs = run_decode(L, env, steps)
    assert env.pool.device_status() == 0
    env.batch.entries.copy_(entries0)
    outs_plan = run_decode(L, env, steps, plan=True)
    assert env.pool.device_status() == 0
    return outs, outs_plan


def _check_decode(cfg, runs, sample):
    ref = Reference(cfg)
    errs = []
    for r in sample:
        want = ref.decode_long(r, len(runs[0]))
        for outs in runs:
            for t in range(len(outs)):
                errs.append(compare(outs[t][r], want[t], "bf16"))
    return errs


def test_rag_decode_full_batch(L):
    cfg = workload.CONFIGS["rag_decode"]
    env = workload.device.setup(cfg, all_docs=False)
    runs = _decode_both(L, env, cfg.decode_steps)
    errs = _check_decode(cfg, runs, [0, 64, 127])
    print("rag_decode full batch, %d steps, both paths: worst max-abs %.3e rel-L2 %.3e"
          % (cfg.decode_steps, max(e[0] for e in errs), max(e[1] for e in errs)))


@pytest.mark.parametrize("name", ["ttft_sweep_20", "ttft_sweep_40"])
def test_ttft_sweep_full_batch(L, name):
    cfg = workload.CONFIGS[name]
    env = workload.device.setup(cfg, all_docs=False)
    b = env.batch
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    ref = Reference(cfg)
    errs = [compare(got[r], ref.prefill(r), "bf16") for r in (0, 31)]
    print("%s full batch worst max-abs %.3e rel-L2 %.3e" % (name, max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_llama3_70b_full_batch(L):
    """64 requests x 32 documents of 1024 tokens plus a 256-token query (group of
    8 query heads per KV head): prefill of the whole batch, then every decode
    step on it; one request checked in prefill, two at every decode step."""
    cfg = workload.CONFIGS["llama3_70b"]
    env = workload.device.setup(cfg, all_docs=False)
    b = env.batch
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    runs = _decode_both(L, env, cfg.decode_steps)
    ref = Reference(cfg)
    errs = [compare(got[5], ref.prefill(5), "bf16")]
    errs += _check_decode(cfg, runs, [5, 63])
    print("llama3_70b full batch, %d decode steps: worst max-abs %.3e rel-L2 %.3e"
          % (cfg.decode_steps, max(e[0] for e in errs), max(e[1] for e in errs)))

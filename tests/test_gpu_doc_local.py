"""GPU parity of the paper's own key layout (§3.2): K stored rotated at
document-local positions, one relative rotation per document offset in
prefill, q rotated per document in decode. Same oracle, same tolerances: by
Fact 3.2 (R_delta R_t = R_(delta+t)) the result is the same attention.

Covers the Llama-3-8B-shaped workload (documents shared by requests at
different offsets, a query segment, decode steps appended into the query
segment's last page and into reserved pages), the stored pages themselves, and
a sampled request of the 70B-shaped workload.
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


def test_store_rotates_at_local_positions(L):
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg, requests=[0], all_docs=False, key_storage="doc_local")
    d = int(env.docs[0][0])
    k, _ = workload.doc_kv(cfg, d)
    want = oracle.rope(k, np.arange(cfg.doc_len)[:, None], cfg.rope_theta)   # [len][Hkv][D]
    pages = env.doc_pages[d]
    got = env.pool.k_pool[torch.tensor(list(pages), device="cuda")].float().cpu().numpy()   # [p][Hkv][16][D]
    got = got.transpose(0, 2, 1, 3).reshape(-1, cfg.n_kv_heads, cfg.head_dim)[:cfg.doc_len]
    # bf16 rounding of the fp32 rotation: within one bf16 ulp
    np.testing.assert_allclose(got, want, rtol=2 ** -7, atol=2 ** -14)


def test_doc_local_llama3_8b_prefill_and_decode(L):
    cfg = workload.CONFIGS["llama3_8b"]
    reqs = [0, 3, 9, 14]
    env = workload.device.setup(cfg, requests=reqs, all_docs=False, key_storage="doc_local")
    ref = Reference(cfg)
    b = env.batch
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(len(reqs), cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    errs = [compare(got[i], ref.prefill(r), "bf16") for i, r in enumerate(reqs)]
    steps = 20   # past the query segment's last page into the reserved pages
    ws_bytes = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, b.c)
    ws = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device="cuda")
    outs = []
    for t in range(steps):
        q, k, v = workload.device.decode_step_tensors(cfg, t, reqs)
        o = torch.empty((len(reqs), cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device="cuda")
        L.lazyattn_decode(env.pool.handle, b.c, q, k, v, o, ws, ws_bytes)
        outs.append(o.float().cpu().numpy())
    torch.cuda.synchronize()
    for i, r in enumerate(reqs):
        want = ref.decode(r, steps)
        for t in range(steps):
            errs.append(compare(outs[t][i], want[t], "bf16"))
    print("doc-local worst max-abs %.3e rel-L2 %.3e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_doc_local_llama3_70b_sampled(L):
    cfg = workload.CONFIGS["llama3_70b"]
    env = workload.device.setup(cfg, requests=[37], all_docs=False, key_storage="doc_local")
    ref = Reference(cfg)
    b = env.batch
    out = torch.full((b.total_q, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=env.pool.tdtype, device="cuda")
    L.lazyattn_prefill(env.pool.handle, b.c, env.q, out)
    torch.cuda.synchronize()
    compare(out.float().cpu().numpy(), ref.prefill(37), "bf16")
    assert env.pool.device_status() == 0


def test_doc_local_rejects_prerotated_flag_and_missing_deltas(L):
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg, requests=[1], all_docs=False, key_storage="doc_local")
    b = env.batch
    out = torch.empty((b.total_q, cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device="cuda")
    pre = b.with_entries(b.entries_host, L.LAZYATTN_KEYS_PREROTATED)
    with pytest.raises(RuntimeError):   # LazyAttnError (EINVAL)
        L.lazyattn_prefill(env.pool.handle, pre.c, env.q, out)
    nod = L.make_batch(b.num_requests, b.max_entries, b.entries, b.entry_offsets, b.q_offsets, b.q_start,
                       b.max_q_len, b.total_q, 0, None)
    with pytest.raises(RuntimeError):   # LazyAttnError (EINVAL)
        L.lazyattn_prefill(env.pool.handle, nod, env.q, out)

"""lazyattn_decode_noalloc, the decode step for callers that cannot allocate
device memory (their host owns every allocation, or they run where cudaMalloc
is unavailable). It must give the same outputs as lazyattn_decode with a
caller-allocated workspace. Kept in a file that pytest collects last."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("name,requests", [("llama3_8b", [0, 3, 6, 9, 12]), ("tiny_fp32", [0, 1])])
def test_noalloc_decode_matches_workspace_decode(L, name, requests):
    cfg = workload.CONFIGS[name]
    a = workload.device.setup(cfg, requests=requests, all_docs=False)   # lazyattn_decode + workspace
    b = workload.device.setup(cfg, requests=requests, all_docs=False)   # lazyattn_decode_noalloc
    nbytes = L.lazyattn_workspace_size(a.pool.handle, L.LAZYATTN_OP_DECODE, a.batch.c)
    assert 0 < nbytes <= L.lazyattn.NOALLOC_SCRATCH_BYTES
    ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device="cuda")
    R = len(requests)
    oa = torch.empty((R, cfg.n_q_heads, cfg.head_dim), dtype=a.pool.tdtype, device="cuda")
    ob = torch.empty_like(oa)
    want = Reference(cfg).decode(requests[0], 2)           # and the oracle, on one request
    for t in range(2):                                   # two calls in a row
        q, k, v = workload.device.decode_step_tensors(cfg, t, requests)
        L.lazyattn_decode(a.pool.handle, a.batch.c, q, k, v, oa, ws, nbytes)
        L.lazyattn_decode_noalloc(b.pool.handle, b.batch.c, q, k, v, ob)
        torch.cuda.synchronize()
        compare(ob.float().cpu().numpy(), oa.float().cpu().numpy(), cfg.dtype)
        compare(ob[0].float().cpu().numpy(), want[t], cfg.dtype)
    assert a.pool.device_status() == 0 and b.pool.device_status() == 0
    assert np.array_equal(a.batch.entries.cpu().numpy(), b.batch.entries.cpu().numpy())


def test_noalloc_rejects_batches_beyond_the_scratch_size(L):
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg, requests=[0], all_docs=False)
    big = L.lazyattn_batch(60000, env.batch.max_entries, 0, 0, env.batch.entries.data_ptr(),
                           env.batch.entry_offsets.data_ptr(), None, None, 0)
    assert L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, big) > L.lazyattn.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    rc = L.lib.lazyattn_decode_noalloc(env.pool.handle, ctypes.byref(big), dummy.data_ptr(), dummy.data_ptr(),
                                       dummy.data_ptr(), dummy.data_ptr(), None)
    assert rc == -7   # LAZYATTN_EWORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert env.pool.device_status() == 0


def test_noalloc_after_a_batch_of_another_shape(L):
    """The array keeps the previous call's contents. A 5-request batch with
    split partials leaves non-zero partial results where a 100-request batch
    keeps its split-combine tickets; the second call must clear them itself
    (with stale tickets the last split to arrive would be misjudged and the
    combine skipped or repeated)."""
    small = workload.CONFIGS["llama3_8b"]
    big = dataclasses.replace(small, n_requests=100)
    env_s = workload.device.setup(small, requests=list(range(5)), all_docs=False)
    env_b = workload.device.setup(big, all_docs=False)
    env_w = workload.device.setup(big, all_docs=False)   # the same batch, decoded with a workspace
    for env in (env_s, env_b):
        n = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, env.batch.c)
        assert 0 < n <= L.lazyattn.NOALLOC_SCRATCH_BYTES
    out_s = torch.empty((5, small.n_q_heads, small.head_dim), dtype=torch.bfloat16, device="cuda")
    q, k, v = workload.device.decode_step_tensors(small, 0, range(5))
    L.lazyattn_decode_noalloc(env_s.pool.handle, env_s.batch.c, q, k, v, out_s)
    nbytes = L.lazyattn_workspace_size(env_w.pool.handle, L.LAZYATTN_OP_DECODE, env_w.batch.c)
    ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device="cuda")
    out_b = torch.empty((100, big.n_q_heads, big.head_dim), dtype=torch.bfloat16, device="cuda")
    out_w = torch.empty_like(out_b)
    want = Reference(big).decode(99, 2)
    for t in range(2):                                   # two calls in a row
        q, k, v = workload.device.decode_step_tensors(big, t, range(100))
        L.lazyattn_decode_noalloc(env_b.pool.handle, env_b.batch.c, q, k, v, out_b)
        L.lazyattn_decode(env_w.pool.handle, env_w.batch.c, q, k, v, out_w, ws, nbytes)
        torch.cuda.synchronize()
        compare(out_b.float().cpu().numpy(), out_w.float().cpu().numpy(), "bf16")
        compare(out_b[99].float().cpu().numpy(), want[t], "bf16")
    for env in (env_s, env_b, env_w):
        assert env.pool.device_status() == 0

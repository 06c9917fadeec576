"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Inputs come from the seeded workload generator; expected values from oracle/
only. Tolerances: fp32 max-abs 1e-4; bf16 max-abs 2e-2 and relative L2 5e-3.
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


def _workspace(L, pool, op, batch):
    n = L.lazyattn_workspace_size(pool.handle, op, batch.c)
    assert n > 0
    return torch.zeros((n + 3) // 4, dtype=torch.int32, device="cuda"), n


def _resolve(L, env):
    b = env.batch
    counts = []
    for r in range(b.num_requests):
        ent = b.entries_host[b.offsets_host[r]:b.offsets_host[r + 1]]
        counts.append(len(oracle.resolve_entries(ent)))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cap = int(offs[-1])
    out = torch.full((max(cap, 1) * 3,), -1, dtype=torch.int32, device="cuda")
    L.lazyattn_resolve(env.pool.handle, b.c, torch.from_numpy(offs).cuda(), out, cap)
    got = out.cpu().numpy()[: cap * 3].reshape(-1, 3)
    ref = []
    for r in range(b.num_requests):
        ref += oracle.resolve_entries(b.entries_host[b.offsets_host[r]:b.offsets_host[r + 1]])
    return got, np.array(ref, dtype=np.int64).reshape(-1, 3)


@pytest.mark.parametrize("name", ["tiny_fp32", "llama3_8b", "tiny_ragged_fp32", "few_shot_skewed"])
def test_resolve_bit_exact(L, name):
    cfg = workload.CONFIGS[name]
    env = workload.device.setup(cfg)
    got, ref = _resolve(L, env)
    assert np.array_equal(got, ref)
    assert env.pool.device_status() == 0


def _run_decode(L, env, steps, batch=None):
    cfg = env.cfg
    batch = batch or env.batch
    ws, nbytes = _workspace(L, env.pool, L.LAZYATTN_OP_DECODE, batch)
    outs = []
    R = len(env.requests)
    out = torch.empty((R, cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device="cuda")
    for t in range(steps):
        q, k, v = workload.device.decode_step_tensors(cfg, t, env.requests)
        L.lazyattn_decode(env.pool.handle, batch.c, q, k, v, out, ws, nbytes)
        outs.append(out.float().cpu().numpy().copy())
    torch.cuda.synchronize()
    return outs


def test_tiny_fp32_prefill_and_decode(L):
    cfg = workload.CONFIGS["tiny_fp32"]
    env = workload.device.setup(cfg)
    ref = Reference(cfg)
    out = torch.empty((env.batch.total_q, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    L.lazyattn_prefill(env.pool.handle, env.batch.c, env.q, out)
    got = out.cpu().numpy().reshape(cfg.n_requests, cfg.q_len, cfg.n_q_heads, cfg.head_dim)
    for r in range(cfg.n_requests):
        compare(got[r], ref.prefill(r), "f32")
    outs = _run_decode(L, env, cfg.decode_steps)
    for r in range(cfg.n_requests):
        refs = ref.decode(r, cfg.decode_steps)
        for t in range(cfg.decode_steps):
            compare(outs[t][r], refs[t], "f32")
    assert env.pool.device_status() == 0


@pytest.fixture(scope="module")
def llama8b(L):
    cfg = workload.CONFIGS["llama3_8b"]
    return cfg, Reference(cfg)


def test_bf16_decode_llama3_8b(L, llama8b):
    cfg, ref = llama8b
    env = workload.device.setup(cfg)
    outs = _run_decode(L, env, cfg.decode_steps)
    errs = []
    for r in range(cfg.n_requests):
        refs = ref.decode(r, cfg.decode_steps)
        for t in range(cfg.decode_steps):
            errs.append(compare(outs[t][r], refs[t], "bf16"))
    print("decode llama3_8b worst max-abs %.3e rel-L2 %.3e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
    assert env.pool.device_status() == 0


def test_bf16_decode_materialised_baseline(L, llama8b):
    """The materialising baseline (copy + eager RoPE, then attention without
    rotation) reaches the same outputs."""
    cfg, ref = llama8b
    reqs = [0, 5, 11]
    env = workload.device.setup(cfg, requests=reqs, baseline=True)
    b = env.batch
    n_ent = len(b.entries_host)
    new_pages = env.pool.alloc_pages(n_ent)
    dst = b.entries_host.copy()
    mask = np.uint64(0xFFFFFFFF)
    dst = (dst & ~mask) | np.array(new_pages, np.uint64)
    dst_dev = torch.from_numpy(dst.view(np.int64).copy()).cuda()
    L.lazyattn_materialize(env.pool.handle, b.c, dst_dev)
    mb = b.with_entries(dst, L.LAZYATTN_KEYS_PREROTATED)
    outs = _run_decode(L, env, 8, batch=mb)
    for i, r in enumerate(reqs):
        refs = ref.decode(r, 8)
        for t in range(8):
            compare(outs[t][i], refs[t], "bf16")
    assert env.pool.device_status() == 0


def test_decode_without_writable_slot_reports_and_zeroes(L):
    cfg = workload.CONFIGS["tiny_fp32"]
    env = workload.device.setup(cfg)
    # strip the writable bit from every entry: nothing to append into
    ent = env.batch.entries_host & ~np.uint64(1 << 63)
    b = env.batch.with_entries(ent, 0)
    ws, nbytes = _workspace(L, env.pool, L.LAZYATTN_OP_DECODE, b)
    q, k, v = workload.device.decode_step_tensors(cfg, 0, env.requests)
    out = torch.full((cfg.n_requests, cfg.n_q_heads, cfg.head_dim), 7.0, device="cuda")
    L.lazyattn_decode(env.pool.handle, b.c, q, k, v, out, ws, nbytes)
    assert float(out.abs().max()) == 0.0
    assert env.pool.device_status() == -8


def test_out_of_range_page_is_skipped_and_reported(L):
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg, requests=[0, 1], all_docs=False)
    ent = env.batch.entries_host.copy()
    ent[3] = (ent[3] & ~np.uint64(0xFFFFFFFF)) | np.uint64(env.pool.num_pages + 5)
    b = env.batch.with_entries(ent, 0)
    ws, nbytes = _workspace(L, env.pool, L.LAZYATTN_OP_DECODE, b)
    q, k, v = workload.device.decode_step_tensors(cfg, 0, env.requests)
    out = torch.empty((2, cfg.n_q_heads, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    L.lazyattn_decode(env.pool.handle, b.c, q, k, v, out, ws, nbytes)
    torch.cuda.synchronize()
    assert env.pool.device_status() == -3
    assert torch.isfinite(out.float()).all()


def test_pool_pages_are_read_only(L):
    """Decode writes only the appended slot; every other pool byte is unchanged."""
    cfg = workload.CONFIGS["llama3_8b"]
    env = workload.device.setup(cfg, requests=[2, 3, 4], all_docs=False)
    before_k = env.pool.k_pool.clone()
    before_v = env.pool.v_pool.clone()
    _run_decode(L, env, 3)
    ek = (env.pool.k_pool != before_k).reshape(env.pool.num_pages, -1).any(dim=1)
    ev = (env.pool.v_pool != before_v).reshape(env.pool.num_pages, -1).any(dim=1)
    changed = set(torch.nonzero(ek | ev).flatten().tolist())
    writable = {int(e & np.uint64(0xFFFFFFFF)) for e in env.batch.entries_host if int(e) >> 63}
    assert changed <= writable

"""Shared helpers of the GPU parity tests: tolerances and oracle references."""
import functools

import numpy as np

import oracle
import workload

# Tolerances (GPU vs fp64 oracle on the same, already rounded, inputs)
F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3


def compare(got, ref, dtype):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = got - ref
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"max-abs {max_abs:.3e} > {F32_MAX_ABS}"
    else:
        assert max_abs <= BF16_MAX_ABS, f"max-abs {max_abs:.3e} > {BF16_MAX_ABS}"
        assert rel <= BF16_REL_L2, f"rel-L2 {rel:.3e} > {BF16_REL_L2}"
    return max_abs, rel


class Reference:
    """fp64 oracle outputs for a workload config, computed per request on demand."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.docs = workload.request_docs(cfg)

    @functools.lru_cache(maxsize=None)
    def doc(self, d):
        return workload.doc_kv(self.cfg, d)

    def ctx(self, r):
        return [self.doc(int(d)) for d in self.docs[r]]

    def qseg(self, r):
        cfg = self.cfg
        if cfg.q_len:
            return workload.query_segment(cfg, r)
        H = np.zeros((0, cfg.n_q_heads, cfg.head_dim), np.float32)
        K = np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
        return H, K, K.copy()

    def prefill(self, r):
        q, kq, vq = self.qseg(r)
        return oracle.prefill_request(self.ctx(r), q, kq, vq, self.cfg.rope_theta)

    def decode(self, r, n_steps):
        _, kq, vq = self.qseg(r)
        steps = [tuple(a[0] for a in workload.decode_inputs(self.cfg, t, [r])) for t in range(n_steps)]
        return oracle.decode_request(self.ctx(r), kq, vq, steps, self.cfg.rope_theta)

    def decode_long(self, r, n_steps):
        """The same outputs as decode(), for long runs: the oracle's eager form
        (every key of the request's final sequence rotated once at its logical
        position by materialize_rotated, then, per step, attention_prerotated
        over the prefix that ends with the step's own token, q rotated at that
        token's position). The oracle pins equate the eager and lazy forms."""
        cfg = self.cfg
        _, kq, vq = self.qseg(r)
        steps = [tuple(a[0] for a in workload.decode_inputs(cfg, t, [r])) for t in range(n_steps)]
        ctx = self.ctx(r)
        k_all = np.concatenate([k for k, _ in ctx] + [kq] + [s[1][None] for s in steps]).astype(np.float64)
        v_all = np.concatenate([v for _, v in ctx] + [vq] + [s[2][None] for s in steps]).astype(np.float64)
        n0 = sum(k.shape[0] for k, _ in ctx) + kq.shape[0]
        pos = np.arange(k_all.shape[0], dtype=np.int64)
        k_rot = oracle.materialize_rotated(k_all, pos, cfg.rope_theta)
        g = cfg.n_q_heads // cfg.n_kv_heads
        kh = [np.ascontiguousarray(k_rot[:, h, :]) for h in range(cfg.n_kv_heads)]
        vh = [np.ascontiguousarray(v_all[:, h, :]) for h in range(cfg.n_kv_heads)]
        scale = oracle.logit_scale(cfg.head_dim, cfg.rope_theta)
        outs = []
        for t, (q, _, _) in enumerate(steps):
            n = n0 + t + 1
            q_rot = oracle.rope(np.asarray(q, np.float64)[None], np.array([[n - 1]]), cfg.rope_theta)
            o = np.empty((cfg.n_q_heads, cfg.head_dim))
            for h in range(cfg.n_kv_heads):
                o[h * g:(h + 1) * g] = oracle.attention_prerotated(
                    q_rot[:, h * g:(h + 1) * g], kh[h][:n, None, :], vh[h][:n, None, :], [n - 1],
                    pos[:n], scale)[0]
            outs.append(o)
        return outs


def run_decode(L, env, steps, batch=None, plan=False):
    """`steps` decode calls (append + attention) over env's requests; the
    outputs of each step, [R][Hq][D] as float arrays. plan: decode through the
    batch's document-major plan (built here)."""
    import torch
    import workload.device  # noqa: F401
    cfg = env.cfg
    batch = batch or env.batch
    if plan:
        batch.plan_decode(env.pool)
    nbytes = L.lazyattn_workspace_size(env.pool.handle, L.LAZYATTN_OP_DECODE, batch.c)
    ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device="cuda")
    out = torch.empty((len(env.requests), cfg.n_q_heads, cfg.head_dim), dtype=env.pool.tdtype, device="cuda")
    outs = []
    for t in range(steps):
        q, k, v = workload.device.decode_step_tensors(cfg, t, env.requests)
        L.lazyattn_decode(env.pool.handle, batch.c, q, k, v, out, ws, nbytes)
        outs.append(out.float().cpu().numpy().copy())
    torch.cuda.synchronize()
    return outs

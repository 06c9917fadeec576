"""Pins of the fp64 oracle to facts fixed outside it (CPU only).

Each test cites what it checks in the LazyAttention paper (LazyAttention:
Efficient Retrieval-Augmented Generation with Deferred Positional Encoding).
The mutation tests at the bottom plant plausible mistakes in the oracle and
check that at least one pin catches each of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workload
from tests.bruteforce import bf_attention, bf_rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rope_golden():
    rows = []
    with open(os.path.join(GOLDEN, "rope_worked_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            head, xs, ys = line.split("|")
            D, th, pos = head.split()
            rows.append((int(D), float(th), int(pos),
                         [float(t) for t in xs.split()], [float(t) for t in ys.split()]))
    return rows


# ---------------------------------------------------------------- RoPE itself

def test_rope_worked_example():
    """§3.2 "Prefilling" rotation formula, hand-derived values (tests/golden)."""
    for D, th, pos, x, y in _read_rope_golden():
        got = oracle.rope(np.array(x), np.array(pos), th)
        np.testing.assert_allclose(got, y, rtol=0, atol=1e-14)


def test_rope_identity_norm_composition():
    """Rotation-group facts: R_0 = I, each pair keeps its norm, R_a R_b = R_{a+b}."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 128))
    assert np.array_equal(oracle.rope(x, np.zeros(64), 5e5), x)
    a = rng.integers(0, 40000, 64)
    b = rng.integers(0, 40000, 64)
    ra = oracle.rope(x, a, 5e5)
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = ra[:, :64] ** 2 + ra[:, 64:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)
    np.testing.assert_allclose(oracle.rope(ra, b, 5e5), oracle.rope(x, a + b, 5e5),
                               rtol=0, atol=1e-9)
    np.testing.assert_allclose(oracle.rope(ra, -a, 5e5), x, rtol=0, atol=1e-9)


def test_fact_3_2_relative_rotation():
    """Fact 3.2: (R_m q)^T (R_n k) = q^T R_{n-m} k."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((32, 128))
    m = rng.integers(0, 30000, 32)
    n = rng.integers(0, 30000, 32)
    lhs = np.sum(oracle.rope(q, m, 5e5) * oracle.rope(k, n, 5e5), axis=1)
    rhs = np.sum(q * oracle.rope(k, n - m, 5e5), axis=1)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-9)


def test_rope_matches_complex_bruteforce():
    rng = np.random.default_rng(2)
    for D in (2, 8, 64):
        x = rng.standard_normal(D)
        for pos in (0, 1, 17, 4099):
            np.testing.assert_allclose(oracle.rope(x, np.array(pos), 1e4),
                                       bf_rope(list(x), pos, 1e4), rtol=0, atol=1e-10)


# ---------------------------------------------------------------- attention

def _rand_case(seed, Lq, L, Hq, Hkv, D):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Lq, Hq, D)), rng.standard_normal((L, Hkv, D)),
            rng.standard_normal((L, Hkv, D)))


def test_textbook_reduction_sdpa():
    """Zero angles: RoPE attention reduces to Eq. 4, checked against PyTorch's
    scaled_dot_product_attention in fp64 (GQA heads expanded by h // g)."""
    q, k, v = _rand_case(3, 7, 19, 4, 2, 16)
    out = oracle.attention(q, k, v, np.zeros(7, np.int64), np.zeros(19, np.int64), 1e4)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def test_causal_rope_against_sdpa():
    """Rotated inputs (complex brute force) plus a causal mask, through SDPA."""
    Lq, L, Hq, Hkv, D, th = 5, 12, 4, 2, 8, 1e4
    q, k, v = _rand_case(4, Lq, L, Hq, Hkv, D)
    k_pos = np.arange(L)
    q_pos = np.arange(L - Lq, L)
    out = oracle.attention(q, k, v, q_pos, k_pos, th)
    qr = np.array([[bf_rope(list(q[i, h]), q_pos[i], th) for h in range(Hq)] for i in range(Lq)])
    kr = np.array([[bf_rope(list(k[j, h]), k_pos[j], th) for h in range(Hkv)] for j in range(L)])
    mask = torch.from_numpy(k_pos[None, :] <= q_pos[:, None])
    tq = torch.from_numpy(qr).permute(1, 0, 2)[None]
    tk = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_eager_equals_lazy():
    """(a) §1: deferred rotation is identical to attention over a materialised,
    re-encoded copy of the keys."""
    q, k, v = _rand_case(5, 9, 40, 8, 2, 32)
    k_pos = np.arange(100, 140)
    q_pos = np.arange(131, 140)
    lazy = oracle.attention(q, k, v, q_pos, k_pos, 5e5)
    k_mat = oracle.materialize_rotated(k, k_pos, 5e5)
    q_rot = oracle.rope(q, q_pos[:, None], 5e5)
    eager = oracle.attention_prerotated(q_rot, k_mat, v, q_pos, k_pos)
    np.testing.assert_allclose(lazy, eager, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("c", [1, 1000, 100000])
def test_shift_invariance(c):
    """(b) Fact 3.2 and Example 3.1: only offsets matter, so shifting every
    logical position by a constant leaves the output unchanged."""
    q, k, v = _rand_case(6, 6, 30, 4, 2, 64)
    k_pos = np.arange(30)
    q_pos = np.arange(24, 30)
    a = oracle.attention(q, k, v, q_pos, k_pos, 1e4)
    b = oracle.attention(q, k, v, q_pos + c, k_pos + c, 1e4)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-9)


def _pack(page, start, nvalid, writable=0):
    return page | (start << 32) | (nvalid << 58) | (writable << 63)


def test_shared_document_two_offsets():
    """(c) Problem statement, §3: two requests read one physical copy of a
    document at different logical offsets; each matches a brute force over
    private copies placed at its own positions."""
    rng = np.random.default_rng(7)
    Hq, Hkv, D, th = 4, 2, 8, 1e4
    doc_k = rng.standard_normal((20, Hkv, D))
    doc_v = rng.standard_normal((20, Hkv, D))
    other_k = rng.standard_normal((16, Hkv, D))
    other_v = rng.standard_normal((16, Hkv, D))
    qs_k = rng.standard_normal((2, 3, Hkv, D))
    qs_v = rng.standard_normal((2, 3, Hkv, D))
    q = rng.standard_normal((2, 3, Hq, D))
    P = oracle.PAGE_SIZE
    kp = np.zeros((8, Hkv, P, D))
    vp = np.zeros((8, Hkv, P, D))

    def put(page, ks, vs):
        kp[page, :, : len(ks)] = np.transpose(ks, (1, 0, 2))
        vp[page, :, : len(vs)] = np.transpose(vs, (1, 0, 2))

    put(0, doc_k[:16], doc_v[:16]); put(1, doc_k[16:], doc_v[16:])   # shared doc: pages 0, 1
    put(2, other_k, other_v)                                           # other doc: page 2
    put(3, qs_k[0], qs_v[0]); put(4, qs_k[1], qs_v[1])                # private query pages
    # request 0: shared doc at 0, other doc at 20, query at 36
    t0 = [_pack(0, 0, 16), _pack(1, 16, 4), _pack(2, 20, 16), _pack(3, 36, 3, 1)]
    # request 1: other doc at 0, shared doc at 16, query at 36
    t1 = [_pack(2, 0, 16), _pack(0, 16, 16), _pack(1, 32, 4), _pack(4, 36, 3, 1)]
    for r, (tab, ctx) in enumerate([(t0, [(doc_k, doc_v), (other_k, other_v)]),
                                    (t1, [(other_k, other_v), (doc_k, doc_v)])]):
        got = oracle.paged_prefill(kp, vp, tab, q[r], 36, th)
        kk = np.concatenate([c[0] for c in ctx] + [qs_k[r]])
        vv = np.concatenate([c[1] for c in ctx] + [qs_v[r]])
        ref = bf_attention(q[r].tolist(), kk.tolist(), vv.tolist(), [36, 37, 38],
                           list(range(39)), th)
        np.testing.assert_allclose(got, np.array(ref), rtol=0, atol=1e-12)
        # and the logical-concatenation form of the oracle agrees
        np.testing.assert_allclose(oracle.prefill_request(ctx, q[r], qs_k[r], qs_v[r], th),
                                   got, rtol=0, atol=1e-12)


def test_resolve_entries_fields():
    e = _pack(123456, 40000, 16, 1)
    assert oracle.unpack_entry(e) == (123456, 40000, 16, 1)
    assert oracle.resolve_entries([_pack(7, 100, 3), _pack(2, 0, 0), _pack(9, 5, 2, 1)]) == [
        (7, 0, 100), (7, 1, 101), (7, 2, 102), (9, 0, 5), (9, 1, 6)]


@pytest.mark.parametrize("name", ["tiny_fp32", "tiny_ragged_fp32"])
def test_tiny_config_against_bruteforce(name):
    """The tiny fp32 workloads (3 docs of 32 tokens + 16 query tokens; 4 distinct
    docs of 5..40 tokens + 21 query tokens): prefill and every decode step by
    direct summation."""
    cfg = workload.CONFIGS[name]
    docs = workload.request_docs(cfg)
    for r in range(cfg.n_requests):
        ctx = [workload.doc_kv(cfg, int(d)) for d in docs[r]]
        q, kq, vq = workload.query_segment(cfg, r)
        got = oracle.prefill_request(ctx, q, kq, vq, cfg.rope_theta)
        kk = np.concatenate([c[0] for c in ctx] + [kq])
        vv = np.concatenate([c[1] for c in ctx] + [vq])
        L0 = sum(c[0].shape[0] for c in ctx)
        # brute force on two query rows (first and last) to keep it quick
        for i in (0, cfg.q_len - 1):
            ref = bf_attention([q[i].tolist()], kk.tolist(), vv.tolist(), [L0 + i],
                               list(range(kk.shape[0])), cfg.rope_theta)
            np.testing.assert_allclose(got[i], np.array(ref[0]), rtol=0, atol=1e-12)
        steps = [tuple(a[0] for a in workload.decode_inputs(cfg, t, [r])) for t in range(cfg.decode_steps)]
        outs = oracle.decode_request(ctx, kq, vq, steps, cfg.rope_theta)
        for t, (qd, kd, vd) in enumerate(steps):
            kk = np.concatenate([kk, kd[None]])
            vv = np.concatenate([vv, vd[None]])
            L = kk.shape[0]
            ref = bf_attention([qd.tolist()], kk.tolist(), vv.tolist(), [L - 1], list(range(L)),
                               cfg.rope_theta)
            np.testing.assert_allclose(outs[t], np.array(ref[0]), rtol=0, atol=1e-12)


def test_paged_decode_matches_logical():
    """Decode through a paged pool with reserved writable tail pages equals the
    logical-concatenation decode; the append fills the first free writable slot."""
    cfg = workload.CONFIGS["tiny_fp32"]
    rng = np.random.default_rng(8)
    Hkv, D, P = cfg.n_kv_heads, cfg.head_dim, oracle.PAGE_SIZE
    dk = [rng.standard_normal((20, Hkv, D)) for _ in range(2)]
    dv = [rng.standard_normal((20, Hkv, D)) for _ in range(2)]
    kq = rng.standard_normal((5, Hkv, D))
    vq = rng.standard_normal((5, Hkv, D))
    kp = np.zeros((10, Hkv, P, D))
    vp = np.zeros((10, Hkv, P, D))
    ent = []
    page = 0
    pos = 0
    for k_, v_ in list(zip(dk, dv)):
        for o in range(0, 20, P):
            n = min(P, 20 - o)
            kp[page, :, :n] = np.transpose(k_[o:o + n], (1, 0, 2))
            vp[page, :, :n] = np.transpose(v_[o:o + n], (1, 0, 2))
            ent.append(_pack(page, pos + o, n))
            page += 1
        pos += 20
    kp[page, :, :5] = np.transpose(kq, (1, 0, 2))
    vp[page, :, :5] = np.transpose(vq, (1, 0, 2))
    ent.append(_pack(page, pos, 5, 1))
    ent.append(_pack(page + 1, pos + P, 0, 1))     # reserved for generated tokens
    steps = [(rng.standard_normal((cfg.n_q_heads, D)), rng.standard_normal((Hkv, D)),
              rng.standard_normal((Hkv, D))) for _ in range(14)]
    ref = oracle.decode_request(list(zip(dk, dv)), kq, vq, steps, cfg.rope_theta)
    for t, (q, k_, v_) in enumerate(steps):
        out, ent = oracle.paged_decode_step(kp, vp, ent, q, k_, v_, cfg.rope_theta)
        np.testing.assert_allclose(out, ref[t], rtol=0, atol=1e-12)
    assert oracle.unpack_entry(ent[-2])[2] == 16 and oracle.unpack_entry(ent[-1])[2] == 3


# ---------------------------------------------------------------- Zipf

def _golden_gap():
    with open(os.path.join(GOLDEN, "hit_ratio_gap.txt")) as f:
        for line in f:
            if not line.startswith("#") and line.strip():
                C, D, gap, digits = line.split()
                return int(C), int(D), float(gap), int(digits)


def test_hit_ratio_harmonic_special_case():
    """Eq. 3 at alpha = 1 is a ratio of harmonic numbers: H_100 / H_5."""
    H5 = 1 + 1 / 2 + 1 / 3 + 1 / 4 + 1 / 5
    H100 = 5.187377517639620261   # harmonic number H_100 to 18 digits
    assert abs(oracle.hit_ratio_gap(100, 20, 1.0) - H100 / H5) < 1e-13
    assert abs(oracle.hit_ratio_agnostic(100, 100, 0.7) - 1.0) < 1e-15


def _harmonic(n, alpha):
    """sum_{i=1..n} i^-alpha as an exact fraction (alpha in {0, 1, 2})."""
    from fractions import Fraction
    return sum((Fraction(1, i ** alpha) for i in range(1, n + 1)), Fraction(0))


@pytest.mark.parametrize("C,D,N,alpha", [(4, 2, 10, 1), (5, 2, 10, 1), (7, 3, 10, 1), (9, 4, 12, 2),
                                         (3, 1, 8, 1), (30, 2, 10, 1), (6, 4, 10, 0), (25, 5, 20, 0)])
def test_hit_ratios_below_pool_size(C, D, N, alpha):
    """Eqs. 1 and 2 at C < N (and C // D < N), against exact sums of i^-alpha:
    Eq. 1 = H(min(C, N)) / H(N); Eq. 2 = H(min(floor(C / D), N)) / H(N). The
    cases tell floor(C / D) from C / D (5 / 2, 7 / 3, 9 / 4), and the
    min(., N) bound (30 / 2 = 15 > N = 10); alpha = 0 (uniform popularity)
    gives the plain coverage fractions min(C, N) / N and floor(C / D) / N."""
    want_agnostic = _harmonic(min(C, N), alpha) / _harmonic(N, alpha)
    want_aware = _harmonic(min(C // D, N), alpha) / _harmonic(N, alpha)
    assert abs(oracle.hit_ratio_agnostic(C, N, float(alpha)) - float(want_agnostic)) < 1e-14
    assert abs(oracle.hit_ratio_aware(C, D, N, float(alpha)) - float(want_aware)) < 1e-14
    if alpha == 0:
        assert abs(oracle.hit_ratio_agnostic(C, N, 0.0) - min(C, N) / N) < 1e-15
        assert abs(oracle.hit_ratio_aware(C, D, N, 0.0) - (C // D) / N) < 1e-15
    # Eq. 3 is the ratio of the two (the normaliser cancels), below the pool size
    if C // D >= 1 and C <= N:
        assert abs(oracle.hit_ratio_gap(C, D, float(alpha)) -
                   oracle.hit_ratio_agnostic(C, N, float(alpha)) / oracle.hit_ratio_aware(C, D, N, float(alpha))) < 1e-13


def test_hit_ratio_hand_values():
    """Two values worked by hand: N = 10, alpha = 1, C = 4, D = 2:
    Eq. 1 = (1 + 1/2 + 1/3 + 1/4) / H_10 = (25/12) / (7381/2520) = 5250/7381,
    Eq. 2 = (1 + 1/2) / H_10 = 3780/7381."""
    assert abs(oracle.hit_ratio_agnostic(4, 10, 1.0) - 5250 / 7381) < 1e-15
    assert abs(oracle.hit_ratio_aware(4, 2, 10, 1.0) - 3780 / 7381) < 1e-15


def test_hit_ratio_printed_value():
    """§1 / §2: the printed 2.86x at D = 20, C = 100. The paper omits alpha;
    the gap is monotone in alpha and equals 2.86 (3 digits) near 0.8526."""
    C, D, gap, digits = _golden_gap()
    got = oracle.hit_ratio_gap(C, D, 0.8526)
    assert abs(got - gap) < 0.5 * 10 ** (1 - digits)
    assert oracle.hit_ratio_gap(C, D, 0.80) > oracle.hit_ratio_gap(C, D, 0.90)


def test_zipf_sampler_reproduces_closed_form():
    """(d) the synthetic document sampler reproduces Eq. 3 empirically:
    P(rank <= C) / P(rank <= C/D) from 10^6 draws over a 100-document pool."""
    rng = np.random.default_rng(9)
    ranks = workload.zipf_ranks(rng, 100, 0.8526, 1_000_000)
    emp = np.mean(ranks <= 100) / np.mean(ranks <= 5)
    assert abs(emp / oracle.hit_ratio_gap(100, 20, 0.8526) - 1) < 0.01


# ---------------------------------------------------------------- mutations

def _mutant_rope_sign(x, pos, theta):
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    ang = np.asarray(pos, np.float64)[..., None] * oracle.rope_inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c + x2 * s, -x1 * s + x2 * c], axis=-1)


def _mutant_rope_interleaved(x, pos, theta):
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    ang = np.asarray(pos, np.float64)[..., None] * oracle.rope_inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x1 * c - x2 * s
    y[..., 1::2] = x1 * s + x2 * c
    return y


@pytest.mark.parametrize("mutant", [_mutant_rope_sign, _mutant_rope_interleaved])
def test_mutant_rope_is_caught(monkeypatch, mutant):
    import oracle.lazyattn_oracle as lo
    monkeypatch.setattr(lo, "rope", mutant)
    with pytest.raises(AssertionError):
        for D, th, pos, x, y in _read_rope_golden():
            np.testing.assert_allclose(lo.rope(np.array(x), np.array(pos), th), y, atol=1e-14)
    with pytest.raises(AssertionError):
        test_tiny_config_against_bruteforce_mut(lo)


def test_tiny_config_against_bruteforce_mut(lo=None):
    """Helper used by the mutation tests (also a plain pass on the real oracle)."""
    import oracle.lazyattn_oracle as real
    lo = lo or real
    rng = np.random.default_rng(10)
    q, k, v = rng.standard_normal((2, 4, 8)), rng.standard_normal((9, 2, 8)), rng.standard_normal((9, 2, 8))
    got = lo.attention(q, k, v, np.array([7, 8]), np.arange(9), 1e4)
    ref = bf_attention(q.tolist(), k.tolist(), v.tolist(), [7, 8], list(range(9)), 1e4)
    np.testing.assert_allclose(got, np.array(ref), rtol=0, atol=1e-12)


def test_mutant_scale_and_grouping_are_caught(monkeypatch):
    import oracle.lazyattn_oracle as lo
    real = lo.attention_prerotated

    def no_scale(q_rot, k_rot, v, q_pos, k_pos, scale=None):
        return real(np.asarray(q_rot) * math.sqrt(q_rot.shape[-1]), k_rot, v, q_pos, k_pos, scale)

    def wrong_group(q_rot, k_rot, v, q_pos, k_pos, scale=None):
        Hq, Hkv = q_rot.shape[1], k_rot.shape[1]
        heads = [real(q_rot[:, h:h + 1], k_rot[:, h % Hkv:h % Hkv + 1], v[:, h % Hkv:h % Hkv + 1],
                      q_pos, k_pos, scale) for h in range(Hq)]
        return np.concatenate(heads, axis=1)

    for m in (no_scale, wrong_group):
        monkeypatch.setattr(lo, "attention_prerotated", m)
        with pytest.raises(AssertionError):
            test_tiny_config_against_bruteforce_mut(lo)
        monkeypatch.setattr(lo, "attention_prerotated", real)

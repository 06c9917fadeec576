"""Pins of the oracle's RoPE-family variants (§3.5 "RoPE-family variants":
scaled/NTK and YaRN keep the score form with variant-specific metadata).

Each variant is checked against what its definition fixes independently of the
oracle's own formula: linear scaling is RoPE at interpolated positions p / s;
NTK-aware scaling keeps the highest frequency and divides the lowest by exactly
s; YaRN and the Llama 3.1 rule keep the high-frequency band, interpolate the
low-frequency band and blend monotonically in between, and reduce to plain RoPE
at s = 1; YaRN's logit scale is (0.1 ln s + 1)^2 / sqrt(D).
"""
import numpy as np
import pytest

import oracle
from oracle import RopeSpec

D = 128
BASE = 5.0e5


def test_linear_is_rope_at_interpolated_positions():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 3, D))
    pos = np.array([0, 1, 5, 100, 4095, 20000, 65535])[:, None]
    for s in (2.0, 4.0, 8.0):
        got = oracle.rope(x, pos, RopeSpec(BASE, "linear", s))
        want = oracle.rope(x, pos / s, BASE)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_ntk_closed_form():
    for s in (2.0, 8.0, 32.0):
        f = RopeSpec(BASE, "ntk", s).inv_freq(D)
        plain = RopeSpec(BASE).inv_freq(D)
        assert f[0] == 1.0 and plain[0] == 1.0
        # lowest frequency: (base * s^(D/(D-2)))^(-(D-2)/D) = base^(-(D-2)/D) / s
        np.testing.assert_allclose(f[-1], BASE ** (-(D - 2) / D) / s, rtol=1e-13)
        assert np.all(np.diff(f) < 0)
        assert np.all(f <= plain) and np.all(f[1:] < plain[1:])


@pytest.mark.parametrize("kind,orig,low,high", [("yarn", 4096, 1.0, 32.0), ("llama3", 8192, 1.0, 4.0)])
def test_band_limits_and_monotone_blend(kind, orig, low, high):
    s = 8.0
    plain = RopeSpec(BASE).inv_freq(D)
    f = RopeSpec(BASE, kind, s, orig, low, high).inv_freq(D)
    wavelength = 2 * np.pi / plain
    if kind == "yarn":
        r = orig / wavelength                  # rotations within the original context
        keep, interp = r > high, r < low
    else:
        keep, interp = wavelength < orig / high, wavelength > orig / low
    mid = ~keep & ~interp
    assert keep.any() and interp.any() and mid.any()
    np.testing.assert_array_equal(f[keep], plain[keep])
    np.testing.assert_allclose(f[interp], plain[interp] / s, rtol=1e-15)
    assert np.all(f[mid] < plain[mid]) and np.all(f[mid] > plain[mid] / s)
    assert np.all(np.diff(f) < 0)             # ordering of the frequencies survives
    # at s = 1 every variant is plain RoPE
    np.testing.assert_allclose(RopeSpec(BASE, kind, 1.0, orig, low, high).inv_freq(D), plain, rtol=1e-15)


def test_yarn_logit_scale():
    for s in (1.0, 4.0, 16.0):
        spec = RopeSpec(BASE, "yarn", s, 4096, 1.0, 32.0)
        t = 0.1 * np.log(s) + 1.0 if s > 1 else 1.0
        assert spec.logit_scale(D) == pytest.approx(t * t / np.sqrt(D), rel=1e-15)
    assert RopeSpec(BASE, "llama3", 8.0, 8192, 1.0, 4.0).logit_scale(D) == pytest.approx(1 / np.sqrt(D))


def test_default_spec_matches_plain_base():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 4, D))
    k = rng.standard_normal((9, 2, D))
    v = rng.standard_normal((9, 2, D))
    a = oracle.attention(q, k, v, np.arange(5, 9), np.arange(9), BASE)
    b = oracle.attention(q, k, v, np.arange(5, 9), np.arange(9), RopeSpec(BASE))
    np.testing.assert_array_equal(a, b)


def test_yarn_temperature_enters_the_logits():
    """Attention with YaRN equals attention over the same rotations with the
    logits multiplied by the temperature (checked by brute force)."""
    rng = np.random.default_rng(2)
    spec = RopeSpec(BASE, "yarn", 8.0, 4096, 1.0, 32.0)
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((6, 1, D))
    v = rng.standard_normal((6, 1, D))
    got = oracle.attention(q, k, v, [5], np.arange(6), spec)[0, 0]
    qr = oracle.rope(q[0, 0], 5, spec)
    logits = np.array([qr @ oracle.rope(k[j, 0], j, spec) for j in range(6)]) * spec.logit_scale(D)
    p = np.exp(logits - logits.max())
    want = (p / p.sum()) @ v[:, 0, :]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_interleaved_pairing_complex_form():
    """Interleaved pairs (x[2i], x[2i+1]) rotate as the complex numbers
    x[2i] + i x[2i+1] multiplied by exp(i p theta_i) (RoFormer's form)."""
    rng = np.random.default_rng(3)
    for Dm in (8, 64, 128):
        x = rng.standard_normal(Dm)
        for pos in (0, 3, 777, 30000):
            spec = RopeSpec(1e4, pairing="interleaved")
            got = oracle.rope(x, pos, spec)
            z = (x[0::2] + 1j * x[1::2]) * np.exp(1j * pos * np.power(1e4, -2.0 * np.arange(Dm // 2) / Dm))
            want = np.empty(Dm)
            want[0::2], want[1::2] = z.real, z.imag
            np.testing.assert_allclose(got, want, rtol=0, atol=1e-10)


def test_interleaved_scores_equal_half_pairing_on_permuted_vectors():
    """A score is a dot product over the head dimension, so interleaved RoPE on
    (q, k) equals rotate-half RoPE on both vectors with evens moved to the first
    half and odds to the second (the layout the library stores)."""
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])
    inter = RopeSpec(BASE, pairing="interleaved")
    for m, n in ((0, 0), (5, 2), (4000, 17), (33000, 32999)):
        a = oracle.rope(q, m, inter) @ oracle.rope(k, n, inter)
        b = oracle.rope(q[perm], m, BASE) @ oracle.rope(k[perm], n, BASE)
        assert a == pytest.approx(b, rel=1e-12, abs=1e-12)


# ---------------------------------------------------------------- ALiBi (§3.5)

def test_alibi_slopes_closed_forms():
    """The slope rule of the ALiBi paper: geometric 2^(-8i/n) for powers of two;
    for 12 heads the 8-head sequence then 2^-0.5, 2^-1.5, 2^-2.5, 2^-3.5."""
    np.testing.assert_array_equal(oracle.alibi_slopes(8), [2.0 ** -i for i in range(1, 9)])
    np.testing.assert_allclose(oracle.alibi_slopes(12),
                               [2.0 ** -i for i in range(1, 9)] + [2.0 ** -(i + 0.5) for i in range(4)], rtol=1e-15)
    s32 = oracle.alibi_slopes(32)
    np.testing.assert_allclose(s32, [2.0 ** (-i / 4) for i in range(1, 33)], rtol=1e-15)
    assert len(oracle.alibi_slopes(24)) == 24


def test_alibi_attention_bruteforce_and_shift():
    """Scores by explicit loops (no rotation, bias -slope (m - n), causal), and
    invariance under a common shift of all positions."""
    rng = np.random.default_rng(5)
    Lq, L, Hq, Hkv, Dm = 3, 7, 4, 2, 16
    q = rng.standard_normal((Lq, Hq, Dm))
    k = rng.standard_normal((L, Hkv, Dm))
    v = rng.standard_normal((L, Hkv, Dm))
    qp, kp = np.arange(4, 7), np.arange(7)
    got = oracle.attention(q, k, v, qp, kp, oracle.AlibiSpec())
    slopes = oracle.alibi_slopes(Hq)
    for i in range(Lq):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            sc = [q[i, h] @ k[j, kv] / np.sqrt(Dm) - slopes[h] * (qp[i] - kp[j]) for j in range(L) if kp[j] <= qp[i]]
            p = np.exp(np.array(sc) - max(sc))
            want = (p / p.sum()) @ v[: len(sc), kv]
            np.testing.assert_allclose(got[i, h], want, rtol=1e-12, atol=1e-12)
    shifted = oracle.attention(q, k, v, qp + 1000, kp + 1000, oracle.AlibiSpec())
    np.testing.assert_allclose(shifted, got, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- mutations
# Each plants a plausible mistake in the oracle's variant code and checks that
# at least one pin above fails on it.

def _pins():
    return [test_linear_is_rope_at_interpolated_positions, test_ntk_closed_form,
            lambda: test_band_limits_and_monotone_blend("yarn", 4096, 1.0, 32.0),
            lambda: test_band_limits_and_monotone_blend("llama3", 8192, 1.0, 4.0),
            test_yarn_logit_scale, test_interleaved_pairing_complex_form,
            test_alibi_slopes_closed_forms, test_alibi_attention_bruteforce_and_shift]


def _failing_pins():
    failed = 0
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            failed += 1
    return failed


def test_every_pin_passes_on_the_oracle():
    assert _failing_pins() == 0


def _freq_mutant(kind, formula):
    real = RopeSpec.inv_freq

    def inv_freq(self, head_dim):
        if self.kind != kind:
            return real(self, head_dim)
        plain = np.power(self.base, -2.0 * np.arange(head_dim // 2) / head_dim)
        return formula(self, plain, head_dim)
    return inv_freq


def _yarn_reversed(self, plain, head_dim):
    r = self.original / (2.0 * np.pi / plain)
    ramp = np.clip((r - self.low) / (self.high - self.low), 0.0, 1.0)
    return ramp * plain / self.factor + (1.0 - ramp) * plain


def _yarn_no_two_pi(self, plain, head_dim):
    r = self.original * plain
    ramp = np.clip((r - self.low) / (self.high - self.low), 0.0, 1.0)
    return (1.0 - ramp) * plain / self.factor + ramp * plain


def _llama3_swapped(self, plain, head_dim):
    wl = 2.0 * np.pi / plain
    blend = (self.original / wl - self.low) / (self.high - self.low)
    mid = (1.0 - blend) * plain / self.factor + blend * plain
    return np.where(wl < self.original / self.low, plain, np.where(wl > self.original / self.high, plain / self.factor, mid))


FREQ_MUTANTS = {
    "linear multiplies": _freq_mutant("linear", lambda self, p, D: p * self.factor),
    "ntk exponent D/(D-1)": _freq_mutant(
        "ntk", lambda self, p, D: np.power(self.base * self.factor ** (D / (D - 1.0)), -2.0 * np.arange(D // 2) / D)),
    "ntk without exponent": _freq_mutant(
        "ntk", lambda self, p, D: np.power(self.base * self.factor, -2.0 * np.arange(D // 2) / D)),
    "yarn ramp reversed": _freq_mutant("yarn", _yarn_reversed),
    "yarn ratio without 2 pi": _freq_mutant("yarn", _yarn_no_two_pi),
    "llama3 bands swapped": _freq_mutant("llama3", _llama3_swapped),
}


@pytest.mark.parametrize("name", list(FREQ_MUTANTS))
def test_frequency_mutants_are_caught(monkeypatch, name):
    monkeypatch.setattr(RopeSpec, "inv_freq", FREQ_MUTANTS[name])
    assert _failing_pins() >= 1


def test_yarn_temperature_not_squared_is_caught(monkeypatch):
    def logit_scale(self, head_dim):
        t = (0.1 * np.log(self.factor) + 1.0) if self.kind == "yarn" and self.factor > 1.0 else 1.0
        return float(t / np.sqrt(head_dim))
    monkeypatch.setattr(RopeSpec, "logit_scale", logit_scale)
    assert _failing_pins() >= 1


def test_interleaved_as_half_pairing_is_caught(monkeypatch):
    import oracle.lazyattn_oracle as lo
    real = lo.rope

    def rope(x, pos, theta):
        if isinstance(theta, RopeSpec) and theta.pairing == "interleaved":
            theta = RopeSpec(theta.base, theta.kind, theta.factor, int(theta.original), theta.low, theta.high)
        return real(x, pos, theta)
    monkeypatch.setattr(lo, "rope", rope)
    monkeypatch.setattr(oracle, "rope", rope)
    assert _failing_pins() >= 1


def test_alibi_mutants_are_caught(monkeypatch):
    import oracle.lazyattn_oracle as lo
    real_slopes, real_attn = lo.alibi_slopes, lo.attention_prerotated

    def even_slopes(n):   # the second half from the wrong positions of the 2p sequence
        p = 1
        while p * 2 <= n:
            p *= 2
        if p == n:
            return real_slopes(n)
        geo = [2.0 ** (-8.0 * (i + 1) / (2 * p)) for i in range(2 * p)]
        return np.array(list(real_slopes(p)) + geo[1::2][: n - p])

    def flipped(q_rot, k_rot, v, q_pos, k_pos, scale=None, alibi=None):
        return real_attn(q_rot, k_rot, v, q_pos, k_pos, scale, None if alibi is None else -alibi)

    def by_kv_head(q_rot, k_rot, v, q_pos, k_pos, scale=None, alibi=None):
        if alibi is not None:
            g = q_rot.shape[1] // k_rot.shape[1]
            alibi = np.repeat(alibi[::g], g)
        return real_attn(q_rot, k_rot, v, q_pos, k_pos, scale, alibi)

    for name, target, mutant in (("alibi_slopes", lo, even_slopes), ("attention_prerotated", lo, flipped),
                                 ("attention_prerotated", lo, by_kv_head)):
        monkeypatch.setattr(target, name, mutant)
        if name == "alibi_slopes":
            monkeypatch.setattr(oracle, "alibi_slopes", mutant)
        assert _failing_pins() >= 1, mutant.__name__
        monkeypatch.undo()

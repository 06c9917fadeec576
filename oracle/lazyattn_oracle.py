"""fp64 oracle: RoPE attention over documents reused at arbitrary logical offsets.

TEST INFRASTRUCTURE ONLY. Imported by tests/, __graft_entry__.smoke() and the
cpu_baseline / reference leg of bench.py; never by the library.

Source: LazyAttention: Efficient Retrieval-Augmented Generation with Deferred
Positional Encoding.
  * §3.1 Eq. 4 and the RoPE form below it: softmax(f(Q,m) f(K,n)^T / sqrt(d_k)) V,
    with d_k the head size.
  * §3.1 "Deferred encoding": Q, K, V are computed without positions; the cache
    holds purely content-based K and V; position is applied at attention time.
  * §1: the result is mathematically identical to re-encoding duplicated caches,
    so the oracle is the plain definition - RoPE attention over the request's
    logical sequence - evaluated in fp64.
  * §3.2 "Prefilling": the rotation of a half-dimension pair,
    k1' = k1 cos(a) - k2 sin(a),  k2' = k1 sin(a) + k2 cos(a).
  * Appendix C.4: angles come from absolute indices (m * theta_i), not from an
    iterated rotation state.
  * §3.5 "GQA/MQA compatibility": query heads share KV heads; no other change.

Readings where the paper is silent:
  * pairing is rotate-half (dims i and i + D/2), as the paper's "half-dimensions"
    K1 / K2 of Figure 3(b) describe;
  * frequencies theta_i = base^(-2i/D) for i < D/2 (RoFormer's definition);
  * query head h reads KV head h // (Hq / Hkv) (contiguous grouping);
  * a key is visible to a query iff its logical position <= the query's;
  * documents are concatenated from position 0 in table order, the query
    segment follows, generated tokens follow the query segment.

Parity pins (tests/test_oracle_pins.py): a hand-derived RoPE example
(tests/golden/), rotation-group identities, equality of the eager (materialised)
and lazy paths, shift invariance (Fact 3.2), document sharing at two offsets
against a complex-number brute force, reduction to PyTorch's
scaled_dot_product_attention at zero angles, and the Zipf closed form.
"""
from __future__ import annotations

from typing import Iterable, List, Sequence, Tuple

import numpy as np

__all__ = [
    "PAGE_SIZE", "unpack_entry", "resolve_entries", "RopeSpec", "AlibiSpec", "alibi_slopes", "rope_inv_freq",
    "logit_scale", "rope",
    "attention", "prefill_request", "decode_request", "materialize_rotated",
    "attention_prerotated", "paged_context", "paged_prefill", "paged_decode_step",
]

PAGE_SIZE = 16


# ----------------------------------------------------------------------------
# block-table entries: one 64-bit word per page
#   bits  0..31  physical page id
#   bits 32..57  logical position of the page's slot 0
#   bits 58..62  number of valid slots (0..16)
#   bit  63      writable (decode appends into writable pages only)
# The paper packs (block_id, offset, mask) into one 64-bit register (§3.2,
# "Decoding"); this is the field layout the library's header fixes.
# ----------------------------------------------------------------------------

def unpack_entry(e: int) -> Tuple[int, int, int, int]:
    e = int(e) & 0xFFFFFFFFFFFFFFFF
    page = e & 0xFFFFFFFF
    start = (e >> 32) & ((1 << 26) - 1)
    nvalid = (e >> 58) & 0x1F
    writable = e >> 63
    return page, start, nvalid, writable


def resolve_entries(entries: Iterable[int]) -> List[Tuple[int, int, int]]:
    """(page, slot, logical position) of every valid token, in table order."""
    out = []
    for e in entries:
        page, start, nvalid, _ = unpack_entry(e)
        for slot in range(nvalid):
            out.append((page, slot, start + slot))
    return out


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

class RopeSpec:
    """A RoPE base with one of the scaled RoPE-family variants that §3.5
    ("Generalization Beyond Standard RoPE") says keep the score
    q^T R_{n-m} k with variant-specific metadata. Each variant, as its
    publication defines it, changes the frequencies:
      "linear"  position interpolation (Chen et al., 2023): every frequency
                divided by the factor s, i.e. positions read as p / s;
      "ntk"     NTK-aware scaling: the base becomes base * s^(D / (D - 2));
      "yarn"    YaRN (Peng et al., 2023): with r_i = (original context) /
                (wavelength 2 pi / theta_i), frequencies with r_i < low are
                interpolated (theta_i / s), those with r_i > high are kept, a
                linear ramp in r blends in between; the logits are multiplied
                by (0.1 ln s + 1)^2 (the attention temperature);
      "llama3"  the Llama 3.1 rule: wavelengths below original / high kept,
                above original / low divided by s, and in between a blend with
                weight (original / wavelength - low) / (high - low) on the
                kept frequency.
    """

    def __init__(self, base: float, kind: str = "default", factor: float = 1.0,
                 original_max_position: int = 0, low: float = 0.0, high: float = 0.0, pairing: str = "half"):
        """pairing: "half" rotates (x[i], x[i + D/2]) (the paper's half-dimensions);
        "interleaved" rotates (x[2i], x[2i+1]) (RoFormer's original form, Llama's
        layout), with the same frequencies theta_i."""
        self.base, self.kind, self.factor = float(base), kind, float(factor)
        self.original, self.low, self.high = float(original_max_position), float(low), float(high)
        self.pairing = pairing

    def inv_freq(self, head_dim: int) -> np.ndarray:
        i = np.arange(head_dim // 2, dtype=np.float64)
        plain = np.power(self.base, -2.0 * i / head_dim)
        s = self.factor
        if self.kind == "default":
            return plain
        if self.kind == "linear":
            return plain / s
        if self.kind == "ntk":
            return np.power(self.base * s ** (head_dim / (head_dim - 2.0)), -2.0 * i / head_dim)
        if self.kind == "yarn":
            r = self.original / (2.0 * np.pi / plain)
            ramp = np.clip((r - self.low) / (self.high - self.low), 0.0, 1.0)
            return (1.0 - ramp) * plain / s + ramp * plain
        if self.kind == "llama3":
            wavelength = 2.0 * np.pi / plain
            blend = (self.original / wavelength - self.low) / (self.high - self.low)
            mid = (1.0 - blend) * plain / s + blend * plain
            return np.where(wavelength < self.original / self.high, plain,
                            np.where(wavelength > self.original / self.low, plain / s, mid))
        raise ValueError(self.kind)

    def logit_scale(self, head_dim: int) -> float:
        scale = 1.0 / np.sqrt(np.float64(head_dim))
        if self.kind == "yarn" and self.factor > 1.0:
            scale *= (0.1 * np.log(self.factor) + 1.0) ** 2
        return float(scale)


class AlibiSpec:
    """ALiBi instead of RoPE (§3.5, "Score-space positional methods": the bias
    is added to the score rather than rotating q and k, so it too can be
    applied lazily from logical positions). Passed where the other functions
    take the RoPE base: q and k are not rotated, and the score of query head h
    at position m with a key at position n gets -slope_h * (m - n)."""


def alibi_slopes(n_heads: int) -> np.ndarray:
    """ALiBi head slopes (Press et al.): for n a power of two, the geometric
    sequence 2^(-8/n), 2^(-16/n), ..., 2^(-8); otherwise the slopes for the
    largest power of two p below n, followed by the 1st, 3rd, 5th, ... slopes
    of the sequence for 2p, up to n in all."""
    def geometric(n):
        return [2.0 ** (-8.0 * (i + 1) / n) for i in range(n)]
    p = 1
    while p * 2 <= n_heads:
        p *= 2
    if p == n_heads:
        return np.array(geometric(n_heads))
    return np.array(geometric(p) + geometric(2 * p)[0::2][: n_heads - p])


def rope_inv_freq(head_dim: int, theta) -> np.ndarray:
    """theta_i, i = 0 .. D/2-1, fp64: base^(-2i/D) for a plain base (a number),
    or the variant's frequencies for a RopeSpec."""
    if isinstance(theta, RopeSpec):
        return theta.inv_freq(head_dim)
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / head_dim)


def logit_scale(head_dim: int, theta) -> float:
    """Scale of q.k in the softmax: 1/sqrt(D) (Eq. 4), times YaRN's temperature."""
    if isinstance(theta, RopeSpec):
        return theta.logit_scale(head_dim)
    return float(1.0 / np.sqrt(np.float64(head_dim)))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate x[..., D] at positions pos (shape x.shape[:-1] or broadcastable).

    Pair (x[i], x[i + D/2]) is rotated by angle pos * theta_i.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    if isinstance(theta, RopeSpec) and theta.pairing == "interleaved":
        x1, x2 = x[..., 0::2], x[..., 1::2]
        out = np.empty(np.broadcast_shapes(x.shape, c.shape[:-1] + (D,)), dtype=np.float64)
        out[..., 0::2] = x1 * c - x2 * s
        out[..., 1::2] = x1 * s + x2 * c
        return out
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


# ----------------------------------------------------------------------------
# attention (Eq. 4 with RoPE applied to already-positioned inputs)
# ----------------------------------------------------------------------------

def attention_prerotated(q_rot: np.ndarray, k_rot: np.ndarray, v: np.ndarray,
                         q_pos: np.ndarray, k_pos: np.ndarray, scale: float = None,
                         alibi: np.ndarray = None) -> np.ndarray:
    """Causal softmax attention over already rotated q and k.

    q_rot: [Lq][Hq][D]; k_rot, v: [L][Hkv][D]; q_pos: [Lq]; k_pos: [L];
    scale: logit scale, 1/sqrt(D) when None; alibi: per query head slopes
    of an ALiBi bias -slope * (q_pos - k_pos), or None.
    Returns [Lq][Hq][D] fp64.
    """
    q_rot = np.asarray(q_rot, np.float64)
    k_rot = np.asarray(k_rot, np.float64)
    v = np.asarray(v, np.float64)
    Lq, Hq, D = q_rot.shape
    Hkv = k_rot.shape[1]
    g = Hq // Hkv
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]   # [Lq][L]
    out = np.zeros((Lq, Hq, D), dtype=np.float64)
    for h in range(Hq):
        kv = h // g
        s = (q_rot[:, h, :] @ k_rot[:, kv, :].T) * (1.0 / np.sqrt(np.float64(D)) if scale is None else scale)
        if alibi is not None:
            s = s - alibi[h] * (np.asarray(q_pos, np.float64)[:, None] - np.asarray(k_pos, np.float64)[None, :])
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kv, :]
    return out


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos, k_pos,
              theta: float) -> np.ndarray:
    """Lazy form: q and k arrive without positions and are rotated here."""
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    if isinstance(theta, AlibiSpec):
        return attention_prerotated(q, k, v, q_pos, k_pos, None, alibi_slopes(np.asarray(q).shape[1]))
    q_rot = rope(q, q_pos[:, None], theta)
    k_rot = rope(k, k_pos[:, None], theta)
    return attention_prerotated(q_rot, k_rot, v, q_pos, k_pos, logit_scale(np.asarray(q).shape[-1], theta))


def materialize_rotated(k: np.ndarray, k_pos, theta: float) -> np.ndarray:
    """Eager form: a private copy of k rotated at its logical positions
    (what re-encoding systems store for each placement of a document)."""
    return rope(np.array(k, dtype=np.float64, copy=True),
                np.asarray(k_pos, np.int64)[:, None], theta)


# ----------------------------------------------------------------------------
# whole requests, from logical contents
# ----------------------------------------------------------------------------

def _concat_context(docs_kv: Sequence[Tuple[np.ndarray, np.ndarray]]):
    ks = [np.asarray(k, np.float64) for k, _ in docs_kv]
    vs = [np.asarray(v, np.float64) for _, v in docs_kv]
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


def prefill_request(docs_kv, q, k_q, v_q, theta: float) -> np.ndarray:
    """Query-segment output of one request.

    docs_kv: list of (k, v) [len][Hkv][D] in prompt order, concatenated from
    position 0; (q, k_q, v_q): the query segment that follows them.
    """
    k_ctx, v_ctx = _concat_context(list(docs_kv) + [(k_q, v_q)])
    L0 = sum(np.asarray(k).shape[0] for k, _ in docs_kv)
    Lq = np.asarray(q).shape[0]
    k_pos = np.arange(k_ctx.shape[0], dtype=np.int64)
    q_pos = np.arange(L0, L0 + Lq, dtype=np.int64)
    return attention(q, k_ctx, v_ctx, q_pos, k_pos, theta)


def decode_request(docs_kv, k_q, v_q, steps, theta: float) -> List[np.ndarray]:
    """Outputs of consecutive decode steps of one request.

    steps: list of (q [Hq][D], k_new [Hkv][D], v_new [Hkv][D]). Step t appends
    its token at position (context + query segment + t), then attends with it.
    """
    k_ctx, v_ctx = _concat_context(list(docs_kv) + [(k_q, v_q)])
    outs = []
    for q, k_new, v_new in steps:
        k_ctx = np.concatenate([k_ctx, np.asarray(k_new, np.float64)[None]], axis=0)
        v_ctx = np.concatenate([v_ctx, np.asarray(v_new, np.float64)[None]], axis=0)
        L = k_ctx.shape[0]
        o = attention(np.asarray(q)[None], k_ctx, v_ctx, [L - 1], np.arange(L), theta)
        outs.append(o[0])
    return outs


# ----------------------------------------------------------------------------
# the same computation through a paged pool and block table
# ----------------------------------------------------------------------------

def paged_context(k_pool: np.ndarray, v_pool: np.ndarray, entries: Iterable[int]):
    """Gather (k, v, positions) of a request from pools [page][Hkv][16][D]."""
    toks = resolve_entries(entries)
    if not toks:
        Hkv, D = k_pool.shape[1], k_pool.shape[3]
        z = np.zeros((0, Hkv, D))
        return z, z.copy(), np.zeros((0,), np.int64)
    pages = np.array([t[0] for t in toks])
    slots = np.array([t[1] for t in toks])
    pos = np.array([t[2] for t in toks], dtype=np.int64)
    k = np.asarray(k_pool[pages, :, slots, :], np.float64)
    v = np.asarray(v_pool[pages, :, slots, :], np.float64)
    return k, v, pos


def paged_prefill(k_pool, v_pool, entries, q, q_start: int, theta: float) -> np.ndarray:
    """Prefill of one request whose K/V (documents and query segment) are in
    the pool; its query tokens sit at q_start, q_start + 1, ..."""
    k, v, k_pos = paged_context(k_pool, v_pool, entries)
    Lq = np.asarray(q).shape[0]
    q_pos = np.arange(q_start, q_start + Lq, dtype=np.int64)
    return attention(q, k, v, q_pos, k_pos, theta)


def paged_decode_step(k_pool, v_pool, entries: List[int], q, k_new, v_new,
                      theta: float):
    """One decode step of one request on a paged pool (modified in place).

    The new token goes into the first writable, non-full entry of the trailing
    run of writable entries; that entry's valid count grows by one. Returns
    (output [Hq][D], new entries list).
    """
    entries = [int(e) for e in entries]
    tail = None
    for i in range(len(entries) - 1, -1, -1):
        page, start, nvalid, writable = unpack_entry(entries[i])
        if not writable:
            break
        if nvalid < PAGE_SIZE:
            tail = i
    if tail is None:
        raise ValueError("no writable page with a free slot")
    page, start, nvalid, writable = unpack_entry(entries[tail])
    k_pool[page, :, nvalid, :] = k_new
    v_pool[page, :, nvalid, :] = v_new
    entries[tail] = (page | (start << 32) | ((nvalid + 1) << 58) | (writable << 63))
    q_pos = start + nvalid
    k, v, k_pos = paged_context(k_pool, v_pool, entries)
    o = attention(np.asarray(q)[None], k, v, [q_pos], k_pos, theta)
    return o[0], entries

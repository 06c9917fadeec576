"""Seeded synthetic RAG workloads for the LazyAttention hot path.

This module only *generates inputs*: document K/V, query segments, decode-step
activations and per-request document lists. It contains none of the attention
arithmetic, so both the fp64 oracle and the CUDA library can consume it without
sharing any of the method's code.

Workload shapes follow the configurations the LazyAttention paper's RAG setting
implies (LazyAttention: Efficient Retrieval-Augmented Generation with Deferred
Positional Encoding, §2 "Hit-ratio impact under limited cache capacity": Zipf
document popularity, p_i proportional to i^-alpha; §4.3: documents concatenated
ahead of a query segment, no common preamble). The few-shot configurations follow
App. C.7 "Beyond RAG: Few-Shot Classification": short exemplar chunks of varying
length recur across requests at different positions and in different orders,
with skewed or uniform popularity.

Every random piece is drawn from its own PCG64 stream keyed by
(seed, tag, index...), so any single document, query segment or decode step can
be regenerated on its own - the oracle recomputes only the requests it samples.

Inputs are drawn in fp32 from N(0, 1). For bf16 workloads they are rounded to
bf16 (round to nearest even) here, once; both sides then consume identical values.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

PAGE_SIZE = 16

# stream tags (stable: changing one changes every input of that kind)
_TAG_DOC = 1
_TAG_REQ_DOCS = 2
_TAG_QSEG = 3
_TAG_DECODE = 4
_TAG_DOC_LEN = 5


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    dtype: str              # "f32" or "bf16"
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rope_theta: float
    n_docs: int             # documents in the pool
    doc_len: int            # tokens per document (the maximum when doc_len_min is set)
    n_requests: int
    docs_per_request: int
    zipf_alpha: Optional[float]   # None: uniform draws
    q_len: int              # query-segment tokens per request (0: none)
    decode_steps: int
    seed: int
    doc_len_min: int = 0    # > 0: document lengths uniform in [doc_len_min, doc_len]
    distinct: bool = False  # documents of one request drawn without replacement, then shuffled

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def doc_pages(self) -> int:
        """Pages of the longest document."""
        return -(-self.doc_len // PAGE_SIZE)

    @property
    def q_pages(self) -> int:
        return -(-self.q_len // PAGE_SIZE)

    @property
    def decode_pages(self) -> int:
        """Pages each request reserves for generated tokens.

        Tokens generated after the query segment first fill the free slots of
        the segment's last page, then these reserved pages.
        """
        free_in_tail = (self.q_pages * PAGE_SIZE - self.q_len)
        extra = max(0, self.decode_steps - free_in_tail)
        return -(-extra // PAGE_SIZE)

    @property
    def context_len(self) -> int:
        """Document tokens per request: the count when all documents have one
        length, else the largest over the requests (request_context_len gives
        each request's own)."""
        if not self.doc_len_min:
            return self.docs_per_request * self.doc_len
        return int(max(request_context_lens(self))) if self.n_requests else 0

    @property
    def max_position(self) -> int:
        """Smallest position-table size that covers every logical position."""
        return self.context_len + self.q_len + self.decode_steps


CONFIGS = {
    # Tiny fp32 single-layer attention (parity only).
    "tiny_fp32": Config("tiny_fp32", "f32", 4, 2, 64, 1.0e4, 4, 32, 2, 3, None, 16, 4, 0),
    # Llama-3-8B-shaped attention layer.
    "llama3_8b": Config("llama3_8b", "bf16", 32, 8, 128, 5.0e5, 200, 256, 16, 8, 1.0, 64, 32, 1),
    # Decode-heavy RAG batch: 128 requests x 20 docs of 512 tokens, no query segment.
    "rag_decode": Config("rag_decode", "bf16", 32, 8, 128, 5.0e5, 1000, 512, 128, 20, 1.0, 0, 256, 2),
    # Prefill-heavy TTFT sweep: 10 / 20 / 40 docs of 1024 tokens per prompt.
    "ttft_sweep_10": Config("ttft_sweep_10", "bf16", 32, 8, 128, 5.0e5, 500, 1024, 32, 10, 1.2, 128, 0, 3),
    "ttft_sweep_20": Config("ttft_sweep_20", "bf16", 32, 8, 128, 5.0e5, 500, 1024, 32, 20, 1.2, 128, 0, 3),
    "ttft_sweep_40": Config("ttft_sweep_40", "bf16", 32, 8, 128, 5.0e5, 500, 1024, 32, 40, 1.2, 128, 0, 3),
    # Llama-3-70B-shaped attention layer, ~16.8 GB of pre-RoPE KV resident.
    "llama3_70b": Config("llama3_70b", "bf16", 64, 8, 128, 5.0e5, 4000, 1024, 64, 32, 0.8, 256, 128, 4),
    # Few-shot classification: 128 prompts of 32 distinct exemplar chunks (32..96
    # tokens each, so entries start off page boundaries and end in partial pages)
    # from a pool of 1000, skewed (Zipf 1.0) or uniform popularity, then a 48-token
    # item to classify and 4 generated label tokens.
    "few_shot_skewed": Config("few_shot_skewed", "bf16", 32, 8, 128, 5.0e5, 1000, 96, 128, 32, 1.0, 48, 4, 5,
                              doc_len_min=32, distinct=True),
    "few_shot_uniform": Config("few_shot_uniform", "bf16", 32, 8, 128, 5.0e5, 1000, 96, 128, 32, None, 48, 4, 6,
                               doc_len_min=32, distinct=True),
    # The same pattern at the tiny fp32 shape (parity only).
    "tiny_ragged_fp32": Config("tiny_ragged_fp32", "f32", 4, 2, 64, 1.0e4, 6, 40, 3, 4, None, 21, 5, 7,
                               doc_len_min=5, distinct=True),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


# ----------------------------------------------------------------------------
# bf16 rounding (input preparation only)
# ----------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + np.uint32(0x7FFF) + lsb) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bf16_bits(x))


def _normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return round_bf16(x) if dtype == "bf16" else x


# ----------------------------------------------------------------------------
# Zipf document popularity
# ----------------------------------------------------------------------------

def zipf_probabilities(n: int, alpha: float) -> np.ndarray:
    """p_i proportional to i^-alpha over ranks i = 1..n."""
    i = np.arange(1, n + 1, dtype=np.float64)
    w = i ** (-float(alpha))
    return w / w.sum()


def zipf_ranks(rng: np.random.Generator, n: int, alpha: float, size) -> np.ndarray:
    """i.i.d. ranks in 1..n drawn by inverting the cumulative distribution."""
    cdf = np.cumsum(zipf_probabilities(n, alpha))
    cdf[-1] = 1.0
    u = rng.random(size)
    return np.searchsorted(cdf, u, side="right").astype(np.int64) + 1


def request_docs(cfg: Config) -> np.ndarray:
    """[n_requests][docs_per_request] document ids, in prompt order.

    Rank i maps to document id i-1. Draws are i.i.d. with replacement, so a
    document may appear in several requests and twice within one request.
    With cfg.distinct, each request instead draws its documents without
    replacement (Zipf or uniform weights, one after another) and then shuffles
    them, so a chunk appears at most once per prompt, in a random order.
    """
    rng = _rng(cfg.seed, _TAG_REQ_DOCS)
    shape = (cfg.n_requests, cfg.docs_per_request)
    if cfg.distinct:
        p = None if cfg.zipf_alpha is None else zipf_probabilities(cfg.n_docs, cfg.zipf_alpha)
        out = np.empty(shape, np.int64)
        for r in range(cfg.n_requests):
            out[r] = rng.permutation(rng.choice(cfg.n_docs, size=cfg.docs_per_request, replace=False, p=p))
        return out
    if cfg.zipf_alpha is None:
        return rng.integers(0, cfg.n_docs, size=shape).astype(np.int64)
    return zipf_ranks(rng, cfg.n_docs, cfg.zipf_alpha, shape) - 1


def doc_lengths(cfg: Config) -> np.ndarray:
    """Token count of every pool document (all cfg.doc_len unless doc_len_min is set)."""
    if not cfg.doc_len_min:
        return np.full(cfg.n_docs, cfg.doc_len, np.int64)
    rng = _rng(cfg.seed, _TAG_DOC_LEN)
    return rng.integers(cfg.doc_len_min, cfg.doc_len + 1, size=cfg.n_docs).astype(np.int64)


def request_context_lens(cfg: Config) -> np.ndarray:
    """Document tokens of each request."""
    return doc_lengths(cfg)[request_docs(cfg)].sum(axis=1).astype(np.int64)


# ----------------------------------------------------------------------------
# activations
# ----------------------------------------------------------------------------

def doc_kv(cfg: Config, doc_id: int):
    """Pre-RoPE (k, v) of one document: two [length][n_kv_heads][head_dim] arrays."""
    rng = _rng(cfg.seed, _TAG_DOC, doc_id)
    n = cfg.doc_len if not cfg.doc_len_min else int(doc_lengths(cfg)[doc_id])
    shape = (n, cfg.n_kv_heads, cfg.head_dim)
    return _normal(rng, shape, cfg.dtype), _normal(rng, shape, cfg.dtype)


def query_segment(cfg: Config, r: int):
    """Pre-RoPE (q, k, v) of request r's query segment.

    q: [q_len][n_q_heads][head_dim]; k, v: [q_len][n_kv_heads][head_dim].
    """
    rng = _rng(cfg.seed, _TAG_QSEG, r)
    q = _normal(rng, (cfg.q_len, cfg.n_q_heads, cfg.head_dim), cfg.dtype)
    k = _normal(rng, (cfg.q_len, cfg.n_kv_heads, cfg.head_dim), cfg.dtype)
    v = _normal(rng, (cfg.q_len, cfg.n_kv_heads, cfg.head_dim), cfg.dtype)
    return q, k, v


def decode_inputs(cfg: Config, step: int, requests: Optional[Sequence[int]] = None):
    """Pre-RoPE (q, k_new, v_new) of one decode step.

    q: [R][n_q_heads][head_dim]; k_new, v_new: [R][n_kv_heads][head_dim], for the
    listed requests (default: all). Each request has its own stream per step.
    """
    if requests is None:
        requests = range(cfg.n_requests)
    qs, ks, vs = [], [], []
    for r in requests:
        rng = _rng(cfg.seed, _TAG_DECODE, step, r)
        qs.append(_normal(rng, (cfg.n_q_heads, cfg.head_dim), cfg.dtype))
        ks.append(_normal(rng, (cfg.n_kv_heads, cfg.head_dim), cfg.dtype))
        vs.append(_normal(rng, (cfg.n_kv_heads, cfg.head_dim), cfg.dtype))
    return np.stack(qs), np.stack(ks), np.stack(vs)


def request_layout(cfg: Config, r: int = 0) -> List[int]:
    """Logical start position of each of request r's documents, then of its query segment.

    Documents are concatenated in table order from position 0 with no gaps; the
    query segment follows them; generated tokens follow the query segment.
    """
    lens = doc_lengths(cfg)[request_docs(cfg)[r]]
    return [0] + np.cumsum(lens).astype(np.int64).tolist()

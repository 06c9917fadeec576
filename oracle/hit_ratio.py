"""Closed-form Zipf hit ratios (test infrastructure only).

LazyAttention: Efficient Retrieval-Augmented Generation with Deferred Positional
Encoding, §2 "Hit-ratio impact under limited cache capacity", Eqs. 1-3: with
document popularity proportional to i^-alpha, a position-agnostic cache holding C
entries covers the top C documents, while a position-aware cache that needs up
to D positional copies per document covers only the top floor(C/D).

Parity pinned by: the harmonic-number special case alpha = 1 and the value the
paper prints for D = 20, C = 100 (2.86, whose alpha the paper does not give).
"""
__all__ = ["zipf_partial_sum", "hit_ratio_agnostic", "hit_ratio_aware", "hit_ratio_gap"]


def zipf_partial_sum(n: int, alpha: float) -> float:
    """sum_{i=1..n} i^-alpha, in fp64, summed smallest term first."""
    s = 0.0
    for i in range(int(n), 0, -1):
        s += float(i) ** (-alpha)
    return s


def hit_ratio_agnostic(C: int, N: int, alpha: float) -> float:
    """Eq. 1: fraction of requests served by a cache of the top C documents."""
    return zipf_partial_sum(min(C, N), alpha) / zipf_partial_sum(N, alpha)


def hit_ratio_aware(C: int, D: int, N: int, alpha: float) -> float:
    """Eq. 2: same budget spent on D positional variants per document."""
    return zipf_partial_sum(min(C // D, N), alpha) / zipf_partial_sum(N, alpha)


def hit_ratio_gap(C: int, D: int, alpha: float) -> float:
    """Eq. 3: the ratio of Eq. 1 to Eq. 2 (the normaliser cancels)."""
    return zipf_partial_sum(C, alpha) / zipf_partial_sum(C // D, alpha)


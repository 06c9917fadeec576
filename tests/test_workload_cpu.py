"""Host-side checks of the seeded workload generator's few-shot pattern
(LazyAttention, App. C.7: exemplar chunks recur across prompts at different
positions and in different orders; skewed or uniform popularity), and that the
fixed-length workloads keep their layout."""
import collections

import numpy as np
import pytest

import workload

FEW_SHOT = ["few_shot_skewed", "few_shot_uniform", "tiny_ragged_fp32"]


@pytest.mark.parametrize("name", FEW_SHOT)
def test_chunks_distinct_lengths_in_range_and_contiguous_layout(name):
    cfg = workload.CONFIGS[name]
    lens = workload.doc_lengths(cfg)
    assert lens.min() >= cfg.doc_len_min and lens.max() <= cfg.doc_len
    assert len(set(lens.tolist())) > 1
    docs = workload.request_docs(cfg)
    assert docs.shape == (cfg.n_requests, cfg.docs_per_request)
    assert all(len(set(row.tolist())) == cfg.docs_per_request for row in docs)
    assert docs.min() >= 0 and docs.max() < cfg.n_docs
    ctx = workload.request_context_lens(cfg)
    assert cfg.context_len == ctx.max()
    assert cfg.max_position == ctx.max() + cfg.q_len + cfg.decode_steps
    for r in (0, cfg.n_requests - 1):
        kv = [workload.doc_kv(cfg, int(d)) for d in docs[r]]
        n = [k.shape[0] for k, _ in kv]
        assert all(k.shape == v.shape == (m, cfg.n_kv_heads, cfg.head_dim) for (k, v), m in zip(kv, n))
        assert workload.request_layout(cfg, r) == [0] + np.cumsum(n).tolist()
        assert ctx[r] == sum(n)
    # some document starts off a page boundary
    starts = [s for r in range(cfg.n_requests) for s in workload.request_layout(cfg, r)[:-1]]
    assert any(s % workload.PAGE_SIZE for s in starts)


@pytest.mark.parametrize("name", ["few_shot_skewed", "few_shot_uniform"])
def test_chunks_recur_at_different_offsets_and_orders(name):
    cfg = workload.CONFIGS[name]
    docs = workload.request_docs(cfg)
    offsets = collections.defaultdict(set)
    for r in range(cfg.n_requests):
        for d, s in zip(docs[r], workload.request_layout(cfg, r)):
            offsets[int(d)].add(s)
    assert sum(len(v) > 1 for v in offsets.values()) > cfg.n_docs // 4
    order = {}
    both = 0
    for r in range(cfg.n_requests):
        pos = {int(d): i for i, d in enumerate(docs[r])}
        for a in pos:
            for b in pos:
                if a < b:
                    o = pos[a] < pos[b]
                    if order.setdefault((a, b), o) != o:
                        both += 1
    assert both > 0


def test_skew_concentrates_reuse():
    top = []
    for name in ("few_shot_skewed", "few_shot_uniform"):
        cfg = workload.CONFIGS[name]
        c = np.bincount(workload.request_docs(cfg).ravel(), minlength=cfg.n_docs)
        top.append(np.sort(c)[::-1][:10].sum() / c.sum())
    assert top[0] > 3 * top[1]
    # without replacement, a document appears at most once per prompt
    cfg = workload.CONFIGS["few_shot_skewed"]
    assert np.bincount(workload.request_docs(cfg).ravel()).max() <= cfg.n_requests


def test_fixed_length_workloads_keep_their_layout():
    cfg = workload.CONFIGS["llama3_8b"]
    assert cfg.context_len == 8 * 256 and cfg.max_position == 2048 + 64 + 32
    assert workload.request_layout(cfg, 3) == [256 * i for i in range(9)]
    assert (workload.request_context_lens(cfg) == 2048).all()
    assert workload.doc_kv(cfg, 5)[0].shape == (256, 8, 128)

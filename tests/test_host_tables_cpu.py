"""Host-side block tables (position_agnostic_kv_lazyattn_gb300.paged) on CPU:
segments become the entries lazyattn_pack_entry defines (page, logical start of
slot 0, valid slots, writable), requests get their entry ranges, document-local
offsets default to each run's start, and the prefill query layout is the
exclusive prefix sum of the query lengths. Entries are decoded with the oracle's
own unpacking, which is pinned separately."""
import numpy as np
import pytest
import torch

import oracle


@pytest.fixture(scope="module")
def P():
    import __graft_entry__
    __graft_entry__.build()
    from position_agnostic_kv_lazyattn_gb300 import paged
    return paged


def test_ragged_segment_entries(P):
    seg = P.Segment([5, 6, 7], start=66, n_tokens=37, writable=True)
    pages, starts, nvalid, wr = P.segment_entries(seg)
    assert (pages, starts, nvalid, wr) == ([5, 6, 7], [66, 82, 98], [16, 16, 5], [1, 1, 1])
    # the tokens resolve to consecutive logical positions 66 .. 102
    ent = P.pack_entries(pages, starts, nvalid, wr)
    toks = oracle.resolve_entries([int(e) for e in ent])
    assert [t[2] for t in toks] == list(range(66, 103))
    assert [(t[0], t[1]) for t in toks][:17] == [(5, s) for s in range(16)] + [(6, 0)]
    # a reserved page for generated tokens: no valid slot yet
    _, starts, nvalid, _ = P.segment_entries(P.Segment([9], start=112, n_tokens=0, writable=True))
    assert starts == [112] and nvalid == [0]
    with pytest.raises(AssertionError):
        P.segment_entries(P.Segment([1], start=0, n_tokens=17))   # more tokens than pages hold


def test_batch_layout(P):
    reqs = [
        [P.Segment([0, 1], 0, 20), P.Segment([2], 20, 7, True)],
        [P.Segment([3], 0, 16), P.Segment([0, 1], 16, 20, delta=10), P.Segment([4, 5], 36, 29, True)],
        [P.Segment([6], 0, 5, True)],
    ]
    b = P.Batch(reqs, q_lens=[7, 29, 5], q_starts=[20, 36, 0], device="cpu")
    assert b.num_requests == 3
    assert b.offsets_host.tolist() == [0, 3, 8, 9]
    assert b.max_entries == 5
    assert b.total_q == 41 and b.max_q_len == 29
    assert b.q_offsets.tolist() == [0, 7, 36, 41]
    assert b.q_start.tolist() == [20, 36, 0]
    got = [oracle.unpack_entry(int(e)) for e in b.entries_host]
    assert got[3:8] == [(3, 0, 16, 0), (0, 16, 16, 0), (1, 32, 4, 0), (4, 36, 16, 1), (5, 52, 13, 1)]
    # document-local offsets: a run's start unless given
    assert b.delta_host.tolist() == [0, 0, 20, 0, 10, 10, 36, 36, 0]
    # the same document (pages 0, 1) serves request 0 at 0 and request 1 at 16
    r0 = oracle.resolve_entries([int(e) for e in b.entries_host[0:3]])
    r1 = oracle.resolve_entries([int(e) for e in b.entries_host[3:8]])
    assert [t[:2] for t in r0[:20]] == [t[:2] for t in r1[16:36]]
    assert [t[2] for t in r1[16:36]] == list(range(16, 36))
    # another entry array with the same requests and query layout (the baseline's copies)
    dst = (b.entries_host & ~np.uint64(0xFFFFFFFF)) | np.arange(100, 109, dtype=np.uint64)
    mb = b.with_entries(dst, 1, device="cpu")
    assert mb.flags == 1 and mb.offsets_host.tolist() == b.offsets_host.tolist()
    assert [oracle.unpack_entry(int(e))[0] for e in mb.entries_host] == list(range(100, 109))
    assert [oracle.unpack_entry(int(e))[1:] for e in mb.entries_host] == \
        [oracle.unpack_entry(int(e))[1:] for e in b.entries_host]
    assert torch.equal(mb.entry_offsets, b.entry_offsets)


def test_decode_only_batch_has_no_query_layout(P):
    b = P.Batch([[P.Segment([0], 0, 3, True)]], device="cpu")
    assert b.q_offsets is None and b.total_q == 0 and b.max_q_len == 0
    assert b.c.num_requests == 1 and b.c.max_entries == 1


def test_host_table_check(P):
    from position_agnostic_kv_lazyattn_gb300 import lazyattn as L
    ok = P.Batch([[P.Segment([0, 1], 0, 20), P.Segment([2], 20, 7, True)],
                  [P.Segment([3], 16, 16), P.Segment([0, 1], 32, 20), P.Segment([4], 0, 16)]],   # any order
                 q_lens=[7, 0], q_starts=[20, 52], device="cpu")
    ok.check(num_pages=8, max_position=64)
    assert L.lazyattn_check_batch_host(ok.entries_host, ok.offsets_host, 8, 64) == (0, -1)
    # an empty entry may sit anywhere (it holds no token)
    P.Batch([[P.Segment([0], 0, 16), P.Segment([5], 8, 0, True)]], device="cpu").check(8, 64)

    def status(reqs, num_pages=8, max_position=64):
        b = P.Batch(reqs, device="cpu")
        return L.lazyattn_check_batch_host(b.entries_host, b.offsets_host, num_pages, max_position)

    good = [P.Segment([0], 0, 16)]
    # two tokens of request 1 at positions 16..19
    assert status([good, [P.Segment([0, 1], 0, 20), P.Segment([2], 16, 7)]]) == (L.LAZYATTN_EINVAL, 1)
    # the same document twice at one offset
    assert status([[P.Segment([0], 0, 10), P.Segment([0], 0, 10)]]) == (L.LAZYATTN_EINVAL, 0)
    # page outside the pool; positions past the table
    assert status([good, good, [P.Segment([8], 0, 3)]]) == (L.LAZYATTN_ERANGE, 2)
    assert status([[P.Segment([1], 60, 5)]]) == (L.LAZYATTN_ERANGE, 0)
    # more than 16 valid slots in one entry (the field holds up to 31)
    e = P.pack_entries([1], [0], [17], [0])
    assert L.lazyattn_check_batch_host(e, [0, 1], 8, 64) == (L.LAZYATTN_ERANGE, 0)
    # malformed offsets
    assert L.lazyattn_check_batch_host(e, [1, 0], 8, 64) == (L.LAZYATTN_EINVAL, -1)
    with pytest.raises(L.LazyAttnError):
        P.Batch([[P.Segment([0], 0, 10), P.Segment([1], 5, 10)]], device="cpu").check(8, 64)


def test_host_table_check_random_tables(P):
    """Random tables against a direct model: decode every entry, fail on the
    first request with an out-of-range entry (ERANGE) or a repeated position
    (EINVAL), range failures taking precedence within a request."""
    from position_agnostic_kv_lazyattn_gb300 import lazyattn as L
    rng = np.random.default_rng(61)
    num_pages, max_position = 40, 300
    for _ in range(300):
        R = int(rng.integers(1, 5))
        ents, offs = [], [0]
        for _r in range(R):
            for _e in range(int(rng.integers(0, 6))):
                ents.append((int(rng.integers(0, 44)), int(rng.integers(0, 300)), int(rng.integers(0, 19)),
                             int(rng.integers(0, 2))))
            offs.append(len(ents))
        packed = P.pack_entries(*zip(*ents)) if ents else np.zeros(0, np.uint64)
        want = (0, -1)
        for r in range(R):
            toks, rc = [], 0
            for e in packed[offs[r]:offs[r + 1]]:
                page, start, n, _w = oracle.unpack_entry(int(e))
                if n == 0:
                    continue
                if page >= num_pages or n > 16 or start + n > max_position:
                    rc = L.LAZYATTN_ERANGE
                    break
                toks += range(start, start + n)
            if rc == 0 and len(set(toks)) != len(toks):
                rc = L.LAZYATTN_EINVAL
            if rc:
                want = (rc, r)
                break
        assert L.lazyattn_check_batch_host(packed, offs, num_pages, max_position) == want

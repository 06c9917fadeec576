"""Host logic of bench.py that needs no GPU: the count of distinct (page,
KV head) tiles each decode call reads, behind the DRAM-level roofline
fraction. Checked against a brute-force replay of the decode appends with the
oracle's paged decode step (its append rule) on small pools."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


def _pack(page, start, nvalid, writable):
    return (page & 0xFFFFFFFF) | (start << 32) | (nvalid << 58) | (int(writable) << 63)


def _tables():
    # request 0: document A (3 pages, the last partial), a 7-token query page, two reserved pages
    r0 = [_pack(0, 0, 16, 0), _pack(1, 16, 16, 0), _pack(2, 32, 5, 0), _pack(20, 37, 7, 1),
          _pack(21, 53, 0, 1), _pack(22, 69, 0, 1)]
    # request 1: A then B, a full query page, one reserved page
    r1 = [_pack(0, 0, 16, 0), _pack(1, 16, 16, 0), _pack(2, 32, 5, 0), _pack(3, 37, 16, 0),
          _pack(4, 53, 9, 0), _pack(30, 62, 16, 1), _pack(31, 78, 0, 1)]
    # request 2: B twice (one document at two offsets), no query segment
    r2 = [_pack(3, 0, 16, 0), _pack(4, 16, 9, 0), _pack(3, 25, 16, 0), _pack(4, 41, 9, 0),
          _pack(40, 50, 0, 1), _pack(41, 66, 0, 1)]
    tables = [r0, r1, r2]
    offs = np.cumsum([0] + [len(t) for t in tables]).astype(np.int32)
    return tables, np.array(sum(tables, []), np.uint64), offs


def test_unique_tiles_against_replayed_appends():
    tables, entries, offs = _tables()
    steps = 16
    got = bench.unique_tiles_per_call(entries, offs, steps)
    kp = np.zeros((64, 1, 16, 2))
    vp = np.zeros_like(kp)
    q = np.zeros((1, 2))
    kv = np.zeros((1, 2))
    ent = [list(t) for t in tables]
    want = []
    for _ in range(steps):
        pages = set()
        for r in range(len(ent)):
            _, ent[r] = oracle.paged_decode_step(kp, vp, ent[r], q, kv, kv, 1.0e4)
            pages |= {oracle.unpack_entry(e)[0] for e in ent[r] if oracle.unpack_entry(e)[2] > 0}
        want.append(len(pages))
    assert got == want
    # shared documents count once: A (3 pages) and B (2 pages) serve 5 placements;
    # then request 0's query page, request 1's full query page and the reserved
    # page its first token goes to, request 2's first reserved page
    assert got[0] == 5 + 1 + 2 + 1

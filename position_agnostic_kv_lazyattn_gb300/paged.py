"""Host-side plumbing around the C ABI: device buffers (torch) and block tables.

DevicePool allocates the caller-owned buffers a lazyattn pool needs (K/V pools,
position table, status word) with torch and creates the pool through the C ABI.
build_batch packs per-request page lists into the 64-bit entry format of
lazyattn_pack_entry and uploads the table. No attention arithmetic happens here.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence

import numpy as np
import torch

from . import lazyattn as L

PAGE_SIZE = L.PAGE_SIZE


def pack_entries(pages, starts, nvalid, writable) -> np.ndarray:
    """Vectorised lazyattn_pack_entry (same bit layout) for whole tables."""
    pages = np.asarray(pages, np.uint64) & np.uint64(0xFFFFFFFF)
    starts = (np.asarray(starts, np.uint64) & np.uint64((1 << 26) - 1)) << np.uint64(32)
    nvalid = (np.asarray(nvalid, np.uint64) & np.uint64(0x1F)) << np.uint64(58)
    writable = (np.asarray(writable, np.uint64) & np.uint64(1)) << np.uint64(63)
    return pages | starts | nvalid | writable


@dataclasses.dataclass
class Segment:
    """A run of tokens stored in consecutive entries: page ids, logical start,
    token count, whether decode may append into its pages, and (doc-local
    pools) the logical position of the run's local position 0, by default its
    start: a run stored by one lazyattn_store_doc call."""
    pages: Sequence[int]
    start: int
    n_tokens: int
    writable: bool = False
    delta: int = None


class DevicePool:
    def __init__(self, num_pages: int, n_q_heads: int, n_kv_heads: int, head_dim: int, dtype: str,
                 rope_theta: float, max_position: int, device="cuda", stream=None, rope_scaling=None,
                 key_storage: str = "position_free", rope_interleaved: bool = False,
                 position_encoding: str = "rope"):
        """rope_scaling: None (plain RoPE) or a dict with "kind" in {"linear", "ntk",
        "yarn", "llama3"}, "factor" and, for yarn / llama3, "original_max_position",
        "low", "high" (see lazyattn.h). key_storage: "position_free" (keys stored
        without RoPE) or "doc_local" (the paper's layout: keys stored rotated at
        document-local positions; bf16 only). rope_interleaved: q and k use
        interleaved RoPE pairs (2i, 2i+1) (bf16 only). position_encoding: "rope" or
        "alibi" (no rotation; score bias -slope_h (m - n); bf16 only)."""
        self.dtype = dtype
        self.tdtype = torch.float32 if dtype == "f32" else torch.bfloat16
        self.n_q_heads, self.n_kv_heads, self.head_dim = n_q_heads, n_kv_heads, head_dim
        self.num_pages = num_pages
        self.max_position = max_position
        shape = (num_pages, n_kv_heads, PAGE_SIZE, head_dim)
        self.k_pool = torch.zeros(shape, dtype=self.tdtype, device=device)
        self.v_pool = torch.zeros(shape, dtype=self.tdtype, device=device)
        self.rope_table = torch.empty(L.lazyattn_rope_table_bytes(head_dim, max_position) // 4,
                                      dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.desc = L.lazyattn_pool_desc(num_pages, PAGE_SIZE, n_q_heads, n_kv_heads, head_dim,
                                         L.LAZYATTN_F32 if dtype == "f32" else L.LAZYATTN_BF16,
                                         float(rope_theta), max_position, self.k_pool.data_ptr(),
                                         self.v_pool.data_ptr(), self.rope_table.data_ptr(),
                                         self.status.data_ptr())
        if rope_scaling:
            kinds = {"linear": L.LAZYATTN_ROPE_LINEAR, "ntk": L.LAZYATTN_ROPE_NTK, "yarn": L.LAZYATTN_ROPE_YARN,
                     "llama3": L.LAZYATTN_ROPE_LLAMA3}
            self.desc.rope_scaling = kinds[rope_scaling["kind"]]
            self.desc.rope_factor = float(rope_scaling["factor"])
            self.desc.rope_original_max_position = int(rope_scaling.get("original_max_position", 0))
            self.desc.rope_low = float(rope_scaling.get("low", 0.0))
            self.desc.rope_high = float(rope_scaling.get("high", 0.0))
        self.key_storage = key_storage
        self.desc.rope_interleaved = int(bool(rope_interleaved))
        self.desc.position_encoding = {"rope": L.LAZYATTN_POS_ROPE, "alibi": L.LAZYATTN_POS_ALIBI}[position_encoding]
        self.desc.key_storage = {"position_free": L.LAZYATTN_KEYS_POSITION_FREE,
                                 "doc_local": L.LAZYATTN_KEYS_DOC_LOCAL}[key_storage]
        self.handle = L.lazyattn_pool_create(self.desc, stream)

    def close(self):
        if self.handle:
            L.lazyattn_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def store_doc(self, k: torch.Tensor, v: torch.Tensor, stream=None) -> List[int]:
        assert k.is_contiguous() and v.is_contiguous() and k.dtype == self.tdtype
        return L.lazyattn_store_doc(self.handle, k, v, int(k.shape[0]), stream)

    def alloc_pages(self, n: int) -> List[int]:
        return L.lazyattn_alloc_pages(self.handle, n)

    def free_pages(self, pages: Sequence[int]):
        L.lazyattn_free_pages(self.handle, list(pages))

    def free_count(self) -> int:
        return L.lazyattn_pool_free_count(self.handle)

    def device_status(self, reset=True, stream=None) -> int:
        return L.lazyattn_get_device_status(self.handle, reset, stream)


def segment_entries(seg: Segment):
    n_pages = len(seg.pages)
    assert n_pages * PAGE_SIZE >= seg.n_tokens
    nvalid = [max(0, min(PAGE_SIZE, seg.n_tokens - j * PAGE_SIZE)) for j in range(n_pages)]
    starts = [seg.start + j * PAGE_SIZE for j in range(n_pages)]
    return list(seg.pages), starts, nvalid, [int(seg.writable)] * n_pages


class Batch:
    """Device-side block table (and prefill query layout) for a set of requests."""

    def __init__(self, requests: Sequence[Sequence[Segment]], q_lens: Sequence[int] = (),
                 q_starts: Sequence[int] = (), device="cuda", flags: int = 0):
        pg, st, nv, wr, dl, offs = [], [], [], [], [], [0]
        for segs in requests:
            for seg in segs:
                a, b, c, d = segment_entries(seg)
                pg += a; st += b; nv += c; wr += d
                dl += [seg.start if seg.delta is None else seg.delta] * len(a)
            offs.append(len(pg))
        self.entries_host = pack_entries(pg, st, nv, wr) if pg else np.zeros(0, np.uint64)
        self.offsets_host = np.array(offs, np.int32)
        self.num_requests = len(requests)
        self.max_entries = int(np.max(np.diff(self.offsets_host))) if len(requests) else 0
        self.entries = torch.from_numpy(self.entries_host.view(np.int64).copy()).to(device)
        if self.entries.numel() == 0:
            self.entries = torch.zeros(1, dtype=torch.int64, device=device)
        self.entry_offsets = torch.from_numpy(self.offsets_host).to(device)
        self.delta_host = np.array(dl if dl else [0], np.int32)
        self.entry_delta = torch.from_numpy(self.delta_host).to(device)
        q_lens = list(q_lens)
        if q_lens:
            qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
            self.q_offsets = torch.from_numpy(qo).to(device)
            self.q_start = torch.tensor(list(q_starts), dtype=torch.int32, device=device)
            self.total_q = int(qo[-1])
            self.max_q_len = int(max(q_lens))
        else:
            self.q_offsets = self.q_start = None
            self.total_q = self.max_q_len = 0
        self.flags = flags
        self.plan = None
        self.c = L.make_batch(self.num_requests, self.max_entries, self.entries, self.entry_offsets,
                              self.q_offsets, self.q_start, self.max_q_len, self.total_q, flags, self.entry_delta)

    def plan_decode(self, pool: "DevicePool", stream=None) -> dict:
        """Build the document-major decode plan of this batch's table
        (lazyattn_decode_plan_create from the host copy), upload it into a
        device buffer and make later decode calls through self.c use it.
        Returns the plan's statistics."""
        self.drop_plan()
        delta = self.delta_host if pool.key_storage == "doc_local" else None
        plan = L.lazyattn_decode_plan_create(pool.handle, self.entries_host, self.offsets_host, delta)
        nbytes = L.lazyattn_decode_plan_device_bytes(plan)
        self.plan_buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.entries.device)
        L.lazyattn_decode_plan_upload(plan, self.plan_buf, nbytes, stream)
        self.plan = plan
        self.c.decode_plan = plan
        return L.lazyattn_decode_plan_get_stats(plan)

    def drop_plan(self):
        if getattr(self, "plan", None):
            self.c.decode_plan = None
            L.lazyattn_decode_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.drop_plan()
        except Exception:
            pass

    def check(self, num_pages: int, max_position: int):
        """Host check of the table (lazyattn_check_batch_host): entries in range
        and no two tokens of a request at one logical position. Raises
        LazyAttnError naming the first failing request."""
        rc, bad = L.lazyattn_check_batch_host(self.entries_host, self.offsets_host, num_pages, max_position)
        if rc != 0:
            raise L.LazyAttnError(rc, f"block table of request {bad}")

    def with_entries(self, entries_host: np.ndarray, flags: int, device="cuda") -> "Batch":
        """Same requests and query layout, another entry array (e.g. materialised pages)."""
        b = Batch.__new__(Batch)
        b.__dict__.update(self.__dict__)
        b.plan = None                      # a plan belongs to one table
        b.entries_host = entries_host.astype(np.uint64)
        b.entries = torch.from_numpy(b.entries_host.view(np.int64).copy()).to(device)
        b.flags = flags
        b.c = L.make_batch(b.num_requests, b.max_entries, b.entries, b.entry_offsets, b.q_offsets, b.q_start,
                           b.max_q_len, b.total_q, flags, b.entry_delta)
        return b

"""ctypes binding of liblazyattn.so (include/lazyattn.h), same names as the C ABI.

Argument marshalling only: every function forwards plain pointers and sizes to
the C library, where all the work happens. Device buffers are torch tensors
(their data_ptr()), streams are torch.cuda streams (their cuda_stream handle).
If the compiled library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "liblazyattn.so")

PAGE_SIZE = 16
LAZYATTN_PAGE_SIZE = PAGE_SIZE
LAZYATTN_MAX_START = (1 << 26) - 1
LAZYATTN_F32 = 0
LAZYATTN_BF16 = 1
LAZYATTN_KEYS_PREROTATED = 1
LAZYATTN_OP_PREFILL = 0
LAZYATTN_OP_DECODE = 1
LAZYATTN_ROPE_DEFAULT = 0
LAZYATTN_ROPE_LINEAR = 1
LAZYATTN_ROPE_NTK = 2
LAZYATTN_ROPE_YARN = 3
LAZYATTN_ROPE_LLAMA3 = 4
LAZYATTN_KEYS_POSITION_FREE = 0
LAZYATTN_KEYS_DOC_LOCAL = 1
LAZYATTN_POS_ROPE = 0
LAZYATTN_POS_ALIBI = 1

STATUS = {
    0: "LAZYATTN_OK", -1: "LAZYATTN_EINVAL", -2: "LAZYATTN_ENOSPC", -3: "LAZYATTN_ERANGE",
    -4: "LAZYATTN_EDTYPE", -5: "LAZYATTN_ECUDA", -6: "LAZYATTN_EDEVICE", -7: "LAZYATTN_EWORKSPACE",
    -8: "LAZYATTN_ENODECODE",
}
(LAZYATTN_OK, LAZYATTN_EINVAL, LAZYATTN_ENOSPC, LAZYATTN_ERANGE, LAZYATTN_EDTYPE, LAZYATTN_ECUDA, LAZYATTN_EDEVICE,
 LAZYATTN_EWORKSPACE, LAZYATTN_ENODECODE) = (0, -1, -2, -3, -4, -5, -6, -7, -8)


class LazyAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({lib.lazyattn_status_string(code).decode()})")


class lazyattn_pool_desc(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("rope_theta", ctypes.c_double), ("max_position", ctypes.c_int32),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("rope_table", ctypes.c_void_p),
        ("status_word", ctypes.c_void_p),
        ("rope_scaling", ctypes.c_int32), ("rope_original_max_position", ctypes.c_int32),
        ("rope_factor", ctypes.c_double), ("rope_low", ctypes.c_double), ("rope_high", ctypes.c_double),
        ("key_storage", ctypes.c_int32), ("rope_interleaved", ctypes.c_int32),
        ("position_encoding", ctypes.c_int32),
    ]


class lazyattn_batch(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32), ("max_entries", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
        ("total_q", ctypes.c_int32), ("entries", ctypes.c_void_p), ("entry_offsets", ctypes.c_void_p),
        ("q_offsets", ctypes.c_void_p), ("q_start", ctypes.c_void_p), ("flags", ctypes.c_int32),
        ("entry_delta", ctypes.c_void_p), ("decode_plan", ctypes.c_void_p),
    ]


class lazyattn_decode_plan_stats(ctypes.Structure):
    _fields_ = [
        ("units", ctypes.c_int32), ("runs", ctypes.c_int32), ("partials", ctypes.c_int32),
        ("max_readers", ctypes.c_int32), ("logical_pages", ctypes.c_int64), ("pass_pages", ctypes.c_int64),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"liblazyattn.so is not built ({LIB_PATH}); run "
                          "python -m position_agnostic_kv_lazyattn_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
    P_i32 = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "lazyattn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "lazyattn_pack_entry": (u64, [i32, i32, i32, i32]),
        "lazyattn_rope_table_bytes": (sz, [i32, i32]),
        "lazyattn_pool_create": (ctypes.c_int, [ctypes.POINTER(lazyattn_pool_desc), vp, ctypes.POINTER(vp)]),
        "lazyattn_pool_destroy": (ctypes.c_int, [vp]),
        "lazyattn_pool_free_count": (ctypes.c_int, [vp, P_i32]),
        "lazyattn_alloc_pages": (ctypes.c_int, [vp, i32, P_i32]),
        "lazyattn_free_pages": (ctypes.c_int, [vp, P_i32, i32]),
        "lazyattn_store_doc": (ctypes.c_int, [vp, vp, vp, i32, vp, P_i32, i32, P_i32]),
        "lazyattn_workspace_size": (sz, [vp, i32, ctypes.POINTER(lazyattn_batch)]),
        "lazyattn_prefill": (ctypes.c_int, [vp, ctypes.POINTER(lazyattn_batch), vp, vp, vp, sz, vp]),
        "lazyattn_decode": (ctypes.c_int, [vp, ctypes.POINTER(lazyattn_batch), vp, vp, vp, vp, vp, sz, vp]),
        "lazyattn_materialize": (ctypes.c_int, [vp, ctypes.POINTER(lazyattn_batch), vp, vp]),
        "lazyattn_resolve": (ctypes.c_int, [vp, ctypes.POINTER(lazyattn_batch), vp, vp, i32, vp]),
        "lazyattn_get_device_status": (ctypes.c_int, [vp, P_i32, i32, vp]),
        "lazyattn_decode_noalloc": (ctypes.c_int, [vp, ctypes.POINTER(lazyattn_batch), vp, vp, vp, vp, vp]),
        "lazyattn_check_batch_host": (ctypes.c_int, [vp, vp, i32, i32, i32, P_i32]),
        "lazyattn_decode_plan_create": (ctypes.c_int, [vp, vp, vp, vp, i32, ctypes.POINTER(vp)]),
        "lazyattn_decode_plan_device_bytes": (sz, [vp]),
        "lazyattn_decode_plan_upload": (ctypes.c_int, [vp, vp, sz, vp]),
        "lazyattn_decode_plan_get_stats": (ctypes.c_int, [vp, ctypes.POINTER(lazyattn_decode_plan_stats)]),
        "lazyattn_decode_plan_destroy": (ctypes.c_int, [vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()
EXPORTS = [
    "lazyattn_status_string", "lazyattn_pack_entry", "lazyattn_rope_table_bytes", "lazyattn_pool_create",
    "lazyattn_pool_destroy", "lazyattn_pool_free_count", "lazyattn_alloc_pages", "lazyattn_free_pages",
    "lazyattn_store_doc", "lazyattn_workspace_size", "lazyattn_prefill", "lazyattn_decode",
    "lazyattn_materialize", "lazyattn_resolve", "lazyattn_get_device_status", "lazyattn_decode_noalloc",
    "lazyattn_check_batch_host", "lazyattn_decode_plan_create", "lazyattn_decode_plan_device_bytes",
    "lazyattn_decode_plan_upload", "lazyattn_decode_plan_get_stats", "lazyattn_decode_plan_destroy",
]
NOALLOC_SCRATCH_BYTES = 16 << 20
LAZYATTN_NOALLOC_SCRATCH_BYTES = NOALLOC_SCRATCH_BYTES


def _check(rc: int, where: str):
    if rc != 0:
        raise LazyAttnError(rc, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr() if hasattr(t, "data_ptr") else int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# --------------------------------------------------------------------- host helpers

def lazyattn_status_string(code: int) -> str:
    return lib.lazyattn_status_string(code).decode()


def lazyattn_pack_entry(page: int, start: int, nvalid: int, writable: int = 0) -> int:
    return int(lib.lazyattn_pack_entry(page, start, nvalid, writable))


def lazyattn_rope_table_bytes(head_dim: int, max_position: int) -> int:
    return int(lib.lazyattn_rope_table_bytes(head_dim, max_position))


# --------------------------------------------------------------------- pool

def lazyattn_pool_create(desc: lazyattn_pool_desc, stream=None) -> int:
    out = ctypes.c_void_p()
    _check(lib.lazyattn_pool_create(ctypes.byref(desc), _stream(stream), ctypes.byref(out)),
           "lazyattn_pool_create")
    return out.value


def lazyattn_pool_destroy(pool: int):
    _check(lib.lazyattn_pool_destroy(pool), "lazyattn_pool_destroy")


def lazyattn_pool_free_count(pool: int) -> int:
    n = ctypes.c_int32()
    _check(lib.lazyattn_pool_free_count(pool, ctypes.byref(n)), "lazyattn_pool_free_count")
    return n.value


def lazyattn_alloc_pages(pool: int, n: int):
    arr = (ctypes.c_int32 * max(n, 1))()
    _check(lib.lazyattn_alloc_pages(pool, n, arr), "lazyattn_alloc_pages")
    return list(arr[:n])


def lazyattn_free_pages(pool: int, pages: Sequence[int]):
    arr = (ctypes.c_int32 * max(len(pages), 1))(*pages)
    _check(lib.lazyattn_free_pages(pool, arr, len(pages)), "lazyattn_free_pages")


def lazyattn_store_doc(pool: int, k, v, n_tokens: int, stream=None):
    cap = (n_tokens + PAGE_SIZE - 1) // PAGE_SIZE
    arr = (ctypes.c_int32 * max(cap, 1))()
    n = ctypes.c_int32()
    _check(lib.lazyattn_store_doc(pool, _ptr(k), _ptr(v), n_tokens, _stream(stream), arr, cap, ctypes.byref(n)),
           "lazyattn_store_doc")
    return list(arr[: n.value])


# --------------------------------------------------------------------- batches

def make_batch(num_requests, max_entries, entries, entry_offsets, q_offsets=None, q_start=None,
               max_q_len=0, total_q=0, flags=0, entry_delta=None, decode_plan=None) -> lazyattn_batch:
    """Fill a lazyattn_batch from device tensors (int64 entries, int32 offsets and deltas)
    and a decode plan handle (or None)."""
    return lazyattn_batch(num_requests, max_entries, max_q_len, total_q, _ptr(entries), _ptr(entry_offsets),
                          _ptr(q_offsets), _ptr(q_start), flags, _ptr(entry_delta), decode_plan)


# --------------------------------------------------------------------- decode plans

def lazyattn_decode_plan_create(pool: int, entries, entry_offsets, entry_delta=None) -> int:
    """Plan handle for a batch from HOST copies of its table (numpy uint64 entries,
    int32 offsets [R+1], and int32 document offsets for doc-local pools)."""
    import numpy as np
    e = np.ascontiguousarray(entries, dtype=np.uint64)
    o = np.ascontiguousarray(entry_offsets, dtype=np.int32)
    d = None if entry_delta is None else np.ascontiguousarray(entry_delta, dtype=np.int32)
    out = ctypes.c_void_p()
    _check(lib.lazyattn_decode_plan_create(pool, e.ctypes.data if e.size else None, o.ctypes.data,
                                           None if d is None else d.ctypes.data, len(o) - 1, ctypes.byref(out)),
           "lazyattn_decode_plan_create")
    return out.value


def lazyattn_decode_plan_device_bytes(plan: int) -> int:
    return int(lib.lazyattn_decode_plan_device_bytes(plan))


def lazyattn_decode_plan_upload(plan: int, device_buffer, nbytes: int, stream=None):
    _check(lib.lazyattn_decode_plan_upload(plan, _ptr(device_buffer), nbytes, _stream(stream)),
           "lazyattn_decode_plan_upload")


def lazyattn_decode_plan_get_stats(plan: int) -> dict:
    st = lazyattn_decode_plan_stats()
    _check(lib.lazyattn_decode_plan_get_stats(plan, ctypes.byref(st)), "lazyattn_decode_plan_get_stats")
    return {name: getattr(st, name) for name, _ in lazyattn_decode_plan_stats._fields_}


def lazyattn_decode_plan_destroy(plan: int):
    _check(lib.lazyattn_decode_plan_destroy(plan), "lazyattn_decode_plan_destroy")


def lazyattn_check_batch_host(entries, entry_offsets, num_pages: int, max_position: int):
    """Host check of a block table (numpy uint64 entries, int32 offsets [R+1]).
    Returns (status, first failing request or -1); raises nothing."""
    import numpy as np
    e = np.ascontiguousarray(entries, dtype=np.uint64)
    o = np.ascontiguousarray(entry_offsets, dtype=np.int32)
    bad = ctypes.c_int32(-1)
    rc = lib.lazyattn_check_batch_host(e.ctypes.data if e.size else None, o.ctypes.data, len(o) - 1, num_pages,
                                       max_position, ctypes.byref(bad))
    return rc, bad.value


def lazyattn_workspace_size(pool: int, op: int, batch: lazyattn_batch) -> int:
    return int(lib.lazyattn_workspace_size(pool, op, ctypes.byref(batch)))


def lazyattn_prefill(pool: int, batch: lazyattn_batch, q, out, workspace=None, workspace_bytes: int = 0,
                     stream=None):
    _check(lib.lazyattn_prefill(pool, ctypes.byref(batch), _ptr(q), _ptr(out), _ptr(workspace),
                                workspace_bytes, _stream(stream)), "lazyattn_prefill")


def lazyattn_decode(pool: int, batch: lazyattn_batch, q, k_new, v_new, out, workspace, workspace_bytes: int,
                    stream=None):
    _check(lib.lazyattn_decode(pool, ctypes.byref(batch), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                               _ptr(workspace), workspace_bytes, _stream(stream)), "lazyattn_decode")


def lazyattn_decode_noalloc(pool: int, batch: lazyattn_batch, q, k_new, v_new, out, stream=None):
    """lazyattn_decode without a workspace, for callers that cannot allocate
    device memory: uses the library's built-in scratch array instead."""
    _check(lib.lazyattn_decode_noalloc(pool, ctypes.byref(batch), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                       _stream(stream)), "lazyattn_decode_noalloc")


def lazyattn_materialize(pool: int, batch: lazyattn_batch, dst_entries, stream=None):
    _check(lib.lazyattn_materialize(pool, ctypes.byref(batch), _ptr(dst_entries), _stream(stream)),
           "lazyattn_materialize")


def lazyattn_resolve(pool: int, batch: lazyattn_batch, out_offsets, out_triples, out_cap: int, stream=None):
    _check(lib.lazyattn_resolve(pool, ctypes.byref(batch), _ptr(out_offsets), _ptr(out_triples), out_cap,
                                _stream(stream)), "lazyattn_resolve")


def lazyattn_get_device_status(pool: int, reset: bool = True, stream=None) -> int:
    s = ctypes.c_int32()
    _check(lib.lazyattn_get_device_status(pool, ctypes.byref(s), 1 if reset else 0, _stream(stream)),
           "lazyattn_get_device_status")
    return s.value

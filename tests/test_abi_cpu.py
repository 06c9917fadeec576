"""The C-ABI library loads, exports what include/lazyattn.h declares, and its
host-only logic (entry packing, argument validation) behaves - no GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from position_agnostic_kv_lazyattn_gb300 import lazyattn
    return lazyattn


def _declared():
    txt = open(os.path.join(ROOT, "include", "lazyattn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(lazyattn_[a-z_0-9]+)\s*\(", txt)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 15
    cdll = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(cdll, n), n
    assert set(names) == set(L.EXPORTS)


def test_pack_entry_matches_oracle_and_numpy(L):
    from position_agnostic_kv_lazyattn_gb300.paged import pack_entries
    rng = np.random.default_rng(0)
    pages = rng.integers(0, 2**31 - 1, 200)
    starts = rng.integers(0, 2**26 - 1, 200)
    nvalid = rng.integers(0, 17, 200)
    wr = rng.integers(0, 2, 200)
    vec = pack_entries(pages, starts, nvalid, wr)
    for i in range(200):
        e = L.lazyattn_pack_entry(int(pages[i]), int(starts[i]), int(nvalid[i]), int(wr[i]))
        assert e == int(vec[i])
        assert oracle.unpack_entry(e) == (pages[i], starts[i], nvalid[i], wr[i])


def test_status_strings(L):
    for code in range(0, -9, -1):
        assert L.lazyattn_status_string(code) != "unknown status"
    assert L.lazyattn_status_string(-99) == "unknown status"


def test_binding_constants_match_the_header(L):
    """Every LAZYATTN_* integer constant of the header (#define or enum value)
    has the same value in the Python binding."""
    txt = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "lazyattn.h")).read(), flags=re.S)
    found = {}
    for name, expr in re.findall(r"#define\s+(LAZYATTN_[A-Z0-9_]+)\s+([-()\d\s<u]+)\n", txt):
        found[name] = eval(expr.replace("u", ""), {})      # integer literals, shifts, minus only
    found.update((n, int(v)) for n, v in re.findall(r"\b(LAZYATTN_[A-Z0-9_]+)\s*=\s*(-?\d+)", txt))
    assert len(found) >= 25
    for name, value in found.items():
        assert hasattr(L, name), name
        assert getattr(L, name) == value, name


def test_rope_table_bytes(L):
    assert L.lazyattn_rope_table_bytes(128, 1000) == 2 * 1000 * 64 * 8   # (cos, sin) rows + paired rows
    assert L.lazyattn_rope_table_bytes(0, 10) == 0


def _desc(L, **kw):
    d = dict(num_pages=8, page_size=16, n_q_heads=4, n_kv_heads=2, head_dim=64, dtype=L.LAZYATTN_F32,
             rope_theta=1e4, max_position=64, k_pool=256, v_pool=512, rope_table=768, status_word=1024)
    d.update(kw)
    return L.lazyattn_pool_desc(**d)


@pytest.mark.parametrize("bad", [
    dict(page_size=8), dict(num_pages=0), dict(n_q_heads=3), dict(head_dim=96), dict(rope_theta=0.0),
    dict(max_position=0), dict(k_pool=0), dict(rope_table=0), dict(status_word=0), dict(k_pool=264),
    dict(dtype=1, head_dim=64), dict(dtype=1, head_dim=128, n_q_heads=32, n_kv_heads=2),
])
def test_pool_create_rejects_bad_desc_before_any_cuda_call(L, bad):
    out = ctypes.c_void_p()
    rc = L.lib.lazyattn_pool_create(ctypes.byref(_desc(L, **bad)), None, ctypes.byref(out))
    assert rc == -1 and not out.value


def test_pool_create_rejects_unknown_dtype(L):
    out = ctypes.c_void_p()
    rc = L.lib.lazyattn_pool_create(ctypes.byref(_desc(L, dtype=7)), None, ctypes.byref(out))
    assert rc == -4


def test_null_handles_are_rejected(L):
    b = L.lazyattn_batch()
    assert L.lib.lazyattn_workspace_size(None, 1, ctypes.byref(b)) == 0
    assert L.lib.lazyattn_prefill(None, ctypes.byref(b), None, None, None, 0, None) == -1
    assert L.lib.lazyattn_decode(None, ctypes.byref(b), None, None, None, None, None, 0, None) == -1
    assert L.lib.lazyattn_pool_destroy(None) == -1
    n = ctypes.c_int32()
    assert L.lib.lazyattn_pool_free_count(None, ctypes.byref(n)) == -1

"""The pool's page allocator (host metadata of lazyattn_pool_create; creating a
pool needs a CUDA device, so these run with the GPU tests). Checked against the
rules include/lazyattn.h states: lazyattn_alloc_pages hands out the lowest free
ids first and takes nothing when it cannot take all (ENOSPC); lazyattn_free_pages
frees nothing when one id is out of range (ERANGE), already free or repeated
(EINVAL); lazyattn_store_doc takes ceil(n / 16) pages or, on ENOSPC, none.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


def _pool(L, n_pages):
    return L.DevicePool(n_pages, 32, 8, 128, "bf16", 5.0e5, 1024)


def _code(fn):
    import position_agnostic_kv_lazyattn_gb300 as L
    try:
        fn()
    except L.LazyAttnError as e:
        return e.code
    return 0


def test_documented_cases(L):
    pool = _pool(L, 8)
    assert pool.free_count() == 8
    assert pool.alloc_pages(3) == [0, 1, 2]
    assert _code(lambda: pool.alloc_pages(6)) == L.LAZYATTN_ENOSPC and pool.free_count() == 5
    pool.free_pages([1])
    assert _code(lambda: pool.free_pages([1])) == L.LAZYATTN_EINVAL          # already free
    assert _code(lambda: pool.free_pages([0, 8])) == L.LAZYATTN_ERANGE       # 8 is outside: 0 stays taken
    assert _code(lambda: pool.free_pages([2, 2])) == L.LAZYATTN_EINVAL       # repeated: 2 stays taken
    assert pool.free_count() == 6
    assert pool.alloc_pages(2) == [1, 3]
    # a document of 81 tokens takes 6 pages; with 4 free it takes none
    k = torch.zeros((81, 8, 128), dtype=torch.bfloat16, device="cuda")
    assert _code(lambda: pool.store_doc(k, k)) == L.LAZYATTN_ENOSPC and pool.free_count() == 4
    pool.free_pages([0, 2])
    assert pool.store_doc(k, k) == [0, 2, 4, 5, 6, 7]
    assert pool.free_count() == 0
    torch.cuda.synchronize()
    assert pool.device_status() == 0


def test_random_sequence_matches_the_rules(L):
    n_pages = 300
    pool = _pool(L, n_pages)
    rng = np.random.default_rng(51)
    free = set(range(n_pages))
    taken = []
    for _ in range(2000):
        if rng.random() < 0.5:
            n = int(rng.integers(0, 40))
            if n > len(free):
                assert _code(lambda: pool.alloc_pages(n)) == L.LAZYATTN_ENOSPC
            else:
                want = sorted(free)[:n]
                assert pool.alloc_pages(n) == want
                free -= set(want)
                taken += want
        else:
            n = int(rng.integers(0, min(len(taken), 30) + 1))
            idx = rng.choice(len(taken), size=n, replace=False) if n else []
            pages = [taken[i] for i in idx]
            bad = rng.random()
            if bad < 0.1 and pages:
                pages.append(pages[0])                              # repeated id
                assert _code(lambda: pool.free_pages(pages)) == L.LAZYATTN_EINVAL
            elif bad < 0.2 and free:
                pages.append(min(free))                             # an id that is free
                assert _code(lambda: pool.free_pages(pages)) == L.LAZYATTN_EINVAL
            elif bad < 0.25:
                pages.append(n_pages + int(rng.integers(0, 5)))     # out of range
                assert _code(lambda: pool.free_pages(pages)) == L.LAZYATTN_ERANGE
            else:
                pool.free_pages(pages)
                free |= set(pages)
                taken = [p for p in taken if p not in set(pages)]
        assert pool.free_count() == len(free)

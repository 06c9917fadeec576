"""The pool's position table, both layouts, against cos/sin computed here in fp64.

lazyattn_pool_create fills the caller's table with (cos, sin)(p * theta_i) for
every position p < max_position and frequency i < D/2 (LazyAttention §3.2
"Prefilling": the kernels table-drive cos/sin), then the same values again with
the cosines and sines of neighbouring frequencies paired, (cos f, cos f+1,
sin f, sin f+1) for even f: the rows the bf16 kernels stage per page. Checked:
* the (cos, sin) rows against fp64 cos/sin of p * theta_i, theta_i from the
  oracle's frequencies of the pool's RoPE variant (plain and Llama 3.1), within
  fp32 rounding;
* the paired rows equal to the (cos, sin) rows, element for element;
* a max_position that is not a multiple of 16 (the kernels' 16-row view stops
  before the table's end; the table itself does not).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

D = 128
THETA = 5.0e5


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import position_agnostic_kv_lazyattn_gb300 as L
    return L


@pytest.mark.parametrize("variant", ["default", "llama3"])
def test_position_table_layouts(L, variant):
    from position_agnostic_kv_lazyattn_gb300 import DevicePool
    max_pos = 3001
    assert max_pos % 16 != 0
    if variant == "default":
        scaling, spec = None, THETA
    else:
        scaling = dict(kind="llama3", factor=8.0, original_max_position=8192, low=1.0, high=4.0)
        spec = oracle.RopeSpec(THETA, "llama3", 8.0, 8192, 1.0, 4.0)
    pool = DevicePool(4, 32, 8, D, "bf16", THETA, max_pos, rope_scaling=scaling)
    tab = pool.rope_table.cpu().numpy()
    assert tab.size == 2 * max_pos * D
    cs = tab[: max_pos * D].reshape(max_pos, D // 2, 2)
    paired = tab[max_pos * D:].reshape(max_pos, D // 4, 4)

    inv = oracle.rope_inv_freq(D, spec)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    err_c = np.abs(cs[:, :, 0] - np.cos(ang)).max()
    err_s = np.abs(cs[:, :, 1] - np.sin(ang)).max()
    print("%s table max-abs error cos %.2e sin %.2e" % (variant, err_c, err_s))
    assert err_c <= 1e-6 and err_s <= 1e-6

    # paired rows: (cos f, cos f+1, sin f, sin f+1), exactly the values above
    assert np.array_equal(paired[:, :, 0], cs[:, 0::2, 0])
    assert np.array_equal(paired[:, :, 1], cs[:, 1::2, 0])
    assert np.array_equal(paired[:, :, 2], cs[:, 0::2, 1])
    assert np.array_equal(paired[:, :, 3], cs[:, 1::2, 1])
    assert pool.device_status() == 0

"""The allocation-free LayerNorm backward (mgb_layernorm_bwd_noalloc) against
the workspace version (mgb_layernorm_bwd), through the C ABI.

This entry point exists for callers that cannot hand the library a scratch
buffer (all device memory reserved up front, or a host framework that owns the
allocator); its dgamma/dbeta partial sums live in a fixed array inside the
library instead. The test checks two calls in a row with different inputs, so
a result that depended on what the previous call left in that shared array
would show up. The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import round_to_bf16
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _built_library(mgb_lib):
    """Builds and loads libmgb.so first when this file runs on its own."""
    return mgb_lib


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dtype)


def _case(rng, rows, cols, dtype):
    td = torch.bfloat16 if dtype == mgb.MGB_BF16 else torch.float32
    rnd = round_to_bf16 if dtype == mgb.MGB_BF16 else (lambda a: a)
    x = _dev(rnd(rng.standard_normal((rows, cols)) * 2.0 + 0.5), td)
    dy = _dev(rnd(rng.standard_normal((rows, cols))), td)
    dres = _dev(rnd(rng.standard_normal((rows, cols))), td)
    gamma = _dev(rnd(1.0 + 0.2 * rng.standard_normal(cols)), td)
    y = torch.empty_like(x)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    mgb.mgb_layernorm_fwd(rows, cols, dtype, 1e-5, x, gamma, None, y, mean, rstd)
    return x, dy, dres, gamma, mean, rstd


def _run_both(rows, cols, dtype, x, dy, dres, gamma, mean, rstd):
    outs = []
    for noalloc in (False, True):
        dx = torch.full_like(x, float("nan"))
        dg = torch.full((cols,), float("nan"), device="cuda", dtype=x.dtype)
        db = torch.full((cols,), float("nan"), device="cuda", dtype=x.dtype)
        if noalloc:
            mgb.mgb_layernorm_bwd_noalloc(rows, cols, dtype, x, mean, rstd, gamma, dy, dres, dx, dg, db)
        else:
            ws = torch.empty(mgb.mgb_layernorm_bwd_ws_bytes(rows, cols), dtype=torch.uint8,
                             device="cuda")
            mgb.mgb_layernorm_bwd(rows, cols, dtype, x, mean, rstd, gamma, dy, dres, dx, dg, db, ws)
        outs.append((to_np(dx), to_np(dg), to_np(db)))
    assert mgb.mgb_device_status() == mgb.MGB_OK
    return outs


@pytest.mark.parametrize("dtype,tol", [(mgb.MGB_BF16, 1e-2), (mgb.MGB_F32, 1e-5)])
def test_noalloc_matches_workspace_version_twice(dtype, tol):
    rng = np.random.default_rng(123)
    # first call: large rows/cols; second: different shape and values, fewer
    # columns, so stale partial sums from the first call would be picked up
    for rows, cols in ((4096, 4096), (300, 1024)):
        args = _case(rng, rows, cols, dtype)
        (dx_w, dg_w, db_w), (dx_n, dg_n, db_n) = _run_both(rows, cols, dtype, *args)
        assert np.isfinite(dx_n).all() and np.isfinite(dg_n).all() and np.isfinite(db_n).all()
        assert rel_l2(dx_n, dx_w) <= tol
        assert rel_l2(dg_n, dg_w) <= tol
        assert rel_l2(db_n, db_w) <= tol


def test_noalloc_rejects_columns_beyond_its_array():
    rows, cols = 8, 16392
    x = torch.zeros((rows, cols), device="cuda", dtype=torch.bfloat16)
    g = torch.ones(cols, device="cuda", dtype=torch.bfloat16)
    st = torch.zeros(rows, device="cuda")
    lib = mgb.load()
    s = lib.mgb_layernorm_bwd_noalloc(rows, cols, mgb.MGB_BF16, x.data_ptr(), st.data_ptr(),
                                      st.data_ptr(), g.data_ptr(), x.data_ptr(), None, x.data_ptr(),
                                      g.data_ptr(), g.data_ptr(), None)
    assert s == mgb.MGB_ERR_UNSUPPORTED

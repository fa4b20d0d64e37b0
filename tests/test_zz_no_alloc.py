"""The allocation-free LayerNorm backward (mgb_layernorm_bwd_noalloc) through
the C ABI, against the float64 oracle and against the workspace version
(mgb_layernorm_bwd).

This entry point is for callers that cannot hand the library a scratch
buffer: a serving engine that reserved all device memory up front and may not
allocate while a request runs, or a plugin inside a framework that owns the
allocator. Its dgamma/dbeta partial sums live in one fixed array inside the
library, shared by every call on the device.

Each case runs two calls in a row with different shapes and values, so a
result that depended on what the previous call left in the shared array, or
on a partial-row count sized for another width, would show up. The file's
name makes pytest collect it after every other test file, so that a run that
stops at the first failure has run all the others first; it passes on its own
in a fresh process as well (the fixture builds and loads the library).
"""
import numpy as np
import pytest
import torch

import oracle
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
    """Inputs on both sides: x, dy, dres, gamma as exact values of the dtype;
    mean/rstd from the library's forward (the backward's own inputs)."""
    td = torch.bfloat16 if dtype == mgb.MGB_BF16 else torch.float32
    rnd = round_to_bf16 if dtype == mgb.MGB_BF16 else (lambda a: a)
    n = max(rows, 1)  # rows = 0 still passes real (unread) device pointers
    h = {"x": rnd(rng.standard_normal((n, cols)) * 2.0 + 0.5),
         "dy": rnd(rng.standard_normal((n, cols))),
         "dres": rnd(rng.standard_normal((n, cols))),
         "gamma": rnd(1.0 + 0.2 * rng.standard_normal(cols))}
    d = {k: _dev(v, td) for k, v in h.items()}
    d["mean"] = torch.empty(max(rows, 1), device="cuda")
    d["rstd"] = torch.empty(max(rows, 1), device="cuda")
    if rows > 0:
        y = torch.empty_like(d["x"])
        mgb.mgb_layernorm_fwd(rows, cols, dtype, 1e-5, d["x"], d["gamma"], None, y, d["mean"],
                              d["rstd"])
    return h, d


def _call(rows, cols, dtype, d, noalloc, with_dres=True, want=(True, True)):
    x = d["x"]
    dx = torch.full_like(x, float("nan"))
    dg = torch.full((cols,), float("nan"), device="cuda", dtype=x.dtype) if want[0] else None
    db = torch.full((cols,), float("nan"), device="cuda", dtype=x.dtype) if want[1] else None
    dres = d["dres"] if with_dres else None
    if noalloc:
        mgb.mgb_layernorm_bwd_noalloc(rows, cols, dtype, x, d["mean"], d["rstd"], d["gamma"], d["dy"],
                                      dres, dx, dg, db)
    else:
        ws = torch.empty(max(mgb.mgb_layernorm_bwd_ws_bytes(rows, cols), 16), dtype=torch.uint8,
                         device="cuda")
        mgb.mgb_layernorm_bwd(rows, cols, dtype, x, d["mean"], d["rstd"], d["gamma"], d["dy"], dres,
                              dx, dg, db, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    return (to_np(dx), None if dg is None else to_np(dg), None if db is None else to_np(db))


def _oracle(h, d, with_dres=True):
    """The oracle's backward on the same x/dy/gamma, with the library's own
    mean/rstd (the statistics are the forward's outputs, checked elsewhere)."""
    rows = h["x"].shape[0]
    mean = to_np(d["mean"])[:rows]
    rstd = to_np(d["rstd"])[:rows]
    dx, dg, db = oracle.ln_bwd(h["dy"], h["x"], mean, rstd, h["gamma"])
    if with_dres:
        dx = dx + h["dres"]
    return dx, dg, db


@pytest.mark.parametrize("dtype,tol", [(mgb.MGB_BF16, 1e-2), (mgb.MGB_F32, 1e-5)])
def test_noalloc_matches_oracle_and_workspace_version_twice(dtype, tol):
    rng = np.random.default_rng(123)
    # first call: 4096 x 4096 (256 partial rows of the array); second: fewer,
    # wider rows (16384 columns: 64 partial rows) with other values
    for rows, cols in ((4096, 4096), (300, 16384)):
        h, d = _case(rng, rows, cols, dtype)
        dx_n, dg_n, db_n = _call(rows, cols, dtype, d, noalloc=True)
        dx_w, dg_w, db_w = _call(rows, cols, dtype, d, noalloc=False)
        rdx, rdg, rdb = _oracle(h, d)
        for got in (dx_n, dg_n, db_n):
            assert np.isfinite(got).all()
        assert rel_l2(dx_n, rdx) <= tol
        assert rel_l2(dg_n, rdg) <= tol
        assert rel_l2(db_n, rdb) <= tol
        assert rel_l2(dx_n, dx_w) <= tol
        assert rel_l2(dg_n, dg_w) <= tol
        assert rel_l2(db_n, db_w) <= tol


@pytest.mark.parametrize("rows", [17, 1])
def test_noalloc_fewer_rows_than_blocks(rows):
    """Fewer rows than row blocks: one partial row per row."""
    rng = np.random.default_rng(rows)
    h, d = _case(rng, rows, 1024, mgb.MGB_F32)
    dx, dg, db = _call(rows, 1024, mgb.MGB_F32, d, noalloc=True)
    rdx, rdg, rdb = _oracle(h, d)
    assert rel_l2(dx, rdx) <= 1e-5 and rel_l2(dg, rdg) <= 1e-5 and rel_l2(db, rdb) <= 1e-5


def test_noalloc_zero_rows_gives_zero_sums():
    """rows = 0 after a call that filled the array: dgamma and dbeta are zero
    (the one partial row reduced is cleared first), nothing else is touched."""
    rng = np.random.default_rng(7)
    _, d = _case(rng, 512, 2048, mgb.MGB_BF16)
    _call(512, 2048, mgb.MGB_BF16, d, noalloc=True)
    _, d0 = _case(rng, 0, 2048, mgb.MGB_BF16)
    _, dg, db = _call(0, 2048, mgb.MGB_BF16, d0, noalloc=True)
    assert (dg == 0).all() and (db == 0).all()


@pytest.mark.parametrize("want", [(True, False), (False, True), (False, False)])
def test_noalloc_without_residual_and_one_sum(want):
    """No residual input, and dgamma or dbeta alone (or neither)."""
    rng = np.random.default_rng(11)
    rows, cols = 700, 3072
    h, d = _case(rng, rows, cols, mgb.MGB_F32)
    dx, dg, db = _call(rows, cols, mgb.MGB_F32, d, noalloc=True, with_dres=False, want=want)
    rdx, rdg, rdb = _oracle(h, d, with_dres=False)
    assert rel_l2(dx, rdx) <= 1e-5
    if want[0]:
        assert rel_l2(dg, rdg) <= 1e-5
    if want[1]:
        assert rel_l2(db, rdb) <= 1e-5


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

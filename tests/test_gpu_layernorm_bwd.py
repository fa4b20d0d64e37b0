"""GPU parity of the LayerNorm backward building block (mgb_layernorm_bwd)
against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import round_to_bf16
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(77)


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dtype)


@pytest.mark.parametrize("dtype,rows,cols,affine,resid", [
    ("bf16", 300, 1024, True, True), ("bf16", 2048, 4096, True, False), ("bf16", 5, 256, False, True),
    ("f32", 130, 256, True, True), ("f32", 64, 64, False, False),
    # rows wider than 1024 vectors: two or four vectors per thread, up to 1024
    # threads a block (the widest rows the layer accepts)
    ("bf16", 40, 12288, True, True), ("bf16", 33, 16384, True, False),
    ("f32", 20, 8192, True, True), ("f32", 17, 16384, True, True),
    # many rows per CTA: the bf16 kernel's shared-memory ring refilled many times
    ("bf16", 8192, 4096, True, True), ("bf16", 3000, 2048, True, False),
    # more than 64 rows per block: row statistics read one row ahead instead
    # of staged up front
    ("bf16", 70000, 256, True, True),
    # widths whose float4 count does not split evenly over a cluster of four
    # (the cluster-combined partial sums) and whose vectors do not fill whole warps
    ("bf16", 300, 1000, True, True), ("f32", 260, 100, True, False)])
@pytest.mark.parametrize("kernel", ["async", "tma", "block"])
def test_layernorm_bwd(mgb_lib, monkeypatch, kernel, dtype, rows, cols, affine, resid):
    """Rows of up to 1024 vectors go through the kernel fed by per-thread
    asynchronous copies (the default), the bf16 kernel fed by bulk copies
    (MGB_LN_KERNEL=tma, rows up to 16384 wide) or the register-prefetch block
    kernel (MGB_LN_KERNEL=block); wider rows always take the block kernel."""
    monkeypatch.setenv("MGB_LN_KERNEL", kernel)
    x = RNG.standard_normal((rows, cols)) * 1.5 + 0.3
    dy = RNG.standard_normal((rows, cols))
    dres = RNG.standard_normal((rows, cols)) if resid else None
    g = 1 + 0.2 * RNG.standard_normal(cols) if affine else None
    if dtype == "bf16":
        x, dy = round_to_bf16(x), round_to_bf16(dy)
        dres = round_to_bf16(dres) if resid else None
        g = round_to_bf16(g) if affine else None
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    mdt = mgb.MGB_BF16 if dtype == "bf16" else mgb.MGB_F32
    tx = _dev(x, td)
    y = torch.empty_like(tx)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    tg = _dev(g, td) if affine else None
    mgb.mgb_layernorm_fwd(rows, cols, mdt, 1e-5, tx, tg, None, y, mean, rstd)
    dx = torch.empty_like(tx)
    dgam = torch.empty(cols, device="cuda", dtype=td) if affine else None
    dbet = torch.empty(cols, device="cuda", dtype=td) if affine else None
    ws = torch.empty(max(mgb.mgb_layernorm_bwd_ws_bytes(rows, cols), 16), dtype=torch.uint8,
                     device="cuda")
    mgb.mgb_layernorm_bwd(rows, cols, mdt, tx, mean, rstd, tg, _dev(dy, td),
                          _dev(dres, td) if resid else None, dx, dgam, dbet, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    _, rm, rr = oracle.ln_fwd(x, g, None, 1e-5)
    rdx, rdg, rdb = oracle.ln_bwd(dy, x, rm, rr, g)
    if resid:
        rdx = rdx + dres
    tol = 1e-2 if dtype == "bf16" else 1e-5
    assert rel_l2(to_np(dx), rdx) < tol
    if affine:
        assert rel_l2(to_np(dgam), rdg) < tol
        assert rel_l2(to_np(dbet), rdb) < tol

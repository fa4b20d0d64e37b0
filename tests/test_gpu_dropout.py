"""GPU parity of dropout ("02 - How a whole Transformer block is split",
section 5) through the C ABI: the device generator's byte stream bit for bit
against the oracle's Philox4x32-10 stream, the elementwise dropout mask
exactly, and the layer with hidden dropout (fused into the projection and
fc2 residual epilogues, replayed in the backward) against the float64 oracle
with the masks the oracle draws from the same tracker."""
import numpy as np
import pytest
import torch

import oracle
from oracle import dropout as od
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import LayerShape, layer_inputs
from megatron_transformer_layer_fwd_gb300.runner import LayerRunner, WEIGHT_KEYS, to_device
from tests.util import TOL, rel_l2, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,offset,n", [(0, 0, 4096), (1234, 7, 1000), (2718, 16 * 1000 + 3, 99999),
                                           (0xFEDCBA9876543210, (1 << 40) + 5, 4096), (5, 0, 1)])
def test_philox_bytes_bit_exact(mgb_lib, seed, offset, n):
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    mgb.mgb_philox_bytes(seed, offset, n, out)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    assert np.array_equal(out.cpu().numpy(), od.uniform_bytes(seed, offset, n))


@pytest.mark.parametrize("pad", [0, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,cols,p", [(64, 256, 0.1), (37, 100, 0.5), (3, 7, 0.9), (8, 32, 0.0)])
def test_dropout_mask_exact(mgb_lib, dtype, rows, cols, p, pad):
    """16-byte-vector rows (cols % 16 == 0, aligned strides) and the general
    element path (ragged cols or an odd output stride)."""
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    dt = mgb.MGB_BF16 if dtype == "bf16" else mgb.MGB_F32
    p32 = float(np.float32(p))
    rng = mgb.RngState(seed=77, offset=16 * 9)
    x = (torch.rand((rows, cols), device="cuda") + 0.5).to(td)  # no zeros
    y = torch.full((rows, cols + pad), float("nan"), device="cuda", dtype=td)
    mgb.mgb_dropout(rows, cols, dt, p32, rng, x, cols, y, cols + pad)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    keep = od.dropout_keep(77, 16 * 9, (rows, cols), p32)
    got = y[:, :cols].float().cpu().numpy()
    assert np.array_equal(got != 0, keep)
    scale = np.float32(256.0) / np.float32(od.keep_threshold(p32))
    want = (x.float().cpu().numpy() * scale).astype(np.float32)
    if dtype == "bf16":
        want = torch.from_numpy(want).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got[keep], want[keep])
    assert torch.isnan(y[:, cols:]).all()  # nothing written outside the site


SHAPES = {
    "pre_gelu": LayerShape(2, 100, 256, 4, 4, 64, 520),
    "post_swiglu_gqa_causal": LayerShape(2, 130, 256, 4, 2, 128, 384, norm_pos="post", act="swiglu",
                                         causal=True),
}


def _dropout_runner(shape, arr, p, seed, p_attn=0.0):
    r = LayerRunner(shape, arr)
    r.desc.hidden_dropout = p
    r.desc.attn_dropout = p_attn
    mgb.mgb_block_dropout_plan(r.desc, mgb.rng_tracker(seed))
    saved, _, bwd = mgb.mgb_block_sizes(r.desc)
    r.saved = torch.empty(max(saved, 16), dtype=torch.uint8, device="cuda")
    r.ws = torch.empty(max(bwd, 16), dtype=torch.uint8, device="cuda")
    return r


@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_hidden_dropout_parity(mgb_lib, name):
    shape = SHAPES[name]
    p = float(np.float32(0.2))
    arr = layer_inputs(shape, seed=31, random_affine=True, random_dy=True)
    r = _dropout_runner(shape, arr, p, seed=4242)
    y = r.fwd().clone()
    dy = to_device(arr["dy"], r.dtype)
    dx, g = r.bwd(dy)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    drop = od.layer_dropout(shape, od.model_parallel_seed(4242), 0.0, p)
    w = {k: arr[k] for k in WEIGHT_KEYS}
    ry, cache = oracle.block_fwd(shape, w, arr["x"], drop=drop)
    rdx, rg = oracle.block_bwd(shape, w, cache, arr["dy"])
    tol_o, tol_g = TOL["bf16"]
    errs = {"y": rel_l2(to_np(y), ry), "dx": rel_l2(to_np(dx), rdx)}
    for k in WEIGHT_KEYS:
        if rg[k] is not None:
            errs[k] = rel_l2(to_np(g[k]), rg[k])
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] < tol_o and all(v < tol_g for k, v in errs.items() if k != "y"), errs
    # the masks matter: the oracle without them is much further off
    ry0, _ = oracle.block_fwd(shape, w, arr["x"])
    assert rel_l2(to_np(y), ry0) > max(2 * tol_o, 5 * errs["y"])


def test_layer_dropout_replay_and_seeds(mgb_lib):
    """The same plan replays bit for bit; another seed gives another output;
    the backward reproduces the forward's masks (checked by parity above)."""
    shape = SHAPES["pre_gelu"]
    arr = layer_inputs(shape, seed=5, random_affine=True)
    r = _dropout_runner(shape, arr, 0.3, seed=1)
    y1 = r.fwd().clone()
    y2 = r.fwd().clone()
    assert torch.equal(y1, y2)
    mgb.mgb_block_dropout_plan(r.desc, mgb.rng_tracker(2))
    y3 = r.fwd().clone()
    assert not torch.equal(y1, y3)
    assert mgb.mgb_device_status() == mgb.MGB_OK


ATTN_SHAPES = {
    "pre_gelu_d64": LayerShape(2, 100, 256, 4, 4, 64, 520),
    "post_swiglu_gqa_causal_d128": LayerShape(2, 130, 256, 4, 2, 128, 384, norm_pos="post",
                                              act="swiglu", causal=True),
    "pre_gqa_causal_multitile": LayerShape(1, 300, 256, 4, 1, 64, 256, causal=True),
}


@pytest.mark.parametrize("name", list(ATTN_SHAPES))
@pytest.mark.parametrize("p_attn,p_hidden", [(0.25, 0.0), (0.1, 0.15)])
def test_layer_attention_dropout_parity(mgb_lib, name, p_attn, p_hidden):
    """Dropout inside the attention kernels (the model-parallel stream): the
    forward draws and stores the keep bits, both backward kernels read them."""
    shape = ATTN_SHAPES[name]
    pa, ph = float(np.float32(p_attn)), float(np.float32(p_hidden))
    arr = layer_inputs(shape, seed=41, random_affine=True, random_dy=True)
    r = _dropout_runner(shape, arr, ph, seed=777, p_attn=pa)
    y = r.fwd().clone()
    dy = to_device(arr["dy"], r.dtype)
    dx, g = r.bwd(dy)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    drop = od.layer_dropout(shape, od.model_parallel_seed(777), pa, ph)
    w = {k: arr[k] for k in WEIGHT_KEYS}
    ry, cache = oracle.block_fwd(shape, w, arr["x"], drop=drop)
    rdx, rg = oracle.block_bwd(shape, w, cache, arr["dy"])
    tol_o, tol_g = TOL["bf16"]
    errs = {"y": rel_l2(to_np(y), ry), "dx": rel_l2(to_np(dx), rdx)}
    for k in WEIGHT_KEYS:
        if rg[k] is not None:
            errs[k] = rel_l2(to_np(g[k]), rg[k])
    print(name, pa, ph, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["y"] < tol_o and all(v < tol_g for k, v in errs.items() if k != "y"), errs
    # without the attention masks the oracle's attention-side gradients are far off
    drop_na = dict(drop, attn=None)
    ry_na, cache_na = oracle.block_fwd(shape, w, arr["x"], drop=drop_na)
    _, rg_na = oracle.block_bwd(shape, w, cache_na, arr["dy"])
    assert rel_l2(to_np(g["w_qkv"]), rg_na["w_qkv"]) > 5 * errs["w_qkv"]

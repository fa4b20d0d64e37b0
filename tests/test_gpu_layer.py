"""GPU parity of the whole layer (mgb_block_fwd / mgb_block_bwd through the C
ABI) against the float64 oracle on the same seeded inputs.

Small shapes span several tiles and ragged tails (tokens not a multiple of
128, seq not a multiple of 64, ffn not a multiple of the column tile) and
every variant (Pre/Post-LN, GELU/SwiGLU, causal, GQA, with/without affine and
bias); the named workloads run at their full sizes.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import (WORKLOADS, LayerShape, layer_inputs,
                                                          mean_loss_dy)
from megatron_transformer_layer_fwd_gb300.runner import LayerRunner, WEIGHT_KEYS, to_device
from tests.util import TOL, rel_l2, to_np

pytestmark = pytest.mark.gpu

SMALL = {
    "bf16_pre_gelu_ragged": LayerShape(2, 100, 256, 4, 4, 64, 520),
    "bf16_pre_swiglu_causal_gqa": LayerShape(2, 130, 256, 4, 2, 128, 384, act="swiglu", causal=True),
    "bf16_post_gelu_causal": LayerShape(1, 192, 128, 2, 2, 64, 256, norm_pos="post", causal=True),
    "bf16_post_swiglu_gqa_gb64": LayerShape(3, 64, 256, 8, 2, 64, 256, norm_pos="post",
                                            act="swiglu", glu_block=64),
    "bf16_pre_noaffine_nobias": LayerShape(2, 96, 128, 2, 1, 128, 256, ln_affine=False,
                                           has_bias=False, causal=True),
    "f32_pre_gelu": LayerShape(2, 40, 64, 2, 2, 32, 128, dtype="f32", causal=True),
    "f32_post_swiglu_gqa": LayerShape(1, 50, 64, 4, 2, 16, 96, dtype="f32", norm_pos="post",
                                      act="swiglu", glu_block=16),
}


def _weights(arr):
    return {k: arr[k] for k in WEIGHT_KEYS}


def run_and_compare(shape, arr, dy_np, check_fwd=True, label=""):
    tol_o, tol_g = TOL[shape.dtype]
    r = LayerRunner(shape, arr)
    y = r.fwd()
    dy = to_device(dy_np, r.dtype)
    dx, g = r.bwd(dy)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    t0 = time.time()
    w = _weights(arr)
    ry, cache = oracle.block_fwd(shape, w, arr["x"])
    rdx, rg = oracle.block_bwd(shape, w, cache, dy_np)
    t_oracle = time.time() - t0
    errs = {}
    if check_fwd:
        errs["y"] = (rel_l2(to_np(y), ry), tol_o)
    errs["dx"] = (rel_l2(to_np(dx), rdx), tol_g)
    for k in WEIGHT_KEYS:
        if rg[k] is not None:
            errs["d_" + k] = (rel_l2(to_np(g[k]), rg[k]), tol_g)
    print(f"{label} oracle {t_oracle:.1f}s", {k: f"{e:.2e}" for k, (e, _) in errs.items()})
    bad = {k: e for k, (e, t) in errs.items() if not e <= t}
    assert not bad, bad
    return r, ry


@pytest.mark.parametrize("name", ["bf16_pre_swiglu_causal_gqa", "bf16_post_gelu_causal",
                                  "bf16_post_swiglu_gqa_gb64"])
def test_small_layer_parity_pair_tiles(mgb_lib, monkeypatch, name):
    """Every GEMM of the layer on CTA-pair tiles (all fused epilogues)."""
    monkeypatch.setenv("MGB_GEMM_PAIR", "1")
    shape = SMALL[name]
    arr = layer_inputs(shape, seed=12, random_affine=True, random_dy=True)
    run_and_compare(shape, arr, arr["dy"], label=f"{name}/pair")


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("dy_kind", ["random", "mean"])
def test_small_layer_parity(mgb_lib, name, dy_kind):
    shape = SMALL[name]
    arr = layer_inputs(shape, seed=11, random_affine=True, random_dy=True)
    if dy_kind == "mean":
        if shape.norm_pos == "post":
            pytest.skip("Post-LN with mean loss has identically zero gradients (checked separately)")
        dy = np.full((shape.tokens, shape.hidden), mean_loss_dy(shape))
    else:
        dy = arr["dy"]
    run_and_compare(shape, arr, dy, label=f"{name}/{dy_kind}")


def test_empty_batch(mgb_lib):
    """batch = 0: forward is a no-op, backward writes zero weight gradients."""
    shape = SMALL["bf16_pre_gelu_ragged"]
    arr = layer_inputs(shape.replace(batch=1), seed=1, random_affine=True)
    r = LayerRunner(shape.replace(batch=1), arr)
    r.desc.batch = 0
    x0 = torch.empty((0, shape.hidden), device="cuda", dtype=torch.bfloat16)
    mgb.mgb_block_fwd(r.desc, r.w, r.x, r.y, r.saved, None)
    for v in r.grads.values():
        v.fill_(1.0)
    mgb.mgb_block_bwd(r.desc, r.w, r.x, r.x, r.saved, r.dx, r.grads, r.ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    for k, v in r.grads.items():
        assert float(v.abs().max()) == 0.0, k
    del x0


def test_deterministic_repeat(mgb_lib, monkeypatch):
    """With MGB_DETERMINISTIC=1 (the attention backward in two kernels, every
    sum in a fixed order) two runs give the same bits."""
    monkeypatch.setenv("MGB_DETERMINISTIC", "1")
    shape = SMALL["bf16_pre_swiglu_causal_gqa"]
    arr = layer_inputs(shape, seed=3, random_affine=True, random_dy=True)
    r = LayerRunner(shape, arr)
    dy = to_device(arr["dy"], r.dtype)
    y1 = r.fwd().clone()
    dx1, g1 = r.bwd(dy)
    dx1 = dx1.clone()
    gw1 = g1["w_qkv"].clone()
    y2 = r.fwd()
    dx2, g2 = r.bwd(dy)
    assert torch.equal(y1, y2) and torch.equal(dx1, dx2) and torch.equal(gw1, g2["w_qkv"])


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dropout", [0.0, 0.15])
def test_graph_capture_replay(mgb_lib, monkeypatch, dropout, deterministic):
    """The layer's forward and backward (including the backward's side streams
    for weight gradients, forked and joined inside the call, and the attention
    backward's zeroed dQ accumulator) captured into one CUDA graph: replaying
    it reproduces the eager results, also after the inputs are changed in
    place; with dropout, the masks come from the descriptor's generator
    states, so the replay draws the same ones. With MGB_DETERMINISTIC=1 the
    results agree bit for bit; without it the attention dQ sums arrive in no
    fixed order, and they agree to bf16 rounding."""
    if deterministic:
        monkeypatch.setenv("MGB_DETERMINISTIC", "1")
    shape = SMALL["bf16_pre_swiglu_causal_gqa"]
    arr = layer_inputs(shape, seed=4, random_affine=True, random_dy=True)
    r = LayerRunner(shape, arr)
    if dropout > 0:
        r.desc.attn_dropout = r.desc.hidden_dropout = dropout
        mgb.mgb_block_dropout_plan(r.desc, mgb.rng_tracker(99))
        saved, _, bwd = mgb.mgb_block_sizes(r.desc)
        r.saved = torch.empty(saved, dtype=torch.uint8, device="cuda")
        r.ws = torch.empty(bwd, dtype=torch.uint8, device="cuda")
    dy = to_device(arr["dy"], r.dtype)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # first calls on this thread: library streams and events
        r.fwd()
        r.bwd(dy)
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        r.fwd()
        r.bwd(dy)
    for scale in (1.0, -0.5):
        r.x.copy_(to_device(arr["x"] * scale, r.dtype))
        g.replay()
        torch.cuda.synchronize()
        got = [r.y.clone(), r.dx.clone()] + [v.clone() for v in r.grads.values() if v is not None]
        r.fwd()
        r.bwd(dy)
        torch.cuda.synchronize()
        want = [r.y, r.dx] + [v for v in r.grads.values() if v is not None]
        for a, b in zip(got, want):
            if deterministic:
                assert torch.equal(a, b)
            else:
                assert rel_l2(to_np(a), to_np(b)) < 1e-2
    assert mgb.mgb_device_status() == mgb.MGB_OK


# ----------------------------------------------------------- named workloads

def test_fp32_page1_layer(mgb_lib):
    """float32 layer with page 1's dataflow, loss = mean(out): all outputs and
    the gradients of x and the six weights within 1e-4."""
    shape = WORKLOADS["fp32_p1_b2s128h256"]
    arr = layer_inputs(shape, seed=0)
    run_and_compare(shape, arr, np.full((shape.tokens, shape.hidden), mean_loss_dy(shape)),
                    label="fp32_p1")


def test_fp32_post_ln_layer(mgb_lib):
    """Textbook Post-LN on the same shapes: mean loss is 0 and every gradient
    vanishes (checked in absolute terms); a random dy checks the backward."""
    shape = WORKLOADS["fp32_postln_b2s128h256"]
    arr = layer_inputs(shape, seed=0, random_dy=True)
    r = LayerRunner(shape, arr)
    y = r.fwd()
    assert abs(float(y.double().mean())) < 1e-6
    dx, g = r.bwd(torch.full_like(y, mean_loss_dy(shape)))
    assert float(dx.abs().max()) < 1e-9
    for k in ("w_qkv", "w_o", "w_1", "w_2"):
        assert float(g[k].abs().max()) < 1e-9, k
    run_and_compare(shape, arr, arr["dy"], label="fp32_post")


@pytest.mark.parametrize("name", ["bf16_preln_b4s512h1024", "bf16_causal_b8s128h2048",
                                  "bf16_causal_b8s256h2048", "bf16_causal_b8s512h2048"])
def test_bf16_workload_full(mgb_lib, name):
    shape = WORKLOADS[name]
    arr = layer_inputs(shape, seed=0)
    run_and_compare(shape, arr, np.full((shape.tokens, shape.hidden), mean_loss_dy(shape)), label=name)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["bf16_causal_b8s1024h2048", "bf16_causal_b8s2048h2048",
                                  "bf16_gqa_swiglu_b2s4096h4096"])
def test_bf16_workload_full_large(mgb_lib, name):
    shape = WORKLOADS[name]
    arr = layer_inputs(shape, seed=0)
    run_and_compare(shape, arr, np.full((shape.tokens, shape.hidden), mean_loss_dy(shape)), label=name)

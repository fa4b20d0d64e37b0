"""Writes tests/golden/*.json from the oracle alone (no GPU code involved).

Run from the repo root:  python tests/golden/make_golden.py
The fixtures lock the oracle's values on tiny seeded cases so that a later
change to its arithmetic shows up as a diff of these files.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from megatron_transformer_layer_fwd_gb300.inputs import LayerShape, CEShape, layer_inputs, ce_inputs  # noqa: E402

KEYS = ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")

LAYER_CASES = {
    "tiny_pre_gelu": LayerShape(2, 4, 8, 2, 2, 4, 16, dtype="f32"),
    "tiny_post_swiglu_causal_gqa": LayerShape(1, 6, 8, 4, 2, 2, 8, dtype="f32", norm_pos="post",
                                              act="swiglu", glu_block=4, causal=True),
}


def layer_case(shape):
    inp = layer_inputs(shape, 0, random_affine=True, random_dy=True)
    w = {k: inp[k] for k in KEYS}
    y, c = oracle.block_fwd(shape, w, inp["x"])
    dx, g = oracle.block_bwd(shape, w, c, inp["dy"])
    return {"y": y.ravel().tolist(), "dx": dx.ravel().tolist(),
            **{"d_" + k: g[k].ravel().tolist() for k in KEYS if g[k] is not None}}


def main():
    out = {name: layer_case(s) for name, s in LAYER_CASES.items()}
    with open(os.path.join(HERE, "layer_tiny.json"), "w") as f:
        json.dump(out, f)
    ce = CEShape(5, 8, 37, 16, dtype="f32")
    inp = ce_inputs(ce, 0)
    loss, lse, mean, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], ce.chunk)
    dh, de = oracle.ce_grads(inp["hidden"], inp["emb"], inp["targets"], lse, 1.0 / ce.tokens)
    with open(os.path.join(HERE, "ce_tiny.json"), "w") as f:
        json.dump({"loss": loss.tolist(), "lse": lse.tolist(), "mean": mean,
                   "d_hidden": dh.ravel().tolist(), "d_emb": de.ravel().tolist()}, f)


if __name__ == "__main__":
    main()

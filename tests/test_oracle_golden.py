"""The oracle reproduces its committed tiny-case fixtures (regression lock)."""
import json
import os

import numpy as np

import oracle
from megatron_transformer_layer_fwd_gb300.inputs import CEShape, ce_inputs, layer_inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_layer_fixtures():
    import importlib.util
    spec = importlib.util.spec_from_file_location("mg", os.path.join(HERE, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    ref = json.load(open(os.path.join(HERE, "layer_tiny.json")))
    for name, shape in mg.LAYER_CASES.items():
        got = mg.layer_case(shape)
        for k, v in ref[name].items():
            np.testing.assert_allclose(got[k], v, rtol=1e-12, atol=1e-15, err_msg=f"{name}.{k}")


def test_ce_fixture():
    ref = json.load(open(os.path.join(HERE, "ce_tiny.json")))
    ce = CEShape(5, 8, 37, 16, dtype="f32")
    inp = ce_inputs(ce, 0)
    loss, lse, mean, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], ce.chunk)
    np.testing.assert_allclose(loss, ref["loss"], rtol=1e-12)
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-12)

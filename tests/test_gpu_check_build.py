"""The checking build of the library (libmgb_check.so, compiled with
-DMGB_CHECK=1): its kernels check their own invariants - every GEMM / TF32 /
attention TMA coordinate a 16-byte multiple, every tile inside its problem,
every bulk-copy address aligned, every CE target id inside the vocabulary -
and a failed check records MGB_ERR_DEVICE_CHECK and skips the access instead
of trapping. compute-sanitizer is not available on these GPUs; this build
and the guard-region tests stand in for it.

The parity suites of the GEMM, attention, LayerNorm and CE run against the
checking build in a child process (the binding loads one library per
process); the checks must pass and the results match the oracle as usual.
A CE call with a target id outside the vocabulary - which the kernels never
use as an address, so it is safe to run - must be reported by the checking
build and not by the normal one.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from megatron_transformer_layer_fwd_gb300 import build, mgb
from megatron_transformer_layer_fwd_gb300.inputs import CEShape, ce_inputs
from megatron_transformer_layer_fwd_gb300.runner import CERunner, to_device

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(code_or_args, env_extra, timeout=900):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, *code_or_args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=timeout)


def test_parity_suites_pass_on_the_checking_build(mgb_lib):
    build.build(check=True)
    r = _child(["-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                "tests/test_gpu_ops.py", "tests/test_gpu_attention.py",
                "tests/test_gpu_layernorm_bwd.py", "tests/test_gpu_ce.py",
                "-k", "not full_size"], {"MGB_LIB": "check"})
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


_BAD_TARGET = r"""
import numpy as np, torch
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import CEShape, ce_inputs
from megatron_transformer_layer_fwd_gb300.runner import CERunner, to_device
shape = CEShape(300, 256, 1000, 136)
inp = ce_inputs(shape, seed=4)
t = inp["targets"].copy()
t[17] = shape.vocab          # one id outside the vocabulary
h = to_device(inp["hidden"], torch.bfloat16)
e = to_device(inp["emb"], torch.bfloat16)
r = CERunner(shape.tokens, shape.hidden, shape.vocab, shape.chunk, h, e,
             torch.from_numpy(t).to("cuda"), mode=mgb.MGB_CE_BLOCKED, token_block=256)
r.run()
print("STATUS", mgb.mgb_device_status())
assert mgb.mgb_device_status() == mgb.MGB_OK   # the word was read and cleared
"""


@pytest.mark.parametrize("lib,want", [("check", mgb.MGB_ERR_DEVICE_CHECK), ("", mgb.MGB_OK)])
def test_out_of_vocabulary_target_is_reported_by_the_checking_build(mgb_lib, lib, want):
    if lib:
        build.build(check=True)
    r = _child(["-c", _BAD_TARGET], {"MGB_LIB": lib}, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert f"STATUS {want}" in r.stdout, r.stdout

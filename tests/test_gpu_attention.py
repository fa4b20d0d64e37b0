"""GPU parity of the attention core (mgb_attention_fwd / mgb_attention_bwd)
against the float64 oracle: MHA, GQA, MQA, causal and not, ragged sequence
lengths (not multiples of the 64/128-row tiles), head_dim 64 and 128, q/k/v
read as column slices of one fused buffer."""
import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import round_to_bf16
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(31)


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dtype)


CASES = [
    (1, 64, 1, 1, 64, False), (2, 100, 4, 2, 64, True), (1, 200, 4, 1, 128, False),
    (2, 130, 2, 2, 128, True), (1, 384, 8, 2, 128, True), (2, 257, 4, 4, 64, False),
    (1, 1000, 4, 1, 128, True),
    # more (batch, head, query tile) items than SMs: every CTA of the persistent
    # forward runs several items through its double-buffered Q and O
    (4, 640, 16, 4, 128, True), (3, 520, 16, 2, 64, False),
]


@pytest.mark.parametrize("bwd", ["one_pass", "split"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,S,nq,nkv,d,causal", CASES)
def test_attention_fwd_bwd(mgb_lib, monkeypatch, bwd, dtype, B, S, nq, nkv, d, causal):
    """The bf16 backward both ways: one pass over key blocks with dQ added up
    in float32 by reduce-add copies (head dim 128), and the two kernels
    (MGB_ATTN_BWD=split; always for head dim 64)."""
    if dtype == "f32" and S > 400:
        pytest.skip("float32 path is for the small float32 layer")
    if bwd == "split" and (dtype == "f32" or d != 128):
        pytest.skip("one backward path only")
    if bwd == "split":
        monkeypatch.setenv("MGB_ATTN_BWD", "split")
    _check(dtype, B, S, nq, nkv, d, causal, 1.0, 0.0)


@pytest.mark.parametrize("B,S,nq,nkv,d,causal", [(2, 130, 4, 2, 128, True), (1, 700, 8, 2, 128, True),
                                                 (2, 200, 2, 2, 128, False)])
def test_attention_bwd_one_pass_matches_split(mgb_lib, monkeypatch, B, S, nq, nkv, d, causal):
    """The one-pass backward against the two-kernel one on the same inputs:
    dK and dV bit for bit (the same products in the same order), dQ to float32
    rounding of its reordered sums (then rounded to bf16), and a second
    one-pass run within the same bound of the first."""
    rng = np.random.default_rng(5)
    qkv = torch.from_numpy(rng.standard_normal((B * S, (nq + 2 * nkv) * d)).astype(np.float32))
    qkv = qkv.to("cuda", torch.bfloat16)
    W = qkv.shape[1]
    qs, ks, vs = qkv, qkv[:, nq * d:], qkv[:, (nq + nkv) * d:]
    o = torch.empty((B * S, nq * d), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((B, nq, S), device="cuda", dtype=torch.float32)
    mgb.mgb_attention_fwd(B, S, nq, nkv, d, causal, mgb.MGB_BF16, qs, ks, vs, W, W, o, lse)
    do = torch.from_numpy(rng.standard_normal((B * S, nq * d)).astype(np.float32)).to("cuda", torch.bfloat16)
    ws = torch.empty(mgb.mgb_attention_bwd_ws_bytes(B, S, nq), dtype=torch.uint8, device="cuda")
    outs = []
    for path in ("split", "one_pass", "one_pass"):
        if path == "split":
            monkeypatch.setenv("MGB_ATTN_BWD", "split")
        else:
            monkeypatch.delenv("MGB_ATTN_BWD", raising=False)
        g = torch.full((B * S, W), float("nan"), device="cuda", dtype=torch.bfloat16)
        mgb.mgb_attention_bwd(B, S, nq, nkv, d, causal, mgb.MGB_BF16, qs, ks, vs, W, W, o, lse, do,
                              nq * d, g, g[:, nq * d:], g[:, (nq + nkv) * d:], W, W, ws)
        torch.cuda.synchronize()
        assert mgb.mgb_device_status() == mgb.MGB_OK
        outs.append(g.float())
    split, one, again = outs
    kv = slice(nq * d, W)
    assert torch.equal(split[:, kv], one[:, kv]) and torch.equal(one[:, kv], again[:, kv])
    dq = slice(0, nq * d)
    scale = float(split[:, dq].abs().max())
    assert float((one[:, dq] - split[:, dq]).abs().max()) <= 2 ** -7 * scale
    assert float((one[:, dq] - again[:, dq]).abs().max()) <= 2 ** -7 * scale


@pytest.mark.parametrize("B,S,nq,nkv,d,causal", [(1, 700, 2, 1, 128, True), (2, 384, 2, 2, 64, False)])
def test_attention_sharp_growing_scores(mgb_lib, B, S, nq, nkv, d, causal):
    """Scores with a spread of ~13 (log2 units) and keys whose norm grows along
    the sequence: a row's running maximum keeps rising tile after tile, so the
    forward's lazily moved softmax reference and the O rescale in TMEM run many
    times per row."""
    _check("bf16", B, S, nq, nkv, d, causal, 3.0, 4.0)


def _check(dtype, B, S, nq, nkv, d, causal, amp, ramp):
    rnd = round_to_bf16 if dtype == "bf16" else (lambda a: a.astype(np.float32).astype(np.float64))
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    mdt = mgb.MGB_BF16 if dtype == "bf16" else mgb.MGB_F32
    grow = 1.0 + ramp * np.arange(S)[None, None, :, None] / S
    q = rnd(amp * RNG.standard_normal((B, nq, S, d)))
    k = rnd(amp * grow * RNG.standard_normal((B, nkv, S, d)))
    v = rnd(RNG.standard_normal((B, nkv, S, d)))
    do = rnd(RNG.standard_normal((B, nq, S, d)))
    pack = lambda t: t.transpose(0, 2, 1, 3).reshape(B * S, -1)
    qkv = _dev(np.concatenate([pack(q), pack(k), pack(v)], axis=1), td)
    W = qkv.shape[1]
    qs, ks, vs = qkv, qkv[:, nq * d:], qkv[:, (nq + nkv) * d:]
    o = torch.empty((B * S, nq * d), device="cuda", dtype=td)
    lse = torch.empty((B, nq, S), device="cuda", dtype=torch.float32)
    mgb.mgb_attention_fwd(B, S, nq, nkv, d, causal, mdt, qs, ks, vs, W, W, o, lse)
    ro, rl = oracle.attention_fwd(q, k, v, causal)
    tol = 1e-2 if dtype == "bf16" else 1e-5
    assert rel_l2(to_np(o), pack(ro)) < tol
    assert np.abs(to_np(lse) - rl).max() < (2e-2 if dtype == "bf16" else 1e-5)
    # backward against the oracle's gradient of sum(do * O) for the same q, k, v
    dqkv = torch.full((B * S, W), float("nan"), device="cuda", dtype=td)
    ws = torch.empty(mgb.mgb_attention_bwd_ws_bytes(B, S, nq), dtype=torch.uint8, device="cuda")
    mgb.mgb_attention_bwd(B, S, nq, nkv, d, causal, mdt, qs, ks, vs, W, W, o, lse,
                          _dev(pack(do), td), nq * d, dqkv, dqkv[:, nq * d:],
                          dqkv[:, (nq + nkv) * d:], W, W, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    rdq, rdk, rdv = oracle.attention_bwd(do, q, k, v, causal)
    g = to_np(dqkv)
    tg = 2e-2 if dtype == "bf16" else 1e-4
    assert rel_l2(g[:, : nq * d], pack(rdq)) < tg
    assert rel_l2(g[:, nq * d: (nq + nkv) * d], pack(rdk)) < tg
    assert rel_l2(g[:, (nq + nkv) * d:], pack(rdv)) < tg

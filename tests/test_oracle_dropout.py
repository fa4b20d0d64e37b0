"""Pins of the dropout oracle (CPU only): the counter-based generator against
an independent library implementation of Philox4x32-10 and the closed forms
of its constants; the keep statistics; the tensor-parallel RNG tracker of
"02 - How a whole Transformer block is split", section 5 (seeds, fork,
replay, the same mask outside the TP region on every rank and different
masks inside); the layer with dropout against finite differences and torch
float64 autograd."""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import dropout as od
from megatron_transformer_layer_fwd_gb300.inputs import LayerShape, layer_inputs

KEYS = ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def _curand():
    for p in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if p and (os.path.exists(p) or not p.startswith("/")):
            try:
                return ctypes.CDLL(p)
            except OSError:
                pass
    pytest.skip("libcurand not available")


def _curand_philox_words(seed, word_offset, n):
    """n 32-bit outputs of the curand host generator CURAND_RNG_PSEUDO_PHILOX4_32_10."""
    lib = _curand()
    g = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(g), 161) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(g, ctypes.c_ulonglong(word_offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(g, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(g)
    return out


def _philox_at_curand_layout(seed, word_offset, n):
    """The oracle's Philox4x32-10 block function on the counters the curand
    host generator visits: its output word i is word i % 4 of counter
    (g >> 16, 0, g & 0xFFFF, 0), g = i // 4 (65536 interleaved subsequences;
    the first word carries into the second)."""
    i = np.arange(word_offset, word_offset + n, dtype=np.uint64)
    g = i // np.uint64(4)
    x = g >> np.uint64(16)
    ctr = np.zeros((n, 4), dtype=np.uint64)
    ctr[:, 0] = x & np.uint64(0xFFFFFFFF)
    ctr[:, 1] = x >> np.uint64(32)
    ctr[:, 2] = g & np.uint64(0xFFFF)
    out = od.philox4x32(ctr, (seed & 0xFFFFFFFF, seed >> 32))
    return out[np.arange(n), (i % np.uint64(4)).astype(np.int64)]


@pytest.mark.parametrize("seed,word_offset", [(0, 0), (1, 0), (2718, 8), (0x123456789ABCDEF, 1000),
                                              (42, 4 * 65536 * 3 + 5), (9, 1 << 50)])
def test_philox_matches_curand_host_generator(seed, word_offset):
    """Counter words 0, 1 and 2 and both key words exercised (the stream
    layout of uniform_bytes uses counter words 0 and 1)."""
    n = 4096
    want = _curand_philox_words(seed, word_offset, n)
    assert np.array_equal(_philox_at_curand_layout(seed, word_offset, n), want)


def test_byte_stream_is_the_philox_counter_sequence():
    """uniform_bytes: counter (q, 0, 0, 0) gives bytes 16q .. 16q+15, words in
    order, each lowest byte first."""
    seed = 0xABCDEF0123
    words = od.philox4x32(np.array([[q, 0, 0, 0] for q in range(8)], dtype=np.uint64),
                          (seed & 0xFFFFFFFF, seed >> 32)).reshape(-1)
    b = od.uniform_bytes(seed, 0, 128)
    for pos in (0, 1, 2, 3, 4, 17, 100, 127):
        assert b[pos] == (int(words[pos // 4]) >> (8 * (pos % 4))) & 0xFF


def test_weyl_constants_closed_forms():
    """Key increments: floor(2^32 (sqrt 5 - 1) / 2) (golden ratio) and
    floor(2^32 (sqrt 3 - 1)), in exact integer arithmetic."""
    assert od.PHILOX_W0 == (math.isqrt(5 << 64) - (1 << 32)) // 2
    assert od.PHILOX_W1 == math.isqrt(3 << 64) - (1 << 32)


def test_stream_positions_are_consistent():
    for off, n in ((0, 100), (5, 37), (31, 1), (4096 + 7, 300)):
        assert np.array_equal(od.uniform_bytes(9, off, n), od.uniform_bytes(9, 0, off + n)[off:])


def test_bytes_uniform_and_keep_fraction():
    u = od.uniform_bytes(123, 0, 1 << 20)
    counts = np.bincount(u, minlength=256)
    e = u.size / 256
    chi2 = float(((counts - e) ** 2 / e).sum())
    assert chi2 < 255 + 8 * math.sqrt(2 * 255)
    for p in (0.1, 0.5, 0.9):
        keep = od.dropout_keep(7, 16, (512, 1024), p)
        q = od.keep_threshold(p) / 256
        n = keep.size
        assert abs(keep.mean() - q) < 6 * math.sqrt(q * (1 - q) / n)
    assert od.keep_threshold(0.0) == 256 and od.dropout_keep(1, 0, (4, 64), 0.0).all()
    assert od.keep_scale(0.5) == 2.0


def test_tracker_seeds_fork_and_draw():
    t = od.model_parallel_seed(1234, tp_rank=3, ep_rank=2, etp_rank=1)
    assert t.states[t.DATA][0] == 1234
    assert t.states[t.MODEL][0] == 1234 + 2718 + 3
    assert t.states[t.EXPERT][0] == 1234 + 1024 + 100 * 2 + 1
    assert t.current == t.DATA
    assert t.draw(10) == (1234, 0) and t.draw(17) == (1234, 16) and t.draw(1) == (1234, 48)
    with t.fork():
        assert t.current == t.MODEL
        assert t.draw(5) == (1234 + 2718 + 3, 0)
    assert t.current == t.DATA
    with pytest.raises(RuntimeError):
        with t.fork(t.EXPERT):
            assert t.current == t.EXPERT
            raise RuntimeError("inside")
    assert t.current == t.DATA  # restored on the way out of an exception too
    assert t.draw(1) == (1234, 64)


SHAPE = LayerShape(2, 6, 8, 4, 2, 3, 10, dtype="f32", causal=True)


def test_tp_ranks_share_outside_masks_and_differ_inside():
    """Section 5's consistency rule on the layer's sites: every TP rank draws
    the same hidden-dropout masks (replicated activations) and its own
    attention masks; a fresh tracker with the same seed replays them."""
    plans = [od.layer_dropout(SHAPE, od.model_parallel_seed(77, tp_rank=r), 0.3, 0.2) for r in range(4)]
    for pl in plans[1:]:
        assert np.array_equal(pl["proj"][0], plans[0]["proj"][0])
        assert np.array_equal(pl["fc2"][0], plans[0]["fc2"][0])
        assert not np.array_equal(pl["attn"][0], plans[0]["attn"][0])
    assert not np.array_equal(plans[0]["proj"][0], plans[0]["fc2"][0])
    again = od.layer_dropout(SHAPE, od.model_parallel_seed(77, tp_rank=2), 0.3, 0.2)
    for site in ("attn", "proj", "fc2"):
        assert np.array_equal(again[site][0], plans[2][site][0])


def test_attention_site_rows_start_on_a_counter():
    """Element (b, h, i, j) of the attention site is byte ((b*nq+h)*S+i)*Sp+j."""
    B, nq, S, p = 1, 2, 5, 0.5
    keep = od.dropout_keep(3, 32, (B, nq, S, S), p, row_pad=od.pad16(S))
    u = od.uniform_bytes(3, 32, B * nq * S * 16)
    for h in range(nq):
        for i in range(S):
            row = u[(h * S + i) * 16:(h * S + i) * 16 + S]
            assert np.array_equal(keep[0, h, i], row < od.keep_threshold(p))


def _inputs(seed=0):
    inp = layer_inputs(SHAPE, seed, random_affine=True, random_dy=True)
    for k in ("w_qkv", "w_o", "w_1", "w_2"):
        inp[k] = inp[k] * 25.0
    return inp


def test_layer_without_drops_is_unchanged():
    inp = _inputs()
    w = {k: inp[k] for k in KEYS}
    y0, c0 = oracle.block_fwd(SHAPE, w, inp["x"])
    T, H, B, S, nq = SHAPE.tokens, SHAPE.hidden, SHAPE.batch, SHAPE.seq, SHAPE.n_q_heads
    ones = {"attn": (np.ones((B, nq, S, S), bool), 1.0), "proj": (np.ones((T, H), bool), 1.0),
            "fc2": (np.ones((T, H), bool), 1.0)}
    y1, c1 = oracle.block_fwd(SHAPE, w, inp["x"], drop=ones)
    assert np.array_equal(y0, y1)
    g0 = oracle.block_bwd(SHAPE, w, c0, inp["dy"])
    g1 = oracle.block_bwd(SHAPE, w, c1, inp["dy"])
    assert np.array_equal(g0[0], g1[0])


def _plan():
    return od.layer_dropout(SHAPE, od.model_parallel_seed(5), 0.3, 0.25)


def test_layer_dropout_backward_finite_differences():
    inp = _inputs(1)
    w = {k: inp[k] for k in KEYS}
    drop = _plan()
    x, dy = inp["x"], inp["dy"]
    _, cache = oracle.block_fwd(SHAPE, w, x, drop=drop)
    dx, g = oracle.block_bwd(SHAPE, w, cache, dy)
    loss = lambda: float((dy * oracle.block_fwd(SHAPE, w, x, drop=drop)[0]).sum())
    h = 1e-6
    rng = np.random.default_rng(11)
    for arr, grad in [(x, dx)] + [(w[k], g[k]) for k in ("w_qkv", "w_o", "b_o", "w_1", "w_2", "b_2")]:
        flat = arr.reshape(-1)
        for i in rng.choice(flat.size, size=min(flat.size, 12), replace=False):
            old = flat[i]
            flat[i] = old + h
            fp = loss()
            flat[i] = old - h
            fm = loss()
            flat[i] = old
            fd = (fp - fm) / (2 * h)
            assert abs(grad.reshape(-1)[i] - fd) <= 1e-6 * max(1.0, abs(fd))


def test_layer_dropout_matches_torch_fp64_autograd():
    """The same layer in torch ops with the same masks, differentiated by
    autograd (explicit attention: softmax, then the probability mask)."""
    inp = _inputs(2)
    w = {k: inp[k] for k in KEYS}
    drop = _plan()
    tw = {k: torch.tensor(v, requires_grad=True) for k, v in w.items()}
    tx = torch.tensor(inp["x"], requires_grad=True)
    B, S, H = SHAPE.batch, SHAPE.seq, SHAPE.hidden
    nq, nkv, d = SHAPE.n_q_heads, SHAPE.n_kv_heads, SHAPE.head_dim
    mask = lambda site: torch.tensor(drop[site][0], dtype=torch.float64) * drop[site][1]
    ln = lambda t, g, b: F.layer_norm(t, (H,), g, b, SHAPE.ln_eps)
    xn = ln(tx, tw["ln1_g"], tw["ln1_b"])
    qkv = F.linear(xn, tw["w_qkv"], tw["b_qkv"])
    q, k, v = torch.split(qkv, [nq * d, nkv * d, nkv * d], dim=1)
    q = q.reshape(B, S, nq, d).transpose(1, 2)
    k = k.reshape(B, S, nkv, d).transpose(1, 2).repeat_interleave(nq // nkv, dim=1)
    v = v.reshape(B, S, nkv, d).transpose(1, 2).repeat_interleave(nq // nkv, dim=1)
    s = q @ k.transpose(-1, -2) / math.sqrt(d)
    s = s.masked_fill(~torch.tril(torch.ones(S, S, dtype=torch.bool)), float("-inf"))
    p = torch.softmax(s, dim=-1) * mask("attn")
    O = (p @ v).transpose(1, 2).reshape(B * S, nq * d)
    h = tx + F.linear(O, tw["w_o"], tw["b_o"]) * mask("proj")
    u = F.linear(ln(h, tw["ln2_g"], tw["ln2_b"]), tw["w_1"], tw["b_1"])
    ty = h + F.linear(F.gelu(u), tw["w_2"], tw["b_2"]) * mask("fc2")
    ty.backward(torch.tensor(inp["dy"]))
    y, cache = oracle.block_fwd(SHAPE, w, inp["x"], drop=drop)
    np.testing.assert_allclose(y, ty.detach().numpy(), rtol=1e-10, atol=1e-11)
    dx, g = oracle.block_bwd(SHAPE, w, cache, inp["dy"])
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-9, atol=1e-10)
    for key in KEYS:
        np.testing.assert_allclose(g[key], tw[key].grad.numpy(), rtol=1e-9, atol=1e-10, err_msg=key)


def test_planted_generator_error_is_caught(monkeypatch):
    """A wrong key increment (a plausible slip) no longer matches the library."""
    want = _curand_philox_words(2718, 0, 64)
    monkeypatch.setattr(od, "PHILOX_W1", od.PHILOX_W1 ^ 1)
    assert not np.array_equal(_philox_at_curand_layout(2718, 0, 64), want)

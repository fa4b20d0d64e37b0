"""GPU parity of the vocab-parallel embedding lookup and its backward
(mgb_embedding_fwd / mgb_embedding_bwd through the C ABI) against the float64
oracle, and the tied-table round trip with the cross-entropy's gradient."""
import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import CEShape, ce_inputs, round_to_bf16
from megatron_transformer_layer_fwd_gb300.runner import CERunner, to_device
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(57)


def _ids(T, V, repeats=False):
    if repeats:  # a few very frequent ids plus a tail, as in text
        return np.minimum((RNG.zipf(1.3, size=T) - 1), V - 1).astype(np.int32)
    return RNG.integers(0, V, size=T).astype(np.int32)


def _dev(a, td):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", td)


def _fwd(ids, E, v0, v1, td, dt):
    T, H = ids.shape[0], E.shape[1]
    out = torch.full((T, H), float("nan"), device="cuda", dtype=td)
    mgb.mgb_embedding_fwd(T, H, v0, v1, dt, torch.from_numpy(ids).cuda(), _dev(E, td), out)
    return out


def _bwd(ids, dout, v0, v1, td, dt, init=None):
    T, H = dout.shape
    d_emb = _dev(init, td) if init is not None else torch.full((v1 - v0, H), float("nan"),
                                                               device="cuda", dtype=td)
    ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(T, v0, v1), dtype=torch.uint8, device="cuda")
    mgb.mgb_embedding_bwd(T, H, v0, v1, dt, torch.from_numpy(ids).cuda(), _dev(dout, td), d_emb,
                          init is not None, ws)
    return d_emb


DT = [("bf16", torch.bfloat16, mgb.MGB_BF16, round_to_bf16, 1e-2),
      ("f32", torch.float32, mgb.MGB_F32, lambda a: a.astype(np.float32).astype(np.float64), 1e-6)]


@pytest.mark.parametrize("name,td,dt,rnd,tol", DT)
@pytest.mark.parametrize("T,H,V", [(333, 64, 1000), (1024, 512, 300), (5, 8, 7)])
def test_lookup_exact_and_shards_sum(mgb_lib, name, td, dt, rnd, tol, T, H, V):
    ids = _ids(T, V, repeats=(V == 300))
    E = rnd(RNG.standard_normal((V, H)))
    full = _fwd(ids, E, 0, V, td, dt)
    assert np.array_equal(to_np(full), oracle.embedding_fwd(ids, E, 0, V))
    # three vocab shards, the last ragged: their outputs sum (exactly) to the full lookup
    b = [0, V // 3, 2 * V // 3 + 1, V]
    parts = [_fwd(ids, E[lo:hi], lo, hi, td, dt) for lo, hi in zip(b[:-1], b[1:])]
    for (lo, hi), p in zip(zip(b[:-1], b[1:]), parts):
        assert np.array_equal(to_np(p), oracle.embedding_fwd(ids, E[lo:hi], lo, hi))
    assert torch.equal(sum(p.float() for p in parts), full.float())
    assert mgb.mgb_device_status() == mgb.MGB_OK


@pytest.mark.parametrize("name,td,dt,rnd,tol", DT)
@pytest.mark.parametrize("T,H,V,v0,v1,rep", [(500, 64, 800, 0, 800, False), (2048, 256, 300, 0, 300, True),
                                             (700, 128, 1000, 250, 613, True), (1, 8, 4, 0, 4, False)])
def test_backward(mgb_lib, name, td, dt, rnd, tol, T, H, V, v0, v1, rep):
    """Overwrite and accumulate; repeated ids; ids outside the shard."""
    ids = _ids(T, V, repeats=rep)
    dout = rnd(RNG.standard_normal((T, H)))
    ref = oracle.embedding_bwd(ids, dout, v0, v1)
    got = to_np(_bwd(ids, dout, v0, v1, td, dt))
    assert rel_l2(got, ref) <= tol
    untouched = np.setdiff1d(np.arange(v0, v1), ids) - v0
    assert np.all(got[untouched] == 0)
    init = rnd(RNG.standard_normal((v1 - v0, H)))
    got = to_np(_bwd(ids, dout, v0, v1, td, dt, init=init))
    assert rel_l2(got, init + ref) <= tol
    assert np.array_equal(got[untouched], to_np(_dev(init, td))[untouched])
    assert mgb.mgb_device_status() == mgb.MGB_OK


def test_backward_deterministic(mgb_lib):
    ids = _ids(4096, 500, repeats=True)
    dout = round_to_bf16(RNG.standard_normal((4096, 256)))
    a = _bwd(ids, dout, 0, 500, torch.bfloat16, mgb.MGB_BF16)
    b = _bwd(ids, dout, 0, 500, torch.bfloat16, mgb.MGB_BF16)
    assert torch.equal(a, b)


@pytest.mark.parametrize("accumulate", [False, True])
def test_backward_token_order_f32(mgb_lib, accumulate):
    """In float32 the backward is bit-exact against adding each token's row in
    token order (starting from the old row when accumulating): the order the
    sums are taken in is fixed, whatever the blocks' schedule. Ids repeat
    across several tiles of the rank computation; some fall outside the shard."""
    T, H, V, v0, v1 = 3000, 64, 400, 37, 381
    ids = _ids(T, V, repeats=True)
    dout = RNG.standard_normal((T, H)).astype(np.float32)
    init = RNG.standard_normal((v1 - v0, H)).astype(np.float32)
    want = init.copy() if accumulate else np.zeros_like(init)
    own = (ids >= v0) & (ids < v1)
    np.add.at(want, ids[own] - v0, dout[own])  # unbuffered, in index order
    got = to_np(_bwd(ids, dout, v0, v1, torch.float32, mgb.MGB_F32, init=init if accumulate else None))
    assert np.array_equal(got.astype(np.float32), want)


def test_prepare_apply_token_order_f32(mgb_lib):
    """The two-step backward: one prepare from the ids, then applies in both
    modes with different d_out, all bit-exact (float32) against adding each
    token's row in token order. The ids are overwritten after the prepare (the
    plan holds everything the applies need), and the applies run on another
    stream, ordered after the prepare by an event."""
    T, H, V, v0, v1 = 3000, 64, 400, 37, 381
    ids = _ids(T, V, repeats=True)
    ids_d = torch.from_numpy(ids).cuda()
    ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(T, v0, v1), dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        plan = mgb.mgb_embedding_bwd_prepare(T, v0, v1, ids_d, ws, stream=s1)
        ids_d.fill_(v0)  # not read again
    ev = torch.cuda.Event()
    ev.record(s1)
    s2.wait_event(ev)
    assert (plan.tokens, plan.v0, plan.v1, plan.ws_bytes) == (T, v0, v1, ws.numel())
    own = (ids >= v0) & (ids < v1)
    d1 = RNG.standard_normal((T, H)).astype(np.float32)
    d2 = RNG.standard_normal((T, H)).astype(np.float32)
    want = np.zeros((v1 - v0, H), dtype=np.float32)
    np.add.at(want, ids[own] - v0, d1[own])
    with torch.cuda.stream(s2):
        d_emb = torch.full((v1 - v0, H), float("nan"), device="cuda", dtype=torch.float32)
        mgb.mgb_embedding_bwd_apply(plan, H, mgb.MGB_F32, _dev(d1, torch.float32), d_emb, 0,
                                    stream=s2)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(d_emb).astype(np.float32), want)
    np.add.at(want, ids[own] - v0, d2[own])
    with torch.cuda.stream(s2):
        mgb.mgb_embedding_bwd_apply(plan, H, mgb.MGB_F32, _dev(d2, torch.float32), d_emb, 1,
                                    stream=s2)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(d_emb).astype(np.float32), want)
    assert mgb.mgb_device_status() == mgb.MGB_OK


@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("T,V,v0,v1,rep", [(2048, 300, 0, 300, True), (700, 1000, 250, 613, True),
                                           (5000, 3000, 0, 3000, False)])
def test_prepare_apply_equals_one_call_bf16(mgb_lib, accumulate, T, V, v0, v1, rep):
    """bf16: the two steps give the one-call backward's result bit for bit."""
    H = 128
    ids = _ids(T, V, repeats=rep)
    dout = round_to_bf16(RNG.standard_normal((T, H)))
    init = round_to_bf16(RNG.standard_normal((v1 - v0, H))) if accumulate else None
    one = _bwd(ids, dout, v0, v1, torch.bfloat16, mgb.MGB_BF16, init=init)
    ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(T, v0, v1), dtype=torch.uint8, device="cuda")
    plan = mgb.mgb_embedding_bwd_prepare(T, v0, v1, torch.from_numpy(ids).cuda(), ws)
    two = (_dev(init, torch.bfloat16) if accumulate else
           torch.full((v1 - v0, H), float("nan"), device="cuda", dtype=torch.bfloat16))
    mgb.mgb_embedding_bwd_apply(plan, H, mgb.MGB_BF16, _dev(dout, torch.bfloat16), two, accumulate)
    assert torch.equal(one, two)
    ref = oracle.embedding_bwd(ids, dout, v0, v1) + (init if accumulate else 0.0)
    assert rel_l2(to_np(two), ref) <= 1e-2
    assert mgb.mgb_device_status() == mgb.MGB_OK


def test_prepare_apply_empty_batch(mgb_lib):
    ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(0, 0, 10), dtype=torch.uint8, device="cuda")
    plan = mgb.mgb_embedding_bwd_prepare(0, 0, 10, None, ws)
    d = torch.full((10, 16), 3.0, device="cuda", dtype=torch.bfloat16)
    mgb.mgb_embedding_bwd_apply(plan, 16, mgb.MGB_BF16, None, d, 1)  # nothing to add
    assert float(d.float().min()) == 3.0 and float(d.float().max()) == 3.0
    mgb.mgb_embedding_bwd_apply(plan, 16, mgb.MGB_BF16, None, d, 0)  # rows written as zeros
    assert float(d.float().abs().max()) == 0.0
    assert mgb.mgb_device_status() == mgb.MGB_OK


def test_empty_batch(mgb_lib):
    ids = np.zeros(0, dtype=np.int32)
    d = _bwd(ids, np.zeros((0, 16)), 0, 10, torch.bfloat16, mgb.MGB_BF16)
    assert float(d.float().abs().max()) == 0.0


def test_tied_table_round_trip(mgb_lib):
    """One table E for the input lookup and the output projection: the CE's
    d_emb, then the lookup's backward accumulated onto it."""
    shape = CEShape(256, 128, 2048, 704)
    inp = ce_inputs(shape, seed=3)
    h = to_device(inp["hidden"], torch.bfloat16)
    e = to_device(inp["emb"], torch.bfloat16)
    t = torch.from_numpy(inp["targets"]).to("cuda")
    r = CERunner(shape.tokens, shape.hidden, shape.vocab, shape.chunk, h, e, t)
    r.run()
    ids = _ids(shape.tokens, shape.vocab, repeats=True)
    dout = round_to_bf16(RNG.standard_normal((shape.tokens, shape.hidden)) * 1e-3)
    ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(shape.tokens, 0, shape.vocab), dtype=torch.uint8,
                     device="cuda")
    mgb.mgb_embedding_bwd(shape.tokens, shape.hidden, 0, shape.vocab, mgb.MGB_BF16,
                          torch.from_numpy(ids).cuda(), _dev(dout, torch.bfloat16), r.d_emb, 1, ws)
    _, lse, _, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], shape.chunk)
    _, de = oracle.ce_grads(inp["hidden"], inp["emb"], inp["targets"], lse, 1.0 / shape.tokens)
    ref = de + oracle.embedding_bwd(ids, dout, 0, shape.vocab)
    assert rel_l2(to_np(r.d_emb), ref) < 2e-2
    assert mgb.mgb_device_status() == mgb.MGB_OK


@pytest.mark.slow
def test_full_size_sampled(mgb_lib):
    """8192 tokens over the 128256 x 4096 table: the lookup is compared whole;
    the backward on windows of 64 rows around sampled ids."""
    T, H, V = 8192, 4096, 128256
    ids = _ids(T, V, repeats=True)
    E = torch.randn((V, H), device="cuda").to(torch.bfloat16)
    out = torch.empty((T, H), device="cuda", dtype=torch.bfloat16)
    mgb.mgb_embedding_fwd(T, H, 0, V, mgb.MGB_BF16, torch.from_numpy(ids).cuda(), E, out)
    assert torch.equal(out, E[torch.from_numpy(ids).long().cuda()])
    dout = torch.randn((T, H), device="cuda").to(torch.bfloat16)
    ws = torch.empty(mgb.mgb_embedding_bwd_ws_bytes(T, 0, V), dtype=torch.uint8, device="cuda")
    d_emb = torch.empty((V, H), device="cuda", dtype=torch.bfloat16)
    mgb.mgb_embedding_bwd(T, H, 0, V, mgb.MGB_BF16, torch.from_numpy(ids).cuda(), dout, d_emb, 0, ws)
    dn = to_np(dout)
    for v in np.unique(np.concatenate([ids[:3], [0, 1, V - 1]])):
        lo = max(0, min(int(v) - 32, V - 64))
        ref = oracle.embedding_bwd(ids, dn, lo, lo + 64)
        assert rel_l2(to_np(d_emb[lo:lo + 64]), ref) < 1e-2
    assert mgb.mgb_device_status() == mgb.MGB_OK

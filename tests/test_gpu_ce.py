"""GPU parity of the vocab-chunked tied-embedding cross-entropy
(mgb_vocab_ce_fwd_bwd through the C ABI) against the float64 oracle."""
import time

import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import CE_WORKLOADS, CEShape, ce_inputs
from megatron_transformer_layer_fwd_gb300.runner import CERunner, to_device
from tests.util import CE_LOSS_ABS, rel_l2, to_np

pytestmark = pytest.mark.gpu


MODES = [mgb.MGB_CE_STREAM, mgb.MGB_CE_FUSED, mgb.MGB_CE_RESIDENT, mgb.MGB_CE_BLOCKED]


def _runner(shape, inp, mode, token_block=0, emb_stream=None):
    h = to_device(inp["hidden"], torch.bfloat16)
    e = to_device(inp["emb"], torch.bfloat16)
    t = torch.from_numpy(inp["targets"]).to("cuda")
    return CERunner(shape.tokens, shape.hidden, shape.vocab, shape.chunk, h, e, t, mode=mode,
                    token_block=token_block, emb_stream=emb_stream)


@pytest.mark.parametrize("T,H,V,C,tb", [(300, 256, 1000, 136, 256), (512, 1024, 8192, 1000, 256),
                                        (1100, 128, 2048, 2048, 512), (130, 64, 520, 64, 256),
                                        # the library's default block (0): 4096 + a ragged 404
                                        (4500, 128, 1024, 520, 0)])
def test_ce_blocked_token_blocks(mgb_lib, T, H, V, C, tb):
    """The token-blocked CE with several blocks (a ragged last one): each
    block's losses from its own partials, d_hidden rows from the split-K
    product, d_emb accumulated in float32 across blocks."""
    shape = CEShape(T, H, V, C)
    inp = ce_inputs(shape, seed=15)
    r = _runner(shape, inp, mgb.MGB_CE_BLOCKED, token_block=tb)
    r.run()
    assert mgb.mgb_device_status() == mgb.MGB_OK
    loss, lse, mean, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], C)
    dh, de = oracle.ce_grads(inp["hidden"], inp["emb"], inp["targets"], lse, 1.0 / T)
    assert np.abs(to_np(r.loss) - loss).max() < CE_LOSS_ABS
    assert np.abs(to_np(r.lse) - lse).max() < CE_LOSS_ABS
    assert abs(float(r.loss_mean[0]) - mean) < CE_LOSS_ABS
    assert rel_l2(to_np(r.d_hidden), dh) < 2e-2
    assert rel_l2(to_np(r.d_emb), de) < 2e-2
    # the same call again gives the same bits (fixed-order sums throughout)
    first = (r.loss.clone(), r.d_hidden.clone(), r.d_emb.clone())
    r.run()
    assert torch.equal(first[0], r.loss) and torch.equal(first[1], r.d_hidden)
    assert torch.equal(first[2], r.d_emb)


def test_ce_blocked_block_size_changes_only_rounding(mgb_lib):
    """The token block is a memory device: token blocks of 256, 768, 1024 and one
    larger than T give the same per-token losses, mean and gradients up to
    float32 rounding order (each also within tolerance of the oracle)."""
    shape = CEShape(1000, 256, 3000, 1000)
    inp = ce_inputs(shape, seed=33)
    loss, lse, mean, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], shape.chunk)
    outs = []
    for tb in (256, 768, 1024, 4096):
        r = _runner(shape, inp, mgb.MGB_CE_BLOCKED, token_block=tb)
        r.run()
        assert mgb.mgb_device_status() == mgb.MGB_OK
        assert np.abs(to_np(r.loss) - loss).max() < CE_LOSS_ABS
        outs.append((to_np(r.loss), float(r.loss_mean[0]), to_np(r.d_hidden), to_np(r.d_emb)))
    for o in outs[1:]:
        assert np.abs(o[0] - outs[0][0]).max() < 1e-5
        assert abs(o[1] - outs[0][1]) < 1e-6
        assert rel_l2(o[2], outs[0][2]) < 1e-2
        assert rel_l2(o[3], outs[0][3]) < 1e-2


@pytest.mark.parametrize("mode", [mgb.MGB_CE_RESIDENT, mgb.MGB_CE_BLOCKED])
def test_ce_kept_logits_through_tma(mgb_lib, monkeypatch, mode):
    """The logits kept by the statistics epilogue, stored by TMA boxes (vocab
    chunks of 32-column multiples, a ragged last chunk and ragged rows) or by
    each thread: the same bits in every output."""
    shape = CEShape(600, 256, 2000, 704)
    inp = ce_inputs(shape, seed=8)
    outs = []
    for tma in ("0", "1"):
        monkeypatch.setenv("MGB_GEMM_TMA_OUT", tma)
        r = _runner(shape, inp, mode, token_block=256)
        r.run()
        torch.cuda.synchronize()
        assert mgb.mgb_device_status() == mgb.MGB_OK
        outs.append([x.clone() for x in (r.loss, r.lse, r.d_hidden, r.d_emb)])
    for x0, x1 in zip(*outs):
        assert torch.equal(x0, x1)


def test_ce_blocked_emb_stream(mgb_lib):
    """Blocked mode with the last block's d_emb left on a caller's stream:
    after joining it, the results equal those of the joined call bit for bit."""
    shape = CEShape(600, 256, 2000, 704)
    inp = ce_inputs(shape, seed=21)
    r0 = _runner(shape, inp, mgb.MGB_CE_BLOCKED, token_block=256)
    r0.run()
    side = torch.cuda.Stream()
    r1 = _runner(shape, inp, mgb.MGB_CE_BLOCKED, token_block=256, emb_stream=side)
    main = torch.cuda.current_stream()
    r1.run(main)
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert mgb.mgb_device_status() == mgb.MGB_OK
    assert torch.equal(r0.d_emb, r1.d_emb) and torch.equal(r0.d_hidden, r1.d_hidden)
    assert torch.equal(r0.loss, r1.loss)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,H,V,C", [(300, 256, 1000, 136), (256, 128, 2048, 2048), (130, 64, 520, 64),
                                     (512, 1024, 8192, 1000)])
def test_ce_small_full_parity(mgb_lib, T, H, V, C, mode):
    """Both places for the statistics and the gradient (streaming kernels over
    stored logits, or the logits GEMM's epilogue): ragged chunks, chunks
    narrower than one 128-column group, one chunk for the whole vocabulary."""
    shape = CEShape(T, H, V, C)
    inp = ce_inputs(shape, seed=5)
    r = _runner(shape, inp, mode)
    r.run()
    assert mgb.mgb_device_status() == mgb.MGB_OK
    loss, lse, mean, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], C)
    dh, de = oracle.ce_grads(inp["hidden"], inp["emb"], inp["targets"], lse, 1.0 / T)
    assert np.abs(to_np(r.loss) - loss).max() < CE_LOSS_ABS
    assert np.abs(to_np(r.lse) - lse).max() < CE_LOSS_ABS
    assert abs(float(r.loss_mean[0]) - mean) < CE_LOSS_ABS
    assert rel_l2(to_np(r.d_hidden), dh) < 2e-2
    assert rel_l2(to_np(r.d_emb), de) < 2e-2


@pytest.mark.parametrize("mode", MODES)
def test_ce_pair_tiles(mgb_lib, monkeypatch, mode):
    """The CE's GEMMs (logits with the statistics or gradient epilogue,
    dgrad, wgrad) on CTA-pair tiles."""
    monkeypatch.setenv("MGB_GEMM_PAIR", "1")
    T, H, V, C = 300, 256, 1000, 136
    shape = CEShape(T, H, V, C)
    inp = ce_inputs(shape, seed=6)
    r = _runner(shape, inp, mode)
    r.run()
    assert mgb.mgb_device_status() == mgb.MGB_OK
    loss, lse, mean, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], C)
    dh, de = oracle.ce_grads(inp["hidden"], inp["emb"], inp["targets"], lse, 1.0 / T)
    assert np.abs(to_np(r.loss) - loss).max() < CE_LOSS_ABS
    assert abs(float(r.loss_mean[0]) - mean) < CE_LOSS_ABS
    assert rel_l2(to_np(r.d_hidden), dh) < 2e-2
    assert rel_l2(to_np(r.d_emb), de) < 2e-2


@pytest.mark.parametrize("mode", MODES)
def test_ce_forward_only(mgb_lib, mode):
    shape = CEShape(128, 64, 256, 96)
    inp = ce_inputs(shape, seed=1)
    h = to_device(inp["hidden"], torch.bfloat16)
    e = to_device(inp["emb"], torch.bfloat16)
    t = torch.from_numpy(inp["targets"]).to("cuda")
    r = CERunner(128, 64, 256, 96, h, e, t, want_grads=False, mode=mode)
    r.run()
    loss, _, _, _ = oracle.ce_chunked(inp["hidden"], inp["emb"], inp["targets"], 96)
    assert np.abs(to_np(r.loss) - loss).max() < CE_LOSS_ABS


_FULL = {}


def _full_size_oracle():
    """The full CE workload's inputs and the oracle's whole forward over it
    (every token's LSE and loss; about 8.6 TFLOP in float64, once per run),
    plus sampled vocab ids: 24 that are some token's target, 24 that are not."""
    if not _FULL:
        shape = CE_WORKLOADS["bf16_ce_t8192h4096v128256"]
        inp = ce_inputs(shape, seed=0)
        t0 = time.time()
        loss, lse, mean = oracle.ce_full(inp["hidden"], inp["emb"], inp["targets"])
        rng = np.random.default_rng(0)
        hit = rng.choice(np.unique(inp["targets"]), 24, replace=False)
        miss_pool = np.setdiff1d(np.arange(shape.vocab), inp["targets"])
        ids = np.sort(np.concatenate([hit, rng.choice(miss_pool, 24, replace=False)]))
        d_emb_rows = oracle.ce_emb_rows(inp["hidden"], inp["emb"], inp["targets"], lse,
                                        1.0 / shape.tokens, ids)
        print(f"oracle full CE forward + {len(ids)} d_emb rows {time.time() - t0:.1f}s")
        _FULL.update(shape=shape, inp=inp, loss=loss, lse=lse, mean=mean, ids=ids,
                     d_emb_rows=d_emb_rows)
    return _FULL


@pytest.mark.slow
@pytest.mark.parametrize("mode", MODES)
def test_ce_full_size_sampled(mgb_lib, mode):
    """Full tied-embedding CE workload against the oracle: every token's loss
    and LSE and the mean loss (the oracle's whole forward); sampled tokens'
    d_hidden rows (one row at a time); sampled d_emb rows, ids that are some
    token's target and ids that are none (each needs every token's LSE)."""
    f = _full_size_oracle()
    shape, inp = f["shape"], f["inp"]
    r = _runner(shape, inp, mode)
    r.run()
    assert mgb.mgb_device_status() == mgb.MGB_OK
    assert np.abs(to_np(r.loss) - f["loss"]).max() < CE_LOSS_ABS
    assert np.abs(to_np(r.lse) - f["lse"]).max() < CE_LOSS_ABS
    assert abs(float(r.loss_mean[0]) - f["mean"]) < CE_LOSS_ABS
    rows = np.random.default_rng(0).choice(shape.tokens, 48, replace=False)
    _, _, dh = oracle.ce_rows(inp["hidden"][rows], inp["emb"], inp["targets"][rows],
                              1.0 / shape.tokens)
    assert rel_l2(to_np(r.d_hidden)[rows], dh) < 2e-2
    assert rel_l2(to_np(r.d_emb[torch.from_numpy(f["ids"]).cuda()]), f["d_emb_rows"]) < 2e-2


def test_ce_modes_agree_and_are_deterministic(mgb_lib):
    """The modes agree to float32 rounding, and each repeats bit for bit
    (the blocked mode with two token blocks)."""
    shape = CEShape(384, 256, 2000, 704)
    inp = ce_inputs(shape, seed=9)
    outs = []
    for mode in MODES:
        r = _runner(shape, inp, mode, token_block=256)
        r.run()
        first = (r.loss.clone(), r.d_hidden.clone(), r.d_emb.clone())
        r.run()
        assert torch.equal(first[0], r.loss) and torch.equal(first[1], r.d_hidden)
        assert torch.equal(first[2], r.d_emb)
        outs.append(first)
    for o in outs[1:]:
        assert float((outs[0][0] - o[0]).abs().max()) < CE_LOSS_ABS
        assert rel_l2(to_np(outs[0][1]), to_np(o[1])) < 2e-2
        assert rel_l2(to_np(outs[0][2]), to_np(o[2])) < 2e-2


def test_ce_resident_emb_stream(mgb_lib):
    """Resident mode with d_emb left on a caller's stream: after joining it the
    results equal those of the joined call bit for bit, while the caller's
    stream went on with other work (here: a GEMM reading d_hidden)."""
    shape = CEShape(384, 256, 2000, 704)
    inp = ce_inputs(shape, seed=13)
    r0 = _runner(shape, inp, mgb.MGB_CE_RESIDENT)
    r0.run()
    side = torch.cuda.Stream()
    h = to_device(inp["hidden"], torch.bfloat16)
    e = to_device(inp["emb"], torch.bfloat16)
    t = torch.from_numpy(inp["targets"]).to("cuda")
    r1 = CERunner(shape.tokens, shape.hidden, shape.vocab, shape.chunk, h, e, t,
                  mode=mgb.MGB_CE_RESIDENT, emb_stream=side)
    main = torch.cuda.current_stream()
    r1.run(main)
    after = r1.d_hidden.float() * 2  # work on the caller's stream meanwhile
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert mgb.mgb_device_status() == mgb.MGB_OK
    assert torch.equal(r0.d_emb, r1.d_emb) and torch.equal(r0.d_hidden, r1.d_hidden)
    assert torch.equal(r0.loss, r1.loss)
    assert torch.equal(after, r0.d_hidden.float() * 2)

"""Out-of-bounds write checks for every entry point (compute-sanitizer is not
available on these GPUs): each output and workspace buffer sits between two
guard regions filled with a byte pattern inside one allocation, and the
guards must come back unchanged. The shapes have ragged edges (rows, columns,
sequence lengths and vocab chunks that are not multiples of the tiles), where
an epilogue or a padded plane could write past the end."""
import numpy as np
import pytest
import torch

from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import CEShape, LayerShape, ce_inputs, layer_inputs
from megatron_transformer_layer_fwd_gb300.runner import WEIGHT_KEYS, to_device
from tests.util import Guarded

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(77)


def _rand(shape, dtype=torch.bfloat16, scale=1.0):
    return (torch.from_numpy(RNG.standard_normal(shape).astype(np.float32)) * scale).to("cuda", dtype)


@pytest.mark.parametrize("tma_out", ["0", "1"])
@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("epi", range(7))
def test_gemm_epilogues_stay_in_bounds(mgb_lib, monkeypatch, tma_out, pair, a_mn, b_mn, epi):
    """Every fused epilogue on both tile kinds, M / N / K ragged, with the
    bf16 outputs stored by each thread and through TMA boxes (clipped at the
    edges by the copy)."""
    monkeypatch.setenv("MGB_GEMM_PAIR", pair)
    monkeypatch.setenv("MGB_GEMM_TMA_OUT", tma_out)
    M, N, K = 328, 200 if epi != mgb.MGB_EPI_BIAS_SWIGLU else 256, 136
    if epi == mgb.MGB_EPI_DSWIGLU:
        N = 192
    g = Guarded()
    a = _rand((K, M) if a_mn else (M, K))
    b = _rand((K, N) if b_mn else (N, K))
    bias = _rand((N,), scale=0.1)
    ldc2 = N // 2 if epi == mgb.MGB_EPI_BIAS_SWIGLU else N
    c_dt = torch.float32 if epi == mgb.MGB_EPI_F32 else torch.bfloat16
    c_cols = 2 * N if epi == mgb.MGB_EPI_DSWIGLU else N
    c = g.empty((M, c_cols), c_dt)
    c2 = g.empty((M, ldc2), torch.bfloat16) if epi in (mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU,
                                                        mgb.MGB_EPI_F32) else None
    resid = _rand((M, N)) if epi == mgb.MGB_EPI_BIAS_RESID else None
    aux = None
    if epi == mgb.MGB_EPI_DGELU:
        aux = _rand((M, N))
    elif epi == mgb.MGB_EPI_DSWIGLU:
        aux = _rand((M, 2 * N))
    use_bias = epi in (mgb.MGB_EPI_STORE, mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU,
                       mgb.MGB_EPI_BIAS_RESID, mgb.MGB_EPI_F32)
    d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=a_mn, b_major=b_mn,
                                      lda=M if a_mn else K, ldb=N if b_mn else K, ldc=c_cols,
                                      dtype=mgb.MGB_BF16, c_f32=0, accumulate=0, alpha=1.0),
                       epilogue=epi, glu_block=64, ldc2=ldc2, ldr=N,
                       ldaux=2 * N if epi == mgb.MGB_EPI_DSWIGLU else N)
    mgb.mgb_gemm_ex(d, a, b, bias if use_bias else None, c, c2=c2, resid=resid, aux=aux)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


@pytest.mark.parametrize("B,S,nq,nkv,d,causal", [(2, 130, 4, 2, 128, True), (1, 257, 2, 2, 64, False),
                                                 (3, 70, 8, 1, 64, True)])
def test_attention_stays_in_bounds(mgb_lib, B, S, nq, nkv, d, causal):
    """Ragged sequence lengths: outputs, LSE, the three gradients and the
    padded per-query workspace planes."""
    g = Guarded()
    q = _rand((B * S, nq * d))
    k = _rand((B * S, nkv * d))
    v = _rand((B * S, nkv * d))
    o = g.empty((B * S, nq * d), torch.bfloat16)
    lse = g.empty((B, nq, S), torch.float32)
    mgb.mgb_attention_fwd(B, S, nq, nkv, d, int(causal), mgb.MGB_BF16, q, k, v, nq * d, nkv * d, o, lse)
    do = _rand((B * S, nq * d))
    dq = g.empty((B * S, nq * d), torch.bfloat16)
    dk = g.empty((B * S, nkv * d), torch.bfloat16)
    dv = g.empty((B * S, nkv * d), torch.bfloat16)
    ws = g.empty((mgb.mgb_attention_bwd_ws_bytes(B, S, nq),), torch.uint8)
    mgb.mgb_attention_bwd(B, S, nq, nkv, d, int(causal), mgb.MGB_BF16, q, k, v, nq * d, nkv * d, o,
                          lse, do, nq * d, dq, dk, dv, nq * d, nkv * d, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


@pytest.mark.parametrize("mode", [mgb.MGB_CE_STREAM, mgb.MGB_CE_FUSED, mgb.MGB_CE_RESIDENT,
                                  mgb.MGB_CE_BLOCKED])
@pytest.mark.parametrize("T,H,V,C", [(300, 256, 1000, 136), (130, 64, 520, 64)])
def test_ce_stays_in_bounds(mgb_lib, mode, T, H, V, C):
    """Ragged tokens and vocab chunks: per-token outputs, both gradients and
    the whole workspace (logits, partial planes, accumulators; the blocked
    mode with 256-token blocks, the last one ragged). The vocab chunks of the
    second shape are multiples of 32, so its kept logits go out through TMA."""
    shape = CEShape(T, H, V, C)
    inp = ce_inputs(shape, seed=2)
    h = to_device(inp["hidden"], torch.bfloat16)
    e = to_device(inp["emb"], torch.bfloat16)
    t = torch.from_numpy(inp["targets"]).to("cuda")
    desc = mgb.ce_desc(T, H, V, C, 1.0 / T, mode, token_block=256)
    g = Guarded()
    ws = g.empty((mgb.mgb_vocab_ce_sizes(desc),), torch.uint8)
    loss, lse = g.empty((T,), torch.float32), g.empty((T,), torch.float32)
    mean = g.empty((1,), torch.float32)
    dh, de = g.like(h), g.like(e)
    mgb.mgb_vocab_ce_fwd_bwd(desc, h, e, t, loss, mean, lse, dh, de, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


@pytest.mark.parametrize("dtype", [mgb.MGB_BF16, mgb.MGB_F32])
def test_layernorm_stays_in_bounds(mgb_lib, dtype):
    rows, cols = 333, 1032
    td = torch.bfloat16 if dtype == mgb.MGB_BF16 else torch.float32
    g = Guarded()
    x, gm, bt = _rand((rows, cols), td), _rand((cols,), td), _rand((cols,), td)
    y, mu, rs = g.empty((rows, cols), td), g.empty((rows,), torch.float32), g.empty((rows,), torch.float32)
    mgb.mgb_layernorm_fwd(rows, cols, dtype, 1e-5, x, gm, bt, y, mu, rs)
    dy = _rand((rows, cols), td)
    dx, dg, db = g.empty((rows, cols), td), g.empty((cols,), td), g.empty((cols,), td)
    ws = g.empty((mgb.mgb_layernorm_bwd_ws_bytes(rows, cols),), torch.uint8)
    mgb.mgb_layernorm_bwd(rows, cols, dtype, x, mu, rs, gm, dy, None, dx, dg, db, ws)
    dx2, dg2, db2 = g.empty((rows, cols), td), g.empty((cols,), td), g.empty((cols,), td)
    mgb.mgb_layernorm_bwd_noalloc(rows, cols, dtype, x, mu, rs, gm, dy, dy, dx2, dg2, db2)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


@pytest.mark.parametrize("shape", [
    LayerShape(2, 100, 256, 4, 2, 64, 520, causal=True),
    LayerShape(1, 130, 256, 4, 2, 128, 384, act="swiglu", causal=True),
    LayerShape(1, 96, 128, 2, 2, 64, 256, norm_pos="post"),
    LayerShape(2, 40, 64, 2, 2, 32, 128, dtype="f32", causal=True),
], ids=["gelu_gqa", "swiglu_gqa", "post_ln", "f32"])
def test_layer_stays_in_bounds(mgb_lib, shape):
    """The whole layer: y, the saved buffer, dx, every gradient and the
    backward workspace."""
    arr = layer_inputs(shape, seed=8, random_affine=True, random_dy=True)
    td = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    desc = mgb.block_desc(shape)
    w = {k: (to_device(arr[k], td) if arr.get(k) is not None else None) for k in WEIGHT_KEYS}
    x = to_device(arr["x"], td)
    dy = to_device(arr["dy"], td)
    saved_b, fwd_b, bwd_b = mgb.mgb_block_sizes(desc)
    g = Guarded()
    saved = g.empty((saved_b,), torch.uint8)
    fws = g.empty((fwd_b,), torch.uint8) if fwd_b > 0 else None  # float32: split operands
    ws = g.empty((max(bwd_b, 16),), torch.uint8)
    y, dx = g.like(x), g.like(x)
    grads = {k: (g.like(v) if v is not None else None) for k, v in w.items()}
    mgb.mgb_block_fwd(desc, w, x, y, saved, fws)
    mgb.mgb_block_bwd(desc, w, x, dy, saved, dx, grads, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


def test_embedding_stays_in_bounds(mgb_lib):
    T, H, v0, v1 = 333, 136, 100, 700
    ids = torch.from_numpy(RNG.integers(0, 800, T).astype(np.int32)).cuda()
    shard = _rand((v1 - v0, H))
    g = Guarded()
    out = g.empty((T, H), torch.bfloat16)
    mgb.mgb_embedding_fwd(T, H, v0, v1, mgb.MGB_BF16, ids, shard, out)
    d_emb = g.empty((v1 - v0, H), torch.bfloat16)
    ws = g.empty((mgb.mgb_embedding_bwd_ws_bytes(T, v0, v1),), torch.uint8)
    mgb.mgb_embedding_bwd(T, H, v0, v1, mgb.MGB_BF16, ids, _rand((T, H)), d_emb, 0, ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


@pytest.mark.parametrize("epi", [mgb.MGB_EPI_STORE, mgb.MGB_EPI_F32, mgb.MGB_EPI_BIAS_RESID])
def test_gemm_f32_tc_stays_in_bounds(mgb_lib, epi):
    """The three-TF32 float32 GEMM: output and the split-operand scratch."""
    M, N, K = 200, 136, 70
    g = Guarded()
    a = _rand((K, M), torch.float32)
    b = _rand((N, K), torch.float32)
    c = g.empty((M, N), torch.float32, fill=0.0)
    ws = g.empty((mgb.mgb_gemm_f32_tc_ws_bytes(M, N, K),), torch.uint8)
    d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=1, b_major=0, lda=M, ldb=K, ldc=N,
                                      dtype=mgb.MGB_F32, c_f32=0, accumulate=0, alpha=1.0),
                       epilogue=epi, glu_block=64, ldc2=N, ldr=N, ldaux=N)
    resid = _rand((M, N), torch.float32) if epi == mgb.MGB_EPI_BIAS_RESID else None
    mgb.mgb_gemm_f32_tc(d, a, b, None, c, resid=resid, ws=ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    g.check()


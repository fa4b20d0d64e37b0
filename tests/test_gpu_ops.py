"""GPU parity of the building blocks through the C ABI: the tcgen05 GEMM in
every operand layout, the float32 GEMM, LayerNorm and the attention core,
against the float64 oracle (or, for the plain product, numpy's matmul of the
same bf16-rounded operands)."""
import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import round_to_bf16
from tests.util import rel_l2, to_np

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(2024)


def _bf16(shape, scale=1.0):
    return round_to_bf16(RNG.standard_normal(shape) * scale)


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda", dtype)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (328, 200, 136), (256, 520, 1000), (1000, 1304, 64)])
def test_gemm_bf16_layouts_f32_out(mgb_lib, monkeypatch, pair, a_mn, b_mn, M, N, K):
    """Every operand layout on one SM (128-row tiles) and on a CTA pair
    (256 x 256 tiles): ragged M, N and K; a pair whose second CTA has no rows."""
    monkeypatch.setenv("MGB_GEMM_PAIR", pair)
    A = _bf16((M, K))
    B = _bf16((N, K))
    a_st = A.T.copy() if a_mn else A
    b_st = B.T.copy() if b_mn else B
    c = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32)
    d = mgb.GemmDesc(m=M, n=N, k=K, a_major=a_mn, b_major=b_mn, lda=a_st.shape[1], ldb=b_st.shape[1],
                     ldc=N, dtype=mgb.MGB_BF16, c_f32=1, accumulate=0, alpha=1.0)
    mgb.mgb_gemm(d, _dev(a_st, torch.bfloat16), _dev(b_st, torch.bfloat16), None, c)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    ref = A @ B.T
    err = rel_l2(to_np(c), ref)
    assert err < 1e-5, err


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("M,N,K", [(384, 768, 256), (200, 136, 72)])
def test_gemm_bf16_bias_out_and_accumulate(mgb_lib, monkeypatch, pair, M, N, K):
    monkeypatch.setenv("MGB_GEMM_PAIR", pair)
    A, B, bias = _bf16((M, K)), _bf16((N, K)), _bf16((N,))
    c = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    d = mgb.GemmDesc(m=M, n=N, k=K, a_major=0, b_major=0, lda=K, ldb=K, ldc=N, dtype=mgb.MGB_BF16,
                     c_f32=0, accumulate=0, alpha=0.5)
    mgb.mgb_gemm(d, _dev(A, torch.bfloat16), _dev(B, torch.bfloat16), _dev(bias, torch.bfloat16), c)
    ref = 0.5 * (A @ B.T) + bias
    assert rel_l2(to_np(c), ref) < 4e-3
    # float32 accumulate: C = C + A B^T
    c32 = _dev(ref, torch.float32)
    d.c_f32, d.accumulate, d.alpha = 1, 1, 1.0
    mgb.mgb_gemm(d, _dev(A, torch.bfloat16), _dev(B, torch.bfloat16), None, c32)
    assert rel_l2(to_np(c32), ref + A @ B.T) < 1e-5
    assert mgb.mgb_device_status() == mgb.MGB_OK


def _f32(shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 128, 32), (200, 136, 70), (300, 520, 1000)])
def test_gemm_f32_tc_layouts(mgb_lib, a_mn, b_mn, M, N, K):
    """The float32 product as three TF32 tensor-core products (hi/lo operand
    splits): every operand layout, ragged M, N and K (K not a multiple of the
    32-wide K block nor of 4), against the float64 product of the same float32
    operands: about 1e-6 at K = 1000 with the accumulator promoted to float32
    registers every 128 K (the tensor core's own accumulation alone gives about
    7e-6 there, one TF32 product about 3e-4)."""
    A, B = _f32((M, K)), _f32((N, K))
    a_st = A.T.copy() if a_mn else A
    b_st = B.T.copy() if b_mn else B
    c = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32)
    ws = torch.empty(mgb.mgb_gemm_f32_tc_ws_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=a_mn, b_major=b_mn, lda=a_st.shape[1],
                                      ldb=b_st.shape[1], ldc=N, dtype=mgb.MGB_F32, c_f32=0,
                                      accumulate=0, alpha=1.0),
                       epilogue=mgb.MGB_EPI_STORE, glu_block=16, ldc2=0, ldr=0, ldaux=0)
    mgb.mgb_gemm_f32_tc(d, _dev(a_st, torch.float32), _dev(b_st, torch.float32), None, c, ws=ws)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    err = rel_l2(to_np(c), A @ B.T)
    assert err < 3e-6, err


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("M,N,K", [(328, 256, 136), (1000, 1280, 200)])
@pytest.mark.parametrize("epi,gb", [(mgb.MGB_EPI_STORE, 0), (mgb.MGB_EPI_BIAS_GELU, 0),
                                    (mgb.MGB_EPI_BIAS_SWIGLU, 128), (mgb.MGB_EPI_BIAS_SWIGLU, 64),
                                    (mgb.MGB_EPI_BIAS_RESID, 0), (mgb.MGB_EPI_DGELU, 0),
                                    (mgb.MGB_EPI_DSWIGLU, 64)])
def test_gemm_tma_out_equals_thread_stores(mgb_lib, monkeypatch, pair, M, N, K, epi, gb):
    """The bf16 epilogues with their outputs staged in shared memory and
    stored by TMA boxes give the same bits as the per-thread stores (the same
    arithmetic; only the store path differs), ragged rows included."""
    monkeypatch.setenv("MGB_GEMM_PAIR", pair)
    a, b = _dev(_bf16((M, K)), torch.bfloat16), _dev(_bf16((N, K)), torch.bfloat16)
    bias = _dev(_bf16((N,), 0.1), torch.bfloat16)
    resid = _dev(_bf16((M, N)), torch.bfloat16)
    w_c = 2 * N if epi == mgb.MGB_EPI_DSWIGLU else N
    w_c2 = N // 2 if epi == mgb.MGB_EPI_BIAS_SWIGLU else N
    aux = _dev(_bf16((M, w_c)), torch.bfloat16)
    outs = []
    for tma in ("0", "1"):
        monkeypatch.setenv("MGB_GEMM_TMA_OUT", tma)
        c = torch.full((M, w_c), float("nan"), device="cuda", dtype=torch.bfloat16)
        c2 = torch.full((M, w_c2), float("nan"), device="cuda", dtype=torch.bfloat16)
        d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=0, b_major=0, lda=K, ldb=K,
                                          ldc=w_c, dtype=mgb.MGB_BF16, c_f32=0, accumulate=0,
                                          alpha=1.0),
                           epilogue=epi, glu_block=gb or 16, ldc2=w_c2, ldr=N, ldaux=w_c)
        two = epi in (mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU)
        has_bias = epi not in (mgb.MGB_EPI_DGELU, mgb.MGB_EPI_DSWIGLU)
        mgb.mgb_gemm_ex(d, a, b, bias if has_bias else None, c, c2=c2 if two else None,
                        resid=resid if epi == mgb.MGB_EPI_BIAS_RESID else None,
                        aux=aux if epi in (mgb.MGB_EPI_DGELU, mgb.MGB_EPI_DSWIGLU) else None)
        assert mgb.mgb_device_status() == mgb.MGB_OK
        outs.append((c.clone(), c2.clone() if two else None))
    assert not torch.isnan(outs[1][0].float()).any()
    assert torch.equal(outs[0][0], outs[1][0])
    if outs[0][1] is not None:
        assert not torch.isnan(outs[1][1].float()).any()
        assert torch.equal(outs[0][1], outs[1][1])


def test_gemm_f32_tc_promotion_long_k(mgb_lib, monkeypatch):
    """At K = 4100 the chunked float32 promotion keeps the 3xTF32 product near
    FFMA accuracy, where one accumulation over the whole K (MGB_TF32_CHUNK=0)
    drifts several times further from the float64 product."""
    M, N, K = 256, 192, 4100
    A, B = _f32((M, K)), _f32((N, K))
    ref = A @ B.T
    errs = {}
    for chunk in ("4", "0"):
        monkeypatch.setenv("MGB_TF32_CHUNK", chunk)
        c = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32)
        ws = torch.empty(mgb.mgb_gemm_f32_tc_ws_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=0, b_major=0, lda=K, ldb=K, ldc=N,
                                          dtype=mgb.MGB_F32, c_f32=0, accumulate=0, alpha=1.0),
                           epilogue=mgb.MGB_EPI_STORE, glu_block=16, ldc2=0, ldr=0, ldaux=0)
        mgb.mgb_gemm_f32_tc(d, _dev(A, torch.float32), _dev(B, torch.float32), None, c, ws=ws)
        assert mgb.mgb_device_status() == mgb.MGB_OK
        errs[chunk] = rel_l2(to_np(c), ref)
    assert errs["4"] < 3e-6, errs
    assert errs["4"] < errs["0"], errs


@pytest.mark.parametrize("epi", [mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU, mgb.MGB_EPI_BIAS_RESID,
                                 mgb.MGB_EPI_DGELU, mgb.MGB_EPI_DSWIGLU, mgb.MGB_EPI_F32])
def test_gemm_f32_tc_epilogues(mgb_lib, epi):
    """The layer's fused epilogues on the three-TF32 product equal the same
    epilogues on the FFMA product (both float32) to float32 rounding."""
    M, N, K = 130, 96, 72
    gb = 16
    A, B, bias = _f32((M, K)), _f32((N, K)), _f32((N,), 0.1)
    w_out = {mgb.MGB_EPI_DSWIGLU: 2 * N}.get(epi, N)
    aux = _f32((M, 2 * N if epi == mgb.MGB_EPI_DSWIGLU else N))
    resid = _f32((M, N))
    outs = []
    for tc in (True, False):
        c = torch.zeros((M, w_out), device="cuda", dtype=torch.float32)
        if epi == mgb.MGB_EPI_F32:
            c.copy_(_dev(resid, torch.float32))
        c2 = torch.zeros((M, N // 2 if epi == mgb.MGB_EPI_BIAS_SWIGLU else N), device="cuda",
                         dtype=torch.float32)
        d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=0, b_major=0, lda=K, ldb=K,
                                          ldc=w_out, dtype=mgb.MGB_F32, c_f32=0,
                                          accumulate=int(epi == mgb.MGB_EPI_F32), alpha=1.0),
                           epilogue=epi, glu_block=gb, ldc2=c2.shape[1], ldr=N, ldaux=aux.shape[1])
        has_bias = epi in (mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU, mgb.MGB_EPI_BIAS_RESID,
                           mgb.MGB_EPI_F32)
        args = (d, _dev(A, torch.float32), _dev(B, torch.float32),
                _dev(bias, torch.float32) if has_bias else None, c)
        kw = dict(c2=c2 if epi in (mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU) else None,
                  resid=_dev(resid, torch.float32) if epi == mgb.MGB_EPI_BIAS_RESID else None,
                  aux=_dev(aux, torch.float32) if epi in (mgb.MGB_EPI_DGELU, mgb.MGB_EPI_DSWIGLU)
                  else None)
        if tc:
            ws = torch.empty(mgb.mgb_gemm_f32_tc_ws_bytes(M, N, K), dtype=torch.uint8, device="cuda")
            mgb.mgb_gemm_f32_tc(*args, ws=ws, **kw)
        else:
            mgb.mgb_gemm_ex(*args, **kw)
        outs.append((to_np(c), to_np(c2)))
    assert mgb.mgb_device_status() == mgb.MGB_OK
    assert rel_l2(outs[0][0], outs[1][0]) < 1e-5
    if epi in (mgb.MGB_EPI_BIAS_GELU, mgb.MGB_EPI_BIAS_SWIGLU):
        assert rel_l2(outs[0][1], outs[1][1]) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
def test_gemm_pair_tiles_many_waves(mgb_lib, a_mn, b_mn):
    """Large enough for the CTA-pair tile to be chosen by itself, with more
    tiles than resident pairs (each pair walks several tiles and reuses both
    TMEM accumulators) and ragged edges in M and N."""
    M, N, K = 2320, 4360, 320
    A = _bf16((M, K))
    B = _bf16((N, K))
    a_st = A.T.copy() if a_mn else A
    b_st = B.T.copy() if b_mn else B
    c = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32)
    d = mgb.GemmDesc(m=M, n=N, k=K, a_major=a_mn, b_major=b_mn, lda=a_st.shape[1], ldb=b_st.shape[1],
                     ldc=N, dtype=mgb.MGB_BF16, c_f32=1, accumulate=0, alpha=1.0)
    mgb.mgb_gemm(d, _dev(a_st, torch.bfloat16), _dev(b_st, torch.bfloat16), None, c)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    err = rel_l2(to_np(c), A @ B.T)
    assert err < 1e-5, err


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
def test_gemm_f32_simt(mgb_lib, a_mn, b_mn):
    M, N, K = 100, 72, 200
    A, B = RNG.standard_normal((M, K)), RNG.standard_normal((N, K))
    a_st = A.T.copy() if a_mn else A
    b_st = B.T.copy() if b_mn else B
    c = torch.empty((M, N), device="cuda", dtype=torch.float32)
    d = mgb.GemmDesc(m=M, n=N, k=K, a_major=a_mn, b_major=b_mn, lda=a_st.shape[1], ldb=b_st.shape[1],
                     ldc=N, dtype=mgb.MGB_F32, c_f32=1, accumulate=0, alpha=1.0)
    mgb.mgb_gemm(d, _dev(a_st, torch.float32), _dev(b_st, torch.float32), None, c)
    assert rel_l2(to_np(c), A.astype(np.float32).astype(np.float64) @ B.astype(np.float32).T) < 1e-6


def test_gemm_zero_k_writes_bias_only(mgb_lib):
    M, N = 130, 64
    bias = _bf16((N,))
    c = torch.full((M, N), 7.0, device="cuda", dtype=torch.bfloat16)
    d = mgb.GemmDesc(m=M, n=N, k=0, a_major=0, b_major=0, lda=8, ldb=8, ldc=N, dtype=mgb.MGB_BF16,
                     c_f32=0, accumulate=0, alpha=1.0)
    dummy = torch.zeros(64, device="cuda", dtype=torch.bfloat16)
    mgb.mgb_gemm(d, dummy, dummy, _dev(bias, torch.bfloat16), c)
    np.testing.assert_array_equal(to_np(c), np.broadcast_to(bias, (M, N)))


@pytest.mark.parametrize("kernel", ["tma", "warp", "block"])
@pytest.mark.parametrize("dtype,rows,cols", [("bf16", 300, 1024), ("bf16", 7, 4096), ("f32", 64, 256),
                                             ("bf16", 5000, 4096), ("bf16", 1000, 256),
                                             ("bf16", 333, 2048), ("bf16", 40, 1032)])
def test_layernorm_fwd(mgb_lib, monkeypatch, kernel, dtype, rows, cols):
    """Each forward kernel (rows streamed into shared memory by bulk copies,
    one warp per row with register prefetch, one block per row): many rows per
    CTA (the shared-memory ring refilled several times), few rows, and widths
    only the block kernel takes."""
    monkeypatch.setenv("MGB_LN_KERNEL", kernel)
    x = RNG.standard_normal((rows, cols)) * 2 + 0.5
    g, b = 1 + 0.1 * RNG.standard_normal(cols), 0.1 * RNG.standard_normal(cols)
    if dtype == "bf16":
        x, g, b = round_to_bf16(x), round_to_bf16(g), round_to_bf16(b)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    y = torch.empty((rows, cols), device="cuda", dtype=td)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    mgb.mgb_layernorm_fwd(rows, cols, mgb.MGB_BF16 if dtype == "bf16" else mgb.MGB_F32, 1e-5,
                          _dev(x, td), _dev(g, td), _dev(b, td), y, mean, rstd)
    ry, rm, rr = oracle.ln_fwd(x, g, b, 1e-5)
    assert rel_l2(to_np(y), ry) < (5e-3 if dtype == "bf16" else 1e-6)
    assert rel_l2(to_np(mean), rm) < 1e-6 and rel_l2(to_np(rstd), rr) < 1e-6


@pytest.mark.parametrize("B,S,nq,nkv,d,causal", [
    (1, 64, 1, 1, 64, False), (2, 100, 4, 2, 64, True), (1, 200, 4, 1, 128, False),
    (2, 130, 2, 2, 128, True)])
def test_attention_fwd_bf16(mgb_lib, B, S, nq, nkv, d, causal):
    q = _bf16((B, nq, S, d))
    k = _bf16((B, nkv, S, d))
    v = _bf16((B, nkv, S, d))
    pack = lambda t: t.transpose(0, 2, 1, 3).reshape(B * S, -1)
    qkv = np.concatenate([pack(q), pack(k), pack(v)], axis=1)
    tq = _dev(qkv, torch.bfloat16)
    W = qkv.shape[1]
    o = torch.empty((B * S, nq * d), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((B, nq, S), device="cuda", dtype=torch.float32)
    e = 2
    mgb.mgb_attention_fwd(B, S, nq, nkv, d, causal, mgb.MGB_BF16, tq, tq[:, nq * d:],
                          tq[:, (nq + nkv) * d:], W, W, o, lse)
    ro, rl = oracle.attention_fwd(q, k, v, causal)
    assert rel_l2(to_np(o), pack(ro)) < 1e-2
    assert rel_l2(to_np(lse), rl) < 1e-3


def test_device_wait_timeout_is_reported(mgb_lib):
    """A bounded wait on a barrier nobody arrives on returns a timeout status
    (no hang, no fault) and the context stays usable."""
    assert mgb.mgb_device_status() == mgb.MGB_OK
    mgb.mgb_selftest_wait_timeout(20_000_000)          # 20 ms
    assert mgb.mgb_device_status() == mgb.MGB_ERR_DEVICE_TIMEOUT
    assert mgb.mgb_device_status() == mgb.MGB_OK        # cleared
    x = torch.ones(16, device="cuda")
    assert float(x.sum()) == 16.0

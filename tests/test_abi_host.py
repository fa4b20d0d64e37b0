"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/mgb.h declares, and rejects bad arguments with the
documented status before touching a device."""
import ctypes
import os

import pytest

from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import WORKLOADS, LayerShape


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mgb.LIB_PATH):
        from megatron_transformer_layer_fwd_gb300 import build
        build.build()
    return mgb.load()


def test_library_exports_every_header_function(lib):
    names = mgb.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(-8, 1):
        assert mgb.status_string(s) not in ("", "unknown status")
    assert mgb.status_string(-99) == "unknown status"


def _desc(**kw):
    return mgb.block_desc(WORKLOADS["bf16_preln_b4s512h1024"].replace(**kw))


@pytest.mark.parametrize("kw,status", [
    (dict(n_kv_heads=3), mgb.MGB_ERR_INVALID_ARG),          # nq % nkv != 0
    (dict(seq=0), mgb.MGB_ERR_INVALID_ARG),
    (dict(batch=-1), mgb.MGB_ERR_INVALID_ARG),
    (dict(head_dim=96), mgb.MGB_ERR_UNSUPPORTED),           # bf16 path: d in {64, 128}
    (dict(hidden=1020), mgb.MGB_ERR_MISALIGNED),             # rows must be 16-byte multiples
    (dict(act="swiglu", ffn=4800, glu_block=48), mgb.MGB_ERR_UNSUPPORTED),
    (dict(act="swiglu", ffn=4000, glu_block=128), mgb.MGB_ERR_INVALID_ARG),
    (dict(ln_eps=-1.0), mgb.MGB_ERR_INVALID_ARG),
])
def test_block_sizes_rejects_bad_descriptors(lib, kw, status):
    d = _desc(**kw)
    s = ctypes.c_size_t()
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == status


def test_block_sizes_cover_saved_activations(lib):
    shape = WORKLOADS["bf16_gqa_swiglu_b2s4096h4096"]
    saved, fwd, bwd = mgb.mgb_block_sizes(mgb.block_desc(shape))
    T, H = shape.tokens, shape.hidden
    # at least: qkv, O, h, u (2F), a (F) in bf16
    floor = 2 * T * (shape.qkv_width + shape.n_q_heads * shape.head_dim + H + 3 * shape.ffn)
    assert saved >= floor and fwd == 0 and bwd > 0


def test_bwd_workspace_holds_the_fused_bias_partials(lib):
    """bf16 with biases: the backward workspace also holds the fc1 bias
    gradient's float32 partial sums, one row of 2F (SwiGLU) or F columns per
    32 tokens, which the fp32 path and bias-free layers do without."""
    shape = WORKLOADS["bf16_gqa_swiglu_b2s4096h4096"]
    d = mgb.block_desc(shape)
    with_bias = mgb.mgb_block_sizes(d)[2]
    d.has_bias = 0
    without = mgb.mgb_block_sizes(d)[2]
    rows = (shape.tokens + 31) // 32
    assert with_bias - without >= 4 * rows * 2 * shape.ffn
    # no tokens: still one zeroed row
    d0 = mgb.block_desc(shape)
    d0.batch = 0
    b0 = mgb.mgb_block_sizes(d0)[2]
    d0.has_bias = 0
    assert b0 - mgb.mgb_block_sizes(d0)[2] >= 4 * 2 * shape.ffn


def test_fwd_argument_errors_before_any_launch(lib):
    d = _desc()
    w = mgb.BlockWeights()
    # missing weights
    assert lib.mgb_block_fwd(ctypes.byref(d), ctypes.byref(w), 16, 16, 16, 1 << 40, None, 0,
                             None) == mgb.MGB_ERR_INVALID_ARG
    # misaligned x
    w = mgb.BlockWeights(**{k: 4096 for k in mgb._WEIGHT_FIELDS})
    assert lib.mgb_block_fwd(ctypes.byref(d), ctypes.byref(w), 4097, 4096, 4096, 1 << 40, None, 0,
                             None) == mgb.MGB_ERR_MISALIGNED
    # saved buffer too small
    assert lib.mgb_block_fwd(ctypes.byref(d), ctypes.byref(w), 4096, 4096, 4096, 16, None, 0,
                             None) == mgb.MGB_ERR_WORKSPACE_TOO_SMALL
    # biases present although has_bias = 0
    d0 = _desc(has_bias=False)
    assert lib.mgb_block_fwd(ctypes.byref(d0), ctypes.byref(w), 4096, 4096, 4096, 1 << 40, None, 0,
                             None) == mgb.MGB_ERR_INVALID_ARG


def test_bwd_workspace_too_small(lib):
    d = _desc()
    w = mgb.BlockWeights(**{k: 4096 for k in mgb._WEIGHT_FIELDS})
    g = mgb.BlockGrads()
    assert lib.mgb_block_bwd(ctypes.byref(d), ctypes.byref(w), 4096, 4096, 4096, 1 << 40, 4096,
                             ctypes.byref(g), 4096, 16, None) == mgb.MGB_ERR_WORKSPACE_TOO_SMALL


def test_ce_validation(lib):
    ok = mgb.ce_desc(8192, 4096, 128256, 16032, 1 / 8192)
    assert mgb.mgb_vocab_ce_sizes(ok) > 2 * 8192 * 16032
    s = ctypes.c_size_t()
    bad = mgb.ce_desc(8192, 4096, 128250, 16032, 1.0)       # vocab not a multiple of 8
    assert lib.mgb_vocab_ce_sizes(ctypes.byref(bad), ctypes.byref(s)) == mgb.MGB_ERR_MISALIGNED
    f32 = mgb.CEDesc(tokens=8, hidden=8, vocab=8, chunk=8, dtype=mgb.MGB_F32, grad_scale=1.0)
    assert lib.mgb_vocab_ce_sizes(ctypes.byref(f32), ctypes.byref(s)) == mgb.MGB_ERR_UNSUPPORTED
    badmode = mgb.ce_desc(8192, 4096, 128256, 16032, 1 / 8192, mode=4)
    assert lib.mgb_vocab_ce_sizes(ctypes.byref(badmode), ctypes.byref(s)) == mgb.MGB_ERR_INVALID_ARG
    badtb = mgb.ce_desc(8192, 4096, 128256, 16032, 1 / 8192, mode=mgb.MGB_CE_BLOCKED, token_block=-1)
    assert lib.mgb_vocab_ce_sizes(ctypes.byref(badtb), ctypes.byref(s)) == mgb.MGB_ERR_INVALID_ARG
    # fused partials: one per token and 128 vocab columns (126 per 16032-wide chunk)
    fused = mgb.mgb_vocab_ce_sizes(mgb.ce_desc(8192, 4096, 128256, 16032, 1 / 8192))
    stream = mgb.mgb_vocab_ce_sizes(mgb.ce_desc(8192, 4096, 128256, 16032, 1 / 8192,
                                                mode=mgb.MGB_CE_STREAM))
    assert fused - stream >= 2 * 4 * 8192 * (8 * 126 - 8) - 4 * 8192 * 8
    # resident logits: 2 bytes per logit of the whole vocabulary, no float32
    # d_hidden accumulator
    resident = mgb.mgb_vocab_ce_sizes(mgb.ce_desc(8192, 4096, 128256, 16032, 1 / 8192,
                                                  mode=mgb.MGB_CE_RESIDENT))
    assert resident >= 2 * 8192 * 128256
    assert resident - fused == 2 * 8192 * (128256 - 16032) - 4 * 8192 * 4096


def test_ce_blocked_workspace_is_bounded_by_the_block(lib):
    """The token-blocked CE holds one block of logits [token_block, vocab] and
    a float32 [vocab, hidden] d_emb accumulator, however many tokens there
    are: its workspace does not grow with the token count (only the per-token
    LSE and loss sums do)."""
    V, H = 128256, 4096
    sizes = {T: mgb.mgb_vocab_ce_sizes(mgb.ce_desc(T, H, V, 16032, 1 / T, mode=mgb.MGB_CE_BLOCKED,
                                                    token_block=2048))
             for T in (8192, 65536)}
    assert sizes[8192] >= 2 * 2048 * V + 4 * V * H
    assert sizes[8192] < 2 * 8192 * V + 4 * V * H     # less than the whole logits beside it
    assert sizes[65536] - sizes[8192] < 16 * (65536 - 8192)  # per-token float32 arrays only
    # one block (all tokens fit): no float32 accumulator
    one = mgb.mgb_vocab_ce_sizes(mgb.ce_desc(2048, H, V, 16032, 1 / 2048, mode=mgb.MGB_CE_BLOCKED,
                                             token_block=2048))
    assert one < 2 * 2048 * V + 4 * V * H


def test_ce_default_token_block(lib):
    """token_block = 0 selects the library's default block, which the binding
    restates (the bench and the runner size their views with it)."""
    V, H, T = 128256, 4096, 16384
    size = lambda tb: mgb.mgb_vocab_ce_sizes(mgb.ce_desc(T, H, V, 16032, 1 / T,
                                                         mode=mgb.MGB_CE_BLOCKED, token_block=tb))
    assert size(0) == size(mgb.CE_DEFAULT_TOKEN_BLOCK)
    assert size(0) != size(mgb.CE_DEFAULT_TOKEN_BLOCK // 2)


def test_gemm_validation(lib):
    d = mgb.GemmDesc(m=128, n=100, k=64, a_major=0, b_major=0, lda=64, ldb=64, ldc=100,
                     dtype=mgb.MGB_BF16, c_f32=0, accumulate=0, alpha=1.0)
    assert lib.mgb_gemm(ctypes.byref(d), 4096, 4096, None, 4096, None) == mgb.MGB_ERR_MISALIGNED
    d.n, d.ldc, d.lda = 128, 128, 32                          # lda < K
    assert lib.mgb_gemm(ctypes.byref(d), 4096, 4096, None, 4096, None) == mgb.MGB_ERR_INVALID_ARG
    d.lda, d.accumulate = 64, 1                               # accumulate needs float32 C
    assert lib.mgb_gemm(ctypes.byref(d), 4096, 4096, None, 4096, None) == mgb.MGB_ERR_INVALID_ARG


def test_gemm_ex_validation(lib):
    """Fused-epilogue GEMM: every error is returned before any device work."""
    g = mgb.GemmDesc(m=256, n=256, k=64, a_major=0, b_major=0, lda=64, ldb=64, ldc=256,
                     dtype=mgb.MGB_BF16, c_f32=0, accumulate=0, alpha=1.0)
    e = mgb.GemmExDesc(g=g, epilogue=7, glu_block=128, ldc2=128, ldr=256, ldaux=256)
    call = lambda c2=4096, resid=None, aux=None: lib.mgb_gemm_ex(
        ctypes.byref(e), 4096, 4096, None, 4096, c2, resid, aux, None)
    assert call() == mgb.MGB_ERR_INVALID_ARG                 # unknown epilogue
    e.epilogue = mgb.MGB_EPI_BIAS_GELU
    assert call(c2=None) == mgb.MGB_ERR_INVALID_ARG          # GELU needs C2
    e.epilogue = mgb.MGB_EPI_BIAS_RESID
    assert call(resid=None) == mgb.MGB_ERR_INVALID_ARG       # residual input missing
    e.epilogue = mgb.MGB_EPI_DSWIGLU
    assert call(aux=None) == mgb.MGB_ERR_INVALID_ARG         # u missing
    e.epilogue, e.glu_block = mgb.MGB_EPI_BIAS_SWIGLU, 96
    assert call() in (mgb.MGB_ERR_INVALID_ARG, mgb.MGB_ERR_UNSUPPORTED)  # 256 % 192 != 0
    e.epilogue, e.glu_block = mgb.MGB_EPI_STORE, 128
    e.g.accumulate = 1                                       # accumulate needs MGB_EPI_F32
    assert call() == mgb.MGB_ERR_INVALID_ARG
    e.g.accumulate, e.g.a_major = 0, 2
    assert call() == mgb.MGB_ERR_INVALID_ARG


def test_rng_tracker_matches_the_oracle_tracker(lib):
    """Seeds of the three states, fork / restore and draws (host-only calls)."""
    from oracle import dropout as od
    t = mgb.rng_tracker(1234, tp_rank=3, ep_rank=2, etp_rank=1)
    o = od.model_parallel_seed(1234, tp_rank=3, ep_rank=2, etp_rank=1)
    assert [t.state[i].seed for i in range(3)] == [o.states[k][0] for k in (o.DATA, o.MODEL, o.EXPERT)]
    assert t.current == mgb.MGB_RNG_DATA_PARALLEL
    for n in (10, 17, 1, 0, 4096):
        r = mgb.mgb_rng_draw(t, n)
        assert (r.seed, r.offset) == o.draw(n)
    prev = mgb.mgb_rng_fork(t, mgb.MGB_RNG_MODEL_PARALLEL)
    with o.fork(o.MODEL):
        r = mgb.mgb_rng_draw(t, 33)
        assert (r.seed, r.offset) == o.draw(33)
    mgb.mgb_rng_restore(t, prev)
    assert t.current == mgb.MGB_RNG_DATA_PARALLEL
    assert lib.mgb_rng_fork(ctypes.byref(t), 3) == mgb.MGB_ERR_INVALID_ARG
    assert lib.mgb_rng_restore(ctypes.byref(t), -2) == mgb.MGB_ERR_INVALID_ARG


def test_block_dropout_plan_matches_the_oracle(lib):
    from oracle import dropout as od
    shape = LayerShape(2, 37, 64, 4, 2, 16, 96)
    d = mgb.block_desc(shape)
    t = mgb.rng_tracker(99, tp_rank=1)
    o = od.model_parallel_seed(99, tp_rank=1)
    for _ in range(2):  # two steps: the offsets move on
        mgb.mgb_block_dropout_plan(d, t)
        want = od.layer_dropout(shape, o, 0.0, 0.0)["states"]
        assert (d.rng_attn.seed, d.rng_attn.offset) == want["attn"]
        assert (d.rng_proj.seed, d.rng_proj.offset) == want["proj"]
        assert (d.rng_fc2.seed, d.rng_fc2.offset) == want["fc2"]
    assert d.rng_attn.seed == 99 + 2718 + 1 and d.rng_proj.seed == 99


def test_dropout_desc_validation(lib):
    s = ctypes.c_size_t()
    d = _desc()
    d.hidden_dropout = 1.0
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_ERR_INVALID_ARG
    d.hidden_dropout = -0.1
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_ERR_INVALID_ARG
    d.hidden_dropout = 0.999  # keeps no byte: rejected before any launch
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_ERR_INVALID_ARG
    d.hidden_dropout, d.attn_dropout = 0.0, 0.1
    s0 = mgb.mgb_block_sizes(_desc())[0]
    s1 = mgb.mgb_block_sizes(d)[0]
    assert s1 - s0 >= 4 * 4 * 16 * 512 * 512 // 32  # one keep bit per query and key
    d.rng_attn.offset = 4
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_ERR_INVALID_ARG
    d.attn_dropout, d.hidden_dropout = 0.0, 0.1
    d.rng_proj.offset = 8
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_ERR_INVALID_ARG
    d.rng_proj.offset = 16
    b0 = mgb.mgb_block_sizes(_desc())[2]
    b1 = mgb.mgb_block_sizes(d)[2]
    assert b1 > b0  # two [T, H] branch-gradient buffers
    f = _desc()
    f.dtype, f.hidden_dropout = mgb.MGB_F32, 0.1
    assert lib.mgb_block_sizes(ctypes.byref(f), ctypes.byref(s), None, None) == mgb.MGB_ERR_UNSUPPORTED
    f.hidden_dropout, f.attn_dropout = 0.0, 0.1
    assert lib.mgb_block_sizes(ctypes.byref(f), ctypes.byref(s), None, None) == mgb.MGB_ERR_UNSUPPORTED
    st = mgb.RngState(seed=1, offset=4)
    assert lib.mgb_dropout(4, 16, mgb.MGB_BF16, ctypes.c_float(0.1), st, 4096, 16, 4096, 16,
                           None) == mgb.MGB_ERR_INVALID_ARG


def test_injected_validation_fault(lib, monkeypatch):
    """MGB_FAULT=validate makes every descriptor check fail (host-side fault injection)."""
    d = _desc()
    s = ctypes.c_size_t()
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_OK
    monkeypatch.setenv("MGB_FAULT", "validate")
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_ERR_INVALID_ARG
    # the allocation-free LayerNorm backward takes the same injection, before
    # anything else (no device is needed to see it)
    p = 4096
    assert lib.mgb_layernorm_bwd_noalloc(8, 64, mgb.MGB_BF16, p, p, p, p, p, None, p, p, p,
                                         None) == mgb.MGB_ERR_INVALID_ARG
    monkeypatch.delenv("MGB_FAULT")
    assert lib.mgb_block_sizes(ctypes.byref(d), ctypes.byref(s), None, None) == mgb.MGB_OK


def test_selftest_limit_is_validated(lib):
    assert lib.mgb_selftest_wait_timeout(10 ** 10, None) == mgb.MGB_ERR_INVALID_ARG


def test_attention_bwd_workspace_size(lib):
    """Two float32 planes with rows padded to 128 queries, then the float32
    dQ accumulator [batch * seq][n_q_heads * 128]; too small a workspace is
    refused before any launch."""
    assert mgb.mgb_attention_bwd_ws_bytes(2, 4096, 32) == 2 * 4 * 2 * 32 * 4096 + 4 * 2 * 4096 * 32 * 128
    assert mgb.mgb_attention_bwd_ws_bytes(1, 130, 4) == 2 * 4 * 4 * 256 + 4 * 130 * 4 * 128
    assert mgb.mgb_attention_bwd_ws_bytes(-1, 8, 1) == 0
    need = mgb.mgb_attention_bwd_ws_bytes(1, 130, 4)
    p = 4096
    s = lib.mgb_attention_bwd(1, 130, 4, 2, 64, 1, mgb.MGB_BF16, p, p, p, 512, 512, p, p, p, 256,
                              p, p, p, 512, 512, p, need - 16, None)
    assert s == mgb.MGB_ERR_WORKSPACE_TOO_SMALL


def test_embedding_validation(lib):
    p = 4096
    # v0 >= v1, negative tokens, bad dtype: invalid before any launch
    assert lib.mgb_embedding_fwd(4, 64, 5, 5, mgb.MGB_BF16, p, p, p, None) == mgb.MGB_ERR_INVALID_ARG
    assert lib.mgb_embedding_fwd(-1, 64, 0, 5, mgb.MGB_BF16, p, p, p, None) == mgb.MGB_ERR_INVALID_ARG
    assert lib.mgb_embedding_fwd(4, 64, 0, 5, 7, p, p, p, None) == mgb.MGB_ERR_INVALID_ARG
    # hidden not a whole number of 16-byte vectors; misaligned table
    assert lib.mgb_embedding_fwd(4, 60, 0, 5, mgb.MGB_BF16, p, p, p, None) == mgb.MGB_ERR_MISALIGNED
    assert lib.mgb_embedding_fwd(4, 64, 0, 5, mgb.MGB_BF16, p, p + 8, p, None) == mgb.MGB_ERR_MISALIGNED
    # tokens present but no ids
    assert lib.mgb_embedding_fwd(4, 64, 0, 5, mgb.MGB_BF16, None, p, p, None) == mgb.MGB_ERR_INVALID_ARG
    # backward workspace: token lists + row offsets
    need = mgb.mgb_embedding_bwd_ws_bytes(100, 10, 60)
    assert need >= 4 * (2 * 100 + 2 * 50 + 1)
    assert mgb.mgb_embedding_bwd_ws_bytes(100, 10, 10) == 0
    assert lib.mgb_embedding_bwd(100, 64, 10, 60, mgb.MGB_BF16, p, p, p, 1, p, need - 16,
                                 None) == mgb.MGB_ERR_WORKSPACE_TOO_SMALL


def test_embedding_prepare_apply_validation(lib):
    """The two-step backward refuses bad arguments before any launch; the plan
    is a host struct that carries the sizes from prepare to apply."""
    import ctypes as ct
    p = 4096
    need = mgb.mgb_embedding_bwd_ws_bytes(100, 10, 60)
    plan = mgb.EmbeddingBwdPlan()
    assert ct.sizeof(plan) == 32
    prep = lib.mgb_embedding_bwd_prepare
    assert prep(100, 10, 10, p, p, need, ct.byref(plan), None) == mgb.MGB_ERR_INVALID_ARG
    assert prep(-1, 10, 60, p, p, need, ct.byref(plan), None) == mgb.MGB_ERR_INVALID_ARG
    assert prep(100, 10, 60, p, p, need, None, None) == mgb.MGB_ERR_INVALID_ARG
    assert prep(100, 10, 60, None, p, need, ct.byref(plan), None) == mgb.MGB_ERR_INVALID_ARG
    assert prep(100, 10, 60, p, None, need, ct.byref(plan), None) == mgb.MGB_ERR_INVALID_ARG
    assert prep(100, 10, 60, p, p + 8, need, ct.byref(plan), None) == mgb.MGB_ERR_MISALIGNED
    assert prep(100, 10, 60, p + 2, p, need, ct.byref(plan), None) == mgb.MGB_ERR_MISALIGNED
    assert prep(100, 10, 60, p, p, need - 16, ct.byref(plan), None) == \
        mgb.MGB_ERR_WORKSPACE_TOO_SMALL
    # nothing was filled in by the refused calls
    assert (plan.tokens, plan.v0, plan.v1, plan.ws, plan.ws_bytes) == (0, 0, 0, None, 0)
    apply = lib.mgb_embedding_bwd_apply
    assert apply(None, 64, mgb.MGB_BF16, p, p, 1, None) == mgb.MGB_ERR_INVALID_ARG
    plan.tokens, plan.v0, plan.v1, plan.ws, plan.ws_bytes = 100, 10, 60, p, need
    assert apply(ct.byref(plan), 60, mgb.MGB_BF16, p, p, 1, None) == mgb.MGB_ERR_MISALIGNED
    assert apply(ct.byref(plan), 64, 7, p, p, 1, None) == mgb.MGB_ERR_INVALID_ARG
    assert apply(ct.byref(plan), 64, mgb.MGB_BF16, None, p, 1, None) == mgb.MGB_ERR_INVALID_ARG
    assert apply(ct.byref(plan), 64, mgb.MGB_BF16, p, p + 8, 1, None) == mgb.MGB_ERR_MISALIGNED
    plan.ws_bytes = need - 16
    assert apply(ct.byref(plan), 64, mgb.MGB_BF16, p, p, 1, None) == \
        mgb.MGB_ERR_WORKSPACE_TOO_SMALL
    plan.ws_bytes, plan.ws = need, None
    assert apply(ct.byref(plan), 64, mgb.MGB_BF16, p, p, 1, None) == mgb.MGB_ERR_INVALID_ARG
    plan.ws = p + 8
    assert apply(ct.byref(plan), 64, mgb.MGB_BF16, p, p, 1, None) == mgb.MGB_ERR_MISALIGNED


def test_checking_build_exports_the_same_calls():
    """The checking build (device-side checks, -DMGB_CHECK=1) compiles and
    exports every call of the header, like the normal build."""
    import ctypes as ct
    from megatron_transformer_layer_fwd_gb300 import build
    path = build.build(check=True)
    lib = ct.CDLL(path)
    for name in mgb.header_functions():
        assert hasattr(lib, name), name
    lib.mgb_status_string.restype = ct.c_char_p
    assert b"check" in lib.mgb_status_string(mgb.MGB_ERR_DEVICE_CHECK)

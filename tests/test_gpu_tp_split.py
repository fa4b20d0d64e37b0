"""The k-way tensor-parallel split of the layer executed on one GPU, through
the C ABI ("LLM Lab 06: build a Megatron-style Transformer Block from
scratch", sections 2-3; "02 - How a whole Transformer block is split",
sections 1-2).

Shard i of k holds query heads [i nq/k, (i+1) nq/k) with their key/value
heads, and fc1 output columns [i W/k, (i+1) W/k) (whole gate/up blocks under
SwiGLU). Each shard runs:
  column-parallel  qkv_i = xn Wqkv[rows_i]^T + b      (3 GEMMs: Q, K, V rows)
                   O_i = attention over its heads
                   u_i, a_i = act(hn W1[rows_i]^T + b1[rows_i])
  row-parallel     partial_i = O_i Wo[:, cols_i]^T,  a_i W2[:, cols_i]^T
The all-reduce of the pages is the sum of the partials, done on the device
by float32-accumulating GEMM launches into one buffer that starts at the
residual plus the row-parallel bias (added once, after the sum, as on the
pages). Backward of the MLP: each shard's weight gradients are slices of the
unsplit ones, and the input gradient of the column-parallel fc1 is the sum
of the shards' partial input gradients (the backward all-reduce).

Checks: the column-parallel outputs equal the matching columns of the
unsplit GEMM / attention bit for bit (the same dot products); the sums of
the row-parallel partials match the unsplit float32 products to float32
rounding; the sharded layer output matches the library's fused layer and
the float64 oracle, whose own shard invariant is pinned in
tests/test_oracle_layer.py.
"""
import numpy as np
import pytest
import torch

import oracle
from megatron_transformer_layer_fwd_gb300 import mgb
from megatron_transformer_layer_fwd_gb300.inputs import LayerShape, layer_inputs
from megatron_transformer_layer_fwd_gb300.runner import LayerRunner, to_device
from tests.util import TOL, rel_l2, to_np

pytestmark = pytest.mark.gpu

BF = torch.bfloat16
SHAPES = {
    "swiglu_gqa_causal": LayerShape(2, 160, 512, 8, 4, 64, 512, act="swiglu", causal=True),
    "gelu_mha": LayerShape(2, 96, 256, 4, 4, 64, 512),
}


def _gemm(M, N, K, a, lda, b, ldb, c, ldc, epi=mgb.MGB_EPI_STORE, bias=None, c2=None, ldc2=0,
          aux=None, ldaux=0, a_mn=0, b_mn=0, accumulate=0, glu_block=128):
    d = mgb.GemmExDesc(g=mgb.GemmDesc(m=M, n=N, k=K, a_major=a_mn, b_major=b_mn, lda=lda, ldb=ldb,
                                      ldc=ldc, dtype=mgb.MGB_BF16, c_f32=0, accumulate=accumulate,
                                      alpha=1.0),
                       epilogue=epi, glu_block=glu_block, ldc2=ldc2, ldr=0, ldaux=ldaux)
    mgb.mgb_gemm_ex(d, a, b, bias, c, c2=c2, aux=aux)


def _ln(x, g, b):
    T, H = x.shape
    y = torch.empty_like(x)
    mgb.mgb_layernorm_fwd(T, H, mgb.MGB_BF16, 1e-5, x, g, b, y, None, None)
    return y


def _attention(sh, qkv, nq, nkv, q0, k0, v0, with_lse=False):
    """Attention over nq query heads starting at column q0 of qkv (K at k0, V at v0)."""
    T, W = qkv.shape
    d = sh.head_dim
    o = torch.empty((T, nq * d), device="cuda", dtype=BF)
    lse = torch.empty((sh.batch * nq * sh.seq,), device="cuda", dtype=torch.float32)
    mgb.mgb_attention_fwd(sh.batch, sh.seq, nq, nkv, d, sh.causal, mgb.MGB_BF16, qkv[:, q0:],
                          qkv[:, k0:], qkv[:, v0:], W, W, o, lse)
    return (o, lse) if with_lse else o


def _attention_bwd(sh, qkv, o, lse, dO, dqkv, nq, nkv, q0, k0, v0):
    """Attention backward over nq query heads into the matching columns of dqkv."""
    T, W = qkv.shape
    d = sh.head_dim
    ws = torch.empty(mgb.mgb_attention_bwd_ws_bytes(sh.batch, sh.seq, nq), dtype=torch.uint8,
                     device="cuda")
    mgb.mgb_attention_bwd(sh.batch, sh.seq, nq, nkv, d, sh.causal, mgb.MGB_BF16, qkv[:, q0:],
                          qkv[:, k0:], qkv[:, v0:], W, W, o, lse, dO, nq * d, dqkv[:, q0:],
                          dqkv[:, k0:], dqkv[:, v0:], W, W, ws)


class Sharded:
    """Forward (and MLP backward) of the layer split k ways."""

    def __init__(self, sh, w, x, k):
        self.sh, self.w, self.x, self.k = sh, w, x, k
        T, H, d = sh.tokens, sh.hidden, sh.head_dim
        nq, nkv = sh.n_q_heads, sh.n_kv_heads
        self.Dq, self.Wqkv, self.W = nq * d, sh.qkv_width, sh.fc1_width
        self.nqs, self.nkvs = nq // k, nkv // k

    def cols(self, i):
        """First columns of shard i's Q, K and V heads in the fused qkv buffer."""
        d, nq, nkv = self.sh.head_dim, self.sh.n_q_heads, self.sh.n_kv_heads
        return (i * self.nqs * d, nq * d + i * self.nkvs * d, (nq + nkv) * d + i * self.nkvs * d)

    def forward(self):
        sh, w, k = self.sh, self.w, self.k
        T, H, d = sh.tokens, sh.hidden, sh.head_dim
        nq, nkv = sh.n_q_heads, sh.n_kv_heads
        xn = _ln(self.x, w["ln1_g"], w["ln1_b"])
        # column-parallel QKV into one fused buffer (each shard writes its columns)
        qkv = torch.full((T, self.Wqkv), float("nan"), device="cuda", dtype=BF)
        Os = []
        for i in range(k):
            for base, nh, h0 in ((0, self.nqs, i * self.nqs), (nq * d, self.nkvs, i * self.nkvs),
                                 ((nq + nkv) * d, self.nkvs, i * self.nkvs)):
                r0, n = base + h0 * d, nh * d
                _gemm(T, n, H, xn, H, w["w_qkv"][r0:r0 + n], H, qkv[:, r0:], self.Wqkv,
                      bias=w["b_qkv"][r0:r0 + n])
        self.lses = []
        for i in range(k):
            o, lse = _attention(sh, qkv, self.nqs, self.nkvs, *self.cols(i), with_lse=True)
            Os.append(o)
            self.lses.append(lse)
        # row-parallel projection: partials summed on the device (float32)
        h32 = self.x.float() + w["b_o"].float()[None, :]
        for i in range(k):
            c0 = i * self.nqs * d
            _gemm(T, H, self.nqs * d, Os[i], self.nqs * d, w["w_o"][:, c0:], self.Dq, h32, H,
                  epi=mgb.MGB_EPI_F32, accumulate=1)
        h = h32.to(BF)
        hn = _ln(h, w["ln2_g"], w["ln2_b"])
        # column-parallel fc1 with the activation fused; row-parallel fc2
        Ws, Fs = self.W // k, sh.ffn // k
        us, As = [], []
        y32 = h.float() + w["b_2"].float()[None, :]
        for i in range(k):
            u = torch.empty((T, Ws), device="cuda", dtype=BF)
            a = torch.empty((T, Fs), device="cuda", dtype=BF)
            epi = mgb.MGB_EPI_BIAS_SWIGLU if sh.act == "swiglu" else mgb.MGB_EPI_BIAS_GELU
            _gemm(T, Ws, H, hn, H, w["w_1"][i * Ws:], H, u, Ws, epi=epi,
                  bias=w["b_1"][i * Ws:(i + 1) * Ws], c2=a, ldc2=Fs, glu_block=sh.glu_block)
            us.append(u)
            As.append(a)
            _gemm(T, H, Fs, a, Fs, w["w_2"][:, i * Fs:], sh.ffn, y32, H, epi=mgb.MGB_EPI_F32,
                  accumulate=1)
        self.xn, self.qkv, self.Os, self.h, self.hn, self.us, self.As = xn, qkv, Os, h, hn, us, As
        self.h32, self.y32 = h32, y32
        return y32.to(BF)

    def mlp_backward(self, dy):
        """Per shard: dW2 slice, du (activation gradient fused), dW1 rows; the
        fc1 input gradient summed over shards in float32."""
        sh, w, k = self.sh, self.w, self.k
        T, H = sh.tokens, sh.hidden
        Ws, Fs = self.W // k, sh.ffn // k
        dW2 = torch.empty((H, sh.ffn), device="cuda", dtype=BF)
        dW1 = torch.empty((self.W, H), device="cuda", dtype=BF)
        dhn32 = torch.zeros((T, H), device="cuda", dtype=torch.float32)
        for i in range(k):
            # dW2[:, cols_i] = dy^T a_i (weight gradient: both operands MN-major)
            _gemm(H, Fs, T, dy, H, self.As[i], Fs, dW2[:, i * Fs:], sh.ffn, a_mn=1, b_mn=1)
            # du_i = (dy W2[:, cols_i]) * act'(u_i)
            du = torch.empty((T, Ws), device="cuda", dtype=BF)
            if sh.act == "swiglu":
                _gemm(T, Fs, H, dy, H, w["w_2"][:, i * Fs:], sh.ffn, du, Ws, epi=mgb.MGB_EPI_DSWIGLU,
                      aux=self.us[i], ldaux=Ws, b_mn=1, glu_block=sh.glu_block)
            else:
                _gemm(T, Fs, H, dy, H, w["w_2"][:, i * Fs:], sh.ffn, du, Ws, epi=mgb.MGB_EPI_DGELU,
                      aux=self.us[i], ldaux=Ws, b_mn=1)
            # dW1[rows_i] = du_i^T hn; d hn += du_i W1[rows_i]
            _gemm(Ws, H, T, du, Ws, self.hn, H, dW1[i * Ws:], H, a_mn=1, b_mn=1)
            _gemm(T, H, Ws, du, Ws, w["w_1"][i * Ws:], H, dhn32, H, b_mn=1, epi=mgb.MGB_EPI_F32,
                  accumulate=1)
        return dW2, dW1, dhn32

    def attention_backward(self, dh):
        """Per shard, from dh = dL/dh at the attention sublayer's output:
        dWo[:, cols_i] = dh^T O_i (row-parallel weight gradient); dO_i =
        dh Wo[:, cols_i]; the attention backward over its heads into its
        columns of dqkv; dWqkv[rows_i] = dqkv_i^T xn (column-parallel weight
        gradient); and the input gradient of the column-parallel QKV,
        d xn = sum over shards of dqkv_i Wqkv[rows_i], summed in float32 (the
        backward all-reduce)."""
        sh, w, k = self.sh, self.w, self.k
        T, H, d = sh.tokens, sh.hidden, sh.head_dim
        dWo = torch.empty((H, self.Dq), device="cuda", dtype=BF)
        dWqkv = torch.empty((self.Wqkv, H), device="cuda", dtype=BF)
        dqkv = torch.full((T, self.Wqkv), float("nan"), device="cuda", dtype=BF)
        dxn32 = torch.zeros((T, H), device="cuda", dtype=torch.float32)
        for i in range(k):
            q0, k0, v0 = self.cols(i)
            n_q = self.nqs * d
            _gemm(H, n_q, T, dh, H, self.Os[i], n_q, dWo[:, q0:], self.Dq, a_mn=1, b_mn=1)
            dO = torch.empty((T, n_q), device="cuda", dtype=BF)
            _gemm(T, n_q, H, dh, H, w["w_o"][:, q0:], self.Dq, dO, n_q, b_mn=1)
            _attention_bwd(sh, self.qkv, self.Os[i], self.lses[i], dO, dqkv, self.nqs, self.nkvs,
                           q0, k0, v0)
            for r0, n in ((q0, n_q), (k0, self.nkvs * d), (v0, self.nkvs * d)):
                _gemm(n, H, T, dqkv[:, r0:], self.Wqkv, self.xn, H, dWqkv[r0:], H, a_mn=1, b_mn=1)
                _gemm(T, H, n, dqkv[:, r0:], self.Wqkv, w["w_qkv"][r0:], H, dxn32, H, b_mn=1,
                      epi=mgb.MGB_EPI_F32, accumulate=1)
        return dWo, dWqkv, dqkv, dxn32


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("k", [2, 4])
def test_tp_split_forward_and_mlp_backward(mgb_lib, name, k):
    sh = SHAPES[name]
    if sh.n_kv_heads % k or (sh.ffn // k) % (sh.glu_block if sh.act == "swiglu" else 1):
        pytest.skip("shards need whole KV heads and whole gate/up blocks")
    arr = layer_inputs(sh, seed=21, random_affine=True, random_dy=True)
    r = LayerRunner(sh, arr)
    y_ref = r.fwd().clone()
    w = r.w
    T, H, d = sh.tokens, sh.hidden, sh.head_dim
    s = Sharded(sh, w, r.x, k)
    y = s.forward()
    assert mgb.mgb_device_status() == mgb.MGB_OK

    # column-parallel outputs: exactly the unsplit columns
    qkv_full = torch.empty_like(s.qkv)
    _gemm(T, s.Wqkv, H, s.xn, H, w["w_qkv"], H, qkv_full, s.Wqkv, bias=w["b_qkv"])
    assert torch.equal(s.qkv, qkv_full)
    O_full = _attention(sh, qkv_full, sh.n_q_heads, sh.n_kv_heads, 0, s.Dq, s.Dq + sh.n_kv_heads * d)
    for i in range(k):
        c0 = i * s.nqs * d
        assert torch.equal(s.Os[i], O_full[:, c0:c0 + s.nqs * d])
    u_full = torch.empty((T, s.W), device="cuda", dtype=BF)
    a_full = torch.empty((T, sh.ffn), device="cuda", dtype=BF)
    epi = mgb.MGB_EPI_BIAS_SWIGLU if sh.act == "swiglu" else mgb.MGB_EPI_BIAS_GELU
    _gemm(T, s.W, H, s.hn, H, w["w_1"], H, u_full, s.W, epi=epi, bias=w["b_1"], c2=a_full,
          ldc2=sh.ffn, glu_block=sh.glu_block)
    Ws, Fs = s.W // k, sh.ffn // k
    for i in range(k):
        assert torch.equal(s.us[i], u_full[:, i * Ws:(i + 1) * Ws])
        assert torch.equal(s.As[i], a_full[:, i * Fs:(i + 1) * Fs])

    # row-parallel sums: the unsplit float32 product to float32 rounding
    h_full = r.x.float() + w["b_o"].float()[None, :]
    _gemm(T, H, s.Dq, O_full, s.Dq, w["w_o"], s.Dq, h_full, H, epi=mgb.MGB_EPI_F32, accumulate=1)
    assert rel_l2(to_np(s.h32), to_np(h_full)) < 1e-6
    y_full = s.h.float() + w["b_2"].float()[None, :]
    _gemm(T, H, sh.ffn, a_full, sh.ffn, w["w_2"], sh.ffn, y_full, H, epi=mgb.MGB_EPI_F32,
          accumulate=1)
    assert rel_l2(to_np(s.y32), to_np(y_full)) < 1e-6

    # the sharded layer against the library's fused layer and the oracle
    tol_o, tol_g = TOL["bf16"]
    assert rel_l2(to_np(y), to_np(y_ref)) < tol_o
    wo = {kk: arr[kk] for kk in w}
    ry, cache = oracle.block_fwd(sh, wo, arr["x"])
    assert rel_l2(to_np(y), ry) < tol_o

    # MLP backward: weight gradients are slices, input gradients sum
    dy = to_device(arr["dy"], BF)
    dW2, dW1, dhn32 = s.mlp_backward(dy)
    dW2_full = torch.empty_like(dW2)
    _gemm(H, sh.ffn, T, dy, H, a_full, sh.ffn, dW2_full, sh.ffn, a_mn=1, b_mn=1)
    assert torch.equal(dW2, dW2_full)
    du_full = torch.empty((T, s.W), device="cuda", dtype=BF)
    if sh.act == "swiglu":
        _gemm(T, sh.ffn, H, dy, H, w["w_2"], sh.ffn, du_full, s.W, epi=mgb.MGB_EPI_DSWIGLU,
              aux=u_full, ldaux=s.W, b_mn=1, glu_block=sh.glu_block)
    else:
        _gemm(T, sh.ffn, H, dy, H, w["w_2"], sh.ffn, du_full, s.W, epi=mgb.MGB_EPI_DGELU,
              aux=u_full, ldaux=s.W, b_mn=1)
    dW1_full = torch.empty_like(dW1)
    _gemm(s.W, H, T, du_full, s.W, s.hn, H, dW1_full, H, a_mn=1, b_mn=1)
    assert torch.equal(dW1, dW1_full)
    dhn_full = torch.empty((T, H), device="cuda", dtype=torch.float32)
    _gemm(T, H, s.W, du_full, s.W, w["w_1"], H, dhn_full, H, b_mn=1, epi=mgb.MGB_EPI_F32)
    assert rel_l2(to_np(dhn32), to_np(dhn_full)) < 1e-5
    # and against the oracle's MLP gradients (from its own forward)
    _, g = oracle.block_bwd(sh, wo, cache, arr["dy"])
    assert rel_l2(to_np(dW2), g["w_2"]) < tol_g
    assert rel_l2(to_np(dW1), g["w_1"]) < tol_g
    assert mgb.mgb_device_status() == mgb.MGB_OK


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("k", [2, 4])
def test_tp_split_attention_backward(mgb_lib, name, k):
    """The attention sublayer's backward split k ways by head: each shard's
    dWqkv rows and dWo columns are exact slices of the unsplit gradients, its
    dqkv columns equal the unsplit attention backward's, and the shards'
    input gradients sum (float32) to the unsplit one; every shard also
    matches the oracle's shard backward."""
    sh = SHAPES[name]
    if sh.n_kv_heads % k:
        pytest.skip("shards need whole KV heads")
    arr = layer_inputs(sh, seed=23, random_affine=True, random_dy=True)
    r = LayerRunner(sh, arr)
    w = r.w
    T, H, d = sh.tokens, sh.hidden, sh.head_dim
    nq, nkv = sh.n_q_heads, sh.n_kv_heads
    s = Sharded(sh, w, r.x, k)
    s.forward()
    dh = to_device(arr["dy"], BF)  # an upstream gradient at the sublayer output
    dWo, dWqkv, dqkv, dxn32 = s.attention_backward(dh)
    assert mgb.mgb_device_status() == mgb.MGB_OK

    # the unsplit sublayer backward from the same tensors
    O_full, lse_full = _attention(sh, s.qkv, nq, nkv, 0, s.Dq, s.Dq + nkv * d, with_lse=True)
    dWo_full = torch.empty_like(dWo)
    _gemm(H, s.Dq, T, dh, H, O_full, s.Dq, dWo_full, s.Dq, a_mn=1, b_mn=1)
    dO_full = torch.empty((T, s.Dq), device="cuda", dtype=BF)
    _gemm(T, s.Dq, H, dh, H, w["w_o"], s.Dq, dO_full, s.Dq, b_mn=1)
    dqkv_full = torch.empty_like(dqkv)
    _attention_bwd(sh, s.qkv, O_full, lse_full, dO_full, dqkv_full, nq, nkv, 0, s.Dq, s.Dq + nkv * d)
    dWqkv_full = torch.empty_like(dWqkv)
    _gemm(s.Wqkv, H, T, dqkv_full, s.Wqkv, s.xn, H, dWqkv_full, H, a_mn=1, b_mn=1)
    dxn_full = torch.empty((T, H), device="cuda", dtype=torch.float32)
    _gemm(T, H, s.Wqkv, dqkv_full, s.Wqkv, w["w_qkv"], H, dxn_full, H, b_mn=1, epi=mgb.MGB_EPI_F32)
    assert mgb.mgb_device_status() == mgb.MGB_OK
    assert torch.equal(dWo, dWo_full)            # row-parallel weight gradient: column slices
    assert torch.equal(dqkv, dqkv_full)          # per-head attention backward: column slices
    assert torch.equal(dWqkv, dWqkv_full)        # column-parallel weight gradient: row slices
    assert rel_l2(to_np(dxn32), to_np(dxn_full)) < 1e-5  # input gradients sum

    # each shard against the oracle's shard backward (from its own float64 forward)
    tol_g = TOL["bf16"][1]
    wo = {kk: arr[kk] for kk in w}
    xn, _, _ = oracle.ln_fwd(arr["x"], arr["ln1_g"], arr["ln1_b"])
    dxn_o = np.zeros((T, H))
    for i in range(k):
        _, c = oracle.shard.attn_partial_fwd(sh, wo, xn, i, k)
        da, dW, _, dWo_i = oracle.shard.attn_partial_bwd(sh, wo, c, arr["dy"])
        rows, o_cols = oracle.shard.head_shard(sh, i, k)
        assert rel_l2(to_np(dWo)[:, o_cols], dWo_i) < tol_g
        assert rel_l2(to_np(dWqkv)[rows], dW) < tol_g
        dxn_o += da
    assert rel_l2(to_np(dxn32), dxn_o) < tol_g


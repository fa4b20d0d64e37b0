"""Seeded synthetic inputs for the layer and the vocab-chunked cross-entropy.

This module is shared by the oracle-side tests and the CUDA-side tests and
bench. It holds workload shapes and random draws only: no step of the method
(no LayerNorm, matmul, softmax, activation or loss) is computed here.

Distributions follow the workloads the pages describe (x ~ N(0,1), weights
~ N(0, 0.02^2), biases zero, LayerNorm gamma = 1 / beta = 0, targets uniform
over the vocabulary; "LLM Lab 06: a Megatron-style Transformer Block from
scratch", section 2, draws x and every weight with torch.randn). Draws come
from numpy's PCG64 in a fixed order so every consumer sees the same values:

    x, Wqkv (Q rows, then K rows, then V rows), Wo, W1, W2,
    then (only when asked for) random biases / LayerNorm affine, then dy.

For bf16 workloads every drawn tensor is rounded to the nearest bf16 (ties to
even) before anyone sees it, so the oracle (float64) and the GPU (bf16
storage) start from identical values.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "LayerShape", "CEShape", "WORKLOADS", "CE_WORKLOADS", "round_to_bf16",
    "layer_inputs", "ce_inputs", "layer_flops", "ce_flops", "ce_stream_bytes",
]


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One transformer layer's shape and options (names follow the pages)."""
    batch: int
    seq: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    dtype: str = "bf16"          # "f32" | "bf16"
    norm_pos: str = "pre"        # "pre" | "post"
    act: str = "gelu"            # "gelu" (erf form) | "swiglu"
    causal: bool = False
    ln_affine: bool = True
    has_bias: bool = True
    glu_block: int = 128
    ln_eps: float = 1e-5

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def qkv_width(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def fc1_width(self) -> int:
        return 2 * self.ffn if self.act == "swiglu" else self.ffn

    def replace(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class CEShape:
    tokens: int
    hidden: int
    vocab: int
    chunk: int
    dtype: str = "bf16"

    def replace(self, **kw) -> "CEShape":
        return dataclasses.replace(self, **kw)


# The five workloads of the layer/CE study. Keys name what they are.
WORKLOADS = {
    # fp32 layer with page 1's dataflow: LN (no affine) -> attention -> +x ->
    # LN -> fc1 -> erf-GELU -> fc2 -> +residual; no biases, no mask.
    "fp32_p1_b2s128h256": LayerShape(2, 128, 256, 4, 4, 64, 1024, dtype="f32",
                                     norm_pos="pre", ln_affine=False, has_bias=False),
    # The same shapes with textbook Post-LN (LN after each residual add).
    "fp32_postln_b2s128h256": LayerShape(2, 128, 256, 4, 4, 64, 1024, dtype="f32",
                                         norm_pos="post", ln_affine=False, has_bias=False),
    "bf16_preln_b4s512h1024": LayerShape(4, 512, 1024, 16, 16, 64, 4096),
    # causal sweep: seq in {128, 256, 512, 1024, 2048} at batch 8
    **{f"bf16_causal_b8s{s}h2048": LayerShape(8, s, 2048, 16, 16, 128, 8192, causal=True)
       for s in (128, 256, 512, 1024, 2048)},
    "bf16_gqa_swiglu_b2s4096h4096": LayerShape(2, 4096, 4096, 32, 8, 128, 11008,
                                               act="swiglu", causal=True),
}

CE_WORKLOADS = {
    "bf16_ce_t8192h4096v128256": CEShape(8192, 4096, 128256, 16032),
}


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bfloat16 (ties to even); returns float64.

    Pure bit manipulation of the float32 encoding: keep the top 16 bits after
    adding 0x7FFF plus the lowest kept bit. Values are finite here.
    """
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _maybe_round(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(a)
    return a.astype(np.float32).astype(np.float64)


def layer_inputs(shape: LayerShape, seed: int = 0, random_affine: bool = False,
                 random_dy: bool = False) -> dict:
    """Draw x, weights (and optionally biases / LN affine, dy) for one layer.

    Weights are [out, in] row-major (the F.linear convention). Wqkv rows are
    [Q heads | K heads | V heads], each head's head_dim rows contiguous.
    W1 is [ffn, hidden] for GELU and [2*ffn, hidden] for SwiGLU, whose rows
    alternate blocks of glu_block gate rows and glu_block up rows.

    Returned arrays are float64 holding values exactly representable in the
    shape's dtype. `dy` is None unless random_dy (then ~N(0,1)).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    T, H = shape.tokens, shape.hidden
    nq, nkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    out = {}
    out["x"] = rng.standard_normal((T, H))
    wq = rng.standard_normal((nq * d, H)) * 0.02
    wk = rng.standard_normal((nkv * d, H)) * 0.02
    wv = rng.standard_normal((nkv * d, H)) * 0.02
    out["w_qkv"] = np.concatenate([wq, wk, wv], axis=0)
    out["w_o"] = rng.standard_normal((H, nq * d)) * 0.02
    out["w_1"] = rng.standard_normal((shape.fc1_width, H)) * 0.02
    out["w_2"] = rng.standard_normal((H, shape.ffn)) * 0.02
    zeros = np.zeros
    if shape.has_bias:
        if random_affine:
            out["b_qkv"] = rng.standard_normal(shape.qkv_width) * 0.02
            out["b_o"] = rng.standard_normal(H) * 0.02
            out["b_1"] = rng.standard_normal(shape.fc1_width) * 0.02
            out["b_2"] = rng.standard_normal(H) * 0.02
        else:
            out["b_qkv"] = zeros(shape.qkv_width)
            out["b_o"] = zeros(H)
            out["b_1"] = zeros(shape.fc1_width)
            out["b_2"] = zeros(H)
    else:
        for k in ("b_qkv", "b_o", "b_1", "b_2"):
            out[k] = None
    if shape.ln_affine:
        if random_affine:
            out["ln1_g"] = 1.0 + 0.1 * rng.standard_normal(H)
            out["ln1_b"] = 0.1 * rng.standard_normal(H)
            out["ln2_g"] = 1.0 + 0.1 * rng.standard_normal(H)
            out["ln2_b"] = 0.1 * rng.standard_normal(H)
        else:
            out["ln1_g"] = np.ones(H)
            out["ln1_b"] = zeros(H)
            out["ln2_g"] = np.ones(H)
            out["ln2_b"] = zeros(H)
    else:
        for k in ("ln1_g", "ln1_b", "ln2_g", "ln2_b"):
            out[k] = None
    out["dy"] = rng.standard_normal((T, H)) if random_dy else None
    for k, v in list(out.items()):
        if v is not None:
            out[k] = _maybe_round(v, shape.dtype)
    return out


def mean_loss_dy(shape: LayerShape) -> float:
    """Upstream gradient of loss = mean(out) over all tokens x hidden entries."""
    return 1.0 / (shape.tokens * shape.hidden)


def ce_inputs(shape: CEShape, seed: int = 0) -> dict:
    """hidden ~ N(0,1) [T,H], embedding ~ N(0,0.02^2) [V,H], targets ~ U[0,V)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    hidden = rng.standard_normal((shape.tokens, shape.hidden), dtype=np.float32)
    emb = rng.standard_normal((shape.vocab, shape.hidden), dtype=np.float32) * np.float32(0.02)
    targets = rng.integers(0, shape.vocab, shape.tokens).astype(np.int32)
    return {"hidden": _maybe_round(hidden, shape.dtype), "emb": _maybe_round(emb, shape.dtype),
            "targets": targets}


# ---- algorithmic work counts (model FLOPs / bytes; no recompute counted) ----

def layer_flops(shape: LayerShape) -> dict:
    """Model FLOPs of one layer: 2*M*N*K per GEMM, attention 4*B*nq*d*pairs.

    pairs = S*S without a mask, S*(S+1)/2 with the causal mask ("Megatron-LM"
    notes, split strategy: attention cost grows as batch*seq^2*heads*head_dim).
    Backward = 2x forward for GEMMs and attention.
    """
    T, H, F = shape.tokens, shape.hidden, shape.ffn
    nq, d, S, B = shape.n_q_heads, shape.head_dim, shape.seq, shape.batch
    gemm = 2 * T * H * shape.qkv_width + 2 * T * nq * d * H \
        + 2 * T * H * shape.fc1_width + 2 * T * F * H
    pairs = S * (S + 1) // 2 if shape.causal else S * S
    attn = 4 * B * nq * d * pairs
    fwd = gemm + attn
    return {"fwd": float(fwd), "bwd": float(2 * fwd), "total": float(3 * fwd),
            "attn_fwd": float(attn), "gemm_fwd": float(gemm)}


def ce_flops(shape: CEShape) -> dict:
    """Logits GEMM (fwd) + dgrad + wgrad = 3 * 2*T*V*H; recompute reported apart."""
    g = 2.0 * shape.tokens * shape.vocab * shape.hidden
    return {"fwd": g, "bwd": 2 * g, "total": 3 * g, "recompute": g}


def ce_stream_bytes(shape: CEShape, elt: int = 2) -> float:
    """Algorithmic bytes of the streaming CE passes: stats reads the logits once
    (elt B/entry); the gradient pass reads them and writes the gradient (2*elt)."""
    return 3.0 * elt * shape.tokens * shape.vocab

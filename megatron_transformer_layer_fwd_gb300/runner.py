"""Device-memory plumbing around the C ABI for one layer and for the CE.

PyTorch allocates the buffers (inputs, weights, outputs, the saved buffer,
the workspace) and provides the stream; every computation is a call into
libmgb.so through `mgb`.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mgb

WEIGHT_KEYS = ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2",
               "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def torch_dtype(name: str) -> torch.dtype:
    return torch.bfloat16 if name == "bf16" else torch.float32


def to_device(a: np.ndarray, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    """float64 array of values exact in `dtype` -> device tensor (exact copy)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=dtype)


class LayerRunner:
    """One layer's device buffers and the fwd/bwd calls."""

    def __init__(self, shape, arrays: dict, device="cuda"):
        self.shape = shape
        self.desc = mgb.block_desc(shape)
        self.dtype = torch_dtype(shape.dtype)
        self.w = {k: (to_device(arrays[k], self.dtype, device) if arrays.get(k) is not None else None)
                  for k in WEIGHT_KEYS}
        self.x = to_device(arrays["x"], self.dtype, device)
        saved, fwd, bwd = mgb.mgb_block_sizes(self.desc)
        self.saved = torch.empty(max(saved, 16), dtype=torch.uint8, device=device)
        self.ws = torch.empty(max(bwd, 16), dtype=torch.uint8, device=device)
        # float32: the forward's GEMMs keep their split operands here
        self.fwd_ws = torch.empty(fwd, dtype=torch.uint8, device=device) if fwd > 0 else None
        self.y = torch.empty_like(self.x)
        self.dx = torch.empty_like(self.x)
        self.grads = {k: (torch.empty_like(v) if v is not None else None) for k, v in self.w.items()}

    def fwd(self, stream=None):
        mgb.mgb_block_fwd(self.desc, self.w, self.x, self.y, self.saved, self.fwd_ws, stream)
        return self.y

    def bwd(self, dy: torch.Tensor, stream=None):
        mgb.mgb_block_bwd(self.desc, self.w, self.x, dy, self.saved, self.dx, self.grads, self.ws,
                          stream)
        return self.dx, self.grads


class CERunner:
    """Tied-embedding CE buffers and the fused fwd+bwd call."""

    def __init__(self, tokens: int, hidden: int, vocab: int, chunk: int, hidden_t: torch.Tensor,
                 emb_t: torch.Tensor, targets_t: torch.Tensor, grad_scale: float | None = None,
                 want_grads: bool = True, mode: int = mgb.MGB_CE_FUSED, emb_stream=None,
                 token_block: int = 0):
        dev = hidden_t.device
        self.desc = mgb.ce_desc(tokens, hidden, vocab, chunk,
                                grad_scale if grad_scale is not None else 1.0 / max(tokens, 1), mode,
                                token_block)
        # resident / blocked mode: d_emb (its last part) is left running on this
        # stream (the caller joins it)
        self.desc.emb_stream = emb_stream.cuda_stream if emb_stream is not None else None
        self.hidden, self.emb, self.targets = hidden_t, emb_t, targets_t
        # the blocked mode's rows per block as the library rounds them
        tb = token_block if token_block > 0 else mgb.CE_DEFAULT_TOKEN_BLOCK
        self.token_block = min((tb + 255) // 256 * 256, (tokens + 255) // 256 * 256)
        self.ws = torch.empty(max(mgb.mgb_vocab_ce_sizes(self.desc), 16), dtype=torch.uint8, device=dev)
        self.loss = torch.empty(max(tokens, 1), dtype=torch.float32, device=dev)
        self.lse = torch.empty(max(tokens, 1), dtype=torch.float32, device=dev)
        self.loss_mean = torch.empty(4, dtype=torch.float32, device=dev)
        self.d_hidden = torch.empty_like(hidden_t) if want_grads else None
        self.d_emb = torch.empty_like(emb_t) if want_grads else None

    def run(self, stream=None):
        mgb.mgb_vocab_ce_fwd_bwd(self.desc, self.hidden, self.emb, self.targets, self.loss,
                                 self.loss_mean, self.lse, self.d_hidden, self.d_emb, self.ws, stream)

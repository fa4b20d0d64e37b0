"""CPU float64 oracle for one Megatron-style transformer layer and the
vocab-chunked tied-embedding cross-entropy.

TEST INFRASTRUCTURE ONLY. This package is the slow, plain, obviously-correct
statement of what the CUDA library computes. Only the test suite,
`__graft_entry__.smoke()` and the `cpu_baseline` / reference leg of `bench.py`
may import it. The product path (the C-ABI library and its Python binding)
never imports, links or executes anything in here, and this package imports
nothing from the product: the two share only the seeded input generator,
which holds no arithmetic of the method.

Everything is numpy float64. Library primitives used as single steps:
matrix product (`@`), `np.exp`, `np.log`, `np.max`, `scipy.special.erf`.
No blocking, fusion or reordering beyond what each definition states.

Sources (web pages on the subject, cited by title and section):
  * "LLM Lab 06: build a Megatron-style Transformer Block from scratch"
    (chat.ai-hpc.org), section 2 code walk-through: the layer's dataflow
    LN -> attention -> residual -> LN -> fc1 -> GELU -> fc2 -> residual,
    loss = out.mean(), end-to-end backward.
  * "02 - How a whole Transformer block is split" (llm-infra-atlas),
    section 1 (MLP column -> row, SwiGLU gate/up kept together by an
    interleaved layout), section 2 (attention split by head, fused
    linear_qkv of width q_proj + 2*kv_proj, GQA, row-parallel linear_proj),
    section 3 (vocab-parallel embedding: masked lookup per vocab shard,
    summed over shards; tied input/output table), section 4 (vocab-parallel
    cross-entropy from per-shard max, target logit and sum-exp partials;
    backward softmax - onehot).
  * "02 - How a whole Transformer block is split", section 5 (the TP RNG
    tracker: data-parallel, model-parallel and expert-parallel generator
    states, fork, replay in recomputation), with Philox4x32-10 (Salmon et
    al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011) as the
    counter-based generator (dropout.py).
  * "Megatron-LM" notes, split strategy section: attention cost grows with
    batch*seq^2*heads*head_dim.

Parity status of each function is listed in its module docstring; all
functions here are pinned by tests/test_oracle_*.py (closed forms,
invariants, finite differences, brute force) unless marked
"parity unpinned" (none currently are).
"""
from .layernorm import ln_fwd, ln_bwd
from .activations import gelu, gelu_grad, silu, silu_grad, swiglu_fwd, swiglu_bwd, glu_split
from .attention import attention_fwd, attention_bwd
from .layer import block_fwd, block_bwd, block_fwd_rows
from .cross_entropy import ce_full, ce_chunked, ce_grads, ce_rows, ce_emb_rows
from .embedding import embedding_fwd, embedding_bwd
from . import dropout
from . import shard

__all__ = [
    "ln_fwd", "ln_bwd", "gelu", "gelu_grad", "silu", "silu_grad", "swiglu_fwd", "swiglu_bwd",
    "glu_split", "attention_fwd", "attention_bwd", "block_fwd", "block_bwd", "block_fwd_rows",
    "ce_full", "ce_chunked", "ce_grads", "ce_rows", "ce_emb_rows", "embedding_fwd", "embedding_bwd", "dropout",
    "shard",
]

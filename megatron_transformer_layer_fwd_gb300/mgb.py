"""ctypes binding of libmgb.so: the C ABI of include/mgb.h, same names.

Argument marshalling only: tensors become device pointers, the stream
becomes a cudaStream_t, and a non-OK status raises MgbError. Every step of
the layer and the cross-entropy runs in the library's CUDA kernels; there is
no other implementation behind these functions. PyTorch supplies device
memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
# MGB_LIB=check loads the checking build (device-side consistency checks)
LIB_PATH = os.path.join(HERE, "libmgb_check.so" if os.environ.get("MGB_LIB") == "check"
                        else "libmgb.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "mgb.h")

MGB_OK = 0
MGB_ERR_INVALID_ARG = -1
MGB_ERR_UNSUPPORTED = -2
MGB_ERR_MISALIGNED = -3
MGB_ERR_WORKSPACE_TOO_SMALL = -4
MGB_ERR_ARCH = -5
MGB_ERR_CUDA = -6
MGB_ERR_DEVICE_TIMEOUT = -7
MGB_ERR_NOT_IMPLEMENTED = -8
MGB_ERR_DEVICE_CHECK = -9

MGB_F32, MGB_BF16 = 0, 1
MGB_CE_STREAM, MGB_CE_FUSED, MGB_CE_RESIDENT, MGB_CE_BLOCKED = 0, 1, 2, 3
# tokens per block of MGB_CE_BLOCKED when mgb_ce_desc.token_block is 0 (the
# library's default, restated here for callers that size their own views)
CE_DEFAULT_TOKEN_BLOCK = 4096
MGB_PRE_LN, MGB_POST_LN = 0, 1
MGB_GELU_ERF, MGB_SWIGLU = 0, 1
MGB_K_MAJOR, MGB_MN_MAJOR = 0, 1
MGB_RNG_DATA_PARALLEL, MGB_RNG_MODEL_PARALLEL, MGB_RNG_EXPERT_PARALLEL = 0, 1, 2
(MGB_EPI_STORE, MGB_EPI_BIAS_GELU, MGB_EPI_BIAS_SWIGLU, MGB_EPI_BIAS_RESID, MGB_EPI_DGELU,
 MGB_EPI_DSWIGLU, MGB_EPI_F32) = range(7)

_WEIGHT_FIELDS = ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2",
                  "ln1_g", "ln1_b", "ln2_g", "ln2_b")


class MgbError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class RngState(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


class RngTracker(ctypes.Structure):
    _fields_ = [("state", RngState * 3), ("current", ctypes.c_int32)]


class BlockDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "seq", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "dtype",
        "norm_pos", "act", "causal", "ln_affine", "has_bias", "glu_block")] + [
        ("ln_eps", ctypes.c_float), ("hidden_dropout", ctypes.c_float),
        ("attn_dropout", ctypes.c_float), ("rng_attn", RngState), ("rng_proj", RngState),
        ("rng_fc2", RngState)]


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class BlockGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


class CEDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int32), ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("dtype", ctypes.c_int32), ("grad_scale", ctypes.c_float),
                ("mode", ctypes.c_int32), ("emb_stream", ctypes.c_void_p),
                ("token_block", ctypes.c_int32)]


class EmbeddingBwdPlan(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int32), ("v0", ctypes.c_int32), ("v1", ctypes.c_int32),
                ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


class GemmDesc(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32), ("k", ctypes.c_int32),
                ("a_major", ctypes.c_int32), ("b_major", ctypes.c_int32),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("c_f32", ctypes.c_int32), ("accumulate", ctypes.c_int32),
                ("alpha", ctypes.c_float)]


class GemmExDesc(ctypes.Structure):
    _fields_ = [("g", GemmDesc), ("epilogue", ctypes.c_int32), ("glu_block", ctypes.c_int32),
                ("ldc2", ctypes.c_int64), ("ldr", ctypes.c_int64), ("ldaux", ctypes.c_int64)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libmgb.so (built in-tree by build.py). Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m megatron_transformer_layer_fwd_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, I64, U64, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t)
        PSZ = ctypes.POINTER(SZ)
        sig = {
            "mgb_block_sizes": [ctypes.POINTER(BlockDesc), PSZ, PSZ, PSZ],
            "mgb_block_fwd": [ctypes.POINTER(BlockDesc), ctypes.POINTER(BlockWeights), P, P, P, SZ,
                              P, SZ, P],
            "mgb_block_bwd": [ctypes.POINTER(BlockDesc), ctypes.POINTER(BlockWeights), P, P, P, SZ,
                              P, ctypes.POINTER(BlockGrads), P, SZ, P],
            "mgb_vocab_ce_sizes": [ctypes.POINTER(CEDesc), PSZ],
            "mgb_vocab_ce_fwd_bwd": [ctypes.POINTER(CEDesc), P, P, P, P, P, P, P, P, P, SZ, P],
            "mgb_gemm": [ctypes.POINTER(GemmDesc), P, P, P, P, P],
            "mgb_gemm_ex": [ctypes.POINTER(GemmExDesc), P, P, P, P, P, P, P, P],
            "mgb_gemm_f32_tc": [ctypes.POINTER(GemmExDesc), P, P, P, P, P, P, P, P, SZ, P],
            "mgb_memcpy_async": [P, P, SZ, P],
            "mgb_layernorm_fwd": [I32, I32, I32, F32, P, P, P, P, P, P, P],
            "mgb_layernorm_bwd": [I32, I32, I32, P, P, P, P, P, P, P, P, P, P, SZ, P],
            "mgb_layernorm_bwd_noalloc": [I32, I32, I32, P, P, P, P, P, P, P, P, P, P],
            "mgb_attention_fwd": [I32, I32, I32, I32, I32, I32, I32, P, P, P, I64, I64, P, P, P],
            "mgb_attention_bwd": [I32, I32, I32, I32, I32, I32, I32, P, P, P, I64, I64, P, P, P,
                                  I64, P, P, P, I64, I64, P, SZ, P],
            "mgb_embedding_fwd": [I32, I32, I32, I32, I32, P, P, P, P],
            "mgb_rng_tracker_init": [ctypes.POINTER(RngTracker), U64, I32, I32, I32],
            "mgb_rng_restore": [ctypes.POINTER(RngTracker), I32],
            "mgb_rng_draw": [ctypes.POINTER(RngTracker), U64, ctypes.POINTER(RngState)],
            "mgb_block_dropout_plan": [ctypes.POINTER(BlockDesc), ctypes.POINTER(RngTracker)],
            "mgb_philox_bytes": [U64, U64, U64, P, P],
            "mgb_dropout": [ctypes.c_int64, ctypes.c_int64, I32, F32, RngState, P, ctypes.c_int64, P,
                            ctypes.c_int64, P],
            "mgb_embedding_bwd": [I32, I32, I32, I32, I32, P, P, P, I32, P, SZ, P],
            "mgb_embedding_bwd_prepare": [I32, I32, I32, P, P, SZ,
                                          ctypes.POINTER(EmbeddingBwdPlan), P],
            "mgb_embedding_bwd_apply": [ctypes.POINTER(EmbeddingBwdPlan), I32, I32, P, P, I32, P],
            "mgb_device_status": [P],
            "mgb_selftest_wait_timeout": [U64, P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.mgb_rng_fork.argtypes = [ctypes.POINTER(RngTracker), I32]
        lib.mgb_rng_fork.restype = I32
        lib.mgb_status_string.argtypes = [ctypes.c_int]
        lib.mgb_status_string.restype = ctypes.c_char_p
        lib.mgb_version.argtypes = []
        lib.mgb_version.restype = ctypes.c_int32
        lib.mgb_layernorm_bwd_ws_bytes.argtypes = [I32, I32]
        lib.mgb_layernorm_bwd_ws_bytes.restype = SZ
        lib.mgb_attention_bwd_ws_bytes.argtypes = [I32, I32, I32]
        lib.mgb_attention_bwd_ws_bytes.restype = SZ
        lib.mgb_gemm_f32_tc_ws_bytes.argtypes = [I32, I32, I32]
        lib.mgb_gemm_f32_tc_ws_bytes.restype = SZ
        lib.mgb_embedding_bwd_ws_bytes.argtypes = [I32, I32, I32]
        lib.mgb_embedding_bwd_ws_bytes.restype = SZ
        lib.mgb_launch_count.argtypes = []
        lib.mgb_launch_count.restype = ctypes.c_uint64
        lib.mgb_profile_enable.argtypes = [I32]
        lib.mgb_profile_enable.restype = ctypes.c_int
        lib.mgb_profile_reset.argtypes = []
        lib.mgb_profile_reset.restype = ctypes.c_int
        lib.mgb_profile_kinds.argtypes = []
        lib.mgb_profile_kinds.restype = I32
        lib.mgb_profile_kind_name.argtypes = [I32]
        lib.mgb_profile_kind_name.restype = ctypes.c_char_p
        lib.mgb_profile_read.argtypes = [I32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)]
        lib.mgb_profile_read.restype = ctypes.c_int
        _lib = lib
    return _lib


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions include/mgb.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(mgb_[a-z0-9_]+)\s*\(", text)))


def status_string(s: int) -> str:
    return load().mgb_status_string(s).decode()


def _check(status: int, where: str) -> None:
    if status != MGB_OK:
        raise MgbError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def block_desc(shape) -> BlockDesc:
    """BlockDesc from any object with the layer-shape attributes."""
    return BlockDesc(
        batch=shape.batch, seq=shape.seq, hidden=shape.hidden, n_q_heads=shape.n_q_heads,
        n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, ffn=shape.ffn,
        dtype=MGB_BF16 if shape.dtype == "bf16" else MGB_F32,
        norm_pos=MGB_PRE_LN if shape.norm_pos == "pre" else MGB_POST_LN,
        act=MGB_SWIGLU if shape.act == "swiglu" else MGB_GELU_ERF,
        causal=int(shape.causal), ln_affine=int(shape.ln_affine), has_bias=int(shape.has_bias),
        glu_block=shape.glu_block, ln_eps=shape.ln_eps)


def mgb_block_sizes(desc: BlockDesc) -> tuple[int, int, int]:
    s, f, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().mgb_block_sizes(ctypes.byref(desc), ctypes.byref(s), ctypes.byref(f),
                                  ctypes.byref(b)), "mgb_block_sizes")
    return s.value, f.value, b.value


def _weights(w: dict) -> BlockWeights:
    return BlockWeights(**{k: _ptr(w.get(k)) for k in _WEIGHT_FIELDS})


def mgb_block_fwd(desc: BlockDesc, weights: dict, x, y, saved, ws=None, stream=None) -> None:
    wt = _weights(weights)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().mgb_block_fwd(ctypes.byref(desc), ctypes.byref(wt), _ptr(x), _ptr(y), _ptr(saved),
                                saved.numel() * saved.element_size(), _ptr(ws), ws_bytes,
                                _stream(stream)), "mgb_block_fwd")


def mgb_block_bwd(desc: BlockDesc, weights: dict, x, dy, saved, dx, grads: dict, ws,
                  stream=None) -> None:
    wt = _weights(weights)
    gr = BlockGrads(**{k: _ptr(grads.get(k)) for k in _WEIGHT_FIELDS})
    _check(load().mgb_block_bwd(ctypes.byref(desc), ctypes.byref(wt), _ptr(x), _ptr(dy), _ptr(saved),
                                saved.numel() * saved.element_size(), _ptr(dx), ctypes.byref(gr),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "mgb_block_bwd")


def ce_desc(tokens: int, hidden: int, vocab: int, chunk: int, grad_scale: float,
            mode: int = MGB_CE_FUSED, token_block: int = 0) -> CEDesc:
    return CEDesc(tokens=tokens, hidden=hidden, vocab=vocab, chunk=chunk, dtype=MGB_BF16,
                  grad_scale=grad_scale, mode=mode, token_block=token_block)


def mgb_vocab_ce_sizes(desc: CEDesc) -> int:
    ws = ctypes.c_size_t()
    _check(load().mgb_vocab_ce_sizes(ctypes.byref(desc), ctypes.byref(ws)), "mgb_vocab_ce_sizes")
    return ws.value


def mgb_vocab_ce_fwd_bwd(desc: CEDesc, hidden, emb, targets, loss_per_token, loss_mean, lse=None,
                         d_hidden=None, d_emb=None, ws=None, stream=None) -> None:
    _check(load().mgb_vocab_ce_fwd_bwd(ctypes.byref(desc), _ptr(hidden), _ptr(emb), _ptr(targets),
                                       _ptr(loss_per_token), _ptr(loss_mean), _ptr(lse),
                                       _ptr(d_hidden), _ptr(d_emb), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)),
           "mgb_vocab_ce_fwd_bwd")


def mgb_gemm(desc: GemmDesc, a, b, bias, c, stream=None) -> None:
    _check(load().mgb_gemm(ctypes.byref(desc), _ptr(a), _ptr(b), _ptr(bias), _ptr(c), _stream(stream)),
           "mgb_gemm")


def mgb_gemm_ex(desc: GemmExDesc, a, b, bias, c, c2=None, resid=None, aux=None, stream=None) -> None:
    _check(load().mgb_gemm_ex(ctypes.byref(desc), _ptr(a), _ptr(b), _ptr(bias), _ptr(c), _ptr(c2),
                              _ptr(resid), _ptr(aux), _stream(stream)), "mgb_gemm_ex")


def mgb_gemm_f32_tc_ws_bytes(m: int, n: int, k: int) -> int:
    return int(load().mgb_gemm_f32_tc_ws_bytes(m, n, k))


def mgb_gemm_f32_tc(desc: GemmExDesc, a, b, bias, c, c2=None, resid=None, aux=None, ws=None,
                    stream=None) -> None:
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().mgb_gemm_f32_tc(ctypes.byref(desc), _ptr(a), _ptr(b), _ptr(bias), _ptr(c),
                                  _ptr(c2), _ptr(resid), _ptr(aux), _ptr(ws), ws_bytes,
                                  _stream(stream)), "mgb_gemm_f32_tc")


def rng_tracker(seed: int, tp_rank: int = 0, ep_rank: int = 0, etp_rank: int = 0) -> RngTracker:
    t = RngTracker()
    _check(load().mgb_rng_tracker_init(ctypes.byref(t), seed, tp_rank, ep_rank, etp_rank),
           "mgb_rng_tracker_init")
    return t


def mgb_rng_fork(t: RngTracker, kind: int) -> int:
    prev = load().mgb_rng_fork(ctypes.byref(t), kind)
    if prev < 0:
        _check(prev, "mgb_rng_fork")
    return prev


def mgb_rng_restore(t: RngTracker, prev: int) -> None:
    _check(load().mgb_rng_restore(ctypes.byref(t), prev), "mgb_rng_restore")


def mgb_rng_draw(t: RngTracker, n: int) -> RngState:
    out = RngState()
    _check(load().mgb_rng_draw(ctypes.byref(t), n, ctypes.byref(out)), "mgb_rng_draw")
    return out


def mgb_block_dropout_plan(desc: BlockDesc, t: RngTracker) -> None:
    _check(load().mgb_block_dropout_plan(ctypes.byref(desc), ctypes.byref(t)), "mgb_block_dropout_plan")


def mgb_philox_bytes(seed: int, offset: int, n: int, out, stream=None) -> None:
    _check(load().mgb_philox_bytes(seed, offset, n, _ptr(out), _stream(stream)), "mgb_philox_bytes")


def mgb_dropout(rows, cols, dtype, p, rng: RngState, x, ldx, y, ldy, stream=None) -> None:
    _check(load().mgb_dropout(rows, cols, dtype, p, rng, _ptr(x), ldx, _ptr(y), ldy, _stream(stream)),
           "mgb_dropout")


def mgb_layernorm_fwd(rows: int, cols: int, dtype: int, eps: float, x, gamma, beta, y, mean, rstd,
                      stream=None) -> None:
    _check(load().mgb_layernorm_fwd(rows, cols, dtype, eps, _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y),
                                    _ptr(mean), _ptr(rstd), _stream(stream)), "mgb_layernorm_fwd")


def mgb_layernorm_bwd_ws_bytes(rows: int, cols: int) -> int:
    return load().mgb_layernorm_bwd_ws_bytes(rows, cols)


def mgb_attention_bwd_ws_bytes(batch: int, seq: int, n_q_heads: int) -> int:
    return load().mgb_attention_bwd_ws_bytes(batch, seq, n_q_heads)


def mgb_embedding_fwd(tokens, hidden, v0, v1, dtype, ids, emb_shard, out, stream=None) -> None:
    _check(load().mgb_embedding_fwd(tokens, hidden, v0, v1, dtype, _ptr(ids), _ptr(emb_shard),
                                    _ptr(out), _stream(stream)), "mgb_embedding_fwd")


def mgb_embedding_bwd_ws_bytes(tokens: int, v0: int, v1: int) -> int:
    return load().mgb_embedding_bwd_ws_bytes(tokens, v0, v1)


def mgb_embedding_bwd(tokens, hidden, v0, v1, dtype, ids, d_out, d_emb_shard, accumulate, ws,
                      stream=None) -> None:
    _check(load().mgb_embedding_bwd(tokens, hidden, v0, v1, dtype, _ptr(ids), _ptr(d_out),
                                    _ptr(d_emb_shard), int(accumulate), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)),
           "mgb_embedding_bwd")


def mgb_embedding_bwd_prepare(tokens, v0, v1, ids, ws, stream=None) -> "EmbeddingBwdPlan":
    """The token order of the backward from the ids alone; returns the plan
    (host struct) that mgb_embedding_bwd_apply takes. `ws` must outlive it."""
    plan = EmbeddingBwdPlan()
    _check(load().mgb_embedding_bwd_prepare(tokens, v0, v1, _ptr(ids), _ptr(ws),
                                            ws.numel() * ws.element_size(), ctypes.byref(plan),
                                            _stream(stream)),
           "mgb_embedding_bwd_prepare")
    return plan


def mgb_embedding_bwd_apply(plan, hidden, dtype, d_out, d_emb_shard, accumulate,
                            stream=None) -> None:
    _check(load().mgb_embedding_bwd_apply(ctypes.byref(plan), hidden, dtype, _ptr(d_out),
                                          _ptr(d_emb_shard), int(accumulate), _stream(stream)),
           "mgb_embedding_bwd_apply")


def mgb_layernorm_bwd(rows: int, cols: int, dtype: int, x, mean, rstd, gamma, dy, dres, dx, dgamma,
                      dbeta, ws, stream=None) -> None:
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().mgb_layernorm_bwd(rows, cols, dtype, _ptr(x), _ptr(mean), _ptr(rstd), _ptr(gamma),
                                    _ptr(dy), _ptr(dres), _ptr(dx), _ptr(dgamma), _ptr(dbeta),
                                    _ptr(ws), ws_bytes, _stream(stream)), "mgb_layernorm_bwd")


def mgb_layernorm_bwd_noalloc(rows: int, cols: int, dtype: int, x, mean, rstd, gamma, dy, dres, dx,
                              dgamma, dbeta, stream=None) -> None:
    """mgb_layernorm_bwd without a workspace (library-held scratch; see mgb.h)."""
    _check(load().mgb_layernorm_bwd_noalloc(rows, cols, dtype, _ptr(x), _ptr(mean), _ptr(rstd),
                                            _ptr(gamma), _ptr(dy), _ptr(dres), _ptr(dx),
                                            _ptr(dgamma), _ptr(dbeta), _stream(stream)),
           "mgb_layernorm_bwd_noalloc")


def mgb_attention_fwd(batch, seq, n_q_heads, n_kv_heads, head_dim, causal, dtype, q, k, v, ld_q,
                      ld_kv, o, lse, stream=None) -> None:
    _check(load().mgb_attention_fwd(batch, seq, n_q_heads, n_kv_heads, head_dim, int(causal), dtype,
                                    _ptr(q), _ptr(k), _ptr(v), ld_q, ld_kv, _ptr(o), _ptr(lse),
                                    _stream(stream)), "mgb_attention_fwd")


def mgb_attention_bwd(batch, seq, n_q_heads, n_kv_heads, head_dim, causal, dtype, q, k, v, ld_q,
                      ld_kv, o, lse, dout, ld_do, dq, dk, dv, ld_dq, ld_dkv, ws,
                      stream=None) -> None:
    _check(load().mgb_attention_bwd(batch, seq, n_q_heads, n_kv_heads, head_dim, int(causal), dtype,
                                    _ptr(q), _ptr(k), _ptr(v), ld_q, ld_kv, _ptr(o), _ptr(lse),
                                    _ptr(dout), ld_do, _ptr(dq), _ptr(dk), _ptr(dv), ld_dq, ld_dkv,
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "mgb_attention_bwd")


def mgb_memcpy_async(dst, src, nbytes: int, stream=None) -> None:
    """Copy nbytes between (pinned host or device) tensors on `stream`."""
    _check(load().mgb_memcpy_async(_ptr(dst), _ptr(src), nbytes, _stream(stream)),
           "mgb_memcpy_async")


def mgb_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return load().mgb_device_status(_stream(stream))


def mgb_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().mgb_selftest_wait_timeout(limit_ns, _stream(stream)), "mgb_selftest_wait_timeout")


def mgb_version() -> int:
    return load().mgb_version()


def mgb_launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return load().mgb_launch_count()


def mgb_profile_enable(on: bool) -> None:
    _check(load().mgb_profile_enable(int(on)), "mgb_profile_enable")


def mgb_profile_reset() -> None:
    _check(load().mgb_profile_reset(), "mgb_profile_reset")


def mgb_profile_read() -> dict:
    """{kind name: (total device ms, launches)} of the profiled launches."""
    lib = load()
    out = {}
    for k in range(lib.mgb_profile_kinds()):
        ms, n = ctypes.c_double(), ctypes.c_int64()
        _check(lib.mgb_profile_read(k, ctypes.byref(ms), ctypes.byref(n)), "mgb_profile_read")
        out[lib.mgb_profile_kind_name(k).decode()] = (ms.value, n.value)
    return out

/*
 * mgb.h - C ABI of the GB300 (sm_103a) Megatron-style transformer layer library.
 *
 * One transformer layer (LayerNorm, fused QKV projection, per-head softmax
 * attention, output projection, residual, LayerNorm, fc1 + GELU/SwiGLU, fc2,
 * residual; Pre-LN or Post-LN) forward and backward, and the tied-embedding
 * cross-entropy computed from per-vocab-chunk partials, on one GPU.
 *
 * Sources the operations follow (web pages on the subject, by title/section):
 *   [P1] "LLM Lab 06: build a Megatron-style Transformer Block from scratch",
 *        section 2 (code walk-through: the layer's dataflow, loss = mean(out),
 *        end-to-end backward), section 5 (Post-LN vs Pre-LN: only the position
 *        of the norm relative to the residual changes).
 *   [P2] "02 - How a whole Transformer block is split", section 1 (MLP
 *        column -> row; SwiGLU gate/up kept together by interleaving),
 *        section 2 (attention split by head; fused linear_qkv of width
 *        q_proj + 2*kv_proj; GQA), section 3 (tied input/output embedding),
 *        section 4 (vocab-parallel cross-entropy: global max, target logit and
 *        sum-exp combined from shard partials; backward softmax - onehot).
 *
 * Conventions for every call:
 *   - All pointers are caller-owned DEVICE pointers unless stated otherwise;
 *     the library allocates no device memory per call and keeps no state
 *     besides a per-process cache of kernel attributes. Scratch memory is the
 *     caller's `ws` buffer; sizes come from the *_sizes queries.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream). Argument errors are returned before
 *     any kernel is launched. Kernel-side failures (a bounded device wait that
 *     ran out) are recorded in a per-device error word read by
 *     mgb_device_status().
 *   - Tensors are dense and row-major: activations [T, features] with token
 *     t = b*S + s (batch-major); weights [out, in] (y = x W^T + b).
 *   - dtype MGB_BF16: every tensor is bfloat16 except LayerNorm statistics,
 *     attention log-sum-exp and losses, which are float32; accumulation is
 *     float32. dtype MGB_F32: every tensor is float32 (SIMT float32 path).
 *   - Device pointers must be 16-byte aligned; feature sizes (hidden, ffn,
 *     head dims, vocab chunk) must keep every row a multiple of 16 bytes.
 *   - Gradients are overwritten, never accumulated into.
 *   - Any status other than MGB_OK leaves outputs unspecified.
 */
#ifndef MGB_H
#define MGB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MGB_OK = 0,
  MGB_ERR_INVALID_ARG = -1,         /* bad shape/flag combination or NULL pointer */
  MGB_ERR_UNSUPPORTED = -2,         /* valid but not supported (e.g. head_dim 96 in bf16) */
  MGB_ERR_MISALIGNED = -3,          /* a pointer or row stride is not 16-byte aligned */
  MGB_ERR_WORKSPACE_TOO_SMALL = -4, /* ws/saved smaller than the *_sizes query */
  MGB_ERR_ARCH = -5,                /* current device is not sm_103 */
  MGB_ERR_CUDA = -6,                /* a CUDA runtime call failed */
  MGB_ERR_DEVICE_TIMEOUT = -7,      /* a bounded device-side wait ran out */
  MGB_ERR_NOT_IMPLEMENTED = -8,
  MGB_ERR_DEVICE_CHECK = -9         /* checking build (libmgb_check.so) only: a kernel's
                                       own consistency check failed (an output address
                                       outside its tensor, a misaligned TMA coordinate,
                                       a CE target outside [0, vocab)); the access it
                                       guards was skipped */
} mgb_status;

typedef enum { MGB_F32 = 0, MGB_BF16 = 1 } mgb_dtype;
typedef enum { MGB_PRE_LN = 0, MGB_POST_LN = 1 } mgb_norm_pos;
typedef enum { MGB_GELU_ERF = 0, MGB_SWIGLU = 1 } mgb_act;

/* State of the counter-based generator behind dropout [P2 section 5]: the
 * stream is Philox4x32-10 (Salmon et al., SC 2011) with key = the seed's two
 * 32-bit halves and counters (q, 0, 0, 0), q = 0, 1, ..., each giving 16
 * bytes (its words in order, lowest byte first). Element e of a dropout site
 * at state (seed, offset) uses the byte at stream position offset + e; it is
 * kept iff the byte < floor((1 - p) * 256 + 1/2), and kept values are scaled
 * by 256 / that threshold. offset must be a multiple of 16. */
typedef struct {
  uint64_t seed, offset;
} mgb_rng_state;

/* Shape and options of one layer [P1 section 2; P2 sections 1-2].
 * Enum-valued fields are int32_t so the struct layout is fixed. */
typedef struct {
  int32_t batch, seq, hidden;
  int32_t n_q_heads, n_kv_heads, head_dim; /* n_q_heads % n_kv_heads == 0 (GQA) */
  int32_t ffn;                             /* fc1 width (SwiGLU: fc1 emits 2*ffn) */
  int32_t dtype;                           /* mgb_dtype */
  int32_t norm_pos;                        /* mgb_norm_pos */
  int32_t act;                             /* mgb_act */
  int32_t causal;                          /* 1: key j visible to query i iff j <= i */
  int32_t ln_affine;                       /* 1: LayerNorms have gamma/beta */
  int32_t has_bias;                        /* 1: the four linears have biases */
  int32_t glu_block;                       /* SwiGLU interleave block (fc1 columns) */
  float ln_eps;                            /* LayerNorm epsilon (1e-5) */
  /* Dropout [P2 section 5]: hidden_dropout on the outputs of the output
   * projection and of fc2 before their residual adds (element t*H + c of the
   * [T, H] branch), attn_dropout on the attention probabilities. 0 = off.
   * bf16 only. The attention site's keep bits (one per query and key) are
   * kept in `saved` for the backward; the hidden sites' masks are
   * regenerated. rng_*: the generator states of the three sites
   * (mgb_block_dropout_plan draws them from a tracker); the backward must get
   * the forward's values. */
  float hidden_dropout, attn_dropout;
  mgb_rng_state rng_attn, rng_proj, rng_fc2;
} mgb_block_desc;

/* Layer parameters. Shapes (H hidden, d head_dim, W = ffn or 2*ffn for SwiGLU):
 *   w_qkv [(nq+2*nkv)*d, H]  rows [Q heads | K heads | V heads]   b_qkv [(nq+2nkv)d]
 *   w_o   [H, nq*d]                                                b_o   [H]
 *   w_1   [W, H]  (SwiGLU: row blocks of glu_block gate, glu_block up, ...)  b_1 [W]
 *   w_2   [H, ffn]                                                 b_2   [H]
 *   ln1_g/ln1_b/ln2_g/ln2_b [H]: LN1 belongs to the attention sublayer, LN2 to the MLP.
 * Biases must be NULL iff !has_bias; LN params NULL iff !ln_affine. */
typedef struct {
  const void *w_qkv, *b_qkv, *w_o, *b_o, *w_1, *b_1, *w_2, *b_2;
  const void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
} mgb_block_weights;

/* Gradient outputs, same shapes/dtype as the weights. Any entry may be NULL
 * (that gradient is not written). */
typedef struct {
  void *w_qkv, *b_qkv, *w_o, *b_o, *w_1, *b_1, *w_2, *b_2;
  void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
} mgb_block_grads;

/* The tensor-parallel RNG tracker [P2 section 5]: three generator states,
 * one current. Outside the TP region activations are replicated, so dropout
 * there draws from the data-parallel state (seed: the same on every TP rank);
 * inside it each rank holds a different shard and draws from the
 * model-parallel state (seed + 2718 + tp_rank); MoE experts use
 * seed + 1024 + 100 * ep_rank + etp_rank. Host-only calls, no device work. */
typedef enum {
  MGB_RNG_DATA_PARALLEL = 0,
  MGB_RNG_MODEL_PARALLEL = 1,
  MGB_RNG_EXPERT_PARALLEL = 2
} mgb_rng_kind;

typedef struct {
  mgb_rng_state state[3]; /* indexed by mgb_rng_kind */
  int32_t current;        /* the state draws come from */
} mgb_rng_tracker;

/* All three states at offset 0; the data-parallel one current. */
mgb_status mgb_rng_tracker_init(mgb_rng_tracker* t, uint64_t seed, int32_t tp_rank,
                                int32_t ep_rank, int32_t etp_rank);
/* Makes `kind` current; returns the previous current kind (pass it to
 * mgb_rng_restore), or MGB_ERR_INVALID_ARG. */
int32_t mgb_rng_fork(mgb_rng_tracker* t, int32_t kind);
mgb_status mgb_rng_restore(mgb_rng_tracker* t, int32_t prev);
/* *out = the current state; its offset then advances by n rounded up to 16. */
mgb_status mgb_rng_draw(mgb_rng_tracker* t, uint64_t n, mgb_rng_state* out);
/* Fills desc->rng_attn (inside the TP region: forked to the model-parallel
 * state; B * n_q_heads * S * Sp elements, element ((b*nq + h)*S + i)*Sp + j,
 * Sp = S rounded up to 16), then rng_proj and rng_fc2 (B*S*H each) from the
 * current state. Every call draws all three, whatever the probabilities. */
mgb_status mgb_block_dropout_plan(mgb_block_desc* desc, mgb_rng_tracker* t);

/* Sizes in bytes of the `saved` buffer (written by fwd, read by bwd) and of
 * the scratch workspaces of fwd and bwd (the forward's is 0 for bf16; for
 * float32 it holds the split operands of the three-TF32 GEMMs, and `ws` of
 * mgb_block_fwd must then be 256-byte aligned). Host-only; no device work. */
mgb_status mgb_block_sizes(const mgb_block_desc* desc, size_t* saved_bytes,
                           size_t* fwd_ws_bytes, size_t* bwd_ws_bytes);

/* Layer forward [P1 section 2; P2 sections 1-2]:
 *   Pre-LN : xn = LN1(x); qkv = xn Wqkv^T + bqkv; O = Attn(qkv);
 *            h = x + O Wo^T + bo; hn = LN2(h); a = act(hn W1^T + b1);
 *            y = h + a W2^T + b2
 *   Post-LN: O = Attn(x Wqkv^T + bqkv); h = LN1(x + O Wo^T + bo);
 *            a = act(h W1^T + b1); y = LN2(h + a W2^T + b2)
 * Attn: per batch and query head h, softmax(Q_h K_g^T / sqrt(d)) V_g with
 * g = h / (nq/nkv), causal mask optional. x, y: [T, H]. `saved` receives what
 * the backward needs (layout private). */
mgb_status mgb_block_fwd(const mgb_block_desc* desc, const mgb_block_weights* w,
                         const void* x, void* y, void* saved, size_t saved_bytes,
                         void* ws, size_t ws_bytes, void* stream);

/* Layer backward [P1 section 2 "end-to-end backward"]: given dy = dL/dy [T, H]
 * and the `saved` buffer of the matching forward (same x and weights), writes
 * dx = dL/dx [T, H] and every non-NULL gradient in `grads`. Attention
 * probabilities are recomputed from the saved log-sum-exp.
 * Weight and bias gradients, and the attention backward's dQ kernel, are
 * computed on side streams that the library owns (two per host thread and
 * device), forked from and joined back into `stream` inside the call: all
 * results are ordered on `stream` as usual. The first call on a thread and
 * device creates those streams and their events; when the call is to be
 * captured into a CUDA graph, make one call before the capture. */
mgb_status mgb_block_bwd(const mgb_block_desc* desc, const mgb_block_weights* w,
                         const void* x, const void* dy, const void* saved, size_t saved_bytes,
                         void* dx, const mgb_block_grads* grads,
                         void* ws, size_t ws_bytes, void* stream);

/* Where the per-chunk statistics and the gradient of the cross-entropy are
 * computed (same results up to float32 rounding order). */
typedef enum {
  MGB_CE_STREAM = 0,  /* the logits GEMM stores a chunk's bf16 logits; streaming
                         kernels read them for the max / sum exp partials and
                         rewrite them into the gradient */
  MGB_CE_FUSED = 1,   /* the logits GEMM's epilogue keeps per-(token, 128-column
                         group) max / sum exp partials of its float32
                         accumulator and stores no logits; the recomputing
                         GEMM's epilogue writes the gradient directly */
  MGB_CE_RESIDENT = 2, /* as MGB_CE_FUSED for the partials, and the epilogue
                         also stores every chunk's bf16 logits into one
                         [tokens, vocab] workspace buffer (2 bytes per logit):
                         the backward rewrites them into the gradient in one
                         streaming pass and runs one input-gradient and one
                         weight-gradient GEMM over the whole vocabulary, with
                         no logits recomputed. Holds the full [tokens, vocab]
                         logits: outside the pages' memory bound */
  MGB_CE_BLOCKED = 3  /* tokens in blocks of token_block rows; per block, the
                         logits GEMM of every vocab chunk keeps per-(token,
                         128-column group) max / sum exp partials (as
                         MGB_CE_FUSED) and stores the block's bf16 logits
                         [token_block, vocab]; the partials are combined into
                         the block's LSE and losses; one streaming pass
                         rewrites the block's logits into G; then
                         d_hidden rows = G E (K split into ranges, float32
                         partial planes summed in fixed order) and
                         d_emb += G^T hidden (float32 accumulator across
                         blocks). Never more than one block of logits is
                         held and none is recomputed: the workspace is
                         O(token_block * vocab + vocab * hidden), whatever
                         the number of tokens */
} mgb_ce_mode;

/* Tied-embedding cross-entropy [P2 sections 3-4]. */
typedef struct {
  int32_t tokens, hidden, vocab;
  int32_t chunk;        /* vocab chunk; the last chunk may be ragged */
  int32_t dtype;        /* MGB_BF16 (hidden/emb/grads bf16) */
  float grad_scale;     /* dL/dloss_t for every token: 1/tokens for the mean */
  int32_t mode;         /* mgb_ce_mode */
  /* MGB_CE_RESIDENT and MGB_CE_BLOCKED, may be NULL: a stream (cudaStream_t
   * as void*) of the caller's for the weight gradient d_emb (BLOCKED: the last
   * block's part of it). It waits for the call's earlier work on `stream` and
   * is not joined back: d_emb, `hidden` and the workspace stay in use on it,
   * so the caller orders their next use after it (e.g. cudaStreamWaitEvent of
   * `stream` on an event recorded on it). The work that follows on `stream`
   * then overlaps d_emb. */
  void* emb_stream;
  /* MGB_CE_BLOCKED only: tokens per block (0 = 4096), rounded up to a
   * multiple of 256; the logits block takes 2 * token_block * vocab bytes of
   * the workspace. Other modes ignore it. */
  int32_t token_block;
} mgb_ce_desc;

mgb_status mgb_vocab_ce_sizes(const mgb_ce_desc* desc, size_t* ws_bytes);

/* logits l = hidden E^T ([T,H] x [V,H]^T), computed chunk by chunk; per chunk
 * the row max m_c, sum exp(l - m_c) and the target logit (0 unless the target
 * falls in the chunk) are kept; LSE = M + log sum_c s_c exp(m_c - M),
 * loss_t = LSE_t - target logit_t, loss_mean = mean_t loss_t. Backward:
 * G = (softmax(l) - onehot(target)) * grad_scale, d_hidden = G E,
 * d_emb = G^T hidden, again chunk by chunk (logits recomputed per chunk).
 * MGB_CE_FUSED keeps one (max, sum) partial per token and 128 vocab columns
 * instead of one per chunk; the combine is the same merge. MGB_CE_BLOCKED
 * walks the tokens in blocks (see mgb_ce_mode) and needs about
 * 2 * token_block * vocab + 4 * vocab * hidden bytes of workspace (the second
 * term only with d_emb and more than one block). MGB_CE_RESIDENT
 * needs a workspace of about 2 * tokens * vocab bytes (mgb_vocab_ce_sizes)
 * and runs the weight gradient on a library-owned second stream, joined back
 * into `stream` before the call returns (as mgb_block_bwd).
 *   targets [T] int32 in [0, vocab) (device); loss_per_token [T] f32;
 *   loss_mean: one f32 (device); lse [T] f32 or NULL;
 *   d_hidden [T,H], d_emb [V,H]: NULL skips that gradient (both NULL = fwd only). */
mgb_status mgb_vocab_ce_fwd_bwd(const mgb_ce_desc* desc, const void* hidden, const void* emb,
                                const int32_t* targets, float* loss_per_token, float* loss_mean,
                                float* lse, void* d_hidden, void* d_emb,
                                void* ws, size_t ws_bytes, void* stream);

/* ---- building blocks of the path (also used by the calls above) ---- */

typedef enum { MGB_K_MAJOR = 0, MGB_MN_MAJOR = 1 } mgb_major;

/* C[M,N] = alpha * op(A) op(B)^T (+ bias[N]) [(+ C if accumulate)]; float32
 * accumulation. A is [M,K] stored row-major with leading dim lda (K_MAJOR)
 * or stored [K,M] (MN_MAJOR); B likewise [N,K] / [K,N]. The dense
 * contractions of every linear layer [P1 section 2; P2 sections 1-2] and their
 * input/weight gradients are this product with one of the three operand
 * layouts (K/K forward, K/MN input grad, MN/MN weight grad).
 * dtype MGB_BF16: A, B, bias bf16; C bf16 unless c_f32 (then float32).
 * dtype MGB_F32: everything float32, on the CUDA cores (FFMA; see
 * mgb_gemm_f32_tc for the tensor-core form). `accumulate` needs c_f32 or
 * MGB_F32. */
typedef struct {
  int32_t m, n, k;
  int32_t a_major, b_major;   /* mgb_major */
  int64_t lda, ldb, ldc;      /* in elements */
  int32_t dtype;
  int32_t c_f32;
  int32_t accumulate;
  float alpha;
} mgb_gemm_desc;

mgb_status mgb_gemm(const mgb_gemm_desc* desc, const void* a, const void* b, const void* bias,
                    void* c, void* stream);

/* Fused epilogues of the same product, as the layer uses them [P1 section 2;
 * P2 section 1]. With acc = alpha * op(A) op(B)^T:
 *   MGB_EPI_STORE        C = acc (+ bias)                         (as mgb_gemm)
 *   MGB_EPI_BIAS_GELU    u = acc + bias; C = u; C2 = gelu_erf(u)  (C2 [M, N])
 *   MGB_EPI_BIAS_SWIGLU  u = acc + bias, the N columns interleaved gate/up in
 *                        blocks of glu_block; C = u [M, N];
 *                        C2 = silu(gate) * up [M, N/2]
 *   MGB_EPI_BIAS_RESID   C = resid + acc + bias                   (resid [M, N])
 *   MGB_EPI_DGELU        C = acc * gelu_erf'(aux)                 (aux = u [M, N])
 *   MGB_EPI_DSWIGLU      acc = d(activation) [M, N]; aux = u [M, 2N] interleaved;
 *                        C [M, 2N] = the interleaved (d gate, d up)
 *   MGB_EPI_F32          C (float32) = (accumulate ? C : 0) + acc (+ bias); C2,
 *                        if not NULL, = C rounded to dtype
 * bias, C2, resid and aux have the dtype of A and B (bf16 or float32); NULL for
 * the ones an epilogue does not use. `g.c_f32` is ignored (MGB_EPI_F32 selects
 * the float32 output); `g.accumulate` needs MGB_EPI_F32. glu_block: bf16 needs
 * a multiple of 32 that divides 128. Errors as mgb_gemm, plus
 * MGB_ERR_INVALID_ARG for an unknown epilogue or a missing pointer. */
typedef enum {
  MGB_EPI_STORE = 0,
  MGB_EPI_BIAS_GELU = 1,
  MGB_EPI_BIAS_SWIGLU = 2,
  MGB_EPI_BIAS_RESID = 3,
  MGB_EPI_DGELU = 4,
  MGB_EPI_DSWIGLU = 5,
  MGB_EPI_F32 = 6
} mgb_epilogue;

typedef struct {
  mgb_gemm_desc g;
  int32_t epilogue;  /* mgb_epilogue */
  int32_t glu_block;
  int64_t ldc2, ldr, ldaux; /* in elements */
} mgb_gemm_ex_desc;

mgb_status mgb_gemm_ex(const mgb_gemm_ex_desc* desc, const void* a, const void* b,
                       const void* bias, void* c, void* c2, const void* resid, const void* aux,
                       void* stream);

/* The float32 product of mgb_gemm_ex (desc->g.dtype MGB_F32, the same
 * operand layouts and epilogues) on the tensor cores [P1 section 2: the
 * float32 layer's linears]: each operand x is split into hi = x rounded to
 * TF32 (10 mantissa bits) and lo = x - hi rounded to TF32, and the product is
 * A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T (tcgen05 kind::tf32, float32
 * accumulation): rel. error about 1e-5 at K ~ 1000 (5.7e-5 at K 8192), where
 * one TF32 product gives a few 1e-4 and FFMA about 1e-6. The split
 * operands are written as K-major copies into `ws` (caller-owned, 256-byte
 * aligned, at least mgb_gemm_f32_tc_ws_bytes(m, n, k) bytes, overwritten).
 * mgb_block_fwd / mgb_block_bwd with dtype MGB_F32 run their GEMMs this way,
 * the split copies in their workspaces. Errors as mgb_gemm_ex, plus
 * MGB_ERR_WORKSPACE_TOO_SMALL. */
size_t mgb_gemm_f32_tc_ws_bytes(int32_t m, int32_t n, int32_t k);
mgb_status mgb_gemm_f32_tc(const mgb_gemm_ex_desc* desc, const void* a, const void* b,
                           const void* bias, void* c, void* c2, const void* resid,
                           const void* aux, void* ws, size_t ws_bytes, void* stream);

/* LayerNorm over the last dim [P1 section 2, F.layer_norm(x, (hidden,))]:
 * y = gamma*(x-mean)*rstd + beta, biased variance. mean/rstd [rows] f32
 * (may be NULL). gamma/beta NULL = no affine. */
mgb_status mgb_layernorm_fwd(int32_t rows, int32_t cols, int32_t dtype, float eps, const void* x,
                             const void* gamma, const void* beta, void* y, float* mean,
                             float* rstd, void* stream);

/* LayerNorm backward [P1 section 2, "end-to-end backward" through
 * F.layer_norm]: with xhat = (x - mean) * rstd and g = dy * gamma,
 *   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat)),
 *   dgamma = sum_rows dy * xhat,  dbeta = sum_rows dy.
 * x, dy, dres (may be NULL), dx: [rows, cols] of dtype; mean/rstd from the
 * forward; gamma NULL = no affine (then dgamma/dbeta must be NULL). dgamma,
 * dbeta (dtype, may be NULL) are summed over rows through float32 partials in
 * `ws` (size from mgb_layernorm_bwd_ws_bytes; deterministic order). */
size_t mgb_layernorm_bwd_ws_bytes(int32_t rows, int32_t cols);
mgb_status mgb_layernorm_bwd(int32_t rows, int32_t cols, int32_t dtype, const void* x,
                             const float* mean, const float* rstd, const void* gamma,
                             const void* dy, const void* dres, void* dx, void* dgamma, void* dbeta,
                             void* ws, size_t ws_bytes, void* stream);

/* LayerNorm backward for callers that cannot allocate device memory. The
 * pages have no counterpart; this is a library-side convenience.
 *
 * Some callers cannot obtain scratch memory at the point where they run this
 * operation: a serving engine that reserved all device memory up front and
 * forbids allocation while a request is in flight, or a plugin inside a host
 * framework that owns the device allocator and offers no workspace. Such a
 * caller cannot supply the `ws` buffer of mgb_layernorm_bwd. This entry point
 * computes the same result (same arguments minus ws/ws_bytes) and keeps the
 * float32 partial sums of dgamma/dbeta in a fixed array inside the library:
 *   - size: 2 x 64 x 16384 floats (8 MiB), held by every GPU that loads the
 *     library until the process exits; cols > 16384 with dgamma or dbeta
 *     requested returns MGB_ERR_UNSUPPORTED before any launch;
 *   - a call uses at most min(the partial rows mgb_layernorm_bwd would use,
 *     2^20 / cols) rows of the array (256 at cols = 4096; the kernel for rows
 *     of up to 1024 vectors combines its partials in clusters of CTAs and
 *     writes one row per cluster), so the backward still spreads over the
 *     whole GPU;
 *   - the library calls no cudaMalloc/cudaFree or allocating routine (keep
 *     the tracing of mgb_profile_enable off: when on, it creates CUDA events);
 *   - the first call on each device looks up the array's device address with
 *     that device current (again after the device's context was destroyed
 *     and created anew, e.g. by cudaDeviceReset); make that first call before
 *     any stream capture;
 *   - every call on a device shares the array: calls that may run at the same
 *     time on the GPU (different streams, no ordering between them) race and
 *     give wrong dgamma/dbeta; serialise them.
 * With fewer partial rows than mgb_layernorm_bwd for wide rows, the two entry
 * points agree to float32 rounding, not always bit for bit. MGB_FAULT=validate
 * makes it fail validation like every other entry point. */
mgb_status mgb_layernorm_bwd_noalloc(int32_t rows, int32_t cols, int32_t dtype, const void* x,
                                     const float* mean, const float* rstd, const void* gamma,
                                     const void* dy, const void* dres, void* dx, void* dgamma,
                                     void* dbeta, void* stream);

/* Attention core [P2 section 2]: q [B*S, nq*d] (head h at columns h*d), k, v
 * [B*S, nkv*d] (row stride ld_q / ld_kv elements, so they may be column slices
 * of one fused qkv buffer); o [B*S, nq*d]; lse [B, nq, S] f32. */
mgb_status mgb_attention_fwd(int32_t batch, int32_t seq, int32_t n_q_heads, int32_t n_kv_heads,
                             int32_t head_dim, int32_t causal, int32_t dtype,
                             const void* q, const void* k, const void* v, int64_t ld_q,
                             int64_t ld_kv, void* o, float* lse, void* stream);

/* Vocab-parallel embedding lookup [P2 section 3]: the table's rows [v0, v1)
 * are held as emb_shard [(v1 - v0), hidden] (row-major, the vocab shard of a
 * tensor-parallel rank; v0 = 0, v1 = vocab for the whole table). For each of
 * `tokens` ids (device int32): out[t] = emb_shard[ids[t] - v0] when
 * v0 <= ids[t] < v1, else a zero row - the masked lookup whose sum over the
 * shards is the full lookup. dtype MGB_BF16 or MGB_F32 for the table and out
 * (16-byte aligned, hidden a multiple of 8 / 4 elements); the copy is exact.
 * Errors: MGB_ERR_INVALID_ARG (sizes, v0 >= v1, NULL), MGB_ERR_MISALIGNED,
 * all before any launch. */
mgb_status mgb_embedding_fwd(int32_t tokens, int32_t hidden, int32_t v0, int32_t v1, int32_t dtype,
                             const int32_t* ids, const void* emb_shard, void* out, void* stream);

/* Bytes of the workspace of mgb_embedding_bwd (0 for invalid sizes). No
 * counterpart on the pages: it sizes the buffer below. */
size_t mgb_embedding_bwd_ws_bytes(int32_t tokens, int32_t v0, int32_t v1);

/* Backward of the lookup (its adjoint) [P2 section 3]: for every shard row v,
 * d_emb_shard[v - v0] = (accumulate ? d_emb_shard[v - v0] : 0) + the sum over
 * the tokens t with ids[t] = v of d_out[t] [tokens, hidden]. accumulate = 1
 * adds onto the existing contents, e.g. the output embedding's gradient from
 * mgb_vocab_ce_fwd_bwd when the input and output tables are tied; rows no
 * token hits are then left untouched (accumulate = 0 writes them as zeros).
 * Each row's tokens are summed in token order in float32 (deterministic, no
 * floating-point atomics), then rounded to dtype. `ws` (16-byte aligned,
 * caller-owned, at least mgb_embedding_bwd_ws_bytes) holds the per-row token
 * lists. Errors as mgb_embedding_fwd, plus MGB_ERR_WORKSPACE_TOO_SMALL. */
mgb_status mgb_embedding_bwd(int32_t tokens, int32_t hidden, int32_t v0, int32_t v1, int32_t dtype,
                             const int32_t* ids, const void* d_out, void* d_emb_shard,
                             int32_t accumulate, void* ws, size_t ws_bytes, void* stream);

/* The backward above in two steps, so that the part that depends on the ids
 * alone can run early (e.g. beside the forward, once the ids are known) and
 * the part that needs d_out is the row sums only [P2 section 3, as
 * mgb_embedding_bwd].
 *
 * mgb_embedding_bwd_prepare writes into `ws` (16-byte aligned, caller-owned, at
 * least mgb_embedding_bwd_ws_bytes(tokens, v0, v1)) the token order of the
 * shard's rows: each token's stable rank among the tokens with the same id,
 * the per-row counts scanned into row offsets, and the tokens placed row by
 * row in token order. It fills *plan (host memory) with tokens, v0, v1, ws and
 * ws_bytes; nothing is read back from the device. The ids are not read again.
 *
 * mgb_embedding_bwd_apply runs the row sums of mgb_embedding_bwd from a plan:
 * d_emb_shard[v - v0] = (accumulate ? d_emb_shard[v - v0] : 0) + the sum over
 * the plan's tokens t with ids[t] = v of d_out[t], in token order, in float32
 * (bit for bit the result of mgb_embedding_bwd with the same ids). A plan
 * serves any number of applies, in either mode, as long as its workspace is
 * left unchanged and each apply is ordered after the prepare (same stream, or
 * an event between the streams).
 * Errors: as mgb_embedding_bwd (a NULL plan or plan->ws is MGB_ERR_INVALID_ARG),
 * all before any launch. */
typedef struct {
  int32_t tokens, v0, v1;
  void* ws;
  size_t ws_bytes;
} mgb_embedding_bwd_plan;

mgb_status mgb_embedding_bwd_prepare(int32_t tokens, int32_t v0, int32_t v1, const int32_t* ids,
                                     void* ws, size_t ws_bytes, mgb_embedding_bwd_plan* plan,
                                     void* stream);
mgb_status mgb_embedding_bwd_apply(const mgb_embedding_bwd_plan* plan, int32_t hidden,
                                   int32_t dtype, const void* d_out, void* d_emb_shard,
                                   int32_t accumulate, void* stream);

/* Bytes of the workspace mgb_attention_bwd needs: two float32 planes
 * [batch * n_q_heads][seq rounded up to a multiple of 128] (LSE * log2(e) and
 * delta = rowsum(dO * O), per query; the padding holds +inf and 0), then the
 * float32 dQ accumulator [batch * seq][n_q_heads * 128] of the one-pass
 * backward (sized for head_dim up to 128). No counterpart on the pages: it
 * sizes the buffer below. 0 for negative sizes. */
size_t mgb_attention_bwd_ws_bytes(int32_t batch, int32_t seq, int32_t n_q_heads);

/* Attention core backward [P1 section 2, end-to-end backward]: given the
 * forward's q, k, v, o, lse and dO = dL/dO (same layouts; do [B*S, nq*d] with
 * row stride ld_do), writes dq (row stride ld_dq) and dk, dv (row stride
 * ld_dkv; the sum over the query heads of each GQA group). P is recomputed
 * from lse. `ws` (16-byte aligned, caller-owned, overwritten) holds the
 * per-query LSE and delta: at least mgb_attention_bwd_ws_bytes(batch, seq,
 * n_q_heads) bytes, else MGB_ERR_WORKSPACE_TOO_SMALL before any launch.
 * bf16, head_dim 128: one pass over key blocks forms dK, dV and each query
 * tile's share of dQ, added into the workspace's float32 accumulator by
 * reduce-add copies in no fixed order (so dq can differ between runs at
 * float32 rounding level), then rounded to bf16. MGB_DETERMINISTIC=1 (or
 * MGB_ATTN_BWD=split) in the environment, and head_dim 64, take two kernels
 * instead, the dQ kernel on a library-owned side stream beside the dK/dV
 * kernel, joined back into `stream` before the call returns; every sum is
 * then in a fixed order and runs repeat bit for bit. mgb_block_bwd inherits
 * both. */
mgb_status mgb_attention_bwd(int32_t batch, int32_t seq, int32_t n_q_heads, int32_t n_kv_heads,
                             int32_t head_dim, int32_t causal, int32_t dtype,
                             const void* q, const void* k, const void* v, int64_t ld_q,
                             int64_t ld_kv, const void* o, const float* lse, const void* dout,
                             int64_t ld_do, void* dq, void* dk, void* dv, int64_t ld_dq,
                             int64_t ld_dkv, void* ws, size_t ws_bytes, void* stream);

/* ---- status and diagnostics ---- */

const char* mgb_status_string(mgb_status s);

/* The generator's bytes at stream positions rng.offset .. + n - 1 of seed
 * rng.seed (any offset) into out[n] (device). */
mgb_status mgb_philox_bytes(uint64_t seed, uint64_t offset, uint64_t n, void* out, void* stream);

/* y = dropout(x) over a [rows, cols] site at state rng (element r*cols + c),
 * probability p in [0, 1) with a keep threshold of at least 1 (p below about
 * 0.998); x, y of dtype with leading dims ldx, ldy (y may be x). The same call
 * with the same rng is the backward (dx from dy). */
mgb_status mgb_dropout(int64_t rows, int64_t cols, int32_t dtype, float p, mgb_rng_state rng,
                       const void* x, int64_t ldx, void* y, int64_t ldy, void* stream);

/* Copies `bytes` from src to dst on `stream` (asynchronous; host pointers
 * must be pinned for the copy to overlap other work): how inputs in host
 * memory (a token batch, targets) reach the device buffers the calls above
 * take, and results (a loss) come back. No counterpart on the pages. */
mgb_status mgb_memcpy_async(void* dst, const void* src, size_t bytes, void* stream);

/* Synchronises `stream`, then returns and clears the current device's error
 * word (MGB_ERR_DEVICE_TIMEOUT if a bounded device wait ran out since the last
 * call; MGB_ERR_DEVICE_CHECK if a device-side check of the checking build
 * failed; else MGB_OK), or MGB_ERR_CUDA if the synchronisation failed. */
mgb_status mgb_device_status(void* stream);

/* Launches one block that waits on a device flag nothing ever sets, bounded
 * by `limit_ns` nanoseconds (<= 5e9), through the same bounded-wait routine the
 * kernels use; the wait runs out and records MGB_ERR_DEVICE_TIMEOUT in the
 * error word. Exists to test that path without hanging or faulting a GPU. */
mgb_status mgb_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* ---- tracing ----
 * Every kernel the library launches is counted; with profiling enabled each
 * launch (or group of launches of one step, e.g. a LayerNorm backward and its
 * partial-sum reduction) is bracketed by CUDA events on the launching stream,
 * grouped by kernel kind (names from mgb_profile_kind_name). Host-side state,
 * process-wide; reading synchronises the recorded events. */
uint64_t mgb_launch_count(void);
mgb_status mgb_profile_enable(int32_t on);
mgb_status mgb_profile_reset(void);
int32_t mgb_profile_kinds(void);
const char* mgb_profile_kind_name(int32_t kind);
mgb_status mgb_profile_read(int32_t kind, double* total_ms, int64_t* launches);

/* Library version (major*10000 + minor*100 + patch). */
int32_t mgb_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MGB_H */

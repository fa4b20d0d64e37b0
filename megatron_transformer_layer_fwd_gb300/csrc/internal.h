// Internal launch interfaces shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "../../include/mgb.h"

namespace mgb {

// Epilogue of the GEMM: what happens to acc[m][n] = alpha * sum_k A(m,k) B(n,k).
enum EpiMode : int {
  EPI_STORE = 0,        // C = acc (+ bias)
  EPI_BIAS_GELU = 1,    // u = acc + bias; C = u; C2 = gelu(u)
  EPI_BIAS_SWIGLU = 2,  // u = acc + bias (interleaved gate/up); C = u; C2 = silu(gate)*up
  EPI_BIAS_RESID = 3,   // C = resid + acc + bias
  EPI_DGELU = 4,        // C = acc * gelu'(aux)             (acc = da, aux = u)
  EPI_DSWIGLU = 5,      // C = interleaved [dgate | dup]     (acc = da, aux = u)
  EPI_F32 = 6,          // Cf = (accumulate ? Cf : 0) + acc (+ bias); optional C2 = bf16(Cf)
  // vocab cross-entropy, logits in float32 straight from the accumulator:
  EPI_CE_STATS = 7,     // no logits stored: per row and 128-column group g of the
                        // N columns, C[g*M + row] = max (natural-log units) and
                        // C2[g*M + row] = sum exp(acc - max) (both float32);
                        // target capture as EPI_STORE
  EPI_CE_GRAD = 8,      // C = bf16((exp(acc - ce_lse[row]) - [column = target]) * ce_scale)
};

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  int a_mn = 0, b_mn = 0;          // operand storage: 0 = K-major, 1 = MN-major
  const void* A = nullptr; int64_t lda = 0;
  const void* B = nullptr; int64_t ldb = 0;
  int dtype = MGB_BF16;            // operand / tensor dtype
  int epi = EPI_STORE;
  float alpha = 1.0f;
  void* C = nullptr; int64_t ldc = 0;       // main output (EPI_F32: float32)
  const void* bias = nullptr;               // [N] (dtype), may be null
  const void* resid = nullptr; int64_t ldr = 0;
  void* C2 = nullptr; int64_t ldc2 = 0;     // second output (dtype)
  const void* aux = nullptr; int64_t ldaux = 0;
  int glu_block = 128;
  int accumulate = 0;
  int prof_kind = -1;  // timing group (-1: by operand layout)
  // EPI_STORE only: for each row m whose target column tgt[m] - tgt_v0 lies in
  // [0, N), tgt_out[m] = that column's float32 value (before bf16 rounding)
  const int32_t* tgt = nullptr;
  int tgt_v0 = 0;
  float* tgt_out = nullptr;
  const float* ce_lse = nullptr;  // EPI_CE_GRAD: LSE per row
  float ce_scale = 1.0f;          // EPI_CE_GRAD: dL/dloss per token
  // EPI_CE_STATS only, may be null: the bf16 logits are also stored here
  void* keep = nullptr; int64_t ld_keep = 0;
  // EPI_BIAS_RESID only: dropout on acc + bias before the residual add, element
  // e = row * N + col of the site at stream state (drop_seed, drop_offset);
  // drop_thr 256 = off (dropout.cu has the definition)
  uint32_t drop_thr = 256;
  float drop_scale = 1.0f;
  uint64_t drop_seed = 0, drop_offset = 0;
  // EPI_DGELU / EPI_DSWIGLU with bf16 operands, may be null: bias-gradient
  // partials of the stored output. For each block p of 32 rows,
  // colsum_part[p * W + c] = the float32 sum over the block's rows (< M) of
  // output column c before bf16 rounding; W = N (DGELU) or 2N (DSWIGLU);
  // ceil(M / 32) blocks. colsum_reduce_launch folds them.
  float* colsum_part = nullptr;
  // split-K, EPI_F32 without accumulate only: the K dimension is cut into
  // k_splits ranges (whole 64-wide K blocks) and range s writes its float32
  // partial product to C + s * split_stride (elements); splitk_reduce_launch
  // sums the planes. gemm_splitk_count picks k_splits for a shape.
  int k_splits = 1;
  int64_t split_stride = 0;
  // EPI_F32 (no split, no C2) through TMA bulk copies of staged 32 x 32 boxes:
  // stores C, or with `accumulate` reduce-adds into C in L2 (no read of C by
  // the SMs). The order in which concurrent tiles add is not fixed, but each
  // element receives exactly one addition per call, so the result of one
  // call is the float32 sum C + acc as with the plain path.
  int f32_tma = 0;
  // EPI_CE_STATS / EPI_CE_GRAD, 0 = off: the N columns are vocab chunks of
  // n_chunk columns (the last may be narrower) handled in one launch; no
  // output tile straddles two chunks, and chunk c's statistics groups are
  // numbered from c * ceil(n_chunk / 128) (the same planes as one launch per
  // chunk); tgt_v0 must be 0 (targets are global columns)
  int n_chunk = 0;
  // dtype MGB_F32, may be null: scratch (256-byte aligned, at least
  // gemm_tf32_scratch_bytes(M, N, K)) for the hi / lo split copies of the
  // operands; with it the product runs as three TF32 tensor-core products
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
};
// Scratch bytes of the three-TF32 float32 GEMM of an M x N x K product.
size_t gemm_tf32_scratch_bytes(int M, int N, int K);

// A library-owned side stream per (host thread, device, slot) for work off a
// call's critical path (slot 0: weight and bias gradients; slot 1: the
// attention backward's dQ kernel beside its dK/dV kernel), so that its kernels
// fill the SMs the critical-path kernels leave idle in their last wave. fork()
// makes the side stream wait for everything issued on the caller's stream so
// far; join() (also run by the destructor, on every return path) makes the
// caller's stream wait for the side stream. Events are reused: a wait takes
// the event's state when it is enqueued. If the stream cannot be created the
// side work runs on the caller's stream. With an `external` stream the side
// work goes there instead and is not joined back (the caller orders it).
// The side streams have the lowest stream priority, so when SMs free up the
// block scheduler starts pending blocks of a caller's stream created with a
// higher priority first. MGB_SIDE_STREAMS=0 in the environment puts all side
// work on the caller's stream (serial order; for timing comparisons).
class SideLane {
 public:
  explicit SideLane(cudaStream_t main, cudaStream_t external = nullptr, int slot = 0,
                    bool serial = false)
      : main_(main), side_(main), ev_(nullptr) {
    if (serial && external == nullptr) return;  // side work on the caller's stream
    struct PerDevice {
      cudaStream_t side = nullptr;
      cudaEvent_t ev[kEvents] = {};
      bool failed = false;
    };
    thread_local PerDevice per[16][2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16 || slot < 0 || slot > 1) return;
    const char* env = getenv("MGB_SIDE_STREAMS");
    if (env != nullptr && env[0] == '0' && external == nullptr) return;
    PerDevice& d = per[dev][slot];
    if (d.side == nullptr && !d.failed) {
      int least = 0, greatest = 0;
      if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) least = 0;
      bool ok = cudaStreamCreateWithPriority(&d.side, cudaStreamNonBlocking, least) == cudaSuccess;
      for (int i = 0; ok && i < kEvents; ++i)
        ok = cudaEventCreateWithFlags(&d.ev[i], cudaEventDisableTiming) == cudaSuccess;
      if (!ok) {
        d.failed = true;
        d.side = nullptr;
        cudaGetLastError();
      }
    }
    if (d.side != nullptr) {
      side_ = external != nullptr ? external : d.side;
      ev_ = d.ev;
      detached_ = external != nullptr;
    }
  }
  ~SideLane() { join(); }
  cudaStream_t side() const { return side_; }
  mgb_status fork() {
    if (side_ == main_) return MGB_OK;
    cudaEvent_t e = ev_[next_++ % (kEvents - 1)];
    if (cudaEventRecord(e, main_) != cudaSuccess || cudaStreamWaitEvent(side_, e, 0) != cudaSuccess)
      return MGB_ERR_CUDA;
    forked_ = true;
    return MGB_OK;
  }
  mgb_status join() {
    if (!forked_ || detached_) return MGB_OK;
    forked_ = false;
    cudaEvent_t e = ev_[kEvents - 1];
    if (cudaEventRecord(e, side_) != cudaSuccess || cudaStreamWaitEvent(main_, e, 0) != cudaSuccess)
      return MGB_ERR_CUDA;
    return MGB_OK;
  }

 private:
  static constexpr int kEvents = 8;
  cudaStream_t main_, side_;
  cudaEvent_t* ev_;
  int next_ = 0;
  bool forked_ = false;
  bool detached_ = false;
};

// Validates operand geometry for the chosen path; returns MGB_OK or an error.
mgb_status gemm_check(const GemmArgs& g);
// K ranges for a bf16 M x N x K product on CTA-pair tiles so that the tiles
// of all ranges fill whole waves of the GPU (at most max_splits, and ranges
// of at least 8 K blocks); 1 when splitting does not help.
int gemm_splitk_count(int M, int N, int K, int max_splits);
// out[m, n] = bf16(sum over s < splits of part[s * split_stride + m * ldp + n])
// in fixed order; N a multiple of 8, 16-byte aligned rows.
mgb_status splitk_reduce_launch(int M, int N, int splits, const float* part, int64_t split_stride,
                                int64_t ldp, void* out, int64_t ldo, cudaStream_t st);
// Launches the bf16 tcgen05 GEMM (dtype MGB_BF16) or the float32 SIMT GEMM.
mgb_status gemm_launch(const GemmArgs& g, cudaStream_t st);

// LayerNorm over `cols` for `rows` rows; x, y of dtype; mean/rstd f32 (nullable).
mgb_status layernorm_fwd_launch(int rows, int cols, int dtype, float eps, const void* x,
                                const void* gamma, const void* beta, void* y, float* mean,
                                float* rstd, cudaStream_t st);
// dx = dres + LN_bwd(dy); partial dgamma/dbeta per block written to part
// ([2, nparts, cols] f32) then reduced into dgamma/dbeta (dtype, nullable).
mgb_status layernorm_bwd_launch(int rows, int cols, int dtype, const void* x, const float* mean,
                                const float* rstd, const void* gamma, const void* dy,
                                const void* dres, void* dx, void* dgamma, void* dbeta,
                                float* part, int nparts, cudaStream_t st);
int layernorm_bwd_parts(int rows);

// db[n] = sum_m dY[m, n] (dY row stride ld); partial buffer [nparts, N] f32.
mgb_status colsum_launch(int M, int N, int dtype, const void* dY, int64_t ld, void* db,
                         float* part, int nparts, cudaStream_t st);
int colsum_parts(int M);
// out[c] = sum over p < nparts of part[p * N + c], fixed order, as dtype; the
// partial buffer is scratch (overwritten). nparts 0: out = 0 (one row zeroed).
mgb_status colsum_reduce_launch(int nparts, int N, int dtype, float* part, void* out,
                                cudaStream_t st);

// Attention (fused online softmax); layouts as mgb_attention_fwd.
struct AttnArgs {
  int B, S, nq, nkv, d, causal, dtype;
  const void *q, *k, *v;
  int64_t ld_q, ld_kv;   // row strides (elements) of q and k/v
  void* o; int64_t ld_o;
  float* lse;            // [B, nq, S]
  // backward
  const void* dout; int64_t ld_do;
  void *dq, *dk, *dv; int64_t ld_dq, ld_dkv;
  float* delta;          // backward scratch (attn_bwd_ws_bytes)
  // dropout on the probabilities (bf16 path; drop_thr 256 = off): the forward
  // keeps element ((b*nq + h)*S + i)*Sp + j of stream (drop_seed, drop_offset),
  // Sp = S rounded up to 16, and writes the keep bits to drop_mask
  // [B*nq*S rows][attn_mask_words(S)] (bit j%32 of word j/32); the backward
  // reads the bits
  uint32_t drop_thr = 256;
  float drop_scale = 1.0f;
  uint64_t drop_seed = 0, drop_offset = 0;
  uint32_t* drop_mask = nullptr;
};
// Words per query row of the attention keep-bit mask (rows padded to 128 keys).
inline int attn_mask_words(int S) { return (S + 127) / 128 * 4; }
inline size_t attn_mask_bytes(int B, int nq, int S) {
  return 4 * (size_t)B * nq * S * attn_mask_words(S);
}
// The bf16 backward's workspace: two float32 planes [B * nq][pad] (LSE *
// log2(e), then delta) with rows padded to a multiple of 128 queries, then the
// one-pass backward's float32 dQ accumulator [B * S][nq * d] (room for d up
// to 128).
inline int attn_bwd_row_pad(int S) { return (S + 127) / 128 * 128; }
inline size_t attn_bwd_ws_bytes(int B, int S, int nq) {
  return 2 * sizeof(float) * (size_t)B * nq * attn_bwd_row_pad(S) +
         sizeof(float) * (size_t)B * S * nq * 128;
}
mgb_status attention_fwd_launch(const AttnArgs& a, cudaStream_t st);
mgb_status attention_bwd_launch(const AttnArgs& a, cudaStream_t st);
// The one-pass bf16 backward (dQ accumulated in float32 by TMA reduce-adds):
// whether it serves these arguments (head dim 128; not with
// MGB_DETERMINISTIC=1 or MGB_ATTN_BWD=split), and the pass itself.
bool attention_bwd_fused_ok(const AttnArgs& a);
// (runs after the pre-pass, which zeroes the accumulator)
mgb_status attention_tc_bwd_fused(const AttnArgs& a, cudaStream_t st);

// Cross-entropy streaming kernels over one logits chunk [T, C] (row stride ldl).
mgb_status ce_stats_launch(int T, int C, int v0, const void* logits, int64_t ldl,
                           const int32_t* targets, float* m, float* s, float* t, cudaStream_t st);
// Merges n_parts (max, sum exp) partials per token ([n_parts][T] each) and
// the target logits ([n_t][T], summed) into LSE, per-token loss and the mean
// (fixed-order reduction through block_loss [ceil(T / 256)] scratch).
// With more than kCeSplits partials, `split` ([2][kCeSplits][T] floats, or
// null for the one-stage merge) holds the per-range pairs of a first stage.
constexpr int kCeSplits = 32;
mgb_status ce_combine_launch(int T, int n_parts, const float* m, const float* s, int n_t,
                             const float* t, float* lse, float* loss, float* loss_mean,
                             float* block_loss, float* split, cudaStream_t st);
inline int ce_combine_blocks(int T) { return (T + 255) / 256; }
// Checking build (MGB_CHECK): records MGB_ERR_DEVICE_CHECK when a target id is
// outside [0, V); no launch in the normal build.
mgb_status ce_check_targets_launch(int T, int V, const int32_t* targets, cudaStream_t st);
// loss_mean = (sum of the first nb block sums, fixed order) / T.
mgb_status ce_mean_launch(int nb, int T, const float* block_loss, float* loss_mean,
                          cudaStream_t st);
mgb_status ce_grad_launch(int T, int C, int v0, void* logits, int64_t ldl, const int32_t* targets,
                          const float* lse, float scale, cudaStream_t st);

// Dropout (dropout.cu): keep threshold of probability p; y = dropout(x) over
// a [rows, cols] site at stream state (seed, offset); the raw byte stream.
uint32_t dropout_threshold(float p);
mgb_status dropout_launch(int64_t rows, int64_t cols, int dtype, float p, uint64_t seed,
                          uint64_t offset, const void* x, int64_t ldx, void* y, int64_t ldy,
                          cudaStream_t st);
mgb_status philox_bytes_launch(uint64_t seed, uint64_t offset, uint64_t n, void* out,
                               cudaStream_t st);

// Vocab-parallel embedding (shard rows [v0, v1)); layouts as mgb_embedding_fwd/bwd.
size_t embedding_bwd_ws(int T, int v0, int v1);
// The backward in two steps: the token order from the ids alone (the full row
// offsets, usable by both apply modes), then the row sums.
mgb_status embedding_bwd_prepare_launch(int T, int v0, int v1, const int32_t* ids, void* ws,
                                        cudaStream_t st);
mgb_status embedding_bwd_apply_launch(int T, int H, int dtype, int v0, int v1, const void* dout,
                                      void* d_emb, int accumulate, const void* ws,
                                      cudaStream_t st);
mgb_status embedding_fwd_launch(int T, int H, int dtype, int v0, int v1, const int32_t* ids,
                                const void* emb, void* out, cudaStream_t st);
mgb_status embedding_bwd_launch(int T, int H, int dtype, int v0, int v1, const int32_t* ids,
                                const void* dout, void* d_emb, int accumulate, void* ws,
                                cudaStream_t st);

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Device address of the current device's error word (nullptr on failure).
int* device_error_word();

// Host-side fault injection: true when MGB_FAULT=validate, which makes every
// entry point's argument validation fail before any launch.
bool fault_injected();
// MGB_OK when the current device is sm_103 (GB300), else MGB_ERR_ARCH /
// MGB_ERR_CUDA.
mgb_status check_arch();
// The current thread's CUDA driver context (a CUcontext), or nullptr. A
// per-device cache of device-symbol addresses is keyed on it, so a context
// that was destroyed and created again (cudaDeviceReset) is noticed.
void* current_cuda_context();

// Kernel kinds for timing (mgb_profile_*).
enum ProfKind : int {
  PROF_GEMM_FWD = 0, PROF_GEMM_DGRAD, PROF_GEMM_WGRAD, PROF_GEMM_F32, PROF_ATTN_FWD,
  PROF_ATTN_BWD, PROF_LN_FWD, PROF_LN_BWD, PROF_COLSUM, PROF_CE_STATS, PROF_CE_COMBINE,
  PROF_CE_GRAD, PROF_GEMM_CE_LOGITS, PROF_EMBEDDING, PROF_DROPOUT,
  // the CE's input-gradient (G E) and weight-gradient (G^T hidden) products
  PROF_GEMM_CE_DGRAD, PROF_GEMM_CE_WGRAD, PROF_SPLITK_REDUCE,
  // stages of the layer (CUDA events around groups of launches, not kernels):
  // attention sublayer forward (LN1, QKV, attention, output projection +
  // residual), MLP sublayer forward (LN2, fc1 + activation, fc2 + residual),
  // the whole backward (side streams joined)
  PROF_STAGE_ATTN, PROF_STAGE_FFN, PROF_STAGE_BWD,
  // token-blocked CE: one block's d_hidden and d_emb products, run side by
  // side (from the fork to the join, on the caller's stream)
  PROF_STAGE_CE_PRODUCTS, PROF_KINDS
};

// Counts `launches` kernel launches and, when profiling is on, brackets them
// with CUDA events on stream `st` (construct right before the launches).
// count_launches = false: a stage timer around launches that have their own
// scopes (counted once per stage in the profile, not in mgb_launch_count).
class LaunchScope {
 public:
  LaunchScope(int kind, cudaStream_t st, int launches = 1, bool count_launches = true);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  int kind_, launches_;
  cudaStream_t st_;
  void* a_;
};

}  // namespace mgb

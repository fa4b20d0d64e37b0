// Streaming kernels of the vocab-chunked cross-entropy.
//
// "02 - How a whole Transformer block is split", section 4: the loss is
// assembled from per-vocab-shard partials - the shard's row max, its sum of
// exp(l - max), and the target logit (nonzero only in the shard owning the
// target) - combined across shards by a max and two sums:
//   M = max_c m_c,  S = sum_c s_c exp(m_c - M),  LSE = M + log S,
//   loss_t = LSE_t - sum_c target_c.
// Backward is local per shard: G = (softmax - onehot(target)) * scale.
// Here the shards are vocab chunks processed one after another on one GPU.
//
//   ce_stats   one warp per token row of a [T, C] bf16 logits chunk: a single
//              pass of 16-byte loads with a running (max, sum) pair per lane
//              (rescaled only when the max passes the reference by more than
//              8 in log2 units: one exponential per logit), merged across the
//              warp.
//   ce_combine one thread per token: partials -> LSE, per-token loss; block
//              sums of the loss then summed in fixed order (deterministic).
// The same combine serves the partials the logits GEMM's epilogue writes when
// the statistics are fused into it (one partial per 128-column group).
//   ce_grad    one block per row: rewrites the logits chunk in place with G.
#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr int CE_THREADS = 256;

// merge running (max, sum) pairs in the log2 domain
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * exp2f(m - mn) + s2 * exp2f(m2 - mn);
  m = mn;
}

// One 8-value vector into a thread's running (max, sum) pair, log2 domain.
// The reference max moves only when the vector's max passes it by more than
// 8 (so terms stay below 2^8), which makes the rescale rare after the first
// vectors: one exponential per value.
__device__ __forceinline__ void ms_vec8(const uint4& w, float& m, float& s) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack_bf16x2(ww[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
  const float mx = fmaxf(fmax3(x[0], x[1], x[2]), fmax3(fmax3(x[3], x[4], x[5]), x[6], x[7])) * LOG2E;
  if (mx > m + 8.0f) {
    s = m == -INFINITY ? 0.0f : s * ex2_ftz(m - mx);
    m = mx;
  }
  if (m == -INFINITY) return;  // nothing but -inf so far
  const float nm = -m;
  float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    float e0, e1;
    fma2(e0, e1, x[i], x[i + 1], LOG2E, LOG2E, nm, nm);
    add2(a0, a1, a0, a1, ex2_ftz(e0), ex2_ftz(e1));
  }
  s += a0 + a1;
}

// One warp per token row (no block-wide barrier): each lane keeps eight
// 16-byte loads in flight and a running (max, sum) pair; the warp merges the
// pairs with shuffles.
__global__ void __launch_bounds__(CE_THREADS) ce_stats_kernel(int T, int C, int v0,
                                                               const bf16* __restrict__ logits,
                                                               int64_t ldl,
                                                               const int32_t* __restrict__ tgt,
                                                               float* m_out, float* s_out,
                                                               float* t_out) {
  const int row = blockIdx.x * (CE_THREADS / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;  // whole warps leave together
  const bf16* l = logits + (int64_t)row * ldl;
  const int nvec = C / 8;
  float m = -INFINITY, s = 0.0f;
  constexpr int U = 8;
  for (int v0i = lane; v0i < nvec; v0i += U * 32) {
    uint4 w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0i + u * 32;
      if (v < nvec) w[u] = __ldg(reinterpret_cast<const uint4*>(l) + v);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0i + u * 32 < nvec) ms_vec8(w[u], m, s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_merge(m, s, m2, s2);
  }
  if (lane == 0) {
    m_out[row] = m * LN2;
    s_out[row] = s;
    // rows whose target lies in this chunk already hold the float32 target
    // logit (written by the logits GEMM epilogue); the rest contribute 0
    const int tc = tgt[row] - v0;
    if (tc < 0 || tc >= C) t_out[row] = 0.0f;
  }
}

// One thread per token: merge its n_parts (max, sum) partials and n_t target
// logits; each block writes the sum of its tokens' losses (fixed order).
__global__ void __launch_bounds__(256) ce_combine_kernel(int T, int n_parts, const float* m,
                                                         const float* s, int n_t, const float* t,
                                                         float* lse, float* loss,
                                                         float* block_loss) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  float li = 0.0f;
  if (i < T) {
    float M = -INFINITY;
    for (int c = 0; c < n_parts; ++c) M = fmaxf(M, m[(int64_t)c * T + i]);
    float S = 0.0f, tl = 0.0f;
    for (int c = 0; c < n_parts; ++c) S += s[(int64_t)c * T + i] * expf(m[(int64_t)c * T + i] - M);
    for (int c = 0; c < n_t; ++c) tl += t[(int64_t)c * T + i];
    const float L = M + logf(S);
    lse[i] = L;
    li = L - tl;
    if (loss) loss[i] = li;
  }
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) li += __shfl_xor_sync(0xffffffffu, li, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = li;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int w = 0; w < 8; ++w) tot += red[w];
    block_loss[blockIdx.x] = tot;
  }
}

// First stage for many partials: split k of blockIdx.y merges partials
// [k*per, (k+1)*per) of each token (natural-log units) into one pair.
__global__ void __launch_bounds__(256) ce_merge_split_kernel(int T, int n_parts, int per,
                                                             const float* m, const float* s,
                                                             float* m2, float* s2) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T) return;
  const int c0 = blockIdx.y * per, c1 = min(n_parts, c0 + per);
  float M = -INFINITY;
  for (int c = c0; c < c1; ++c) M = fmaxf(M, m[(int64_t)c * T + i]);
  float S = 0.0f;
  if (M != -INFINITY)
    for (int c = c0; c < c1; ++c) S += s[(int64_t)c * T + i] * expf(m[(int64_t)c * T + i] - M);
  m2[(int64_t)blockIdx.y * T + i] = M;
  s2[(int64_t)blockIdx.y * T + i] = S;
}

// loss_mean = sum of the block sums (one warp, fixed order) / T
__global__ void ce_mean_kernel(int nb, int T, const float* block_loss, float* loss_mean) {
  float v = 0.0f;
  for (int b = threadIdx.x; b < nb; b += 32) v += block_loss[b];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (threadIdx.x == 0 && loss_mean) *loss_mean = T > 0 ? v / T : 0.0f;
}

__global__ void __launch_bounds__(CE_THREADS) ce_grad_kernel(int T, int C, int v0,
                                                              bf16* __restrict__ logits,
                                                              int64_t ldl,
                                                              const int32_t* __restrict__ tgt,
                                                              const float* __restrict__ lse,
                                                              float scale) {
  const int row = blockIdx.x;
  bf16* l = logits + (int64_t)row * ldl;
  const float L2 = lse[row] * LOG2E;
  const int tc = tgt[row] - v0;
  const int nvec = C / 8;
  constexpr int U = 4;  // 16-byte vectors in flight per thread
  for (int v0i = threadIdx.x; v0i < nvec; v0i += U * CE_THREADS) {
    uint4 w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0i + u * CE_THREADS;
      if (v < nvec) w[u] = *(reinterpret_cast<const uint4*>(l) + v);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0i + u * CE_THREADS;
      if (v >= nvec) break;
      uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_bf16x2(ww[i]);
        float g0 = ex2_ftz(fmaf(f.x, LOG2E, -L2));
        float g1 = ex2_ftz(fmaf(f.y, LOG2E, -L2));
        const int c0 = v * 8 + 2 * i;
        if (c0 == tc) g0 -= 1.0f;
        if (c0 + 1 == tc) g1 -= 1.0f;
        ww[i] = pack_bf16x2(g0 * scale, g1 * scale);
      }
      *(reinterpret_cast<uint4*>(l) + v) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
    }
  }
}

// Checking build: every target id lies in [0, vocab).
__global__ void ce_check_targets_kernel(int T, int V, const int32_t* __restrict__ tgt, int* err) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T; i += gridDim.x * blockDim.x)
    dcheck(tgt[i] >= 0 && tgt[i] < V, err);
}

}  // namespace

mgb_status ce_check_targets_launch(int T, int V, const int32_t* targets, cudaStream_t st) {
#if MGB_CHECK
  if (T > 0) {
    LaunchScope scope(PROF_CE_COMBINE, st);
    ce_check_targets_kernel<<<(T + 255) / 256 < 1024 ? (T + 255) / 256 : 1024, 256, 0, st>>>(
        T, V, targets, device_error_word());
  }
#else
  (void)T; (void)V; (void)targets; (void)st;
#endif
  return MGB_OK;
}

mgb_status ce_stats_launch(int T, int C, int v0, const void* logits, int64_t ldl,
                           const int32_t* targets, float* m, float* s, float* t, cudaStream_t st) {
  if (T == 0) return MGB_OK;
  LaunchScope scope(PROF_CE_STATS, st);
  constexpr int rows_per_block = CE_THREADS / 32;
  ce_stats_kernel<<<(T + rows_per_block - 1) / rows_per_block, CE_THREADS, 0, st>>>(
      T, C, v0, (const bf16*)logits, ldl, targets, m, s, t);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status ce_combine_launch(int T, int n_parts, const float* m, const float* s, int n_t,
                             const float* t, float* lse, float* loss, float* loss_mean,
                             float* block_loss, float* split, cudaStream_t st) {
  const int nb = ce_combine_blocks(T);
  const bool two = n_parts > kCeSplits && split != nullptr && nb > 0;
  LaunchScope scope(PROF_CE_COMBINE, st, (nb > 0 ? 1 : 0) + 1 + (two ? 1 : 0));
  if (two) {
    // many partials (one per 128 vocab columns): merge them in kCeSplits
    // parallel ranges first, then combine the per-range pairs
    const int per = (n_parts + kCeSplits - 1) / kCeSplits;
    float* m2 = split;
    float* s2 = split + (size_t)kCeSplits * T;
    ce_merge_split_kernel<<<dim3(nb, kCeSplits), 256, 0, st>>>(T, n_parts, per, m, s, m2, s2);
    m = m2;
    s = s2;
    n_parts = kCeSplits;
  }
  if (nb > 0)
    ce_combine_kernel<<<nb, 256, 0, st>>>(T, n_parts, m, s, n_t, t, lse, loss, block_loss);
  ce_mean_kernel<<<1, 32, 0, st>>>(nb, T, block_loss, loss_mean);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status ce_mean_launch(int nb, int T, const float* block_loss, float* loss_mean,
                          cudaStream_t st) {
  LaunchScope scope(PROF_CE_COMBINE, st);
  ce_mean_kernel<<<1, 32, 0, st>>>(nb, T, block_loss, loss_mean);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status ce_grad_launch(int T, int C, int v0, void* logits, int64_t ldl, const int32_t* targets,
                          const float* lse, float scale, cudaStream_t st) {
  if (T == 0) return MGB_OK;
  LaunchScope scope(PROF_CE_GRAD, st);
  ce_grad_kernel<<<T, CE_THREADS, 0, st>>>(T, C, v0, (bf16*)logits, ldl, targets, lse, scale);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

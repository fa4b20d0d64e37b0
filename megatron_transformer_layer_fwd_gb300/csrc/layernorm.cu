// LayerNorm over the hidden dimension (forward and backward) and column sums.
//
// "LLM Lab 06: build a Megatron-style Transformer Block from scratch",
// section 2: F.layer_norm(x, (hidden,)) - per token, mean and biased variance
// over the hidden features, eps 1e-5; optional affine gamma/beta.
//
// Forward: one block per row; each thread keeps up to 4 16-byte vectors of the
// row in registers (one global read, one write), warp-shuffle + shared-memory
// block reduction for the mean, then for the centred sum of squares (two-pass
// in registers; no E[x^2]-E[x]^2 cancellation).
// Backward (per row, xhat = (x - mean) * rstd, g = dy * gamma):
//   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat))
// rows are strided over a fixed number of blocks; each thread accumulates the
// dgamma = sum dy*xhat and dbeta = sum dy partials of its own columns in
// registers, written per block and reduced by a second small kernel.
// Column sums db[n] = sum_m dY[m, n] (bias gradients) use the same
// partial-then-reduce scheme with coalesced 16-byte row reads. Many partial
// rows (the backward's 1024) are folded in two stages: 16 splits of rows
// folded in place, then the split results.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

constexpr int MAXV = 4;  // 16-byte vectors per thread
// Widest row whose dgamma/dbeta partial sums fit one block's shared memory.
constexpr int kLnBwdMaxCols = 16384;

template <typename T> struct Vec;
template <> struct Vec<bf16> { static constexpr int N = 8; };
template <> struct Vec<float> { static constexpr int N = 4; };

template <typename T>
__device__ __forceinline__ void vload(const T* p, float* f) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = unpack_bf16x2(w[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  } else {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
}
template <typename T>
__device__ __forceinline__ void vstore(T* p, const float* f) {
  uint4 v;
  if constexpr (sizeof(T) == 2) {
    v.x = pack_bf16x2(f[0], f[1]); v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]); v.w = pack_bf16x2(f[6], f[7]);
  } else {
    v.x = __float_as_uint(f[0]); v.y = __float_as_uint(f[1]);
    v.z = __float_as_uint(f[2]); v.w = __float_as_uint(f[3]);
  }
  *reinterpret_cast<uint4*>(p) = v;
}

// Sum over the block; `red` holds >= 32 floats. All threads get the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

template <typename T>
__global__ void ln_fwd_kernel(int rows, int cols, float eps, const T* __restrict__ x,
                              const T* __restrict__ gamma, const T* __restrict__ beta,
                              T* __restrict__ y, float* __restrict__ mean_out,
                              float* __restrict__ rstd_out) {
  constexpr int VN = Vec<T>::N;
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int nvec = cols / VN;
  const T* xr = x + (int64_t)row * cols;
  float v[MAXV][VN];
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      vload(xr + vi * VN, v[i]);
#pragma unroll
      for (int j = 0; j < VN; ++j) s += v[i][j];
    }
  }
  const float mean = block_sum(s, red) / cols;
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
#pragma unroll
      for (int j = 0; j < VN; ++j) {
        const float d = v[i][j] - mean;
        ss += d * d;
      }
    }
  }
  const float var = block_sum(ss, red) / cols;
  const float rstd = rsqrtf(var + eps);
  T* yr = y + (int64_t)row * cols;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
    if (vi < nvec) {
      float o[VN];
      float g[VN], b[VN];
      if (gamma) vload(gamma + vi * VN, g);
      if (beta) vload(beta + vi * VN, b);
#pragma unroll
      for (int j = 0; j < VN; ++j) {
        float t = (v[i][j] - mean) * rstd;
        if (gamma) t *= g[j];
        if (beta) t += b[j];
        o[j] = t;
      }
      vstore(yr + vi * VN, o);
    }
  }
  if (threadIdx.x == 0) {
    if (mean_out) mean_out[row] = mean;
    if (rstd_out) rstd_out[row] = rstd;
  }
}

// Sum of a float2 over the block (one pass of shuffles + shared memory).
__device__ __forceinline__ float2 block_sum2(float2 v, float2* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float2 t = lane < nw ? red[lane] : make_float2(0.0f, 0.0f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    t.x += __shfl_xor_sync(0xffffffffu, t.x, o);
    t.y += __shfl_xor_sync(0xffffffffu, t.y, o);
  }
  return t;
}

// Row blocks stride over the rows; thread t owns the VPT 16-byte vectors
// t, t + blockDim, ... of every row, so gamma and the dgamma/dbeta partial sums
// of those columns stay in registers for the whole block. A row's x, dy and
// dres are all requested before the row reduction, so each thread keeps
// 3 * VPT loads in flight.
template <typename T, int VPT>
__device__ __forceinline__ void ln_bwd_rows(int rows, int cols, const T* __restrict__ x,
                                            const float* __restrict__ mean,
                                            const float* __restrict__ rstd,
                                            const T* __restrict__ gamma, const T* __restrict__ dy,
                                            const T* __restrict__ dres, T* __restrict__ dx,
                                            float* __restrict__ part) {
  constexpr int VN = Vec<T>::N;
  __shared__ float2 red[32];
  const int nvec = cols / VN;
  float gm[VPT][VN], pg[VPT][VN], pb[VPT][VN];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int vi = threadIdx.x + i * blockDim.x;
#pragma unroll
    for (int j = 0; j < VN; ++j) {
      gm[i][j] = 1.0f;
      pg[i][j] = pb[i][j] = 0.0f;
    }
    if (gamma && vi < nvec) vload(gamma + vi * VN, gm[i]);
  }
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const float mu = mean[row], rs = rstd[row];
    const int64_t ro = (int64_t)row * cols;
    float xv[VPT][VN], dv[VPT][VN], rv[VPT][VN];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
        vload(x + ro + vi * VN, xv[i]);
        vload(dy + ro + vi * VN, dv[i]);
        if (dres) vload(dres + ro + vi * VN, rv[i]);
      }
    }
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
#pragma unroll
        for (int j = 0; j < VN; ++j) {
          const float xh = (xv[i][j] - mu) * rs;
          const float g = dv[i][j] * gm[i][j];
          s1 += g;
          s2 += g * xh;
          pg[i][j] += dv[i][j] * xh;
          pb[i][j] += dv[i][j];
          xv[i][j] = xh;  // keep xhat
          dv[i][j] = g;   // keep g
        }
      }
    }
    const float2 tot = block_sum2(make_float2(s1, s2), red);
    const float mg = tot.x / cols;
    const float mgx = tot.y / cols;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
        float o[VN];
#pragma unroll
        for (int j = 0; j < VN; ++j) {
          o[j] = rs * (dv[i][j] - mg - xv[i][j] * mgx);
          if (dres) o[j] += rv[i][j];
        }
        vstore(dx + ro + vi * VN, o);
      }
    }
  }
  if (part) {
    float* pgr = part + (int64_t)blockIdx.x * cols;
    float* pbr = part + (int64_t)(gridDim.x + blockIdx.x) * cols;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
#pragma unroll
        for (int j = 0; j < VN; j += 4) {
          *reinterpret_cast<float4*>(pgr + vi * VN + j) =
              make_float4(pg[i][j], pg[i][j + 1], pg[i][j + 2], pg[i][j + 3]);
          *reinterpret_cast<float4*>(pbr + vi * VN + j) =
              make_float4(pb[i][j], pb[i][j + 1], pb[i][j + 2], pb[i][j + 3]);
        }
      }
    }
  }
}

// Rows of up to 1024 vectors: one vector per thread.
template <typename T, int VPT>
__global__ void ln_bwd_kernel(int rows, int cols, const T* __restrict__ x,
                              const float* __restrict__ mean, const float* __restrict__ rstd,
                              const T* __restrict__ gamma, const T* __restrict__ dy,
                              const T* __restrict__ dres, T* __restrict__ dx,
                              float* __restrict__ part) {
  ln_bwd_rows<T, VPT>(rows, cols, x, mean, rstd, gamma, dy, dres, dx, part);
}

// Wider rows (VPT 2 or 4 vectors per thread, up to 1024 threads): the register
// count is held to 64 a thread so a full block always launches; these spill a
// little instead.
template <typename T, int VPT>
__global__ void __launch_bounds__(1024, 1) ln_bwd_wide_kernel(
    int rows, int cols, const T* __restrict__ x, const float* __restrict__ mean,
    const float* __restrict__ rstd, const T* __restrict__ gamma, const T* __restrict__ dy,
    const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ part) {
  ln_bwd_rows<T, VPT>(rows, cols, x, mean, rstd, gamma, dy, dres, dx, part);
}

// out0[c] = sum_p part[p * stride, c] and out1[c] = sum_p part[half + p * stride, c]
// for p < nparts (rows of `cols` floats), written as T (nullable outputs
// skipped). Block (32 x 8): lane = column (coalesced 128-byte rows of the
// partial buffer), the 8 warps split the partials, fixed order of summation
// (deterministic).
template <typename T>
__global__ void reduce_parts_kernel(int nparts, int stride, int64_t half, int cols,
                                    const float* __restrict__ part, T* __restrict__ out0,
                                    T* __restrict__ out1) {
  __shared__ float red[2][8][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  float s0 = 0.0f, s1 = 0.0f;
  if (c < cols) {
    for (int p = threadIdx.y; p < nparts; p += 8) {
      const int64_t o = (int64_t)p * stride * cols + c;
      if (out0) s0 += part[o];
      if (out1) s1 += part[half + o];
    }
  }
  red[0][threadIdx.y][threadIdx.x] = s0;
  red[1][threadIdx.y][threadIdx.x] = s1;
  __syncthreads();
  if (threadIdx.y == 0 && c < cols) {
    float a = 0.0f, b = 0.0f;
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      a += red[0][y][threadIdx.x];
      b += red[1][y][threadIdx.x];
    }
    if (out0) out0[c] = from_f<T>(a);
    if (out1) out1[c] = from_f<T>(b);
  }
}

// First stage for many partial rows: split blockIdx.y folds rows
// [p0, p0 + per) of 128 columns (four per lane, 16-byte loads) into row p0,
// in place, and the same rows of the second half when `two` is set. Each block
// alone reads and writes its rows and columns, so the in-place write races
// with nothing. Fixed order of summation.
__global__ void __launch_bounds__(256) fold_parts_kernel(int nparts, int per, int cols,
                                                         float* __restrict__ part, int two) {
  __shared__ float4 red[2][8][32];
  const int c = (blockIdx.x * 32 + threadIdx.x) * 4;
  const int p0 = blockIdx.y * per, p1 = min(nparts, p0 + per);
  const int64_t half = (int64_t)nparts * cols;
  float4 a0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), a1 = a0;
  if (c < cols) {
    for (int p = p0 + threadIdx.y; p < p1; p += 8) {
      const float4 v = *reinterpret_cast<const float4*>(part + (int64_t)p * cols + c);
      a0.x += v.x; a0.y += v.y; a0.z += v.z; a0.w += v.w;
      if (two) {
        const float4 w = *reinterpret_cast<const float4*>(part + half + (int64_t)p * cols + c);
        a1.x += w.x; a1.y += w.y; a1.z += w.z; a1.w += w.w;
      }
    }
  }
  red[0][threadIdx.y][threadIdx.x] = a0;
  red[1][threadIdx.y][threadIdx.x] = a1;
  __syncthreads();
  if (threadIdx.y == 0 && c < cols && p0 < p1) {
    float4 s0 = red[0][0][threadIdx.x], s1 = red[1][0][threadIdx.x];
#pragma unroll
    for (int y = 1; y < 8; ++y) {
      const float4 u = red[0][y][threadIdx.x], w = red[1][y][threadIdx.x];
      s0.x += u.x; s0.y += u.y; s0.z += u.z; s0.w += u.w;
      s1.x += w.x; s1.y += w.y; s1.z += w.z; s1.w += w.w;
    }
    *reinterpret_cast<float4*>(part + (int64_t)p0 * cols + c) = s0;
    if (two) *reinterpret_cast<float4*>(part + half + (int64_t)p0 * cols + c) = s1;
  }
}

constexpr int kFoldSplits = 16;
// Partial counts from which the reduction folds in two stages.
bool fold_first(int nparts, int cols) { return nparts >= 8 * kFoldSplits && cols % 4 == 0; }
int reduce_launches(int nparts, int cols) { return fold_first(nparts, cols) ? 2 : 1; }

// out0/out1 from [2][nparts][cols] float32 partials (the second half only read
// when out1 is set); the partial buffer may be overwritten (first stage).
template <typename T>
void reduce_parts_go(int nparts, int cols, float* part, T* out0, T* out1, cudaStream_t st) {
  const int64_t half = (int64_t)nparts * cols;
  const dim3 block(32, 8);
  if (fold_first(nparts, cols)) {
    const int per = (nparts + kFoldSplits - 1) / kFoldSplits;
    const int splits = (nparts + per - 1) / per;
    fold_parts_kernel<<<dim3((cols + 127) / 128, splits), block, 0, st>>>(nparts, per, cols, part,
                                                                          out1 != nullptr);
    reduce_parts_kernel<T><<<(cols + 31) / 32, block, 0, st>>>(splits, per, half, cols, part,
                                                               out0, out1);
  } else {
    reduce_parts_kernel<T><<<(cols + 31) / 32, block, 0, st>>>(nparts, 1, half, cols, part, out0,
                                                               out1);
  }
}

// part[p, n] = sum over rows m in split p of dY[m, n]; block (32 x 8): x covers
// 32 vectors of a row, y strides rows.
template <typename T>
__global__ void colsum_kernel(int M, int N, const T* __restrict__ dY, int64_t ld,
                              float* __restrict__ part) {
  constexpr int VN = Vec<T>::N;
  __shared__ float red[8][32 * 8 + 1];
  const int n = (blockIdx.x * 32 + threadIdx.x) * VN;
  float acc[VN];
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = 0.0f;
  const int rows_per = (M + gridDim.y - 1) / gridDim.y;
  const int r0 = blockIdx.y * rows_per, r1 = min(M, r0 + rows_per);
  if (n < N) {
    // four rows' loads in flight per thread before they are summed
    int m = r0 + threadIdx.y;
    for (; m + 24 < r1; m += 32) {
      float v[4][VN];
#pragma unroll
      for (int u = 0; u < 4; ++u) vload(dY + (int64_t)(m + 8 * u) * ld + n, v[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < VN; ++j) acc[j] += v[u][j];
    }
    for (; m < r1; m += 8) {
      float v[VN];
      vload(dY + (int64_t)m * ld + n, v);
#pragma unroll
      for (int j = 0; j < VN; ++j) acc[j] += v[j];
    }
  }
#pragma unroll
  for (int j = 0; j < VN; ++j) red[threadIdx.y][threadIdx.x * VN + j] = acc[j];
  __syncthreads();
  if (threadIdx.y == 0 && n < N) {
#pragma unroll
    for (int j = 0; j < VN; ++j) {
      float s = 0.0f;
#pragma unroll
      for (int y = 0; y < 8; ++y) s += red[y][threadIdx.x * VN + j];
      part[(int64_t)blockIdx.y * N + n + j] = s;
    }
  }
}

int ln_threads(int cols, int vn) {
  const int nvec = cols / vn;
  int t = (nvec + MAXV - 1) / MAXV;
  t = ((t + 31) / 32) * 32;
  return t < 32 ? 32 : t;
}

}  // namespace

// Row blocks of the backward: about one resident wave (several blocks per SM)
// to hide the latency of the per-row reductions; each writes one partial
// dgamma/dbeta row.
int layernorm_bwd_parts(int rows) { return rows < 1024 ? (rows > 0 ? rows : 1) : 1024; }
int colsum_parts(int M) { return M < 64 * 8 ? 1 : 64; }

mgb_status layernorm_fwd_launch(int rows, int cols, int dtype, float eps, const void* x,
                                const void* gamma, const void* beta, void* y, float* mean,
                                float* rstd, cudaStream_t st) {
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  if (rows < 0 || cols <= 0 || cols % vn) return MGB_ERR_INVALID_ARG;
  const int threads = ln_threads(cols, vn);
  if (threads > 1024) return MGB_ERR_UNSUPPORTED;
  if (rows == 0) return MGB_OK;
  LaunchScope scope(PROF_LN_FWD, st);
  if (dtype == MGB_BF16)
    ln_fwd_kernel<bf16><<<rows, threads, 0, st>>>(
        rows, cols, eps, (const bf16*)x, (const bf16*)gamma, (const bf16*)beta, (bf16*)y, mean, rstd);
  else
    ln_fwd_kernel<float><<<rows, threads, 0, st>>>(rows, cols, eps, (const float*)x,
                                                    (const float*)gamma, (const float*)beta,
                                                    (float*)y, mean, rstd);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

namespace {

template <typename T, int VPT>
void ln_bwd_go(int nparts, int threads, int rows, int cols, const void* x, const float* mean,
               const float* rstd, const void* gamma, const void* dy, const void* dres, void* dx,
               float* part, cudaStream_t st) {
  if constexpr (VPT == 1)
    ln_bwd_kernel<T, 1><<<nparts, threads, 0, st>>>(rows, cols, (const T*)x, mean, rstd,
                                                    (const T*)gamma, (const T*)dy,
                                                    (const T*)dres, (T*)dx, part);
  else
    ln_bwd_wide_kernel<T, VPT><<<nparts, threads, 0, st>>>(rows, cols, (const T*)x, mean, rstd,
                                                           (const T*)gamma, (const T*)dy,
                                                           (const T*)dres, (T*)dx, part);
}

template <typename T>
mgb_status ln_bwd_dispatch(int nparts, int rows, int cols, const void* x, const float* mean,
                           const float* rstd, const void* gamma, const void* dy, const void* dres,
                           void* dx, float* part, cudaStream_t st) {
  // one 16-byte vector per thread (64 registers: full occupancy), two or four
  // for rows wider than 1024 vectors
  const int nvec = cols / Vec<T>::N;
  auto thr = [&](int vpt) { return ((nvec + vpt - 1) / vpt + 31) / 32 * 32; };
  if (nvec <= 1024)
    ln_bwd_go<T, 1>(nparts, thr(1), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  else if (nvec <= 2048)
    ln_bwd_go<T, 2>(nparts, thr(2), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  else if (nvec <= 4096)
    ln_bwd_go<T, 4>(nparts, thr(4), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  else
    return MGB_ERR_UNSUPPORTED;
  return MGB_OK;
}

}  // namespace

mgb_status layernorm_bwd_launch(int rows, int cols, int dtype, const void* x, const float* mean,
                                const float* rstd, const void* gamma, const void* dy,
                                const void* dres, void* dx, void* dgamma, void* dbeta,
                                float* part, int nparts, cudaStream_t st) {
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  if (rows < 0 || cols <= 0 || cols % vn) return MGB_ERR_INVALID_ARG;
  if (cols / vn > 4096) return MGB_ERR_UNSUPPORTED;
  const bool want = (dgamma || dbeta) && part;
  // the dgamma/dbeta partial rows of the workspace are sized for this width
  if (want && cols > kLnBwdMaxCols) return MGB_ERR_UNSUPPORTED;
  if (rows == 0) nparts = 1;
  LaunchScope scope(PROF_LN_BWD, st, (rows > 0 ? 1 : 0) + (want ? reduce_launches(nparts, cols) : 0));
  if (rows > 0) {
    const mgb_status s =
        dtype == MGB_BF16
            ? ln_bwd_dispatch<bf16>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                                    want ? part : nullptr, st)
            : ln_bwd_dispatch<float>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                                     want ? part : nullptr, st);
    if (s != MGB_OK) return s;
  } else if (want) {
    cudaMemsetAsync(part, 0, sizeof(float) * 2 * cols, st);
  }
  if (want) {
    if (dtype == MGB_BF16)
      reduce_parts_go<bf16>(nparts, cols, part, (bf16*)dgamma, (bf16*)dbeta, st);
    else
      reduce_parts_go<float>(nparts, cols, part, (float*)dgamma, (float*)dbeta, st);
  }
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

// ------------------------------------------- LayerNorm backward, no allocation
// Scratch of mgb_layernorm_bwd_noalloc: the float32 partial sums of dgamma and
// dbeta, [2][nparts][cols] in a file-scope device array of kNoAllocFloats
// floats (8 MiB). Every GPU that loads the library holds it until the process
// exits, and every call on a device shares it. A call with cols columns uses
// nparts = min(the workspace version's row blocks, kNoAllocFloats / (2 cols))
// partial rows: 256 at cols 4096, 64 at the widest row, 16384.
constexpr int kNoAllocFloats = 2 * 64 * 16384;
constexpr int kNoAllocMaxCols = 16384;
static __device__ __align__(256) float g_ln_bwd_scratch[kNoAllocFloats];

// Device address of g_ln_bwd_scratch on the current device. Looked up on the
// first call on each device, with that device current, and again only when
// the device's context changed (a reset device gets a new one); host code
// never passes the symbol itself to a kernel.
static float* ln_bwd_scratch_address() {
  static float* addr[64] = {};
  static void* ctx_of[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  void* ctx = current_cuda_context();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == nullptr || ctx_of[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ln_bwd_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(p);
    ctx_of[dev] = current_cuda_context();
  }
  return addr[dev];
}

// Partial rows the no-allocation backward uses for `rows` x `cols`.
static int noalloc_parts(int rows, int cols) {
  const int fit = kNoAllocFloats / (2 * (cols > 0 ? cols : 1));
  const int want = layernorm_bwd_parts(rows);
  return want < fit ? want : fit;
}

mgb_status colsum_launch(int M, int N, int dtype, const void* dY, int64_t ld, void* db,
                         float* part, int nparts, cudaStream_t st) {
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  if (N % vn || ld % vn) return MGB_ERR_INVALID_ARG;
  if (N == 0) return MGB_OK;
  if (M == 0) nparts = 1;
  LaunchScope scope(PROF_COLSUM, st, (M == 0 ? 0 : 1) + reduce_launches(nparts, N));
  if (M == 0) {
    cudaMemsetAsync(part, 0, sizeof(float) * N, st);
  } else {
    dim3 grid((N / vn + 31) / 32, nparts);
    dim3 block(32, 8);
    if (dtype == MGB_BF16)
      colsum_kernel<bf16><<<grid, block, 0, st>>>(M, N, (const bf16*)dY, ld, part);
    else
      colsum_kernel<float><<<grid, block, 0, st>>>(M, N, (const float*)dY, ld, part);
  }
  if (dtype == MGB_BF16)
    reduce_parts_go<bf16>(nparts, N, part, (bf16*)db, nullptr, st);
  else
    reduce_parts_go<float>(nparts, N, part, (float*)db, nullptr, st);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status colsum_reduce_launch(int nparts, int N, int dtype, float* part, void* out,
                                cudaStream_t st) {
  if (N < 0 || nparts < 0) return MGB_ERR_INVALID_ARG;
  if (N == 0) return MGB_OK;
  if (nparts == 0) {
    if (cudaMemsetAsync(part, 0, sizeof(float) * N, st) != cudaSuccess) return MGB_ERR_CUDA;
    nparts = 1;
  }
  LaunchScope scope(PROF_COLSUM, st, reduce_launches(nparts, N));
  if (dtype == MGB_BF16)
    reduce_parts_go<bf16>(nparts, N, part, (bf16*)out, nullptr, st);
  else
    reduce_parts_go<float>(nparts, N, part, (float*)out, nullptr, st);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

extern "C" mgb_status mgb_layernorm_bwd_noalloc(int32_t rows, int32_t cols, int32_t dtype,
                                                const void* x, const float* mean,
                                                const float* rstd, const void* gamma,
                                                const void* dy, const void* dres, void* dx,
                                                void* dgamma, void* dbeta, void* stream) {
  using namespace mgb;
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (rows < 0 || cols < 1 || !x || !mean || !rstd || !dy || !dx) return MGB_ERR_INVALID_ARG;
  if (!gamma && (dgamma || dbeta)) return MGB_ERR_INVALID_ARG;
  const void* ps[] = {x, mean, rstd, gamma, dy, dres, dx, dgamma, dbeta};
  for (const void* q : ps)
    if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return MGB_ERR_MISALIGNED;
  const bool want = dgamma || dbeta;
  // at least one partial row of the widest allowed row must fit the array
  if (want && cols > kNoAllocMaxCols) return MGB_ERR_UNSUPPORTED;
  const mgb_status arch = check_arch();
  if (arch != MGB_OK) return arch;
  float* part = nullptr;
  if (want) {
    part = ln_bwd_scratch_address();
    if (part == nullptr) return MGB_ERR_CUDA;
  }
  // each row block overwrites its whole partial row, so nothing left in the
  // array by an earlier call is read (rows == 0 zeroes the one row it reduces)
  const int nparts = want ? noalloc_parts(rows, cols) : layernorm_bwd_parts(rows);
  return layernorm_bwd_launch(rows, cols, dtype, x, mean, rstd, gamma, dy, dres, dx, dgamma, dbeta,
                              part, nparts, reinterpret_cast<cudaStream_t>(stream));
}

// LayerNorm over the hidden dimension (forward and backward) and column sums.
//
// "LLM Lab 06: build a Megatron-style Transformer Block from scratch",
// section 2: F.layer_norm(x, (hidden,)) - per token, mean and biased variance
// over the hidden features, eps 1e-5; optional affine gamma/beta.
//
// Forward: for bf16 rows of 256..4096 columns, rows streamed into a shared-
// memory ring by bulk copies and normalised one warp per row (ln_fwd_tma);
// otherwise one warp per row from registers, or one block per row (each
// thread up to 4 16-byte vectors). Mean, then the centred sum of squares, both
// from registers (two passes, no E[x^2]-E[x]^2 cancellation).
// Backward (per row, xhat = (x - mean) * rstd, g = dy * gamma):
//   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat))
// rows are strided over a fixed number of blocks; each thread accumulates the
// dgamma = sum dy*xhat and dbeta = sum dy partials of its own columns in
// registers. Rows of up to 1024 vectors stream through per-thread
// asynchronous copies (ln_bwd_async), and clusters of four CTAs combine their
// partials in distributed shared memory; a second small kernel sums the
// partial rows in a fixed order.
// Column sums db[n] = sum_m dY[m, n] (bias gradients) use the same
// partial-then-reduce scheme with coalesced 16-byte row reads. Many partial
// rows are folded in two stages: 16 splits of rows folded in place, then the
// split results.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

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
__device__ __forceinline__ void vunpack(const uint4& v, float* f) {
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

// Forward, one warp per row, bf16 rows of VPL * 256 elements (each lane holds
// VPL 16-byte vectors: columns 8 * (lane + 32 * i) .. + 7). Persistent warps
// stride over the rows and issue the next row's loads before normalising the
// current one, so about two rows per warp are in flight and the row's
// reductions (warp shuffles only, no block barrier) overlap that traffic.
// Two-pass mean / variance from registers, as the block kernel.
__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = unpack_bf16x2(w[j]);
    v[2 * j] = t.x;
    v[2 * j + 1] = t.y;
  }
}

template <int VPL>
__global__ void __launch_bounds__(256) ln_fwd_warp_kernel(int rows, int cols, float eps,
                                                          const bf16* __restrict__ x,
                                                          const bf16* __restrict__ gamma,
                                                          const bf16* __restrict__ beta,
                                                          bf16* __restrict__ y,
                                                          float* __restrict__ mean_out,
                                                          float* __restrict__ rstd_out) {
  const int lane = threadIdx.x & 31;
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const float inv_cols = 1.0f / (float)cols;
  uint4 cur[VPL], nxt[VPL];
  int row = wid;
  if (row < rows) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)row * cols);
#pragma unroll
    for (int i = 0; i < VPL; ++i) cur[i] = __ldg(xr + lane + 32 * i);
  }
  for (; row < rows; row += nw) {
    const int nrow = row + nw;
    if (nrow < rows) {
      const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)nrow * cols);
#pragma unroll
      for (int i = 0; i < VPL; ++i) nxt[i] = __ldg(xr + lane + 32 * i);
    }
    // the row stays packed (bf16 pairs) in registers and is unpacked on each
    // of the three passes: half the registers of a float copy
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      float v[8];
      unpack8(cur[i], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) s += v[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s * inv_cols;
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      float v[8];
      unpack8(cur[i], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = v[j] - mean;
        ss += d * d;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = rsqrtf(ss * inv_cols + eps);
    uint4* yr = reinterpret_cast<uint4*>(y + (int64_t)row * cols);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int c = 8 * (lane + 32 * i);
      float g[8], b[8];
      if (gamma) vload(gamma + c, g);
      if (beta) vload(beta + c, b);
      float o8[8], v[8];
      unpack8(cur[i], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float t = (v[j] - mean) * rstd;
        if (gamma) t *= g[j];
        if (beta) t += b[j];
        o8[j] = t;
      }
      uint4 ov;
      ov.x = pack_bf16x2(o8[0], o8[1]); ov.y = pack_bf16x2(o8[2], o8[3]);
      ov.z = pack_bf16x2(o8[4], o8[5]); ov.w = pack_bf16x2(o8[6], o8[7]);
      yr[lane + 32 * i] = ov;
    }
    if (lane == 0) {
      if (mean_out) mean_out[row] = mean;
      if (rstd_out) rstd_out[row] = rstd;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) cur[i] = nxt[i];
  }
}

template <int VPL>
void ln_fwd_warp_go(int rows, int cols, float eps, const void* x, const void* gamma,
                    const void* beta, void* y, float* mean, float* rstd, cudaStream_t st) {
  // persistent: as many 8-warp blocks as are resident at once (by the
  // kernel's registers), never more than the rows need
  static int per_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (per_sm[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ln_fwd_warp_kernel<VPL>, 256, 0) !=
            cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = 1;
    }
    per_sm[dev] = n;
  }
  const int want_blocks = (rows + 7) / 8;
  const int cap = per_sm[dev] * device_sm_count();
  const int blocks = want_blocks < cap ? want_blocks : cap;
  ln_fwd_warp_kernel<VPL><<<blocks, 256, 0, st>>>(rows, cols, eps, (const bf16*)x,
                                                  (const bf16*)gamma, (const bf16*)beta, (bf16*)y,
                                                  mean, rstd);
}

// ------------------------------------------------ rows streamed by TMA bulk copies
// The two bf16 kernels below keep their rows in a ring of shared-memory slots
// filled by cp.async.bulk copies (one producer lane per CTA, completion on an
// mbarrier per slot), so many rows per SM are in flight without registers
// holding them. Every wait is bounded; a wait that runs out records the
// error, sets the CTA's abort flag, and the CTA waits 10 ms for copies still
// in flight before it exits.
constexpr int kLnConsumers = 8;  // consumer warps per CTA (plus one producer warp)

__device__ __forceinline__ void ln_abort_drain(volatile int* abort) {
  __syncthreads();
  if (*abort && threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
}

// Forward: consumer warp w of the CTA normalises the CTA's rows i = w, w + 8,
// ... (row = blockIdx.x + i * gridDim.x), each from slot i % nslot; it copies
// the row into registers (VPL 16-byte vectors per lane) and frees the slot
// before the reductions, then writes y with 16-byte stores.
template <int VPL>
__global__ void __launch_bounds__(32 * (1 + kLnConsumers), VPL >= 16 ? 1 : 2) ln_fwd_tma_kernel(
    int rows, int cols, float eps, const bf16* __restrict__ x, const bf16* __restrict__ gamma,
    const bf16* __restrict__ beta, bf16* __restrict__ y, float* __restrict__ mean_out,
    float* __restrict__ rstd_out, int nslot, int* err) {
  extern __shared__ __align__(128) uint8_t ln_smem[];
  const uint32_t slot_bytes = (uint32_t)cols * 2;
  const uint32_t slots = smem_u32(ln_smem);
  const uint32_t full0 = slots + nslot * slot_bytes;  // 8-byte aligned (slot_bytes % 16 == 0)
  const uint32_t empty0 = full0 + 8 * nslot;
  volatile int* abort = reinterpret_cast<volatile int*>(ln_smem + nslot * slot_bytes + 16 * nslot);
  // gamma and beta of the whole row as float32 (1 and 0 when absent), staged
  // once (16-byte aligned after the flag)
  float4* sgb = reinterpret_cast<float4*>(ln_smem + nslot * slot_bytes + 16 * nslot + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = cols / 8;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nslot; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    fence_mbar_init();
    *abort = 0;
  }
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float g[8], b[8];
    if (gamma) {
      unpack8(reinterpret_cast<const uint4*>(gamma)[v], g);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) g[e] = 1.0f;
    }
    if (beta) {
      unpack8(reinterpret_cast<const uint4*>(beta)[v], b);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) b[e] = 0.0f;
    }
    sgb[2 * v] = make_float4(g[0], g[1], g[2], g[3]);
    sgb[2 * v + 1] = make_float4(g[4], g[5], g[6], g[7]);
    sgb[2 * (nvec + v)] = make_float4(b[0], b[1], b[2], b[3]);
    sgb[2 * (nvec + v) + 1] = make_float4(b[4], b[5], b[6], b[7]);
  }
  __syncthreads();
  const int n = rows > (int)blockIdx.x ? (rows - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < n && !*abort; ++i) {
        const int s = i % nslot;
        if (i >= nslot && !mbar_wait(empty0 + 8 * s, ((i / nslot) - 1) & 1, err)) {
          *abort = 1;
          break;
        }
        const int row = blockIdx.x + i * gridDim.x;
        const bf16* src = x + (int64_t)row * cols;
        // bulk copies need 16-byte aligned addresses and sizes
        if (!dcheck(row < rows && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                        (slot_bytes & 15) == 0,
                    err)) {
          *abort = 1;
          break;
        }
        mbar_arrive_expect_tx(full0 + 8 * s, slot_bytes);
        bulk_load(slots + s * slot_bytes, src, slot_bytes, full0 + 8 * s);
      }
    }
  } else {
    const float inv_cols = 1.0f / (float)cols;
    for (int i = warp - 1; i < n; i += kLnConsumers) {
      const int s = i % nslot;
      const bool ok = !*abort && mbar_wait(full0 + 8 * s, (i / nslot) & 1, err);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort = 1;
        break;
      }
      uint4 cur[VPL];
      const uint4* src = reinterpret_cast<const uint4*>(ln_smem + s * slot_bytes);
#pragma unroll
      for (int j = 0; j < VPL; ++j) cur[j] = src[lane + 32 * j];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);  // slot free: the producer refills it
      const int row = blockIdx.x + i * gridDim.x;
      // eight independent partial sums (one per element of a vector): short
      // dependency chains instead of one chain over the lane's elements;
      // element pairs in packed float32x2 arithmetic
      float a8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        float v[8];
        unpack8(cur[j], v);
#pragma unroll
        for (int e = 0; e < 8; e += 2) add2(a8[e], a8[e + 1], a8[e], a8[e + 1], v[e], v[e + 1]);
      }
      float sm = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      const float mean = sm * inv_cols;
#pragma unroll
      for (int e = 0; e < 8; ++e) a8[e] = 0.0f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        float v[8];
        unpack8(cur[j], v);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          add2(v[e], v[e + 1], v[e], v[e + 1], -mean, -mean);
          fma2(a8[e], a8[e + 1], v[e], v[e + 1], v[e], v[e + 1], a8[e], a8[e + 1]);
        }
      }
      float ss = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rstd = rsqrtf(ss * inv_cols + eps);
      uint4* yr = reinterpret_cast<uint4*>(y + (int64_t)row * cols);
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int vi = lane + 32 * j;
        float v[8], o8[8];
        unpack8(cur[j], v);
        const float4 g0 = sgb[2 * vi], g1 = sgb[2 * vi + 1];
        const float4 b0 = sgb[2 * (nvec + vi)], b1 = sgb[2 * (nvec + vi) + 1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        // y = (x - mean) rstd gamma + beta
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          add2(o8[e], o8[e + 1], v[e], v[e + 1], -mean, -mean);
          mul2(o8[e], o8[e + 1], o8[e], o8[e + 1], rstd, rstd);
          fma2(o8[e], o8[e + 1], o8[e], o8[e + 1], g[e], g[e + 1], b[e], b[e + 1]);
        }
        uint4 ov;
        ov.x = pack_bf16x2(o8[0], o8[1]); ov.y = pack_bf16x2(o8[2], o8[3]);
        ov.z = pack_bf16x2(o8[4], o8[5]); ov.w = pack_bf16x2(o8[6], o8[7]);
        yr[vi] = ov;
      }
      if (lane == 0) {
        if (mean_out) mean_out[row] = mean;
        if (rstd_out) rstd_out[row] = rstd;
      }
    }
  }
  ln_abort_drain(abort);
}

// Backward: the CTA's 8 consumer warps (256 threads, VPT vectors each) take
// the CTA's rows one after another, each from slot i % nslot holding x, dy and
// dres (three bulk copies); the row reduction uses two float2 slots per warp
// in shared memory (alternating by row) and one named barrier of the 256
// consumer threads; dgamma/dbeta partials stay in registers and are written
// once at the end as partial row blockIdx.x.
template <int VPT>
__global__ void __launch_bounds__(32 * (1 + kLnConsumers)) ln_bwd_tma_kernel(
    int rows, int cols, const bf16* __restrict__ x, const float* __restrict__ mean,
    const float* __restrict__ rstd, const bf16* __restrict__ gamma, const bf16* __restrict__ dy,
    const bf16* __restrict__ dres, bf16* __restrict__ dx, float* __restrict__ part, int nslot,
    int* err) {
  extern __shared__ __align__(128) uint8_t ln_smem[];
  const uint32_t row_bytes = (uint32_t)cols * 2;
  const uint32_t slot_bytes = 3 * row_bytes;
  const uint32_t slots = smem_u32(ln_smem);
  const uint32_t full0 = slots + nslot * slot_bytes;
  const uint32_t empty0 = full0 + 8 * nslot;
  float2* red = reinterpret_cast<float2*>(ln_smem + nslot * slot_bytes + 16 * nslot);  // [2][8]
  volatile int* abort = reinterpret_cast<volatile int*>(red + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = cols / 8;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nslot; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kLnConsumers);
    }
    fence_mbar_init();
    *abort = 0;
  }
  __syncthreads();
  const int n = rows > (int)blockIdx.x ? (rows - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (warp == 0) {
    if (lane == 0) {
      const uint32_t bytes = dres ? slot_bytes : 2 * row_bytes;
      for (int i = 0; i < n && !*abort; ++i) {
        const int s = i % nslot;
        if (i >= nslot && !mbar_wait(empty0 + 8 * s, ((i / nslot) - 1) & 1, err)) {
          *abort = 1;
          break;
        }
        const int64_t ro = (int64_t)(blockIdx.x + i * gridDim.x) * cols;
        const uint32_t dst = slots + s * slot_bytes, fb = full0 + 8 * s;
        mbar_arrive_expect_tx(fb, bytes);
        bulk_load(dst, x + ro, row_bytes, fb);
        bulk_load(dst + row_bytes, dy + ro, row_bytes, fb);
        if (dres) bulk_load(dst + 2 * row_bytes, dres + ro, row_bytes, fb);
      }
    }
  } else {
    const int t = threadIdx.x - 32, cw = warp - 1;  // consumer thread / warp
    float pg[VPT][8], pb[VPT][8];
#pragma unroll
    for (int q = 0; q < VPT; ++q)
#pragma unroll
      for (int e = 0; e < 8; ++e) pg[q][e] = pb[q][e] = 0.0f;
    const float inv_cols = 1.0f / (float)cols;
    for (int i = 0; i < n; ++i) {
      const int s = i % nslot;
      // every consumer thread takes the same decision (a barrier with an OR
      // vote), so none is left waiting at the row barrier below
      const bool ok = !*abort && mbar_wait(full0 + 8 * s, (i / nslot) & 1, err);
      int bad = 0;
      asm volatile(
          "{\n .reg .pred p, q;\n setp.eq.u32 p, %1, 0;\n"
          " bar.red.or.pred q, 2, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
          : "=r"(bad)
          : "r"((uint32_t)ok), "r"(32 * kLnConsumers)
          : "memory");
      if (bad) {
        *abort = 1;
        break;
      }
      const uint8_t* sl = ln_smem + s * slot_bytes;
      uint4 rx[VPT], rd[VPT], rr[VPT];
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        const int vi = t + 256 * q;
        if (vi < nvec) {
          rx[q] = reinterpret_cast<const uint4*>(sl)[vi];
          rd[q] = reinterpret_cast<const uint4*>(sl + row_bytes)[vi];
          if (dres) rr[q] = reinterpret_cast<const uint4*>(sl + 2 * row_bytes)[vi];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      const int row = blockIdx.x + i * gridDim.x;
      const float mu = mean[row], rs = rstd[row];
      float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        const int vi = t + 256 * q;
        if (vi < nvec) {
          float xv[8], dv[8], gm[8];
          unpack8(rx[q], xv);
          unpack8(rd[q], dv);
          if (gamma) vload(gamma + vi * 8, gm);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float xh = (xv[e] - mu) * rs;
            const float g = gamma ? dv[e] * gm[e] : dv[e];
            s1 += g;
            s2 += g * xh;
            pg[q][e] += dv[e] * xh;
            pb[q][e] += dv[e];
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      }
      float2* rb = red + 8 * (i & 1);
      if (lane == 0) rb[cw] = make_float2(s1, s2);
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kLnConsumers) : "memory");
      float a = 0.0f, b2 = 0.0f;
#pragma unroll
      for (int w = 0; w < kLnConsumers; ++w) {
        const float2 v = rb[w];
        a += v.x;
        b2 += v.y;
      }
      const float mg = a * inv_cols, mgx = b2 * inv_cols;
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        const int vi = t + 256 * q;
        if (vi < nvec) {
          float xv[8], dv[8], gm[8], rv[8], o[8];
          unpack8(rx[q], xv);
          unpack8(rd[q], dv);
          if (gamma) vload(gamma + vi * 8, gm);
          if (dres) unpack8(rr[q], rv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float xh = (xv[e] - mu) * rs;
            const float g = gamma ? dv[e] * gm[e] : dv[e];
            o[e] = rs * (g - mg - xh * mgx);
            if (dres) o[e] += rv[e];
          }
          vstore(dx + (int64_t)row * cols + vi * 8, o);
        }
      }
    }
    if (part) {
      float* pgr = part + (int64_t)blockIdx.x * cols;
      float* pbr = part + (int64_t)(gridDim.x + blockIdx.x) * cols;
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        const int vi = t + 256 * q;
        if (vi < nvec) {
#pragma unroll
          for (int e = 0; e < 8; e += 4) {
            *reinterpret_cast<float4*>(pgr + vi * 8 + e) =
                make_float4(pg[q][e], pg[q][e + 1], pg[q][e + 2], pg[q][e + 3]);
            *reinterpret_cast<float4*>(pbr + vi * 8 + e) =
                make_float4(pb[q][e], pb[q][e + 1], pb[q][e + 2], pb[q][e + 3]);
          }
        }
      }
    }
  }
  ln_abort_drain(abort);
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
template <typename T, int VPT, bool PF>
__device__ __forceinline__ void ln_bwd_rows(int rows, int cols, const T* __restrict__ x,
                                            const float* __restrict__ mean,
                                            const float* __restrict__ rstd,
                                            const T* __restrict__ gamma, const T* __restrict__ dy,
                                            const T* __restrict__ dres, T* __restrict__ dx,
                                            float* __restrict__ part) {
  constexpr int VN = Vec<T>::N;
  __shared__ float2 red[32];
  const int nvec = cols / VN;
  float pg[VPT][VN], pb[VPT][VN];
#pragma unroll
  for (int i = 0; i < VPT; ++i)
#pragma unroll
    for (int j = 0; j < VN; ++j) pg[i][j] = pb[i][j] = 0.0f;
  // The row is kept as raw 16-byte vectors (x, dy, dres) and unpacked in each
  // of the two passes; with PF the next row's vectors are requested before
  // this row's reduction. gamma is read per row (an L1 hit after the first).
  uint4 rx[VPT], rd[VPT], rr[VPT], nx[VPT], nd[VPT], nr[VPT];
  auto fetch = [&](int row, uint4 (&ax)[VPT], uint4 (&ad)[VPT], uint4 (&ar)[VPT]) {
    const int64_t ro = (int64_t)row * cols;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
        ax[i] = *reinterpret_cast<const uint4*>(x + ro + vi * VN);
        ad[i] = *reinterpret_cast<const uint4*>(dy + ro + vi * VN);
        if (dres) ar[i] = *reinterpret_cast<const uint4*>(dres + ro + vi * VN);
      }
    }
  };
  if (PF && blockIdx.x < rows) fetch(blockIdx.x, rx, rd, rr);
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const float mu = mean[row], rs = rstd[row];
    const int64_t ro = (int64_t)row * cols;
    if (PF) {
      if (row + (int)gridDim.x < rows) fetch(row + gridDim.x, nx, nd, nr);
    } else {
      fetch(row, rx, rd, rr);
    }
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
        float xv[VN], dv[VN], gm[VN];
        vunpack<T>(rx[i], xv);
        vunpack<T>(rd[i], dv);
        if (gamma) vload(gamma + vi * VN, gm);
#pragma unroll
        for (int j = 0; j < VN; ++j) {
          const float xh = (xv[j] - mu) * rs;
          const float g = gamma ? dv[j] * gm[j] : dv[j];
          s1 += g;
          s2 += g * xh;
          pg[i][j] += dv[j] * xh;
          pb[i][j] += dv[j];
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
        float xv[VN], dv[VN], gm[VN], rv[VN], o[VN];
        vunpack<T>(rx[i], xv);
        vunpack<T>(rd[i], dv);
        if (gamma) vload(gamma + vi * VN, gm);
        if (dres) vunpack<T>(rr[i], rv);
#pragma unroll
        for (int j = 0; j < VN; ++j) {
          const float xh = (xv[j] - mu) * rs;
          const float g = gamma ? dv[j] * gm[j] : dv[j];
          o[j] = rs * (g - mg - xh * mgx);
          if (dres) o[j] += rv[j];
        }
        vstore(dx + ro + vi * VN, o);
      }
    }
    if (PF) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        rx[i] = nx[i];
        rd[i] = nd[i];
        rr[i] = nr[i];
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

// Rows of up to 1024 vectors: one vector per thread (64 registers: two
// 512-thread blocks per SM).
template <typename T, int VPT>
__global__ void __launch_bounds__(1024, 1) ln_bwd_kernel(int rows, int cols, const T* __restrict__ x,
                              const float* __restrict__ mean, const float* __restrict__ rstd,
                              const T* __restrict__ gamma, const T* __restrict__ dy,
                              const T* __restrict__ dres, T* __restrict__ dx,
                              float* __restrict__ part) {
  ln_bwd_rows<T, VPT, true>(rows, cols, x, mean, rstd, gamma, dy, dres, dx, part);
}

// Wider rows (VPT 2 or 4 vectors per thread, up to 1024 threads): the register
// count is held to 64 a thread so a full block always launches; these spill a
// little instead.
template <typename T, int VPT>
__global__ void __launch_bounds__(1024, 1) ln_bwd_wide_kernel(
    int rows, int cols, const T* __restrict__ x, const float* __restrict__ mean,
    const float* __restrict__ rstd, const T* __restrict__ gamma, const T* __restrict__ dy,
    const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ part) {
  ln_bwd_rows<T, VPT, false>(rows, cols, x, mean, rstd, gamma, dy, dres, dx, part);
}

// 16-byte asynchronous copy global -> shared (bypassing L1); completion is
// tracked per thread by commit groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Backward for rows of up to 1024 vectors, fed by per-thread asynchronous
// copies. Blocks stride over the rows as in ln_bwd_kernel (thread t owns
// vector t of every row; gamma and the dgamma/dbeta partial sums stay in its
// registers). Each thread copies its own vector of x, dy and dres of the
// block's next P - 1 rows into its private slots of a P-row shared-memory ring
// and reads them back itself, so no barrier guards the ring: only the row
// reduction synchronises the block (once per row, alternating between two
// reduction buffers). P - 1 rows per block are in flight while one is worked
// on, without registers holding them.
// With CL > 1 the grid is launched in clusters of CL CTAs, which combine their
// dgamma/dbeta partial sums through distributed shared memory before they are
// written: partial row blockIdx.x / CL, CTA rank r of the cluster summing the
// r-th share of the columns over the cluster's CTAs in rank order.
template <typename T, int P, int CL>
__global__ void __launch_bounds__(1024, 1) ln_bwd_async_kernel(
    int rows, int cols, const T* __restrict__ x, const float* __restrict__ mean,
    const float* __restrict__ rstd, const T* __restrict__ gamma, const T* __restrict__ dy,
    const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ part) {
  constexpr int VN = Vec<T>::N;
  extern __shared__ uint4 ln_ring[];  // [P][3][blockDim.x]
  __shared__ float2 red[2][32];
  const int nt = blockDim.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int nvec = cols / VN;
  const bool have = t < nvec;
  const int nrow = rows > (int)blockIdx.x ? (rows - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  // the block's i-th row into slot i % P (an empty group past the end keeps
  // one group per row)
  auto issue = [&](int i) {
    if (i < nrow && have) {
      const int64_t o = (int64_t)((int)blockIdx.x + (int64_t)i * gridDim.x) * cols + t * VN;
      uint4* s = ln_ring + (i % P) * 3 * nt + t;
      cp_async16(s, x + o);
      cp_async16(s + nt, dy + o);
      if (dres) cp_async16(s + 2 * nt, dres + o);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < P - 1; ++i) issue(i);
  float gm[VN], pg[VN], pb[VN];
#pragma unroll
  for (int j = 0; j < VN; ++j) {
    gm[j] = 1.0f;
    pg[j] = pb[j] = 0.0f;
  }
  if (gamma && have) vload(gamma + t * VN, gm);
  const float inv_cols = 1.0f / (float)cols;
  // the block's row statistics: staged in shared memory up front when the
  // block has at most 64 rows, else loaded one row ahead into registers
  __shared__ float2 stat[64];
  const bool staged = nrow <= 64;
  float mu_n = 0.0f, rs_n = 0.0f;
  if (staged) {
    for (int k = t; k < nrow; k += nt) {
      const int r = (int)blockIdx.x + k * (int)gridDim.x;
      stat[k] = make_float2(mean[r], rstd[r]);
    }
    __syncthreads();
  } else if (nrow > 0) {
    mu_n = mean[blockIdx.x];
    rs_n = rstd[blockIdx.x];
  }
  for (int i = 0; i < nrow; ++i) {
    const int row = (int)blockIdx.x + i * (int)gridDim.x;
    float mu = mu_n, rs = rs_n;
    if (staged) {
      const float2 m = stat[i];
      mu = m.x;
      rs = m.y;
    } else if (i + 1 < nrow) {
      mu_n = mean[row + gridDim.x];
      rs_n = rstd[row + gridDim.x];
    }
    // refill the slot of row i - 1 (read into registers last iteration) with
    // row i + P - 1; then row i's own copies are complete
    issue(i + P - 1);
    cp_async_wait<P - 1>();
    float xv[VN], dv[VN];
    float s1 = 0.0f, s2 = 0.0f;
    const uint4* slot = ln_ring + (i % P) * 3 * nt + t;
    if (have) {
      vunpack<T>(slot[0], xv);
      vunpack<T>(slot[nt], dv);
      // column pairs in packed float32x2 arithmetic (half the instructions)
      float s1b = 0.0f, s2b = 0.0f;
#pragma unroll
      for (int j = 0; j < VN; j += 2) {
        float g0, g1;
        add2(xv[j], xv[j + 1], xv[j], xv[j + 1], -mu, -mu);
        mul2(xv[j], xv[j + 1], xv[j], xv[j + 1], rs, rs);  // x-hat
        mul2(g0, g1, dv[j], dv[j + 1], gm[j], gm[j + 1]);
        add2(s1, s1b, s1, s1b, g0, g1);
        fma2(s2, s2b, g0, g1, xv[j], xv[j + 1], s2, s2b);
        fma2(pg[j], pg[j + 1], dv[j], dv[j + 1], xv[j], xv[j + 1], pg[j], pg[j + 1]);
        add2(pb[j], pb[j + 1], pb[j], pb[j + 1], dv[j], dv[j + 1]);
      }
      s1 += s1b;
      s2 += s2b;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    float2* rb = red[i & 1];
    if (lane == 0) rb[warp] = make_float2(s1, s2);
    __syncthreads();
    float2 tot = lane < (nt >> 5) ? rb[lane] : make_float2(0.0f, 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot.x += __shfl_xor_sync(0xffffffffu, tot.x, o);
      tot.y += __shfl_xor_sync(0xffffffffu, tot.y, o);
    }
    if (have) {
      const float nmg = -tot.x * inv_cols, nmgx = -tot.y * inv_cols;
      float rv[VN], o[VN];
      if (dres) {
        // (the slot is refilled only in the next iteration)
        vunpack<T>(slot[2 * nt], rv);
      } else {
#pragma unroll
        for (int j = 0; j < VN; ++j) rv[j] = 0.0f;
      }
      // dx = rs (g - mean(g) - x-hat mean(g x-hat)) (+ dres)
#pragma unroll
      for (int j = 0; j < VN; j += 2) {
        mul2(o[j], o[j + 1], dv[j], dv[j + 1], gm[j], gm[j + 1]);
        add2(o[j], o[j + 1], o[j], o[j + 1], nmg, nmg);
        fma2(o[j], o[j + 1], xv[j], xv[j + 1], nmgx, nmgx, o[j], o[j + 1]);
        fma2(o[j], o[j + 1], o[j], o[j + 1], rs, rs, rv[j], rv[j + 1]);
      }
      vstore(dx + (int64_t)row * cols + t * VN, o);
    }
  }
  cp_async_wait<0>();
  if (part == nullptr) return;
  if constexpr (CL == 1) {
    if (have) {
      float* pgr = part + (int64_t)blockIdx.x * cols + t * VN;
      float* pbr = part + (int64_t)(gridDim.x + blockIdx.x) * cols + t * VN;
#pragma unroll
      for (int j = 0; j < VN; j += 4) {
        *reinterpret_cast<float4*>(pgr + j) = make_float4(pg[j], pg[j + 1], pg[j + 2], pg[j + 3]);
        *reinterpret_cast<float4*>(pbr + j) = make_float4(pb[j], pb[j + 1], pb[j + 2], pb[j + 3]);
      }
    }
  } else {
    // this CTA's partials as [2][cols] float32 over the start of the ring
    // (every thread's copies into it have completed)
    __syncthreads();
    float4* sp = reinterpret_cast<float4*>(ln_ring);
    const int c4n = cols / 4;
    if (have) {
#pragma unroll
      for (int j = 0; j < VN; j += 4) {
        sp[(t * VN + j) / 4] = make_float4(pg[j], pg[j + 1], pg[j + 2], pg[j + 3]);
        sp[c4n + (t * VN + j) / 4] = make_float4(pb[j], pb[j + 1], pb[j + 2], pb[j + 3]);
      }
    }
    cluster_sync();  // every CTA's partials are in its shared memory
    const int rank = (int)cluster_ctarank();
    const int share = (c4n + CL - 1) / CL;
    const int c_end = min(c4n, (rank + 1) * share);
    const int64_t prow = blockIdx.x / CL, nrows = gridDim.x / CL;
    const uint32_t sp_addr = smem_u32(sp);
    for (int c = rank * share + t; c < c_end; c += nt) {
      float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f), b = a;
#pragma unroll 1
      for (int k = 0; k < CL; ++k) {
        const uint32_t ra = mapa_shared(sp_addr + c * 16, k);
        const uint32_t rb = mapa_shared(sp_addr + (c4n + c) * 16, k);
        float4 u, w;
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(u.x), "=f"(u.y), "=f"(u.z), "=f"(u.w) : "r"(ra) : "memory");
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(w.x), "=f"(w.y), "=f"(w.z), "=f"(w.w) : "r"(rb) : "memory");
        a.x += u.x; a.y += u.y; a.z += u.z; a.w += u.w;
        b.x += w.x; b.y += w.y; b.z += w.z; b.w += w.w;
      }
      reinterpret_cast<float4*>(part + prow * cols)[c] = a;
      reinterpret_cast<float4*>(part + (nrows + prow) * cols)[c] = b;
    }
    cluster_sync();  // no CTA leaves while the others still read its shared memory
  }
}

// out0[c] = sum_p part[p * stride, c] and out1[c] = sum_p part[half + p * stride, c]
// for p < nparts (rows of `cols` floats), written as T (nullable outputs
// skipped). Block (32 x 16), grid (column blocks, 2): lane = column (coalesced
// 128-byte rows of the partial buffer), blockIdx.y = which output, the 16
// warps split the partials (four rows' loads in flight per thread), fixed
// order of summation (deterministic).
template <typename T>
__global__ void __launch_bounds__(512) reduce_parts_kernel(int nparts, int stride, int64_t half,
                                                           int cols, const float* __restrict__ part,
                                                           T* __restrict__ out0,
                                                           T* __restrict__ out1) {
  __shared__ float red[16][33];
  T* out = blockIdx.y == 0 ? out0 : out1;
  if (out == nullptr) return;
  const float* src = part + (blockIdx.y == 0 ? 0 : half);
  const int c = blockIdx.x * 32 + threadIdx.x;
  float s = 0.0f;
  if (c < cols) {
#pragma unroll 4
    for (int p = threadIdx.y; p < nparts; p += 16) s += src[(int64_t)p * stride * cols + c];
  }
  red[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && c < cols) {
    float a = 0.0f;
#pragma unroll
    for (int y = 0; y < 16; ++y) a += red[y][threadIdx.x];
    out[c] = from_f<T>(a);
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
    reduce_parts_kernel<T><<<dim3((cols + 31) / 32, 2), dim3(32, 16), 0, st>>>(
        splits, per, half, cols, part, out0, out1);
  } else {
    reduce_parts_kernel<T><<<dim3((cols + 31) / 32, 2), dim3(32, 16), 0, st>>>(
        nparts, 1, half, cols, part, out0, out1);
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
// (608 = four 512-thread blocks on each of 152 SMs: one resident wave)
int layernorm_bwd_parts(int rows) { return rows < 608 ? (rows > 0 ? rows : 1) : 608; }
int colsum_parts(int M) { return M < 64 * 8 ? 1 : 64; }

namespace {

// Resident CTAs per SM of a kernel at `smem` bytes of dynamic shared memory.
template <typename K>
int resident_ctas(K kern, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

template <int VPL>
mgb_status ln_fwd_tma_vpl(int rows, int cols, float eps, const void* x, const void* gamma,
                          const void* beta, void* y, float* mean, float* rstd, cudaStream_t st) {
  const int slot = cols * 2;
  const int nslot = std::max(2, std::min(16, (96 << 10) / slot));
  // ring, barriers, abort flag, float32 gamma and beta
  const size_t smem = (size_t)nslot * slot + 16 * nslot + 16 + 2 * (size_t)cols * 4;
  auto kern = ln_fwd_tma_kernel<VPL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MGB_ERR_CUDA;
  const int threads = 32 * (1 + kLnConsumers);
  const int cap = resident_ctas(kern, threads, smem) * device_sm_count();
  const int want = (rows + kLnConsumers - 1) / kLnConsumers;
  const int grid = std::max(1, std::min(cap, want));
  kern<<<grid, threads, smem, st>>>(rows, cols, eps, (const bf16*)x, (const bf16*)gamma,
                                    (const bf16*)beta, (bf16*)y, mean, rstd, nslot,
                                    device_error_word());
  return MGB_OK;
}

mgb_status ln_fwd_tma_go(int rows, int cols, float eps, const void* x, const void* gamma,
                         const void* beta, void* y, float* mean, float* rstd, cudaStream_t st) {
  switch (cols / 256) {
    case 1: return ln_fwd_tma_vpl<1>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st);
    case 2: return ln_fwd_tma_vpl<2>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st);
    case 4: return ln_fwd_tma_vpl<4>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st);
    case 8: return ln_fwd_tma_vpl<8>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st);
    case 16: return ln_fwd_tma_vpl<16>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st);
    default: return MGB_ERR_UNSUPPORTED;
  }
}

template <int VPT>
int ln_bwd_tma_vpt(int nparts, int rows, int cols, const void* x, const float* mean,
                   const float* rstd, const void* gamma, const void* dy, const void* dres,
                   void* dx, float* part, cudaStream_t st) {
  const int slot = 3 * cols * 2;
  const int nslot = std::max(2, std::min(8, (96 << 10) / slot));
  const size_t smem = (size_t)nslot * slot + 16 * nslot + 16 * 8 + 32;
  auto kern = ln_bwd_tma_kernel<VPT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return -1;
  const int threads = 32 * (1 + kLnConsumers);
  const int cap = resident_ctas(kern, threads, smem) * device_sm_count();
  const int grid = std::max(1, std::min(cap, nparts));
  kern<<<grid, threads, smem, st>>>(rows, cols, (const bf16*)x, mean, rstd, (const bf16*)gamma,
                                    (const bf16*)dy, (const bf16*)dres, (bf16*)dx, part, nslot,
                                    device_error_word());
  return grid;
}

// Launches the TMA-fed backward when it applies; returns the partial rows it
// wrote (its grid), 0 when it does not apply, -1 on a launch-setup error.
int ln_bwd_tma_go(int nparts, int rows, int cols, const void* x, const float* mean,
                  const float* rstd, const void* gamma, const void* dy, const void* dres,
                  void* dx, float* part, cudaStream_t st) {
  const int nvec = cols / 8;
  if (nvec <= 256) return ln_bwd_tma_vpt<1>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  if (nvec <= 512) return ln_bwd_tma_vpt<2>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  if (nvec <= 1024) return ln_bwd_tma_vpt<4>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  return 0;
}

}  // namespace

mgb_status layernorm_fwd_launch(int rows, int cols, int dtype, float eps, const void* x,
                                const void* gamma, const void* beta, void* y, float* mean,
                                float* rstd, cudaStream_t st) {
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  if (rows < 0 || cols <= 0 || cols % vn) return MGB_ERR_INVALID_ARG;
  const int threads = ln_threads(cols, vn);
  if (threads > 1024) return MGB_ERR_UNSUPPORTED;
  if (rows == 0) return MGB_OK;
  LaunchScope scope(PROF_LN_FWD, st);
  // MGB_LN_KERNEL=block / warp picks the block-per-row or register-prefetch
  // kernel instead of the TMA-fed one (comparisons)
  const char* kenv = getenv("MGB_LN_KERNEL");
  const bool force_block = kenv && strcmp(kenv, "block") == 0;
  const bool force_warp = kenv && strcmp(kenv, "warp") == 0;
  if (dtype == MGB_BF16 && cols % 256 == 0 && cols <= 4096 && !force_block && !force_warp) {
    const mgb_status s = ln_fwd_tma_go(rows, cols, eps, x, gamma, beta, y, mean, rstd, st);
    if (s != MGB_ERR_UNSUPPORTED) return s;
  }
  const bool warp_ok = dtype == MGB_BF16 && cols % 256 == 0 && !force_block;
  if (warp_ok) {
    switch (cols / 256) {
      case 1: ln_fwd_warp_go<1>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st); break;
      case 2: ln_fwd_warp_go<2>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st); break;
      case 4: ln_fwd_warp_go<4>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st); break;
      case 8: ln_fwd_warp_go<8>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st); break;
      case 16: ln_fwd_warp_go<16>(rows, cols, eps, x, gamma, beta, y, mean, rstd, st); break;
      default: goto block_kernel;
    }
    return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
  }
block_kernel:
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

// Launches with at most as many blocks as are resident at once (the blocks
// stride over the rows, so a second wave would only serialise); returns the
// grid, which is the number of partial rows written.
template <typename T, int VPT>
int ln_bwd_go(int nparts, int threads, int rows, int cols, const void* x, const float* mean,
              const float* rstd, const void* gamma, const void* dy, const void* dres, void* dx,
              float* part, cudaStream_t st) {
  int per_sm = 0;
  auto k1 = ln_bwd_kernel<T, VPT>;
  auto kw = ln_bwd_wide_kernel<T, VPT>;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, VPT == 1 ? k1 : kw, threads, 0) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int grid = std::max(1, std::min(nparts, per_sm * device_sm_count()));
  if constexpr (VPT == 1)
    k1<<<grid, threads, 0, st>>>(rows, cols, (const T*)x, mean, rstd, (const T*)gamma,
                                 (const T*)dy, (const T*)dres, (T*)dx, part);
  else
    kw<<<grid, threads, 0, st>>>(rows, cols, (const T*)x, mean, rstd, (const T*)gamma,
                                 (const T*)dy, (const T*)dres, (T*)dx, part);
  return grid;
}

// The asynchronous-copy backward (rows of up to 1024 vectors): a ring of 4 rows
// while it fits in 100 KB of shared memory (two blocks of 512 threads per SM at
// bf16 H = 4096), else 2. Returns the grid (partial rows written), -2 on a
// launch-setup error.
//
// With partial sums wanted and enough rows, the CTAs run in clusters of four
// (partial rows: a quarter of the CTAs, so the final reduction is one small
// pass) when clusters of four still fill the machine to within 6 %.
template <typename T, int P, int CL>
int ln_bwd_async_cl(int clusters, int threads, size_t smem, int rows, int cols, const void* x,
                    const float* mean, const float* rstd, const void* gamma, const void* dy,
                    const void* dres, void* dx, float* part, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * clusters, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(ln_bwd_async_kernel<T, P, CL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -2;
  if (cudaLaunchKernelEx(&cfg, ln_bwd_async_kernel<T, P, CL>, rows, cols, (const T*)x, mean, rstd,
                         (const T*)gamma, (const T*)dy, (const T*)dres, (T*)dx, part) != cudaSuccess)
    return -2;
  return clusters;
}

// Clusters of CL resident at once for this launch shape (0 if the query fails).
template <typename T, int P, int CL>
int ln_bwd_max_clusters(int threads, size_t smem) {
  auto kern = ln_bwd_async_kernel<T, P, CL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * 64, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Launch shape of the asynchronous-copy backward for a block size: the plain
// kernel's resident CTAs and the clusters of CL resident at once. Queried once
// per CUDA context and block size, so that a call costs no occupancy queries
// on the host. (The shared-memory size attribute is still set before every
// launch: another block size may have lowered it since.)
struct AsyncShape {
  bool ok = false;
  int resident = 0, clusters = 0;
};
template <typename T, int P, int CL>
AsyncShape ln_bwd_async_shape(int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<void*, int>, AsyncShape> cache;
  const std::pair<void*, int> key(current_cuda_context(), threads);
  std::lock_guard<std::mutex> lock(mu);
  const auto it = cache.find(key);
  if (it != cache.end() && key.first != nullptr) return it->second;
  AsyncShape sh;
  auto kern = ln_bwd_async_kernel<T, P, 1>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
      cudaSuccess) {
    sh.ok = true;
    sh.resident = resident_ctas(kern, threads, smem) * device_sm_count();
    sh.clusters = ln_bwd_max_clusters<T, P, CL>(threads, smem);
  } else {
    cudaGetLastError();
  }
  if (key.first != nullptr) cache[key] = sh;
  return sh;
}

template <typename T, int P>
int ln_bwd_async_p(int nparts, int threads, int rows, int cols, const void* x, const float* mean,
                   const float* rstd, const void* gamma, const void* dy, const void* dres,
                   void* dx, float* part, cudaStream_t st) {
  constexpr int CL = 4;
  const size_t smem = (size_t)P * 3 * threads * 16;
  auto kern = ln_bwd_async_kernel<T, P, 1>;
  const AsyncShape sh = ln_bwd_async_shape<T, P, CL>(threads, smem);
  if (!sh.ok) return -2;
  const int resident = sh.resident;
  // the partials of a cluster fit in its CTAs' rings
  if (part && std::min(nparts, rows) >= 2 * CL && 2 * (size_t)cols * 4 <= smem) {
    const int mc = sh.clusters;
    if (mc > 0 && (int64_t)mc * CL * 100 >= (int64_t)resident * 94) {
      // one partial row per cluster: at most nparts of them
      const int clusters = std::min(mc, std::min(nparts, (rows + CL - 1) / CL));
      return ln_bwd_async_cl<T, P, CL>(clusters, threads, smem, rows, cols, x, mean, rstd, gamma,
                                       dy, dres, dx, part, st);
    }
  }
  const int grid = std::max(1, std::min(nparts, resident));
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return -2;
  kern<<<grid, threads, smem, st>>>(rows, cols, (const T*)x, mean, rstd, (const T*)gamma,
                                    (const T*)dy, (const T*)dres, (T*)dx, part);
  return grid;
}

template <typename T>
int ln_bwd_async_go(int nparts, int threads, int rows, int cols, const void* x, const float* mean,
                    const float* rstd, const void* gamma, const void* dy, const void* dres,
                    void* dx, float* part, cudaStream_t st) {
  if ((size_t)4 * 3 * threads * 16 <= (100u << 10))
    return ln_bwd_async_p<T, 4>(nparts, threads, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                                part, st);
  return ln_bwd_async_p<T, 2>(nparts, threads, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                              part, st);
}

// Returns the partial rows written (the grid), -1 for an unsupported width,
// -2 on a launch-setup error.
template <typename T>
int ln_bwd_dispatch(int nparts, int rows, int cols, const void* x, const float* mean,
                    const float* rstd, const void* gamma, const void* dy, const void* dres,
                    void* dx, float* part, cudaStream_t st) {
  // one 16-byte vector per thread (64 registers: full occupancy), two or four
  // for rows wider than 1024 vectors
  const int nvec = cols / Vec<T>::N;
  auto thr = [&](int vpt) { return ((nvec + vpt - 1) / vpt + 31) / 32 * 32; };
  if (nvec <= 1024) {
    // MGB_LN_KERNEL=block: the register-prefetch kernel instead of the
    // asynchronous-copy one
    const char* kenv = getenv("MGB_LN_KERNEL");
    if (kenv && strcmp(kenv, "block") == 0)
      return ln_bwd_go<T, 1>(nparts, thr(1), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part,
                             st);
    return ln_bwd_async_go<T>(nparts, thr(1), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part,
                              st);
  }
  if (nvec <= 2048)
    return ln_bwd_go<T, 2>(nparts, thr(2), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  if (nvec <= 4096)
    return ln_bwd_go<T, 4>(nparts, thr(4), rows, cols, x, mean, rstd, gamma, dy, dres, dx, part, st);
  return -1;
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
  // the TMA-fed bf16 kernel writes as many partial rows as its grid (at most
  // nparts); the reduction then folds that many
  // (MGB_LN_KERNEL=tma selects the bulk-copy kernel; otherwise rows of up to
  // 1024 vectors take the asynchronous-copy kernel, wider ones the block kernel)
  const char* kenv = getenv("MGB_LN_KERNEL");
  const bool tma = dtype == MGB_BF16 && rows > 0 && cols * 2 * 3 <= (96 << 10) && kenv &&
                   strcmp(kenv, "tma") == 0;
  if (tma) {
    int used;
    {
      LaunchScope pre(PROF_LN_BWD, st);
      used = ln_bwd_tma_go(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                           want ? part : nullptr, st);
    }
    if (used < 0) return MGB_ERR_CUDA;
    if (used > 0) {
      if (want) {
        LaunchScope scope(PROF_LN_BWD, st, reduce_launches(used, cols));
        if (dtype == MGB_BF16)
          reduce_parts_go<bf16>(used, cols, part, (bf16*)dgamma, (bf16*)dbeta, st);
      }
      return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
    }
  }
  if (rows > 0) {
    int used;
    {
      LaunchScope scope(PROF_LN_BWD, st);
      used = dtype == MGB_BF16
                 ? ln_bwd_dispatch<bf16>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                                         want ? part : nullptr, st)
                 : ln_bwd_dispatch<float>(nparts, rows, cols, x, mean, rstd, gamma, dy, dres, dx,
                                          want ? part : nullptr, st);
    }
    if (used == -2) return MGB_ERR_CUDA;
    if (used < 0) return MGB_ERR_UNSUPPORTED;
    nparts = used;
  }
  LaunchScope scope(PROF_LN_BWD, st, want ? reduce_launches(nparts, cols) : 0);
  if (rows > 0) {
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

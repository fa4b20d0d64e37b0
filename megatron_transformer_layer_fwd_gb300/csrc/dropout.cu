// Dropout from a counter-based generator, and the tensor-parallel RNG
// tracker ("02 - How a whole Transformer block is split", section 5).
//
// A generator state is (seed, offset). The stream is Philox4x32-10 (SC 2011)
// with key = the seed's two 32-bit halves, counters (q, 0, 0, 0) for
// q = 0, 1, ...; each counter gives 16 bytes (its four words, lowest byte
// first). Element e of a dropout site whose state is (seed, offset) uses the
// byte at stream position offset + e and is kept iff that byte is below
// thr = floor((1 - p) * 256 + 1/2); kept values are scaled by 256 / thr. A
// mask is a function of (seed, offset, e) only, so a recomputation with the
// same state reproduces it exactly.
//
// Tracker: three states - data-parallel (seed: the same on every rank of a
// tensor-parallel group, for dropout outside the TP region), model-parallel
// (seed + 2718 + tp_rank, inside the region) and expert-parallel
// (seed + 1024 + 100 ep_rank + etp_rank) - one of them current; fork()
// makes another current and returns the previous one for restore(); draw(n)
// hands out the current state and advances its offset by n rounded up to 16.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

// out[i] = stream byte (offset + i), i < n: one thread per 16-byte block
__global__ void philox_bytes_kernel(uint64_t seed, uint64_t offset, uint64_t n,
                                    uint8_t* __restrict__ out) {
  const uint64_t q0 = offset / 16, q1 = (offset + n - 1) / 16;
  for (uint64_t q = q0 + blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q <= q1;
       q += (uint64_t)gridDim.x * blockDim.x) {
    const uint4 w = philox_block(seed, q);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const uint64_t pos = q * 16 + b;
      if (pos >= offset && pos < offset + n) out[pos - offset] = (uint8_t)(ws[b >> 2] >> (8 * (b & 3)));
    }
  }
}

template <typename T>
__device__ __forceinline__ float ldf(const T* p) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(*p);
  else return *p;
}
template <typename T>
__device__ __forceinline__ void stf(T* p, float v) {
  if constexpr (sizeof(T) == 2) *p = __float2bfloat16_rn(v);
  else *p = v;
}

// y[r, c] = keep(offset + r*cols + c) ? x[r, c] * scale : 0, offset % 16 == 0:
// one thread per 16 consecutive elements of the site (one Philox block)
template <typename T>
__global__ void dropout_kernel(int64_t rows, int64_t cols, uint64_t seed, uint64_t offset,
                               uint32_t thr, float scale, const T* __restrict__ x, int64_t ldx,
                               T* __restrict__ y, int64_t ldy) {
  const int64_t total = rows * cols;
  const int64_t groups = (total + 15) / 16;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
       g += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = philox_block(seed, offset / 16 + (uint64_t)g);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    const int64_t e0 = 16 * g;
    int64_t r = e0 / cols, c = e0 - r * cols;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (e0 + i < total) {
        const bool keep = keep_byte(ws[i >> 2], i & 3, thr);
        stf(y + r * ldy + c, keep ? ldf(x + r * ldx + c) * scale : 0.0f);
      }
      if (++c == cols) {
        c = 0;
        ++r;
      }
    }
  }
}

// As dropout_kernel for rows of a multiple of 16 elements and 16-byte aligned
// rows: group g = 16 elements of row g / gpr (the site's element 16 g), moved
// as 16-byte vectors.
template <typename T>
__global__ void dropout_rows_kernel(int64_t rows, int gpr, uint64_t seed, uint64_t q0, uint32_t thr,
                                    float scale, const T* __restrict__ x, int64_t ldx,
                                    T* __restrict__ y, int64_t ldy) {
  constexpr int VN = 16 / sizeof(T);  // elements per 16-byte vector
  const int64_t total = rows * gpr;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / gpr;
    const int c = (int)(g - r * gpr) * 16;
    const uint4* xs = reinterpret_cast<const uint4*>(x + r * ldx + c);
    uint4* ys = reinterpret_cast<uint4*>(y + r * ldy + c);
    uint4 v[16 / VN];
#pragma unroll
    for (int i = 0; i < 16 / VN; ++i) v[i] = xs[i];
    const uint4 w = philox_block(seed, q0 + (uint64_t)g);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 16 / VN; ++i) {
      uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if constexpr (sizeof(T) == 2) {
          const int e = i * 8 + 2 * k;  // element of the group
          const float2 f = unpack_bf16x2(u[k]);
          u[k] = pack_bf16x2(keep_byte(ws[e >> 2], e & 3, thr) ? f.x * scale : 0.0f,
                             keep_byte(ws[e >> 2], (e & 3) + 1, thr) ? f.y * scale : 0.0f);
        } else {
          const int e = i * 4 + k;
          u[k] = __float_as_uint(keep_byte(ws[e >> 2], e & 3, thr) ? __uint_as_float(u[k]) * scale
                                                                   : 0.0f);
        }
      }
      ys[i] = make_uint4(u[0], u[1], u[2], u[3]);
    }
  }
}

}  // namespace

uint32_t dropout_threshold(float p) {
  return (uint32_t)std::floor((1.0 - (double)p) * 256.0 + 0.5);
}

mgb_status dropout_launch(int64_t rows, int64_t cols, int dtype, float p, uint64_t seed,
                          uint64_t offset, const void* x, int64_t ldx, void* y, int64_t ldy,
                          cudaStream_t st) {
  if (rows == 0 || cols == 0) return MGB_OK;
  const uint32_t thr = dropout_threshold(p);
  const float scale = 256.0f / (float)thr;
  const int64_t groups = (rows * cols + 15) / 16;
  const int threads = 256;
  const int64_t want = (groups + threads - 1) / threads;
  const int grid = (int)(want < device_sm_count() * 8 ? want : device_sm_count() * 8);
  LaunchScope scope(PROF_DROPOUT, st);
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  const bool vec = cols % 16 == 0 && ldx % vn == 0 && ldy % vn == 0 &&
                   (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && cols / 16 < (1 << 30);
  if (vec) {
    if (dtype == MGB_BF16)
      dropout_rows_kernel<bf16><<<grid, threads, 0, st>>>(rows, (int)(cols / 16), seed, offset / 16,
                                                          thr, scale, static_cast<const bf16*>(x),
                                                          ldx, static_cast<bf16*>(y), ldy);
    else
      dropout_rows_kernel<float><<<grid, threads, 0, st>>>(rows, (int)(cols / 16), seed, offset / 16,
                                                           thr, scale, static_cast<const float*>(x),
                                                           ldx, static_cast<float*>(y), ldy);
  } else if (dtype == MGB_BF16)
    dropout_kernel<bf16><<<grid, threads, 0, st>>>(rows, cols, seed, offset, thr, scale,
                                                   static_cast<const bf16*>(x), ldx,
                                                   static_cast<bf16*>(y), ldy);
  else
    dropout_kernel<float><<<grid, threads, 0, st>>>(rows, cols, seed, offset, thr, scale,
                                                    static_cast<const float*>(x), ldx,
                                                    static_cast<float*>(y), ldy);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status philox_bytes_launch(uint64_t seed, uint64_t offset, uint64_t n, void* out,
                               cudaStream_t st) {
  if (n == 0) return MGB_OK;
  const uint64_t blocks16 = (offset + n - 1) / 16 - offset / 16 + 1;
  const uint64_t want = (blocks16 + 255) / 256;
  const int grid = (int)(want < (uint64_t)device_sm_count() * 8 ? want : device_sm_count() * 8);
  LaunchScope scope(PROF_DROPOUT, st);
  philox_bytes_kernel<<<grid, 256, 0, st>>>(seed, offset, n, static_cast<uint8_t*>(out));
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

using namespace mgb;

extern "C" {

mgb_status mgb_rng_tracker_init(mgb_rng_tracker* t, uint64_t seed, int32_t tp_rank, int32_t ep_rank,
                                int32_t etp_rank) {
  if (t == nullptr || tp_rank < 0 || ep_rank < 0 || etp_rank < 0) return MGB_ERR_INVALID_ARG;
  t->state[MGB_RNG_DATA_PARALLEL] = {seed, 0};
  t->state[MGB_RNG_MODEL_PARALLEL] = {seed + 2718u + (uint64_t)tp_rank, 0};
  t->state[MGB_RNG_EXPERT_PARALLEL] = {seed + 1024u + 100u * (uint64_t)ep_rank + (uint64_t)etp_rank,
                                       0};
  t->current = MGB_RNG_DATA_PARALLEL;
  return MGB_OK;
}

int32_t mgb_rng_fork(mgb_rng_tracker* t, int32_t kind) {
  if (t == nullptr || kind < 0 || kind > MGB_RNG_EXPERT_PARALLEL) return MGB_ERR_INVALID_ARG;
  const int32_t prev = t->current;
  t->current = kind;
  return prev;
}

mgb_status mgb_rng_restore(mgb_rng_tracker* t, int32_t prev) {
  if (t == nullptr || prev < 0 || prev > MGB_RNG_EXPERT_PARALLEL) return MGB_ERR_INVALID_ARG;
  t->current = prev;
  return MGB_OK;
}

mgb_status mgb_rng_draw(mgb_rng_tracker* t, uint64_t n, mgb_rng_state* out) {
  if (t == nullptr || out == nullptr || t->current < 0 || t->current > MGB_RNG_EXPERT_PARALLEL)
    return MGB_ERR_INVALID_ARG;
  mgb_rng_state& s = t->state[t->current];
  *out = s;
  s.offset += (n + 15) / 16 * 16;
  return MGB_OK;
}

mgb_status mgb_block_dropout_plan(mgb_block_desc* d, mgb_rng_tracker* t) {
  if (d == nullptr || t == nullptr || d->batch < 0 || d->seq < 1 || d->hidden < 1 ||
      d->n_q_heads < 1)
    return MGB_ERR_INVALID_ARG;
  const uint64_t B = (uint64_t)d->batch, S = (uint64_t)d->seq, H = (uint64_t)d->hidden;
  const uint64_t Sp = (S + 15) / 16 * 16;
  // attention probabilities: inside the tensor-parallel region
  const int32_t prev = mgb_rng_fork(t, MGB_RNG_MODEL_PARALLEL);
  if (prev < 0) return MGB_ERR_INVALID_ARG;
  mgb_status s = mgb_rng_draw(t, B * (uint64_t)d->n_q_heads * S * Sp, &d->rng_attn);
  const mgb_status r = mgb_rng_restore(t, prev);
  if (s != MGB_OK) return s;
  if (r != MGB_OK) return r;
  // hidden dropouts after the projection and fc2: outside the region
  s = mgb_rng_draw(t, B * S * H, &d->rng_proj);
  if (s != MGB_OK) return s;
  return mgb_rng_draw(t, B * S * H, &d->rng_fc2);
}

}  // extern "C"

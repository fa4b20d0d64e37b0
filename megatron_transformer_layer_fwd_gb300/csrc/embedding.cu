// Vocab-parallel embedding lookup and its backward.
//
// "02 - How a whole Transformer block is split", section 3: the [vocab, h]
// table is split along the vocabulary; a shard holds rows [v0, v1), looks up
// the tokens whose id falls in its range and writes zero rows for the others,
// so the sum of all shards' outputs is the full lookup. Input and output
// embeddings are tied: the table's gradient is the lookup's gradient plus the
// output projection's (the cross-entropy's).
//
//   forward   out[t] = E_shard[ids[t] - v0] if v0 <= ids[t] < v1 else 0
//             (a 16-byte-vector row copy; blocks stride over the tokens)
//   backward  dE_shard[v - v0] (+)= sum over tokens t with ids[t] = v of dout[t]
//
// The backward is deterministic without floating-point atomics: every row's
// tokens are summed in token order, in float32, by one block. To find them,
// each token gets its stable rank among the tokens with the same id (tiles of
// ids compared in shared memory), the per-row counts (integer atomics: the
// totals do not depend on order) are scanned into row offsets, and
// each token writes its index at offset + rank. Rows without tokens are
// written as zeros (overwrite) or left alone (accumulate).
#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

template <typename T> struct EVec;
template <> struct EVec<bf16> { static constexpr int N = 8; };
template <> struct EVec<float> { static constexpr int N = 4; };

template <typename T>
__device__ __forceinline__ void eload(const T* p, float* f) {
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
__device__ __forceinline__ void estore(T* p, const float* f) {
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

// Masked row copy: one 16-byte vector per thread per step; blocks stride
// over the tokens (whole rows are moved as raw bytes: the copy is exact).
__global__ void emb_fwd_kernel(int T, int H, int elt, int v0, int v1, const int32_t* __restrict__ ids,
                               const uint8_t* __restrict__ emb, uint8_t* __restrict__ out) {
  const int64_t row_bytes = (int64_t)H * elt;
  const int nvec = (int)(row_bytes / 16);
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const int v = ids[t];
    const bool own = v >= v0 && v < v1;
    const uint4* src = reinterpret_cast<const uint4*>(emb + (own ? (int64_t)(v - v0) * row_bytes : 0));
    uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)t * row_bytes);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x)
      dst[i] = own ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
  }
}

constexpr int RANK_TILE = 1024;

// rank[t] = number of earlier tokens with the same id (ids outside the
// shard get -1); counts[v - v0] += 1 for tokens the shard owns.
__global__ void __launch_bounds__(256) emb_rank_kernel(int T, int v0, int v1,
                                                       const int32_t* __restrict__ ids,
                                                       int32_t* __restrict__ rank,
                                                       int32_t* __restrict__ counts) {
  __shared__ int32_t tile[RANK_TILE];
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int v = t < T ? ids[t] : -1;
  const bool own = t < T && v >= v0 && v < v1;
  int r = 0;
  const int last = min(T, (int)((blockIdx.x + 1) * blockDim.x));  // tokens before this block's end
  for (int base = 0; base < last; base += RANK_TILE) {
    const int n = min(RANK_TILE, last - base);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) tile[i] = ids[base + i];
    __syncthreads();
    if (own) {
      const int lim = min(n, t - base);  // only tokens t' < t
      for (int i = 0; i < lim; ++i) r += tile[i] == v;
    }
  }
  if (t < T) {
    rank[t] = own ? r : -1;
    if (own) atomicAdd(counts + (v - v0), 1);
  }
}

// Exclusive scan of the per-row counts, in three steps:
//   emb_scan_chunks  each block scans SCAN_CHUNK counts (4 per thread, 16-byte
//                    loads) into local offsets and writes the chunk's total
//   emb_scan_totals  one block scans the chunk totals (fixed order)
//   emb_scan_add     adds each chunk's base; offsets[n] = the grand total
constexpr int SCAN_THREADS = 1024, SCAN_CHUNK = 4 * SCAN_THREADS;

// inclusive block scan of one value per thread (warp shuffles, then the warp totals)
__device__ __forceinline__ int block_incl_scan(int v, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += x;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  return v + (warp > 0 ? wsum[warp - 1] : 0);
}

__global__ void __launch_bounds__(SCAN_THREADS) emb_scan_chunks(int n, const int32_t* __restrict__ counts,
                                                                int32_t* __restrict__ offsets,
                                                                int32_t* __restrict__ totals) {
  __shared__ int wsum[32];
  const int base = blockIdx.x * SCAN_CHUNK + threadIdx.x * 4;
  int c[4] = {0, 0, 0, 0};
  if (base + 3 < n) {
    const int4 q = *reinterpret_cast<const int4*>(counts + base);
    c[0] = q.x; c[1] = q.y; c[2] = q.z; c[3] = q.w;
  } else {
    for (int j = 0; j < 4; ++j)
      if (base + j < n) c[j] = counts[base + j];
  }
  const int mine = c[0] + c[1] + c[2] + c[3];
  const int incl = block_incl_scan(mine, wsum);
  int run = incl - mine;
  for (int j = 0; j < 4; ++j) {
    if (base + j < n) offsets[base + j] = run;
    run += c[j];
  }
  if (threadIdx.x == blockDim.x - 1) totals[blockIdx.x] = incl;
}

__global__ void __launch_bounds__(SCAN_THREADS) emb_scan_totals(int nchunks,
                                                                int32_t* __restrict__ totals) {
  __shared__ int wsum[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int b = 0; b < nchunks; b += blockDim.x) {
    const int i = b + threadIdx.x;
    const int v = i < nchunks ? totals[i] : 0;
    const int incl = block_incl_scan(v, wsum);
    const int c0 = carry;
    __syncthreads();
    if (i < nchunks) totals[i] = c0 + incl - v;  // exclusive base of chunk i
    if (threadIdx.x == blockDim.x - 1) carry = c0 + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) totals[nchunks] = carry;
}

__global__ void emb_scan_add(int n, const int32_t* __restrict__ totals, int nchunks,
                             int32_t* __restrict__ offsets) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) offsets[i] += totals[i / SCAN_CHUNK];
  if (i == 0) offsets[n] = totals[nchunks];
}

__global__ void emb_place_kernel(int T, int v0, const int32_t* __restrict__ ids,
                                 const int32_t* __restrict__ rank,
                                 const int32_t* __restrict__ offsets, int32_t* __restrict__ order) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T && rank[t] >= 0) order[offsets[ids[t] - v0] + rank[t]] = t;
}

// One block per shard row: sum its tokens' gradient rows in token order.
template <typename T>
__global__ void emb_accum_kernel(int rows, int H, const int32_t* __restrict__ offsets,
                                 const int32_t* __restrict__ order, const T* __restrict__ dout,
                                 T* __restrict__ d_emb, int accumulate) {
  constexpr int VN = EVec<T>::N;
  const int nvec = H / VN;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int a = offsets[row], b = offsets[row + 1];
    if (a == b && accumulate) continue;
    T* dst = d_emb + (int64_t)row * H;
    for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
      float acc[VN];
      if (accumulate) {
        eload(dst + vi * VN, acc);
      } else {
#pragma unroll
        for (int j = 0; j < VN; ++j) acc[j] = 0.0f;
      }
      for (int i = a; i < b; ++i) {
        float g[VN];
        eload(dout + (int64_t)order[i] * H + vi * VN, g);
#pragma unroll
        for (int j = 0; j < VN; ++j) acc[j] += g[j];
      }
      estore(dst + vi * VN, acc);
    }
  }
}

}  // namespace

size_t embedding_bwd_ws(int T, int v0, int v1) {
  const size_t rows = v1 > v0 ? (size_t)(v1 - v0) : 0;
  const size_t chunks = (rows + SCAN_CHUNK - 1) / SCAN_CHUNK;
  // rank, order [T]; counts [rows] (padded to 16 bytes); offsets [rows + 1]; chunk totals
  return 4 * (2 * (size_t)T + (rows + 3) / 4 * 4 + rows + 1 + chunks + 1) + 256;
}

mgb_status embedding_fwd_launch(int T, int H, int dtype, int v0, int v1, const int32_t* ids,
                                const void* emb, void* out, cudaStream_t st) {
  if (T == 0) return MGB_OK;
  const int elt = dtype == MGB_BF16 ? 2 : 4;
  const int nvec = H * elt / 16;
  const int threads = nvec >= 256 ? 256 : ((nvec + 31) / 32) * 32;
  const int grid = T < device_sm_count() * 16 ? T : device_sm_count() * 16;
  LaunchScope scope(PROF_EMBEDDING, st);
  emb_fwd_kernel<<<grid, threads, 0, st>>>(T, H, elt, v0, v1, ids,
                                            static_cast<const uint8_t*>(emb),
                                            static_cast<uint8_t*>(out));
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status embedding_bwd_launch(int T, int H, int dtype, int v0, int v1, const int32_t* ids,
                                const void* dout, void* d_emb, int accumulate, void* ws,
                                cudaStream_t st) {
  const int rows = v1 - v0;
  const int nchunks = (rows + SCAN_CHUNK - 1) / SCAN_CHUNK;
  int32_t* rank = static_cast<int32_t*>(ws);
  int32_t* order = rank + T;
  int32_t* counts = order + T;
  counts += (4 - (reinterpret_cast<uintptr_t>(counts) / 4) % 4) % 4;  // 16-byte aligned
  int32_t* offsets = counts + (rows + 3) / 4 * 4;
  int32_t* totals = offsets + rows + 1;
  LaunchScope scope(PROF_EMBEDDING, st, 6);
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * rows, st) != cudaSuccess) return MGB_ERR_CUDA;
  if (T > 0) emb_rank_kernel<<<(T + 63) / 64, 64, 0, st>>>(T, v0, v1, ids, rank, counts);
  emb_scan_chunks<<<nchunks, SCAN_THREADS, 0, st>>>(rows, counts, offsets, totals);
  emb_scan_totals<<<1, SCAN_THREADS, 0, st>>>(nchunks, totals);
  emb_scan_add<<<(rows + 255) / 256, 256, 0, st>>>(rows, totals, nchunks, offsets);
  if (T > 0) emb_place_kernel<<<(T + 255) / 256, 256, 0, st>>>(T, v0, ids, rank, offsets, order);
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  const int nvec = H / vn;
  const int threads = nvec >= 256 ? 256 : ((nvec + 31) / 32) * 32;
  const int grid = rows < device_sm_count() * 32 ? rows : device_sm_count() * 32;
  if (dtype == MGB_BF16)
    emb_accum_kernel<bf16><<<grid, threads, 0, st>>>(rows, H, offsets, order,
                                                     static_cast<const bf16*>(dout),
                                                     static_cast<bf16*>(d_emb), accumulate);
  else
    emb_accum_kernel<float><<<grid, threads, 0, st>>>(rows, H, offsets, order,
                                                      static_cast<const float*>(dout),
                                                      static_cast<float*>(d_emb), accumulate);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

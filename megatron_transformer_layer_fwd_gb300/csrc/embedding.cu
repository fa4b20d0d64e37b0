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

constexpr int RANK_I = 128, RANK_J = 512;

// rank[t] += number of tokens t' < t with ids[t'] = ids[t], over the tokens t'
// of tile blockIdx.y (RANK_J of them) and the tokens t of tile blockIdx.x
// (RANK_I, one per thread); rank starts at zero and the partial counts are
// added with integer atomics, so the result does not depend on block order.
// Tiles of blockIdx.y == 0 also count the shard's tokens per row.
__global__ void __launch_bounds__(RANK_I) emb_rank_kernel(int T, int v0, int v1,
                                                          const int32_t* __restrict__ ids,
                                                          int32_t* __restrict__ rank,
                                                          int32_t* __restrict__ counts) {
  __shared__ __align__(16) int32_t tile[RANK_J];
  const int i0 = blockIdx.x * RANK_I, j0 = blockIdx.y * RANK_J;
  if (j0 >= min(T, i0 + RANK_I) - 1 && blockIdx.y > 0) return;  // no t' < t in this tile
  const int t = i0 + threadIdx.x;
  const int v = t < T ? ids[t] : -1;
  const bool own = t < T && v >= v0 && v < v1;
  if (blockIdx.y == 0 && own) atomicAdd(counts + (v - v0), 1);
  const int n = min(RANK_J, T - j0);
  for (int i = threadIdx.x; i < n; i += RANK_I) tile[i] = ids[j0 + i];
  __syncthreads();
  const int lim = own ? max(0, min(n, t - j0)) : 0;  // tokens t' < t of this tile
  int r = 0;
  const int4* tile4 = reinterpret_cast<const int4*>(tile);
#pragma unroll 4
  for (int q = 0; q < lim / 4; ++q) {
    const int4 x = tile4[q];
    r += (x.x == v) + (x.y == v) + (x.z == v) + (x.w == v);
  }
  for (int i = lim & ~3; i < lim; ++i) r += tile[i] == v;
  if (r > 0) atomicAdd(rank + t, r);
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

// Token t goes to order[offsets[row] + rank[t]]; the first token of a row
// also records the row and the end of its segment at that position.
__global__ void emb_place_kernel(int T, int v0, int v1, const int32_t* __restrict__ ids,
                                 const int32_t* __restrict__ rank,
                                 const int32_t* __restrict__ offsets, int32_t* __restrict__ order,
                                 int32_t* __restrict__ seg_row, int32_t* __restrict__ seg_end) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int v = ids[t];
  if (v < v0 || v >= v1) return;
  const int row = v - v0, rk = rank[t], pos = offsets[row] + rk;
  order[pos] = t;
  seg_row[pos] = rk == 0 ? row : -1;
  if (rk == 0) seg_end[pos] = offsets[row + 1];
}

// As emb_place_kernel, for accumulate mode, from the chunk-local offsets of
// emb_scan_chunks and the raw chunk totals (nchunks <= 1024): each block scans
// the chunk totals itself (fixed order), so the last two scan steps are not
// launched. *npos = the in-shard tokens (written by block 0).
__global__ void __launch_bounds__(256) emb_place_chunked_kernel(
    int T, int v0, int v1, const int32_t* __restrict__ ids, const int32_t* __restrict__ rank,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ local_off,
    const int32_t* __restrict__ totals, int nchunks, int32_t* __restrict__ order,
    int32_t* __restrict__ seg_row, int32_t* __restrict__ seg_end, int32_t* __restrict__ npos) {
  __shared__ int cbase[1025];  // exclusive chunk bases, then the grand total
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nchunks ? totals[c] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (c < nchunks) cbase[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      cbase[nchunks] = carry;
      if (blockIdx.x == 0) *npos = carry;
    }
  }
  __syncthreads();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int v = ids[t];
  if (v < v0 || v >= v1) return;
  const int row = v - v0, rk = rank[t];
  const int start = local_off[row] + cbase[row / SCAN_CHUNK];
  const int pos = start + rk;
  order[pos] = t;
  seg_row[pos] = rk == 0 ? row : -1;
  if (rk == 0) seg_end[pos] = start + counts[row];
}

// Sum of one row's token gradients in token order (float32), added to or
// written over the row.
template <typename T>
__device__ __forceinline__ void emb_row_sum(int H, int a, int b, const int32_t* __restrict__ order,
                                            const T* __restrict__ dout, T* __restrict__ dst,
                                            bool accumulate) {
  constexpr int VN = EVec<T>::N;
  const int nvec = H / VN;
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

// 16 bytes of a row as raw bits (converted to float32 where they are added).
template <typename T>
__device__ __forceinline__ uint4 eraw(const T* p) {
  return *reinterpret_cast<const uint4*>(p);
}
// f[j] = x[j] + y[j] from two raw vectors.
template <typename T>
__device__ __forceinline__ void eadd_raw(const uint4& x, const uint4& y, float* f) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t wx[4] = {x.x, x.y, x.z, x.w}, wy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = unpack_bf16x2(wx[i]), b = unpack_bf16x2(wy[i]);
      f[2 * i] = a.x + b.x;
      f[2 * i + 1] = a.y + b.y;
    }
  } else {
    f[0] = __uint_as_float(x.x) + __uint_as_float(y.x);
    f[1] = __uint_as_float(x.y) + __uint_as_float(y.y);
    f[2] = __uint_as_float(x.z) + __uint_as_float(y.z);
    f[3] = __uint_as_float(x.w) + __uint_as_float(y.w);
  }
}
// f[j] += y[j] from a raw vector.
template <typename T>
__device__ __forceinline__ void eacc_raw(const uint4& y, float* f) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t wy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 b = unpack_bf16x2(wy[i]);
      f[2 * i] += b.x;
      f[2 * i + 1] += b.y;
    }
  } else {
    f[0] += __uint_as_float(y.x); f[1] += __uint_as_float(y.y);
    f[2] += __uint_as_float(y.z); f[3] += __uint_as_float(y.w);
  }
}

// Accumulate mode, one block per position of the token order (T blocks, *npos
// positions used): the block at the head of a row's segment adds
// the row's tokens in token order onto the row, the others return. Two
// vectors per thread per step, with the row's and the first token's vectors
// requested together and held as raw bits until they are added, so that the
// kernel fits six 256-thread blocks per SM (40 registers a thread).
template <typename T>
__global__ void __launch_bounds__(256, 6) emb_accum_heads_kernel(
    int H, const int32_t* __restrict__ npos, const int32_t* __restrict__ order,
    const int32_t* __restrict__ seg_row, const int32_t* __restrict__ seg_end,
    const T* __restrict__ dout, T* __restrict__ d_emb) {
  constexpr int VN = EVec<T>::N;
  const int p = blockIdx.x;
  // the position's entries are requested together with the position count
  // (one round trip instead of three; p < T, so every read is in bounds, and
  // the values past *npos are not used)
  const int n = *npos;
  const int row = seg_row[p], end = seg_end[p], t0 = order[p];
  if (p >= n || row < 0) return;
  const int nvec = H / VN;
  T* dst = d_emb + (int64_t)row * H;
  const T* g0 = dout + (int64_t)t0 * H;
  for (int vi = threadIdx.x; vi < nvec; vi += 2 * blockDim.x) {
    const int vj = vi + blockDim.x;
    const bool two = vj < nvec;
    const uint4 ra = eraw(dst + vi * VN), qa = eraw(g0 + vi * VN);
    uint4 rb = make_uint4(0u, 0u, 0u, 0u), qb = rb;
    if (two) {
      rb = eraw(dst + vj * VN);
      qb = eraw(g0 + vj * VN);
    }
    float a[VN], b[VN];
    eadd_raw<T>(ra, qa, a);
    eadd_raw<T>(rb, qb, b);
    for (int i = p + 1; i < end; ++i) {
      const T* gi = dout + (int64_t)order[i] * H;
      const uint4 ga = eraw(gi + vi * VN);
      uint4 gb = make_uint4(0u, 0u, 0u, 0u);
      if (two) gb = eraw(gi + vj * VN);
      eacc_raw<T>(ga, a);
      eacc_raw<T>(gb, b);
    }
    estore(dst + vi * VN, a);
    if (two) estore(dst + vj * VN, b);
  }
}

// Overwrite mode: blocks stride over all shard rows; rows without tokens are
// written as zeros.
template <typename T>
__global__ void emb_write_rows_kernel(int rows, int H, const int32_t* __restrict__ offsets,
                                      const int32_t* __restrict__ order, const T* __restrict__ dout,
                                      T* __restrict__ d_emb) {
  for (int row = blockIdx.x; row < rows; row += gridDim.x)
    emb_row_sum<T>(H, offsets[row], offsets[row + 1], order, dout, d_emb + (int64_t)row * H, false);
}

}  // namespace

size_t embedding_bwd_ws(int T, int v0, int v1) {
  const size_t rows = v1 > v0 ? (size_t)(v1 - v0) : 0;
  const size_t chunks = (rows + SCAN_CHUNK - 1) / SCAN_CHUNK;
  // counts [rows] (padded to a multiple of 4), rank, order, seg_row, seg_end
  // [T]; offsets [rows + 1]; chunk totals [chunks + 1]; positions [1]
  return 4 * ((rows + 3) / 4 * 4 + 4 * (size_t)T + rows + 1 + chunks + 1 + 1) + 256;
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

namespace {

// The workspace's arrays (layout of embedding_bwd_ws).
struct EmbWs {
  int32_t *counts, *rank, *order, *seg_row, *seg_end, *offsets, *totals, *npos;
  EmbWs(void* ws, int T, int rows) {
    const int nchunks = (rows + SCAN_CHUNK - 1) / SCAN_CHUNK;
    // counts and rank side by side (one zeroing); counts first, so 16-byte aligned
    counts = static_cast<int32_t*>(ws);
    rank = counts + (rows + 3) / 4 * 4;
    order = rank + T;
    seg_row = order + T;
    seg_end = seg_row + T;
    offsets = seg_end + T;
    totals = offsets + rows + 1;
    npos = totals + nchunks + 1;
  }
};

// The token order: ranks, the scan of the per-row counts and the placement.
// chunked (accumulate mode only, at most 1024 scan chunks): the placement
// finishes the scan itself and writes *npos, and the row offsets stay
// chunk-local; otherwise the full scan, offsets[rows] = the in-shard tokens.
mgb_status emb_plan(int T, int v0, int v1, const int32_t* ids, bool chunked, const EmbWs& w,
                    cudaStream_t st) {
  const int rows = v1 - v0;
  const int nchunks = (rows + SCAN_CHUNK - 1) / SCAN_CHUNK;
  if (cudaMemsetAsync(w.counts, 0, sizeof(int32_t) * ((rows + 3) / 4 * 4 + (size_t)T), st) !=
      cudaSuccess)
    return MGB_ERR_CUDA;
  if (T > 0) {
    const dim3 grid((T + RANK_I - 1) / RANK_I, (T + RANK_J - 1) / RANK_J);
    emb_rank_kernel<<<grid, RANK_I, 0, st>>>(T, v0, v1, ids, w.rank, w.counts);
  }
  emb_scan_chunks<<<nchunks, SCAN_THREADS, 0, st>>>(rows, w.counts, w.offsets, w.totals);
  if (chunked) {
    emb_place_chunked_kernel<<<(T + 255) / 256, 256, 0, st>>>(
        T, v0, v1, ids, w.rank, w.counts, w.offsets, w.totals, nchunks, w.order, w.seg_row,
        w.seg_end, w.npos);
  } else {
    emb_scan_totals<<<1, SCAN_THREADS, 0, st>>>(nchunks, w.totals);
    emb_scan_add<<<(rows + 255) / 256, 256, 0, st>>>(rows, w.totals, nchunks, w.offsets);
    if (T > 0)
      emb_place_kernel<<<(T + 255) / 256, 256, 0, st>>>(T, v0, v1, ids, w.rank, w.offsets,
                                                        w.order, w.seg_row, w.seg_end);
  }
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

// The row sums from a token order made by emb_plan (chunked as there).
mgb_status emb_apply(int T, int H, int dtype, int rows, const void* dout, void* d_emb,
                     bool accumulate, bool chunked, const EmbWs& w, cudaStream_t st) {
  const int vn = dtype == MGB_BF16 ? 8 : 4;
  const int nvec = H / vn;
  if (accumulate) {
    if (T == 0) return MGB_OK;  // nothing to add
    // one block per position; two vectors per thread per step
    const int athreads = std::min(256, ((nvec + 1) / 2 + 31) / 32 * 32);
    const int32_t* np = chunked ? w.npos : w.offsets + rows;
    if (dtype == MGB_BF16)
      emb_accum_heads_kernel<bf16><<<T, athreads, 0, st>>>(H, np, w.order, w.seg_row, w.seg_end,
                                                           static_cast<const bf16*>(dout),
                                                           static_cast<bf16*>(d_emb));
    else
      emb_accum_heads_kernel<float><<<T, athreads, 0, st>>>(H, np, w.order, w.seg_row, w.seg_end,
                                                            static_cast<const float*>(dout),
                                                            static_cast<float*>(d_emb));
  } else {
    const int threads = nvec >= 256 ? 256 : ((nvec + 31) / 32) * 32;
    const int grid = rows < device_sm_count() * 32 ? rows : device_sm_count() * 32;
    if (dtype == MGB_BF16)
      emb_write_rows_kernel<bf16><<<grid, threads, 0, st>>>(rows, H, w.offsets, w.order,
                                                            static_cast<const bf16*>(dout),
                                                            static_cast<bf16*>(d_emb));
    else
      emb_write_rows_kernel<float><<<grid, threads, 0, st>>>(rows, H, w.offsets, w.order,
                                                             static_cast<const float*>(dout),
                                                             static_cast<float*>(d_emb));
  }
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

mgb_status embedding_bwd_launch(int T, int H, int dtype, int v0, int v1, const int32_t* ids,
                                const void* dout, void* d_emb, int accumulate, void* ws,
                                cudaStream_t st) {
  const int rows = v1 - v0;
  const int nchunks = (rows + SCAN_CHUNK - 1) / SCAN_CHUNK;
  if (accumulate && T == 0) return MGB_OK;  // nothing to add
  // accumulate: rank, chunk scan, placement (finishing the scan), sums;
  // overwrite: rank, the three scan steps, placement, every row written
  const bool chunked = accumulate && nchunks <= 1024;
  LaunchScope scope(PROF_EMBEDDING, st, chunked ? 4 : 3 + (T > 0 ? 3 : 1));
  const EmbWs w(ws, T, rows);
  const mgb_status planned = emb_plan(T, v0, v1, ids, chunked, w, st);
  if (planned != MGB_OK) return planned;
  return emb_apply(T, H, dtype, rows, dout, d_emb, accumulate != 0, chunked, w, st);
}

mgb_status embedding_bwd_prepare_launch(int T, int v0, int v1, const int32_t* ids, void* ws,
                                        cudaStream_t st) {
  LaunchScope scope(PROF_EMBEDDING, st, 3 + (T > 0 ? 2 : 0));
  return emb_plan(T, v0, v1, ids, false, EmbWs(ws, T, v1 - v0), st);
}

mgb_status embedding_bwd_apply_launch(int T, int H, int dtype, int v0, int v1, const void* dout,
                                      void* d_emb, int accumulate, const void* ws,
                                      cudaStream_t st) {
  if (accumulate && T == 0) return MGB_OK;
  LaunchScope scope(PROF_EMBEDDING, st, 1);
  return emb_apply(T, H, dtype, v1 - v0, dout, d_emb, accumulate != 0, false,
                   EmbWs(const_cast<void*>(ws), T, v1 - v0), st);
}

}  // namespace mgb

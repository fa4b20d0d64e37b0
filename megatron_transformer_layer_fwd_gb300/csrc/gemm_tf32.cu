// float32 GEMM on the 5th-generation tensor cores with three TF32 products
// (tcgen05.mma kind::tf32), for the float32 layer.
//
// acc[m][n] = alpha * sum_k A(m,k) B(n,k) close to float32 accuracy: each
// operand x is split into hi = x rounded to tf32 (10 mantissa bits) and lo =
// (x - hi) rounded to tf32, both exact in their 32-bit containers, and
// acc = A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T with float32 accumulation in
// TMEM. Every product of two tf32 values is exact in float32; the dropped
// A_lo B_lo^T term and the rounding of lo are each about 2^-22 relative to
// |a||b| per product. The tensor core's own float32 accumulation loses more
// as K grows (6e-5 relative at K 8192 when it runs over the whole K), so the
// accumulator is promoted every 128 K: the MMA warp starts each K chunk in the
// next of four TMEM buffers, and the epilogue warps add the chunks in float32
// registers (9e-7 relative at K 8192, below the FFMA product's 1.6e-6; one
// TF32 product gives 3e-4).
//
// A pre-pass writes hi and lo of both operands as K-major float32 copies
// (transposing an MN-major operand) into the caller's scratch, with K padded
// to a multiple of 4 (16-byte rows for TMA) by zeros. The product kernel then
// only ever reads K-major tf32 tiles: per 32-wide K block, TMA brings the four
// tiles A_hi, A_lo, B_hi, B_lo (128 x 32 float32 each, 128-byte swizzle: the
// same byte layout as a 128 x 64 bf16 tile) into one stage of a 3-stage ring,
// and the MMA warp issues three M=128 N=128 K=8 products per 8-wide K step.
// One persistent CTA per SM walks 128 x 128 output tiles, six warps as in the
// bf16 GEMM: producer, MMA issuer, four epilogue warps reading the two
// double-buffered TMEM accumulators; the epilogue is the float32 one of the
// SIMT GEMM (bias, activation, residual, activation gradient, accumulate).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "f32_epilogue.cuh"
#include "internal.h"

namespace mgb {

namespace {

constexpr int TBM = 128, TBN = 128, TBK = 32;  // tile rows, tile columns, K per block
constexpr int TSTAGES = 3;
constexpr int TACC = 4;  // accumulator buffers in TMEM (one per K chunk in turn)

constexpr int TILE4 = TBM * TBK * 4;           // one 128 x 32 float32 tile: 16 KB
constexpr int TSTAGE = 4 * TILE4;              // A_hi, A_lo, B_hi, B_lo
constexpr int TSMEM = TSTAGES * TSTAGE + 1024 + 1024;

struct Tf32Params {
  SimtParams e;  // epilogue (C, bias, ...; A/B fields unused)
  int tiles_m, tiles_n, num_k;
  // K blocks per accumulation chunk: the tensor core sums one chunk in its
  // float32 accumulator, the epilogue adds the chunks in float32 registers
  int kchunk;
  int* err;
};

// x rounded to the nearest tf32 value (10 mantissa bits; halfway cases away
// from zero), as a float32 whose 13 low mantissa bits are zero.
__device__ __forceinline__ float round_tf32(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// hi / lo of one float32 value, both exact tf32 values (so the tensor core
// reads them unchanged): hi = x rounded to tf32, lo = (x - hi) rounded to
// tf32; |x - hi - lo| <= 2^-22 |x| (about).
__device__ __forceinline__ void tf32_split(float x, float& hi, float& lo) {
  hi = round_tf32(x);
  lo = round_tf32(x - hi);
}

// out_hi / out_lo [R][Kp] (K-major, row stride Kp, columns K..Kp-1 zero) from
// X(r, k) = src[r * ld + k] (src_mn = 0) or src[k * ld + r] (src_mn = 1).
// 32 x 32 tiles through shared memory: reads coalesced along src's
// contiguous index, writes coalesced along k.
__global__ void __launch_bounds__(256) tf32_split_kernel(int R, int K, int Kp, const float* src,
                                                         int64_t ld, int src_mn, float* out_hi,
                                                         float* out_lo) {
  __shared__ float t[32][33];
  const int r0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < 32; i += 8) {
    if (src_mn) {  // contiguous along r: lane = r
      const int k = k0 + i, r = r0 + tx;
      t[tx][i] = (r < R && k < K) ? src[(int64_t)k * ld + r] : 0.0f;
    } else {       // contiguous along k: lane = k
      const int r = r0 + i, k = k0 + tx;
      t[i][tx] = (r < R && k < K) ? src[(int64_t)r * ld + k] : 0.0f;
    }
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i, k = k0 + tx;
    if (r < R && k < Kp) {
      float hi, lo;
      tf32_split(t[i][tx], hi, lo);
      out_hi[(int64_t)r * Kp + k] = hi;
      out_lo[(int64_t)r * Kp + k] = lo;
    }
  }
}

// Persistent CTA per SM, six warps (see the file comment). Barriers: full[s]
// (the stage's four tiles landed), empty[s] (its products done), accf[b] /
// acce[b] (accumulator b ready / drained). Every wait is bounded.
__global__ void __launch_bounds__(192, 1)
    gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap tmAh,
                       const __grid_constant__ CUtensorMap tmAl,
                       const __grid_constant__ CUtensorMap tmBh,
                       const __grid_constant__ CUtensorMap tmBl, const Tf32Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TSTAGES * TSTAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * TSTAGES + 2 * TACC);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t tiles = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * TSTAGES;
  const uint32_t accf0 = empty0 + 8 * TSTAGES;
  const uint32_t acce0 = accf0 + 8 * TACC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = p.tiles_m * p.tiles_n;
  const int nkc = p.num_k > 0 ? p.num_k : 1;  // K blocks, or one empty chunk when K = 0

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmAh);
    tma_prefetch_desc(&tmAl);
    tma_prefetch_desc(&tmBh);
    tma_prefetch_desc(&tmBl);
    for (int s = 0; s < TSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < TACC; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4);
    }
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TACC * TBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t kg = 0;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        const int m0 = (tile % p.tiles_m) * TBM, n0 = (tile / p.tiles_m) * TBN;
        for (int kb = 0; kb < p.num_k; ++kb, ++kg) {
          const int s = kg % TSTAGES;
          if (!mbar_wait(empty0 + 8 * s, ((kg / TSTAGES) & 1) ^ 1, p.err)) {
            *abort = 1;
            break;
          }
          const uint32_t st = tiles + s * TSTAGE;
          const uint32_t fb = full0 + 8 * s;
          const int k0 = kb * TBK;
          // x coordinates multiples of 4 float32 (16 bytes), tile inside the problem
          if (!dcheck((k0 & 3) == 0 && m0 < p.e.M && n0 < p.e.N, p.err)) {
            *abort = 1;
            break;
          }
          mbar_arrive_expect_tx(fb, TSTAGE);
          tma_load_2d(st, &tmAh, k0, m0, fb);
          tma_load_2d(st + TILE4, &tmAl, k0, m0, fb);
          tma_load_2d(st + 2 * TILE4, &tmBh, k0, n0, fb);
          tma_load_2d(st + 3 * TILE4, &tmBl, k0, n0, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: per 8-wide K step, A_lo B_hi, A_hi B_lo,
      // then A_hi B_hi (small terms first)
      constexpr uint32_t idesc = idesc_tf32_f32(TBM, TBN);
      uint32_t kg = 0;
      int t = 0;
      bool good = true;
      for (int tile = blockIdx.x; tile < total && !*abort && good; tile += gridDim.x) {
       for (int c0 = 0; c0 < nkc; c0 += p.kchunk, ++t) {  // one accumulator buffer per chunk
        const int buf = t % TACC;
        if (!mbar_wait_spin(acce0 + 8 * buf, ((t / TACC) & 1) ^ 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * TBN;
        const int c1 = min(c0 + p.kchunk, p.num_k);
        for (int kb = c0; kb < c1; ++kb, ++kg) {
          const int s = kg % TSTAGES;
          if (!mbar_wait(full0 + 8 * s, (kg / TSTAGES) & 1, p.err)) {
            good = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = tiles + s * TSTAGE;
#pragma unroll
          for (int kk = 0; kk < TBK / 8; ++kk) {
            const uint64_t ah = smem_desc_sw128(st + 32 * kk, 16, 1024);
            const uint64_t al = smem_desc_sw128(st + TILE4 + 32 * kk, 16, 1024);
            const uint64_t bh = smem_desc_sw128(st + 2 * TILE4 + 32 * kk, 16, 1024);
            const uint64_t bl = smem_desc_sw128(st + 3 * TILE4 + 32 * kk, 16, 1024);
            tc_mma_tf32(acc, al, bh, idesc, (kb != c0 || kk != 0) ? 1u : 0u);
            tc_mma_tf32(acc, ah, bl, idesc, 1u);
            tc_mma_tf32(acc, ah, bh, idesc, 1u);
          }
          tc_commit(empty0 + 8 * s);
        }
        if (!good) break;
        tc_commit(accf0 + 8 * buf);
       }
      }
      if (!good) *abort = 1;
    }
  } else {
    // ---------------- epilogue warps 2..5: one output row per thread, the
    // tile's K chunks summed in float32 registers, then the epilogue
    const int q = warp & 3;
    int t = 0;
    bool good = true;
    for (int tile = blockIdx.x; tile < total && good; tile += gridDim.x) {
      const int m0 = (tile % p.tiles_m) * TBM, n0 = (tile / p.tiles_m) * TBN;
      const int row = m0 + q * 32 + lane;
      float sum[TBN];
#pragma unroll
      for (int j = 0; j < TBN; ++j) sum[j] = 0.0f;
      for (int c0 = 0; c0 < nkc; c0 += p.kchunk, ++t) {
        const int buf = t % TACC;
        const bool ready = !*abort && mbar_wait_spin(accf0 + 8 * buf, (t / TACC) & 1, p.err);
        if (!__all_sync(0xffffffffu, ready)) {
          good = false;
          break;
        }
        tc_fence_after();
        const uint32_t trow = tmem + buf * TBN + ((uint32_t)(q * 32) << 16);
#pragma unroll
        for (int lc = 0; lc < TBN; lc += 32) {
          uint32_t r[32];
          tmem_ld32(trow + lc, r);
          tmem_ld_wait();
          if (p.num_k > 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[lc + j] += __uint_as_float(r[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce0 + 8 * buf);
      }
      if (!good) break;
      if (row < p.e.M) {
#pragma unroll
        for (int j = 0; j < TBN; ++j) {
          const int n = n0 + j;
          if (n < p.e.N) epi_elem(p.e, row, n, p.e.alpha * sum[j]);
        }
      }
    }
    if (!good) *abort = 1;
  }

  __syncthreads();
  if (*abort && threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TACC * TBN);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_tf32() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// K-major float32 operand [rows][Kp]: boxes of 32 K-elements (128 bytes) x 128
// rows, 128-byte swizzle, zero fill past the edges.
bool tmap_f32_kmajor(CUtensorMap* tm, const float* base, int rows, int Kp) {
  auto fn = encode_fn_tf32();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)Kp * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t gemm_tf32_scratch_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const size_t Kp = (size_t)(K + 3) / 4 * 4;
  return 2 * al256(4 * (size_t)M * Kp) + 2 * al256(4 * (size_t)N * Kp);
}

mgb_status gemm_tf32_launch(const GemmArgs& g, cudaStream_t st) {
  if (g.scratch == nullptr || g.scratch_bytes < gemm_tf32_scratch_bytes(g.M, g.N, g.K))
    return MGB_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(g.scratch) & 255u) != 0) return MGB_ERR_MISALIGNED;
  const int Kp = (g.K + 3) / 4 * 4;
  char* sc = static_cast<char*>(g.scratch);
  float* ah = reinterpret_cast<float*>(sc);
  float* al = reinterpret_cast<float*>(sc + al256(4 * (size_t)g.M * Kp));
  float* bh = reinterpret_cast<float*>(sc + 2 * al256(4 * (size_t)g.M * Kp));
  float* bl = reinterpret_cast<float*>(sc + 2 * al256(4 * (size_t)g.M * Kp) +
                                       al256(4 * (size_t)g.N * Kp));
  LaunchScope scope(PROF_GEMM_F32, st, g.K > 0 ? 3 : 1);
  if (g.K > 0) {
    const dim3 blk(256);
    tf32_split_kernel<<<dim3((Kp + 31) / 32, (g.M + 31) / 32), blk, 0, st>>>(
        g.M, g.K, Kp, static_cast<const float*>(g.A), g.lda, g.a_mn, ah, al);
    tf32_split_kernel<<<dim3((Kp + 31) / 32, (g.N + 31) / 32), blk, 0, st>>>(
        g.N, g.K, Kp, static_cast<const float*>(g.B), g.ldb, g.b_mn, bh, bl);
  }
  CUtensorMap tah, tal, tbh, tbl;
  const int kp_map = Kp > 0 ? Kp : 4;  // K = 0: maps over the scratch, never read
  if (!tmap_f32_kmajor(&tah, ah, g.M, kp_map) || !tmap_f32_kmajor(&tal, al, g.M, kp_map) ||
      !tmap_f32_kmajor(&tbh, bh, g.N, kp_map) || !tmap_f32_kmajor(&tbl, bl, g.N, kp_map))
    return MGB_ERR_CUDA;
  Tf32Params p{};
  SimtParams& e = p.e;
  e.M = g.M; e.N = g.N; e.K = g.K;
  e.epi = g.epi; e.alpha = g.alpha;
  e.C = static_cast<float*>(g.C); e.ldc = g.ldc;
  e.bias = static_cast<const float*>(g.bias);
  e.resid = static_cast<const float*>(g.resid); e.ldr = g.ldr;
  e.C2 = static_cast<float*>(g.C2); e.ldc2 = g.ldc2;
  e.aux = static_cast<const float*>(g.aux); e.ldaux = g.ldaux;
  e.glu_block = g.glu_block; e.accumulate = g.accumulate;
  p.tiles_m = (g.M + TBM - 1) / TBM;
  p.tiles_n = (g.N + TBN - 1) / TBN;
  p.num_k = (g.K + TBK - 1) / TBK;
  // 4 K blocks (128 K) per chunk: at 8192^3 the relative error is 9e-7
  // against 5.7e-5 with one chunk over the whole K (FFMA: 1.6e-6), for about
  // 40 % more time; MGB_TF32_CHUNK=<blocks> for another length, 0 for one
  // chunk over the whole K
  p.kchunk = 4;
  if (const char* e = getenv("MGB_TF32_CHUNK")) p.kchunk = atoi(e);
  if (p.kchunk <= 0) p.kchunk = p.num_k > 0 ? p.num_k : 1;
  p.err = device_error_word();
  if (cudaFuncSetAttribute(gemm_tf32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           TSMEM) != cudaSuccess)
    return MGB_ERR_CUDA;
  const long total = (long)p.tiles_m * p.tiles_n;
  const int grid = (int)std::max(1L, std::min<long>(total, device_sm_count()));
  gemm_tf32x3_kernel<<<grid, 192, TSMEM, st>>>(tah, tal, tbh, tbl, p);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

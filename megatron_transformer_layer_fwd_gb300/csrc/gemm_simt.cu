// float32 GEMM on the CUDA cores (FFMA), for the float32 layer.
//
// Same contract as the tensor-core GEMM (internal.h GemmArgs): acc[m][n] =
// alpha * sum_k A(m,k) B(n,k) with either operand K-major or MN-major, and the
// same epilogues (f32_epilogue.cuh). gemm_launch sends float32 products to the
// three-TF32 tensor-core kernel (gemm_tf32.cu) when the caller provides its
// split-operand scratch, and here otherwise.
//
// 64 x 64 output tile per 256-thread block, 4 x 4 outputs per thread, K
// staged through shared memory 16 at a time.
#include "common.cuh"
#include "f32_epilogue.cuh"
#include "internal.h"

namespace mgb {

mgb_status gemm_tc_launch(const GemmArgs& g, cudaStream_t st);
mgb_status gemm_tf32_launch(const GemmArgs& g, cudaStream_t st);

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__global__ void __launch_bounds__(256) gemm_simt_kernel(const SimtParams p) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      int mm, kk;
      if (p.a_mn) { kk = i / TM; mm = i % TM; } else { mm = i / TK; kk = i % TK; }
      const int m = m0 + mm, k = k0 + kk;
      float v = 0.0f;
      if (m < p.M && k < p.K) v = p.a_mn ? p.A[(int64_t)k * p.lda + m] : p.A[(int64_t)m * p.lda + k];
      As[kk][mm] = v;
    }
    for (int i = threadIdx.x; i < TN * TK; i += 256) {
      int nn, kk;
      if (p.b_mn) { kk = i / TN; nn = i % TN; } else { nn = i / TK; kk = i % TK; }
      const int n = n0 + nn, k = k0 + kk;
      float v = 0.0f;
      if (n < p.N && k < p.K) v = p.b_mn ? p.B[(int64_t)k * p.ldb + n] : p.B[(int64_t)n * p.ldb + k];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n < p.N) epi_elem(p, m, n, p.alpha * acc[i][j]);
    }
  }
}

// a[m, i*gb + c] = silu(u[m, 2i*gb + c]) * u[m, (2i+1)*gb + c]   (float32)
__global__ void swiglu_f32_kernel(int M, int F, int gb, const float* u, int64_t ldu, float* a,
                                  int64_t lda) {
  const int64_t total = (int64_t)M * F;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / F), c = (int)(idx % F);
    const int i = c / gb, cc = c % gb;
    const float g = u[(int64_t)m * ldu + 2 * i * gb + cc];
    const float up = u[(int64_t)m * ldu + (2 * i + 1) * gb + cc];
    a[(int64_t)m * lda + c] = g / (1.0f + expf(-g)) * up;
  }
}

}  // namespace

mgb_status gemm_check(const GemmArgs& g) {
  if (g.M < 0 || g.N < 0 || g.K < 0 || g.k_splits < 1) return MGB_ERR_INVALID_ARG;
  if (g.k_splits > 1 && g.dtype != MGB_BF16) return MGB_ERR_UNSUPPORTED;
  if (g.dtype != MGB_BF16 && g.dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (g.epi < EPI_STORE || g.epi > EPI_CE_GRAD) return MGB_ERR_INVALID_ARG;
  if (g.epi == EPI_CE_STATS || g.epi == EPI_CE_GRAD) {
    // cross-entropy epilogues: bf16 operands only, per-row inputs present
    if (g.dtype != MGB_BF16) return MGB_ERR_UNSUPPORTED;
    if (g.epi == EPI_CE_STATS && g.M > 0 && g.N > 0 && g.C2 == nullptr) return MGB_ERR_INVALID_ARG;
    if (g.epi == EPI_CE_GRAD && g.M > 0 && g.N > 0 && (g.tgt == nullptr || g.ce_lse == nullptr))
      return MGB_ERR_INVALID_ARG;
  }
  if ((g.M > 0 && g.N > 0) && (g.C == nullptr)) return MGB_ERR_INVALID_ARG;
  if (g.K > 0 && g.M > 0 && g.N > 0 && (g.A == nullptr || g.B == nullptr)) return MGB_ERR_INVALID_ARG;
  const int64_t a_inner = g.a_mn ? g.M : g.K, b_inner = g.b_mn ? g.N : g.K;
  if (g.lda < a_inner || g.ldb < b_inner) return MGB_ERR_INVALID_ARG;
  if ((g.epi == EPI_BIAS_GELU || g.epi == EPI_BIAS_SWIGLU) && g.C2 == nullptr) return MGB_ERR_INVALID_ARG;
  if (g.epi == EPI_BIAS_RESID && g.resid == nullptr) return MGB_ERR_INVALID_ARG;
  if ((g.epi == EPI_DGELU || g.epi == EPI_DSWIGLU) && g.aux == nullptr) return MGB_ERR_INVALID_ARG;
  // fused bias-gradient partials: activation-backward epilogues, tensor-core path
  if (g.colsum_part != nullptr &&
      (g.dtype != MGB_BF16 || (g.epi != EPI_DGELU && g.epi != EPI_DSWIGLU)))
    return MGB_ERR_INVALID_ARG;
  if (g.epi == EPI_BIAS_SWIGLU || g.epi == EPI_DSWIGLU) {
    const int gb = g.glu_block;
    if (gb <= 0) return MGB_ERR_INVALID_ARG;
    const int width = g.epi == EPI_BIAS_SWIGLU ? g.N : 2 * g.N;
    if (width % (2 * gb) != 0) return MGB_ERR_INVALID_ARG;
    if (g.dtype == MGB_BF16 && (gb % 32 != 0 || 256 % (2 * gb) != 0)) return MGB_ERR_UNSUPPORTED;
  }
  if (g.dtype == MGB_BF16) {
    // TMA: 16-byte aligned bases and row strides; 16-byte epilogue vectors.
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    // (EPI_CE_STATS writes single floats to C and C2: any 4-byte alignment)
    const bool vec_out = g.epi != EPI_CE_STATS;
    if (!al(g.A) || !al(g.B) || (vec_out && (!al(g.C) || !al(g.C2))) || !al(g.resid) ||
        !al(g.aux) || !al(g.bias))
      return MGB_ERR_MISALIGNED;
    if (g.lda % 8 || g.ldb % 8 || g.N % 8) return MGB_ERR_MISALIGNED;
    const int64_t c_mult = g.epi == EPI_F32 ? 4 : g.epi == EPI_CE_STATS ? 1 : 8;
    if (g.ldc % c_mult || (g.C2 && g.ldc2 % 8) || (g.resid && g.ldr % 8) || (g.aux && g.ldaux % 8))
      return MGB_ERR_MISALIGNED;
    if (g.accumulate && g.epi != EPI_F32) return MGB_ERR_INVALID_ARG;
    if (g.f32_tma && (g.epi != EPI_F32 || g.C2 != nullptr || g.k_splits > 1 || g.ldc % 4))
      return MGB_ERR_INVALID_ARG;
    if (g.n_chunk != 0 && (g.n_chunk < 0 || g.n_chunk % 8 || g.tgt_v0 != 0 ||
                           (g.epi != EPI_CE_STATS && g.epi != EPI_CE_GRAD)))
      return MGB_ERR_INVALID_ARG;
    if (g.k_splits > 1 && (g.epi != EPI_F32 || g.accumulate || g.C2 != nullptr ||
                           g.bias != nullptr || g.split_stride % 4 ||
                           g.split_stride < (int64_t)g.M * g.ldc))
      return MGB_ERR_INVALID_ARG;
    if (g.keep != nullptr && (g.epi != EPI_CE_STATS || !al(g.keep) || g.ld_keep % 8 ||
                              g.ld_keep < g.N))
      return MGB_ERR_INVALID_ARG;
  }
  if (g.drop_thr < 256) {
    // dropout in the residual epilogue: bf16, whole 16-element stream blocks
    if (g.epi != EPI_BIAS_RESID || g.dtype != MGB_BF16) return MGB_ERR_UNSUPPORTED;
    if (g.N % 16 || g.drop_offset % 16 || g.drop_thr == 0) return MGB_ERR_INVALID_ARG;
  }
  return MGB_OK;
}

mgb_status gemm_launch(const GemmArgs& g, cudaStream_t st) {
  mgb_status s = gemm_check(g);
  if (s != MGB_OK) return s;
  if (g.M == 0 || g.N == 0) return MGB_OK;
  if (g.dtype == MGB_BF16) return gemm_tc_launch(g, st);
  // float32: three TF32 products on the tensor cores when the caller gave the
  // split operands' scratch, else the FFMA kernel (MGB_F32_SIMT=1 forces it)
  const char* simt = getenv("MGB_F32_SIMT");
  if (g.scratch != nullptr && g.K > 0 && !(simt != nullptr && simt[0] == '1')) {
    s = gemm_tf32_launch(g, st);
    if (s != MGB_OK) return s;
  } else {
    SimtParams p{};
    p.M = g.M; p.N = g.N; p.K = g.K; p.a_mn = g.a_mn; p.b_mn = g.b_mn;
    p.A = static_cast<const float*>(g.A); p.lda = g.lda;
    p.B = static_cast<const float*>(g.B); p.ldb = g.ldb;
    p.epi = g.epi; p.alpha = g.alpha;
    p.C = static_cast<float*>(g.C); p.ldc = g.ldc;
    p.bias = static_cast<const float*>(g.bias);
    p.resid = static_cast<const float*>(g.resid); p.ldr = g.ldr;
    p.C2 = static_cast<float*>(g.C2); p.ldc2 = g.ldc2;
    p.aux = static_cast<const float*>(g.aux); p.ldaux = g.ldaux;
    p.glu_block = g.glu_block; p.accumulate = g.accumulate;
    dim3 grid((g.N + TN - 1) / TN, (g.M + TM - 1) / TM);
    LaunchScope scope(PROF_GEMM_F32, st);
    gemm_simt_kernel<<<grid, 256, 0, st>>>(p);
  }
  if (g.epi == EPI_BIAS_SWIGLU) {
    LaunchScope scope(PROF_GEMM_F32, st);
    const int F = g.N / 2;
    swiglu_f32_kernel<<<1024, 256, 0, st>>>(g.M, F, g.glu_block, static_cast<const float*>(g.C),
                                            g.ldc, static_cast<float*>(g.C2), g.ldc2);
  }
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

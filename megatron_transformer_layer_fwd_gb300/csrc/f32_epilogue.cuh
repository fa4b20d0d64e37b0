// Per-element float32 epilogues of the GEMM (internal.h EpiMode), shared by
// the SIMT float32 GEMM and the 3xTF32 tensor-core GEMM: the accumulator
// acc[m][n] of one output element goes through bias / activation / residual /
// activation gradient / float32 accumulate into C (and C2).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace mgb {

struct SimtParams {
  int M, N, K, a_mn, b_mn;
  const float* A; int64_t lda;
  const float* B; int64_t ldb;
  int epi; float alpha;
  float* C; int64_t ldc;
  const float* bias;
  const float* resid; int64_t ldr;
  float* C2; int64_t ldc2;
  const float* aux; int64_t ldaux;
  int glu_block, accumulate;
};

__device__ __forceinline__ void epi_elem(const SimtParams& p, int m, int n, float acc) {
  switch (p.epi) {
    case EPI_STORE:
    case EPI_F32: {
      float v = acc + (p.bias ? p.bias[n] : 0.0f);
      float* c = p.C + (int64_t)m * p.ldc + n;
      if (p.accumulate) v += *c;
      *c = v;
      if (p.C2) p.C2[(int64_t)m * p.ldc2 + n] = v;
      break;
    }
    case EPI_BIAS_GELU: {
      const float u = acc + (p.bias ? p.bias[n] : 0.0f);
      p.C[(int64_t)m * p.ldc + n] = u;
      p.C2[(int64_t)m * p.ldc2 + n] = gelu_erf(u);
      break;
    }
    case EPI_BIAS_SWIGLU:  // u only; the activation is a separate pass
      p.C[(int64_t)m * p.ldc + n] = acc + (p.bias ? p.bias[n] : 0.0f);
      break;
    case EPI_BIAS_RESID:
      p.C[(int64_t)m * p.ldc + n] =
          p.resid[(int64_t)m * p.ldr + n] + acc + (p.bias ? p.bias[n] : 0.0f);
      break;
    case EPI_DGELU:
      p.C[(int64_t)m * p.ldc + n] = acc * gelu_erf_grad(p.aux[(int64_t)m * p.ldaux + n]);
      break;
    case EPI_DSWIGLU: {
      const int gb = p.glu_block;
      const int i = n / gb, cc = n % gb;
      const int64_t cg = (int64_t)2 * i * gb + cc, cu = cg + gb;
      const float g = p.aux[(int64_t)m * p.ldaux + cg], u = p.aux[(int64_t)m * p.ldaux + cu];
      const float s = 1.0f / (1.0f + expf(-g));
      p.C[(int64_t)m * p.ldc + cg] = acc * u * s * (1.0f + g * (1.0f - s));
      p.C[(int64_t)m * p.ldc + cu] = acc * g * s;
      break;
    }
    default:
      break;
  }
}

}  // namespace mgb

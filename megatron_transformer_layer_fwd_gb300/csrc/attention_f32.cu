// float32 attention core on the CUDA cores (the float32 layer's path).
//
// Same definition as the bf16 kernels ("02 - How a whole Transformer block is
// split", section 2: per-head softmax(Q K^T / sqrt(d)) V, GQA, optional causal
// mask). One warp per query row (forward, dQ) or per key row (dK/dV); a row's
// scores live in shared memory, so seq <= 2048 on this path. Exact float32
// exp/log keep it within 1e-4 of the float64 definition.
#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

constexpr int WPB = 4;  // warps per block
constexpr int MAXD = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float dot_rows(const float* x, const float* y, int d) {
  float s = 0.0f;
  for (int i = 0; i < d; ++i) s = fmaf(x[i], y[i], s);
  return s;
}

// scores (already softmaxed into probabilities) of query row qi against keys
// [0, n_keys) of one KV head; returns (max, sum) through refs; p in sc[].
__device__ void row_probs(const float* q, const float* K, int64_t ld_kv, int d, int n_keys,
                          float scale, float* sc, float& mx, float& sum) {
  const int lane = threadIdx.x & 31;
  mx = -INFINITY;
  for (int j = lane; j < n_keys; j += 32) {
    const float s = dot_rows(q, K + (int64_t)j * ld_kv, d) * scale;
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
  mx = warp_max(mx);
  sum = 0.0f;
  for (int j = lane; j < n_keys; j += 32) {
    const float p = expf(sc[j] - mx);
    sc[j] = p;
    sum += p;
  }
  sum = warp_sum(sum);
  __syncwarp();
}

__global__ void attn_f32_fwd_kernel(const AttnArgs a) {
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = sh + warp * a.S;
  float* qs = sh + WPB * a.S + warp * a.d;
  const int qi = blockIdx.x * WPB + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  if (qi >= a.S) return;
  const int kvh = h / (a.nq / a.nkv);
  const float* Q = reinterpret_cast<const float*>(a.q) + ((int64_t)b * a.S + qi) * a.ld_q + h * a.d;
  const float* K = reinterpret_cast<const float*>(a.k) + (int64_t)b * a.S * a.ld_kv + kvh * a.d;
  const float* V = reinterpret_cast<const float*>(a.v) + (int64_t)b * a.S * a.ld_kv + kvh * a.d;
  for (int i = lane; i < a.d; i += 32) qs[i] = Q[i];
  __syncwarp();
  const int n_keys = a.causal ? qi + 1 : a.S;
  float mx, sum;
  row_probs(qs, K, a.ld_kv, a.d, n_keys, rsqrtf((float)a.d), sc, mx, sum);
  float* O = reinterpret_cast<float*>(a.o) + ((int64_t)b * a.S + qi) * a.ld_o + h * a.d;
  for (int c = lane; c < a.d; c += 32) {
    float o = 0.0f;
    for (int j = 0; j < n_keys; ++j) o = fmaf(sc[j], V[(int64_t)j * a.ld_kv + c], o);
    O[c] = o / sum;
  }
  if (lane == 0) a.lse[((int64_t)b * a.nq + h) * a.S + qi] = mx + logf(sum);
}

__global__ void attn_f32_delta_kernel(const AttnArgs a) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= a.B * a.S * a.nq) return;
  const int tok = w / a.nq, h = w % a.nq;
  const float* O = reinterpret_cast<const float*>(a.o) + (int64_t)tok * a.ld_o + h * a.d;
  const float* dO = reinterpret_cast<const float*>(a.dout) + (int64_t)tok * a.ld_do + h * a.d;
  float s = 0.0f;
  for (int i = lane; i < a.d; i += 32) s = fmaf(O[i], dO[i], s);
  s = warp_sum(s);
  if (lane == 0) a.delta[((int64_t)(tok / a.S) * a.nq + h) * a.S + tok % a.S] = s;
}

__global__ void attn_f32_dq_kernel(const AttnArgs a) {
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = sh + warp * a.S;
  float* qs = sh + WPB * a.S + warp * 2 * a.d;
  float* os = qs + a.d;
  const int qi = blockIdx.x * WPB + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  if (qi >= a.S) return;
  const int kvh = h / (a.nq / a.nkv);
  const int64_t tok = (int64_t)b * a.S + qi;
  const float* Q = reinterpret_cast<const float*>(a.q) + tok * a.ld_q + h * a.d;
  const float* dO = reinterpret_cast<const float*>(a.dout) + tok * a.ld_do + h * a.d;
  const float* K = reinterpret_cast<const float*>(a.k) + (int64_t)b * a.S * a.ld_kv + kvh * a.d;
  const float* V = reinterpret_cast<const float*>(a.v) + (int64_t)b * a.S * a.ld_kv + kvh * a.d;
  for (int i = lane; i < a.d; i += 32) {
    qs[i] = Q[i];
    os[i] = dO[i];
  }
  __syncwarp();
  const int n_keys = a.causal ? qi + 1 : a.S;
  const float scale = rsqrtf((float)a.d);
  float mx, sum;
  row_probs(qs, K, a.ld_kv, a.d, n_keys, scale, sc, mx, sum);
  const float delta = a.delta[((int64_t)b * a.nq + h) * a.S + qi];
  for (int j = lane; j < n_keys; j += 32) {
    const float p = sc[j] / sum;
    const float dp = dot_rows(os, V + (int64_t)j * a.ld_kv, a.d);
    sc[j] = p * (dp - delta);
  }
  __syncwarp();
  float* dQ = reinterpret_cast<float*>(a.dq) + tok * a.ld_dq + h * a.d;
  for (int c = lane; c < a.d; c += 32) {
    float s = 0.0f;
    for (int j = 0; j < n_keys; ++j) s = fmaf(sc[j], K[(int64_t)j * a.ld_kv + c], s);
    dQ[c] = s * scale;
  }
}

__global__ void attn_f32_dkdv_kernel(const AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kj = blockIdx.x * WPB + warp;
  const int kvh = blockIdx.y, b = blockIdx.z;
  if (kj >= a.S) return;
  const int rep = a.nq / a.nkv;
  const float scale = rsqrtf((float)a.d);
  const int64_t ktok = (int64_t)b * a.S + kj;
  const float* Kr = reinterpret_cast<const float*>(a.k) + ktok * a.ld_kv + kvh * a.d;
  const float* Vr = reinterpret_cast<const float*>(a.v) + ktok * a.ld_kv + kvh * a.d;
  constexpr int PL = MAXD / 32;
  float kr[PL], vr[PL], dk[PL], dv[PL];
#pragma unroll
  for (int u = 0; u < PL; ++u) {
    const int c = lane + 32 * u;
    kr[u] = c < a.d ? Kr[c] : 0.0f;
    vr[u] = c < a.d ? Vr[c] : 0.0f;
    dk[u] = dv[u] = 0.0f;
  }
  for (int hh = 0; hh < rep; ++hh) {
    const int h = kvh * rep + hh;
    const int64_t lrow = ((int64_t)b * a.nq + h) * a.S;
    for (int qi = a.causal ? kj : 0; qi < a.S; ++qi) {
      const int64_t tok = (int64_t)b * a.S + qi;
      const float* Q = reinterpret_cast<const float*>(a.q) + tok * a.ld_q + h * a.d;
      const float* dO = reinterpret_cast<const float*>(a.dout) + tok * a.ld_do + h * a.d;
      float qv[PL], ov[PL], s = 0.0f, dp = 0.0f;
#pragma unroll
      for (int u = 0; u < PL; ++u) {
        const int c = lane + 32 * u;
        qv[u] = c < a.d ? Q[c] : 0.0f;
        ov[u] = c < a.d ? dO[c] : 0.0f;
        s = fmaf(qv[u], kr[u], s);
        dp = fmaf(ov[u], vr[u], dp);
      }
      s = warp_sum(s);
      dp = warp_sum(dp);
      const float p = expf(s * scale - a.lse[lrow + qi]);
      const float ds = p * (dp - a.delta[lrow + qi]);
#pragma unroll
      for (int u = 0; u < PL; ++u) {
        dv[u] = fmaf(p, ov[u], dv[u]);
        dk[u] = fmaf(ds, qv[u], dk[u]);
      }
    }
  }
  float* dK = reinterpret_cast<float*>(a.dk) + ktok * a.ld_dkv + kvh * a.d;
  float* dV = reinterpret_cast<float*>(a.dv) + ktok * a.ld_dkv + kvh * a.d;
#pragma unroll
  for (int u = 0; u < PL; ++u) {
    const int c = lane + 32 * u;
    if (c < a.d) {
      dK[c] = dk[u] * scale;
      dV[c] = dv[u];
    }
  }
}

}  // namespace

mgb_status attention_f32_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.S > 2048 || a.d > MAXD) return MGB_ERR_UNSUPPORTED;
  const int smem = (WPB * a.S + WPB * a.d) * 4;
  if (cudaFuncSetAttribute(attn_f32_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 grid((a.S + WPB - 1) / WPB, a.nq, a.B);
  attn_f32_fwd_kernel<<<grid, 32 * WPB, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status attention_f32_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.S > 2048 || a.d > MAXD) return MGB_ERR_UNSUPPORTED;
  const int warps = a.B * a.S * a.nq;
  attn_f32_delta_kernel<<<(warps + 7) / 8, 256, 0, st>>>(a);
  const int smem = (WPB * a.S + WPB * 2 * a.d) * 4;
  if (cudaFuncSetAttribute(attn_f32_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 g1((a.S + WPB - 1) / WPB, a.nq, a.B);
  attn_f32_dq_kernel<<<g1, 32 * WPB, smem, st>>>(a);
  dim3 g2((a.S + WPB - 1) / WPB, a.nkv, a.B);
  attn_f32_dkdv_kernel<<<g2, 32 * WPB, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

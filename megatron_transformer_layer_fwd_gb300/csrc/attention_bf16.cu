// bf16 attention backward: the per-query pre-pass and the launch sequence.
//
// delta_i = sum_d dO_i,d * O_i,d per query row and head (the rowsum that turns
// dP into dS = P (dP - delta) without forming P^T dP; it equals
// sum_j P_ij dP_ij because O = P V). Eight lanes per (batch, head, position),
// float32 sum of bf16 products. The pass also stores LSE * log2(e) next to it:
// two planes [B * nq][pad] with rows padded to a multiple of 128 positions
// (+inf and 0 in the padding, where P must vanish), so the tensor-core kernels
// (attention_tc_bwd.cu) fetch any query tile's values as one aligned block.
#include "common.cuh"
#include "internal.h"

namespace mgb {

mgb_status attention_tc_bwd_main(const AttnArgs& a, cudaStream_t st, cudaStream_t st_dq);

namespace {

// acc (the one-pass backward's float32 dQ accumulator [B*S][nq*128], or
// null): each slot of a real position also zeroes its head's 128 floats.
template <int D>
__global__ void attn_delta_kernel(const AttnArgs a, int pad, float* acc) {
  // 8 lanes per (batch, head, position) slot, positions fastest (the planes'
  // order), each lane a 16-byte vector of O and dO per 64 head dims
  constexpr int NV = D / 64;
  const int64_t g = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 3;
  const int sub = threadIdx.x & 7;
  if (g >= (int64_t)a.B * a.nq * pad) return;  // whole 8-lane groups leave together
  const int si = (int)(g % pad);
  const int64_t bh = g / pad;
  const int h = (int)(bh % a.nq), b = (int)(bh / a.nq);
  float* lse2 = a.delta;
  float* dl = a.delta + (size_t)a.B * a.nq * pad;
  if (si >= a.S) {
    if (sub == 0) {
      lse2[g] = INFINITY;
      dl[g] = 0.0f;
    }
    return;
  }
  const int64_t tok = (int64_t)b * a.S + si;
  if (acc != nullptr) {
    float4* z = reinterpret_cast<float4*>(acc + (tok * a.nq + h) * 128 + sub * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const bf16* O = reinterpret_cast<const bf16*>(a.o) + tok * a.ld_o + h * D;
  const bf16* dO = reinterpret_cast<const bf16*>(a.dout) + tok * a.ld_do + h * D;
  uint4 x[NV], y[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    x[v] = *reinterpret_cast<const uint4*>(O + (sub + 8 * v) * 8);
    y[v] = *reinterpret_cast<const uint4*>(dO + (sub + 8 * v) * 8);
  }
  float s = 0.0f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint32_t xs[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
    const uint32_t ys[4] = {y[v].x, y[v].y, y[v].z, y[v].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 p = unpack_bf16x2(xs[k]), q = unpack_bf16x2(ys[k]);
      s += p.x * q.x + p.y * q.y;
    }
  }
  const unsigned mask = 0xFFu << (threadIdx.x & 24);  // this 8-lane group
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) s += __shfl_xor_sync(mask, s, off);
  if (sub == 0) {
    dl[g] = s;
    lse2[g] = a.lse[bh * a.S + si] * 1.4426950408889634f;
  }
}

}  // namespace

mgb_status attention_bf16_bwd(const AttnArgs& a, cudaStream_t st) {
  const int pad = attn_bwd_row_pad(a.S);
  const int64_t slots = (int64_t)a.B * pad * a.nq;  // 8 threads each
  const int blocks = (int)((slots * 8 + 255) / 256);
  const bool one_pass = attention_bwd_fused_ok(a);
  // the one-pass backward's dQ accumulator follows the two planes
  float* acc = one_pass ? a.delta + 2 * (size_t)a.B * a.nq * pad : nullptr;
  if (a.d == 64)
    attn_delta_kernel<64><<<blocks, 256, 0, st>>>(a, pad, nullptr);
  else if (a.d == 128)
    attn_delta_kernel<128><<<blocks, 256, 0, st>>>(a, pad, acc);
  else
    return MGB_ERR_UNSUPPORTED;
  if (cudaGetLastError() != cudaSuccess) return MGB_ERR_CUDA;
  if (one_pass) return attention_tc_bwd_fused(a, st);
  // two kernels: dK/dV and dQ are independent, dQ on a side stream, so each
  // fills the SMs the other leaves idle in its last wave
  SideLane lane(st, nullptr, 1);
  const mgb_status f = lane.fork();
  if (f != MGB_OK) return f;
  const mgb_status r = attention_tc_bwd_main(a, st, lane.side());
  const mgb_status j = lane.join();
  return r != MGB_OK ? r : j;
}

}  // namespace mgb

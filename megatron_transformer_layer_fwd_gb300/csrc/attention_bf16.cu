// bf16 attention backward: the per-query pre-pass and the launch sequence.
//
// delta_i = sum_d dO_i,d * O_i,d per query row and head (the rowsum that turns
// dP into dS = P (dP - delta) without forming P^T dP; it equals
// sum_j P_ij dP_ij because O = P V). One warp per (batch, position, head),
// float32 sum of bf16 products. The pass also stores LSE * log2(e) next to it:
// two planes [B * nq][pad] with rows padded to a multiple of 128 positions
// (+inf and 0 in the padding, where P must vanish), so the tensor-core kernels
// (attention_tc_bwd.cu) fetch any query tile's values as one aligned block.
#include "common.cuh"
#include "internal.h"

namespace mgb {

mgb_status attention_tc_bwd_main(const AttnArgs& a, cudaStream_t st, cudaStream_t st_dq);

namespace {

template <int D>
__global__ void attn_delta_kernel(const AttnArgs a, int pad) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  // warp -> (b, s, h), h fastest: neighbouring warps read one token's heads
  if (warp >= a.B * pad * a.nq) return;
  const int h = warp % a.nq, bs = warp / a.nq;
  const int si = bs % pad, b = bs / pad;
  float* lse2 = a.delta;
  float* dl = a.delta + (size_t)a.B * a.nq * pad;
  const int64_t o = ((int64_t)b * a.nq + h) * pad + si;
  if (si >= a.S) {
    if (lane == 0) {
      lse2[o] = INFINITY;
      dl[o] = 0.0f;
    }
    return;
  }
  const int64_t tok = (int64_t)b * a.S + si;
  const bf16* O = reinterpret_cast<const bf16*>(a.o) + tok * a.ld_o + h * D;
  const bf16* dO = reinterpret_cast<const bf16*>(a.dout) + tok * a.ld_do + h * D;
  float s = 0.0f;
  for (int i = lane * 2; i < D; i += 64) {
    const float2 x = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(O + i));
    const float2 y = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(dO + i));
    s += x.x * y.x + x.y * y.y;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    dl[o] = s;
    lse2[o] = a.lse[((int64_t)b * a.nq + h) * a.S + si] * 1.4426950408889634f;
  }
}

}  // namespace

mgb_status attention_bf16_bwd(const AttnArgs& a, cudaStream_t st) {
  const int pad = attn_bwd_row_pad(a.S);
  const int warps = a.B * pad * a.nq;
  if (a.d == 64)
    attn_delta_kernel<64><<<(warps + 7) / 8, 256, 0, st>>>(a, pad);
  else if (a.d == 128)
    attn_delta_kernel<128><<<(warps + 7) / 8, 256, 0, st>>>(a, pad);
  else
    return MGB_ERR_UNSUPPORTED;
  if (cudaGetLastError() != cudaSuccess) return MGB_ERR_CUDA;
  // the dK/dV and dQ kernels are independent: dQ on a side stream, so each
  // fills the SMs the other leaves idle in its last wave
  SideLane lane(st, nullptr, 1);
  const mgb_status f = lane.fork();
  if (f != MGB_OK) return f;
  const mgb_status r = attention_tc_bwd_main(a, st, lane.side());
  const mgb_status j = lane.join();
  return r != MGB_OK ? r : j;
}

}  // namespace mgb

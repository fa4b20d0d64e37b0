// bf16 attention backward: the delta pre-pass and the launch sequence.
//
// delta_i = sum_d dO_i,d * O_i,d per query row and head (the rowsum that turns
// dP into dS = P (dP - delta) without forming P^T dP; it equals
// sum_j P_ij dP_ij because O = P V). One warp per (token, head), float32 sum of
// bf16 products. The matrix products of the backward run on the tensor cores
// (attention_tc_bwd.cu).
#include "common.cuh"
#include "internal.h"

namespace mgb {

mgb_status attention_tc_bwd_main(const AttnArgs& a, cudaStream_t st);

namespace {

template <int D>
__global__ void attn_delta_kernel(const AttnArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.B * a.S;
  if (warp >= T * a.nq) return;
  const int tok = warp / a.nq, h = warp % a.nq;
  const bf16* O = reinterpret_cast<const bf16*>(a.o) + (int64_t)tok * a.ld_o + h * D;
  const bf16* dO = reinterpret_cast<const bf16*>(a.dout) + (int64_t)tok * a.ld_do + h * D;
  float s = 0.0f;
  for (int i = lane * 2; i < D; i += 64) {
    const float2 x = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(O + i));
    const float2 y = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(dO + i));
    s += x.x * y.x + x.y * y.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    const int b = tok / a.S, si = tok % a.S;
    a.delta[((int64_t)b * a.nq + h) * a.S + si] = s;
  }
}

}  // namespace

mgb_status attention_bf16_bwd(const AttnArgs& a, cudaStream_t st) {
  const int warps = a.B * a.S * a.nq;
  if (a.d == 64)
    attn_delta_kernel<64><<<(warps + 7) / 8, 256, 0, st>>>(a);
  else if (a.d == 128)
    attn_delta_kernel<128><<<(warps + 7) / 8, 256, 0, st>>>(a);
  else
    return MGB_ERR_UNSUPPORTED;
  if (cudaGetLastError() != cudaSuccess) return MGB_ERR_CUDA;
  return attention_tc_bwd_main(a, st);
}

}  // namespace mgb

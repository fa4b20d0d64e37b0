// bf16 attention forward on the 5th-generation tensor cores (tcgen05).
//
// Definition ("LLM Lab 06: build a Megatron-style Transformer Block from
// scratch", section 2; "02 - How a whole Transformer block is split",
// section 2): O_h = softmax(Q_h K_g^T / sqrt(d)) V_g per batch and query head h,
// g = h / (nq / nkv), optional causal mask; LSE = log sum_j exp(s_j) is saved
// for the backward. FlashAttention-style (page 1, section 5): the [S, S] score
// matrix never leaves the chip.
//
// One CTA = 128 query rows of one (batch, head); 4 warps, thread t owns query
// row t (= TMEM lane t). KV tiles of 64 keys are loaded by TMA (128-byte
// swizzle): K double-buffered (it feeds the next score product early), V
// single-buffered (it is needed only after the softmax). Per KV tile j:
//   S   = Q K^T      tcgen05.mma M=128 N=64 K=d   -> TMEM columns [0, 64)
//   softmax          tcgen05.ld the row; running max m and sum l (log2
//                    domain); P = exp2(s - m) rounded to bf16 into a K-major
//                    swizzled smem tile, the A operand of the next product
//   O_j = P V        tcgen05.mma M=128 N=d K=64   -> TMEM columns [COL_PV, +d)
//   O   = O * exp2(m_old - m_new) + O_j            float32 registers
// Thread 0 issues the copies and the MMAs; S_{j+1} is issued as soon as every
// thread has read S_j, so it runs during the PV product and the accumulation.
// About 97 KB of smem and 256 TMEM columns per CTA: two CTAs share an SM and
// one CTA's softmax overlaps the other's MMAs. Q and K are K-major operands;
// the same V tile bytes are read as an MN-major operand (d contiguous).
// Every wait is bounded; a wait that runs out sets a shared abort flag that
// all threads read only right after a CTA barrier.
#include "common.cuh"
#include "internal.h"

namespace mgb {

CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int TQ = 128;  // query rows per CTA (TMEM lanes)
constexpr int TK = 64;   // keys per KV tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int KB = D / 64;              // 64-wide d blocks
  static constexpr int Q_BYTES = TQ * D * 2;     // KB boxes of [128 rows][64]
  static constexpr int KV_BYTES = TK * D * 2;    // KB boxes of [64 keys][64]
  static constexpr int P_BYTES = TQ * TK * 2;    // [128][64] K-major
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;  // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_P = OFF_V + KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 128 + 1024;  // barriers + alignment slack
  static constexpr int TMEM_COLS = D == 128 ? 256 : 128;
  static constexpr int COL_PV = D == 128 ? 128 : 64;
};

struct FwdParams {
  int B, S, nq, nkv, causal;
  bf16* o;
  int64_t ld_o;
  float* lse;
  int* err;
  float sl2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int D>
__global__ void __launch_bounds__(128, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V, sP = sb + C::OFF_P;
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t q_full = bar, k_full0 = bar + 8, k_empty0 = bar + 24, v_full = bar + 40,
                 v_empty = bar + 48, s_full = bar + 56, pv_full = bar + 64;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 72);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 76);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int nqt = (p.S + TQ - 1) / TQ;
  // grid: x = (head, batch) pairs, y = query tile from the last (longest causal
  // rows) to the first, so the heaviest tiles of every head start first
  const int qt = nqt - 1 - (int)blockIdx.y;
  const int h = blockIdx.x % p.nq, b = blockIdx.x / p.nq;
  const int g = h / (p.nq / p.nkv);
  const int q0 = qt * TQ;
  const int row = q0 + tid;  // this thread's query position in the sequence
  const int kv_end = p.causal ? min(p.S, q0 + TQ) : p.S;
  const int nkt = (kv_end + TK - 1) / TK;
  const int grow0 = b * p.S;  // first token row of this batch

  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    const uint32_t bars[] = {q_full, k_full0, k_full0 + 8, k_empty0, k_empty0 + 8,
                             v_full, v_empty, s_full, pv_full};
    for (uint32_t bb : bars) mbar_init(bb, 1);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem, t_pv = tmem + C::COL_PV;

  auto load_k = [&](int j) {
    const uint32_t fb = k_full0 + 8 * (j & 1);
    mbar_arrive_expect_tx(fb, C::KV_BYTES);
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_2d(sK + (j & 1) * C::KV_BYTES + kb * 8192, &tmK, g * D + kb * 64, grow0 + j * TK, fb);
  };
  auto load_v = [&](int j) {
    mbar_arrive_expect_tx(v_full, C::KV_BYTES);
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_2d(sV + kb * 8192, &tmV, g * D + kb * 64, grow0 + j * TK, v_full);
  };
  constexpr uint32_t idesc_s = idesc_bf16_f32(TQ, TK, 0, 0);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(TQ, D, 0, 1);
  auto issue_s = [&](int j) {
    const uint32_t kbase = sK + (j & 1) * C::KV_BYTES;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk & 3) * 32;  // K offset inside a 64-wide d block
      const uint64_t ad = smem_desc_sw128(sQ + (kk >> 2) * (TQ * 128) + off, 16, 1024);
      const uint64_t bd = smem_desc_sw128(kbase + (kk >> 2) * 8192 + off, 16, 1024);
      tc_mma_f16(t_s, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
    }
    tc_commit(s_full);
    tc_commit(k_empty0 + 8 * (j & 1));
  };
  auto issue_pv = [&]() {
#pragma unroll
    for (int kk = 0; kk < TK / 16; ++kk) {
      const uint64_t ad = smem_desc_sw128(sP + kk * 32, 16, 1024);
      const uint64_t bd = smem_desc_sw128(sV + kk * 2048, 8192, 1024);
      tc_mma_f16(t_pv, ad, bd, idesc_pv, kk > 0 ? 1u : 0u);
    }
    tc_commit(pv_full);
    tc_commit(v_empty);
  };

  if (tid == 0) {
    mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_2d(sQ + kb * (TQ * 128), &tmQ, h * D + kb * 64, grow0 + q0, q_full);
    load_k(0);
    load_v(0);
    if (nkt > 1) load_k(1);
    if (mbar_wait(q_full, 0, p.err) && mbar_wait(k_full0, 0, p.err)) {
      tc_fence_after();
      issue_s(0);
    } else {
      *abort = 1;
    }
  }
  __syncthreads();

  float o[D];
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  uint8_t* prow = smem + C::OFF_P + tid * 128;  // this row of P (128 bytes)

  for (int j = 0; j < nkt && !*abort; ++j) {
    // ---- S_j -> registers
    if (!mbar_wait(s_full, j & 1, p.err)) *abort = 1;
    tc_fence_after();
    float s[TK];
    {
      uint32_t r[32];
      tmem_ld32(t_s + lane_base, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
      tmem_ld32(t_s + lane_base + 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(r[i]);
    }
    // ---- online softmax of this row (log2 domain)
    const int kv0 = j * TK;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < TK; ++i) {
      const int kv = kv0 + i;
      const bool masked = kv >= p.S || (p.causal && kv > row);
      s[i] = masked ? -INFINITY : s[i] * p.sl2;
      mx = fmaxf(mx, s[i]);
    }
    const float m_new = fmaxf(m_run, mx);
    const float ref = m_new == -INFINITY ? 0.0f : m_new;
    const float alpha = exp2f(m_run - ref);
    m_run = m_new;
    float rs = 0.0f;
#pragma unroll
    for (int c = 0; c < TK / 8; ++c) {
      float e[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        e[i] = exp2f(s[8 * c + i] - ref);
        rs += e[i];
      }
      uint4 v;
      v.x = pack_bf16x2(e[0], e[1]);
      v.y = pack_bf16x2(e[2], e[3]);
      v.z = pack_bf16x2(e[4], e[5]);
      v.w = pack_bf16x2(e[6], e[7]);
      // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7)
      *reinterpret_cast<uint4*>(prow + ((c ^ (tid & 7)) << 4)) = v;
    }
    l_run = l_run * alpha + rs;
    // P writes (generic proxy) must be visible to the tensor core (async proxy)
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (*abort) break;
    if (tid == 0) {
      tc_fence_after();
      if (mbar_wait(v_full, j & 1, p.err)) {
        issue_pv();
        if (j + 1 < nkt) {
          // every thread read S_j before the barrier above: S may be rewritten
          if (mbar_wait(k_full0 + 8 * ((j + 1) & 1), ((j + 1) >> 1) & 1, p.err)) issue_s(j + 1);
          else *abort = 1;
        }
        if (j + 2 < nkt) {
          // K stage (j & 1) is free once S_j completed
          if (mbar_wait(k_empty0 + 8 * (j & 1), (j >> 1) & 1, p.err)) load_k(j + 2);
          else *abort = 1;
        }
      } else {
        *abort = 1;
      }
    }
    __syncwarp();
    // ---- O = O * alpha + P V_j
    const bool pv_ok = !*abort && mbar_wait(pv_full, j & 1, p.err);
    if (!pv_ok) *abort = 1;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(t_pv + lane_base + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) o[c * 32 + i] = fmaf(o[c * 32 + i], alpha, __uint_as_float(r[i]));
    }
    // V is free once PV_j completed: load V_{j+1}
    if (tid == 0 && pv_ok && j + 1 < nkt) {
      if (mbar_wait(v_empty, j & 1, p.err)) load_v(j + 1);
      else *abort = 1;
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();  // TMEM PV columns and the P tile are reused next iteration
    tc_fence_after();
  }

  const bool ok = !*abort;
  if (!ok && tid == 0) {
    // give tensor-core work and copies still in flight time to finish (bounded)
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  // ---- epilogue: normalise, store O (bf16) and LSE
  if (ok && row < p.S) {
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    bf16* out = p.o + (int64_t)(grow0 + row) * p.ld_o + h * D;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v;
      v.x = pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv);
      v.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
      v.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
      v.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
      *reinterpret_cast<uint4*>(out + 8 * c) = v;
    }
    p.lse[((int64_t)b * p.nq + h) * p.S + row] = (m_run + log2f(l_run)) * LN2;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
mgb_status fwd_tc_d(const AttnArgs& a, cudaStream_t st) {
  using C = FwdCfg<D>;
  const uint64_t T = (uint64_t)a.B * a.S;
  CUtensorMap tq, tk, tv;
  if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TQ) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TK) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TK) != CUDA_SUCCESS)
    return MGB_ERR_CUDA;
  FwdParams p{};
  p.B = a.B; p.S = a.S; p.nq = a.nq; p.nkv = a.nkv; p.causal = a.causal;
  p.o = reinterpret_cast<bf16*>(a.o); p.ld_o = a.ld_o; p.lse = a.lse;
  p.err = device_error_word();
  p.sl2 = LOG2E / sqrtf((float)D);
  auto k = attn_fwd_tc_kernel<D>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 grid(a.nq * a.B, (a.S + TQ - 1) / TQ);
  k<<<grid, 128, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

mgb_status attention_tc_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.d == 64) return fwd_tc_d<64>(a, st);
  if (a.d == 128) return fwd_tc_d<128>(a, st);
  return MGB_ERR_UNSUPPORTED;
}

}  // namespace mgb

// bf16 attention backward on the 5th-generation tensor cores (tcgen05).
//
// From the saved LSE ("02 - How a whole Transformer block is split",
// section 2 defines the forward; page 1, section 2 asks for the end-to-end
// backward): with s = q.k / sqrt(d), P = exp(s - LSE) recomputed, dP = dO V^T,
// delta = rowsum(dO * O) (precomputed), dS = P * (dP - delta):
//   dV_g = sum_h P^T dO_h,   dK_g = sum_h dS^T Q_h / sqrt(d),   dQ_h = dS K_g / sqrt(d),
// summing over the query heads h of the GQA group g.
//
// Kernel A (dK, dV): one CTA = 128 keys of one KV head (key row = TMEM lane).
// It loops over every query head of the group and every 64-query tile that
// can see its keys (Q/dO tiles in a 3-stage TMA ring):
//   S^T  = K Q^T     M=128 N=64 K=d     TMEM buffer i & 1, columns [0, 64)
//   dP^T = V dO^T    M=128 N=64 K=d     TMEM buffer i & 1, columns [64, 128)
//   registers: P^T = exp2(S^T*log2e/sqrt(d) - LSE*log2e), dS^T = P^T (dP^T - delta)
//   (bf16, K-major 128-byte-swizzled smem tiles)
//   dV  += P^T dO    M=128 N=d K=64     TMEM [256, 256+d)
//   dK  += dS^T Q    M=128 N=d K=64     TMEM [256+d, 256+2d)
// The Q and dO tiles are read as K-major operands by the first two products and
// as MN-major operands (d contiguous) by the last two: the same smem bytes.
// dK and dV stay in TMEM across the whole loop, so the GQA sum costs nothing.
//
// Kernel B (dQ): one CTA = 128 queries of one head; per 64-key tile (K/V in a
// 3-stage ring): S = Q K^T, dP = dO V^T (TMEM buffer i & 1), dS in registers
// -> smem, dQ += dS K (TMEM [256, 256+d); the K tile read as MN-major).
//
// Warp-specialised, 10 warps:
//   warps 0-7  compute: warps w and w+4 share TMEM lane quarter w%4 (32 rows)
//              and take one 32-column half of each 64-column tile
//   warp 8     producer: TMA ring refills (and, in kernel A, the per-query LSE
//              and delta of each tile into a double-buffered smem slot)
//   warp 9     MMA issuer (one lane)
// No CTA barrier inside the loop: the roles hand tiles to each other through
// mbarriers only. The score products of a tile are double-buffered in TMEM and
// issued two tiles ahead, so the compute warps find them ready. Every wait is
// bounded; a wait that runs out sets a shared abort flag and every role leaves
// its loop (warp-uniformly) before the single closing barrier.
#include "common.cuh"
#include "internal.h"

namespace mgb {

CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int TR = 128;        // rows (keys in A, queries in B) per CTA
constexpr int TC = 64;         // columns per inner tile (queries in A, keys in B)
constexpr int NS = 3;          // stages of the streamed operand ring
constexpr int COL_ACC = 256;   // first TMEM column of the accumulators
constexpr int NCOMPUTE = 256;  // compute threads (warps 0-7)
constexpr int NTHREADS = 320;  // + producer warp + MMA warp

struct BwdParams {
  int B, S, nq, nkv, causal;
  const float* lse;    // [B, nq, S]
  const float* delta;  // [B, nq, S]
  bf16 *d0, *d1;       // A: dk, dv; B: dq
  int64_t ld_out;
  int* err;
  float sl2, scale;
};

// ------------------------------------------------------------ kernel A: dK, dV
template <int D>
struct DkvCfg {
  static constexpr int KB = D / 64;
  static constexpr int KV_BYTES = TR * D * 2;   // K or V rows of this CTA
  static constexpr int QT_BYTES = TC * D * 2;   // one Q or dO tile
  static constexpr int PT_BYTES = TR * TC * 2;  // P^T or dS^T tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;         // NS stages
  static constexpr int OFF_DO = OFF_Q + NS * QT_BYTES;   // NS stages
  static constexpr int OFF_P = OFF_DO + NS * QT_BYTES;
  static constexpr int OFF_DS = OFF_P + PT_BYTES;
  static constexpr int OFF_LD = OFF_DS + PT_BYTES;       // [2][lse2 64 | delta 64] f32
  static constexpr int OFF_BAR = OFF_LD + 2 * 2 * TC * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int COL_DV = COL_ACC, COL_DK = COL_ACC + D;
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO, const BwdParams p) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V, sQ = sb + C::OFF_Q, sO = sb + C::OFF_DO,
                 sP = sb + C::OFF_P, sS = sb + C::OFF_DS;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t kv_full = bar;                // K, V loaded            (tx)
  const uint32_t qd_full0 = bar + 8;           // [3] Q/dO stage loaded (tx)
  const uint32_t qd_empty0 = bar + 32;         // [3] stage read by dV/dK (commit)
  const uint32_t sp_full0 = bar + 56;          // [2] S^T/dP^T ready   (commit)
  const uint32_t pds_full = bar + 72;          // P^T/dS^T written      (256 arrivals)
  const uint32_t pds_empty = bar + 80;         // dV/dK read them       (commit)
  const uint32_t ld_full0 = bar + 88;          // [2] LSE/delta slot written (32)
  const uint32_t ld_empty0 = bar + 104;        // [2] slot read          (256)
  const uint32_t acc_done = bar + 120;         // all products done     (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 128);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 132);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: x = (KV head, batch) pairs, y = key tile (the first key tiles see the
  // most causal queries, so they start first)
  const int kt = blockIdx.y, g = blockIdx.x % p.nkv, b = blockIdx.x / p.nkv;
  const int rep = p.nq / p.nkv;
  const int kv0 = kt * TR;
  const int nqt = (p.S + TC - 1) / TC;
  const int qt_start = p.causal ? kv0 / TC : 0;
  const int per_head = nqt - qt_start;
  const int n_it = per_head * rep;  // >= 1: the query tile at kv0 sees key kv0
  const int grow0 = b * p.S;
  auto it_head = [&](int it) { return g * rep + it / per_head; };
  auto it_q0 = [&](int it) { return (qt_start + it % per_head) * TC; };

  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
    for (int i = 0; i < 9; ++i) mbar_init(bar + 8 * i, 1);  // kv, qd_full, qd_empty, sp_full
    mbar_init(pds_full, NCOMPUTE);
    mbar_init(pds_empty, 1);
    mbar_init(ld_full0, 32);
    mbar_init(ld_full0 + 8, 32);
    mbar_init(ld_empty0, NCOMPUTE);
    mbar_init(ld_empty0 + 8, NCOMPUTE);
    mbar_init(acc_done, 1);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_2d(sK + kb * (TR * 128), &tmK, g * D + kb * 64, grow0 + kv0, kv_full);
        tma_load_2d(sV + kb * (TR * 128), &tmV, g * D + kb * 64, grow0 + kv0, kv_full);
      }
    }
    for (int it = 0; it < n_it; ++it) {
      if (warp_aborted(abort)) break;
      // Q/dO of tile it into stage it % 3 once dV/dK of tile it - 3 read it
      if (lane == 0) {
        const int s = it % NS;
        if (it >= NS && !mbar_wait(qd_empty0 + 8 * s, ((it - NS) / NS) & 1, p.err)) *abort = 1;
        if (!*abort) {
          const uint32_t fb = qd_full0 + 8 * s;
          const int h = it_head(it), q0 = it_q0(it);
          mbar_arrive_expect_tx(fb, 2 * C::QT_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_2d(sQ + s * C::QT_BYTES + kb * 8192, &tmQ, h * D + kb * 64, grow0 + q0, fb);
            tma_load_2d(sO + s * C::QT_BYTES + kb * 8192, &tmO, h * D + kb * 64, grow0 + q0, fb);
          }
        }
      }
      __syncwarp();
      // per-query LSE (log2 units) and delta of tile it into slot it & 1
      if (it >= 2 && !warp_wait(ld_empty0 + 8 * (it & 1), ((it - 2) >> 1) & 1, p.err)) {
        *abort = 1;
        break;
      }
      const int h = it_head(it);
      float* dst = sLD + (it & 1) * 2 * TC;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u, q = it_q0(it) + c;
        const int64_t off = ((int64_t)b * p.nq + h) * p.S + q;
        dst[c] = q < p.S ? p.lse[off] * LOG2E : INFINITY;
        dst[TC + c] = q < p.S ? p.delta[off] : 0.0f;
      }
      mbar_arrive(ld_full0 + 8 * (it & 1));
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_sp = idesc_bf16_f32(TR, TC, 0, 0);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(TR, D, 0, 1);
      auto issue_sp = [&](int it) -> bool {
        const int s = it % NS;
        if (!mbar_wait(qd_full0 + 8 * s, (it / NS) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t tb = tmem + (it & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (TR * 128) + (kk & 3) * 32;
          const uint32_t offq = (kk >> 2) * 8192 + (kk & 3) * 32;
          tc_mma_f16(tb, smem_desc_sw128(sK + off, 16, 1024),
                     smem_desc_sw128(sQ + s * C::QT_BYTES + offq, 16, 1024), idesc_sp, kk > 0);
          tc_mma_f16(tb + 64, smem_desc_sw128(sV + off, 16, 1024),
                     smem_desc_sw128(sO + s * C::QT_BYTES + offq, 16, 1024), idesc_sp, kk > 0);
        }
        tc_commit(sp_full0 + 8 * (it & 1));
        return true;
      };
      bool good = mbar_wait(kv_full, 0, p.err) && issue_sp(0) && (n_it < 2 || issue_sp(1));
      for (int it = 0; it < n_it && good && !*abort; ++it) {
        // P^T / dS^T of tile it written by every compute thread (which also
        // means every thread has read tile it's scores out of TMEM)
        if (!mbar_wait(pds_full, it & 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        const int s = it % NS;
#pragma unroll
        for (int kk = 0; kk < TC / 16; ++kk) {
          const uint32_t b_off = s * C::QT_BYTES + kk * 2048;
          tc_mma_f16(tmem + C::COL_DV, smem_desc_sw128(sP + kk * 32, 16, 1024),
                     smem_desc_sw128(sO + b_off, 8192, 1024), idesc_acc, (it > 0 || kk > 0));
          tc_mma_f16(tmem + C::COL_DK, smem_desc_sw128(sS + kk * 32, 16, 1024),
                     smem_desc_sw128(sQ + b_off, 8192, 1024), idesc_acc, (it > 0 || kk > 0));
        }
        tc_commit(qd_empty0 + 8 * s);
        tc_commit(pds_empty);
        if (it + 2 < n_it && !issue_sp(it + 2)) good = false;
      }
      if (good && !*abort) tc_commit(acc_done);
      else *abort = 1;
    }
  } else {
    // ---------------- compute warps 0-7
    const int rrow = (warp & 3) * 32 + lane, half = warp >> 2;
    const int kr = kv0 + rrow;  // this thread's key position
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t col0 = half * 32;  // this warp's columns of the 64-wide tiles
    bool good = true;
    for (int it = 0; it < n_it; ++it) {
      if (warp_aborted(abort) || !warp_wait(sp_full0 + 8 * (it & 1), (it >> 1) & 1, p.err) ||
          !warp_wait(ld_full0 + 8 * (it & 1), (it >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      float st[32], dp[32], L[32], Dl[32];
      const uint32_t tb = tmem + (it & 1) * 128;
      ld_cols32(tb + lane_base + col0, st);
      ld_cols32(tb + lane_base + 64 + col0, dp);
      const float* ldp = sLD + (it & 1) * 2 * TC + col0;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 a = *reinterpret_cast<const float4*>(ldp + c);
        const float4 d = *reinterpret_cast<const float4*>(ldp + TC + c);
        L[c] = a.x; L[c + 1] = a.y; L[c + 2] = a.z; L[c + 3] = a.w;
        Dl[c] = d.x; Dl[c + 1] = d.y; Dl[c + 2] = d.z; Dl[c + 3] = d.w;
      }
      mbar_arrive(ld_empty0 + 8 * (it & 1));
      // P^T and dS^T of this key row against its 32 queries of the tile
      const int q0 = it_q0(it) + col0;
      const bool full = q0 + 32 <= p.S && kv0 + TR <= p.S && (!p.causal || q0 >= kv0 + TR - 1);
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float pt = exp2f(fmaf(st[c], p.sl2, -L[c]));
          st[c] = pt;
          dp[c] = pt * (dp[c] - Dl[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int q = q0 + c;
          const bool vis = q < p.S && kr < p.S && !(p.causal && q < kr);
          const float pt = vis ? exp2f(fmaf(st[c], p.sl2, -L[c])) : 0.0f;
          st[c] = pt;
          dp[c] = pt * (dp[c] - Dl[c]);
        }
      }
      // the P / dS tiles were last read by dV/dK of tile it - 1
      if (it >= 1 && !warp_wait(pds_empty, (it - 1) & 1, p.err)) {
        good = false;
        break;
      }
      store_half_row_sw128(smem + C::OFF_P + rrow * 128, rrow, half, st);
      store_half_row_sw128(smem + C::OFF_DS + rrow * 128, rrow, half, dp);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(pds_full);
    }
    if (!good) *abort = 1;
    // ---- all products done: dK (scaled) and dV rows out of TMEM
    if (good && warp_wait(acc_done, 0, p.err) && !warp_aborted(abort)) {
      tc_fence_after();
      const bool row_ok = kr < p.S;
      const int64_t orow = (int64_t)(grow0 + kr) * p.ld_out + g * D;
      const int c0 = half * (D / 2);  // the two warps of a quarter split the d columns
      store_tmem_row<D / 2>(tmem + lane_base + C::COL_DK + c0, p.scale,
                            row_ok ? p.d0 + orow + c0 : nullptr);
      store_tmem_row<D / 2>(tmem + lane_base + C::COL_DV + c0, 1.0f,
                            row_ok ? p.d1 + orow + c0 : nullptr);
    } else {
      *abort = 1;
    }
  }
  __syncthreads();
  if (*abort && tid == 0) spin_10ms();  // let work and copies still in flight finish
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------- kernel B: dQ
template <int D>
struct DqCfg {
  static constexpr int KB = D / 64;
  static constexpr int QO_BYTES = TR * D * 2;  // Q or dO rows of this CTA
  static constexpr int KV_BYTES = TC * D * 2;  // one K or V tile
  static constexpr int DS_BYTES = TR * TC * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + QO_BYTES;
  static constexpr int OFF_K = OFF_DO + QO_BYTES;      // NS stages
  static constexpr int OFF_V = OFF_K + NS * KV_BYTES;  // NS stages
  static constexpr int OFF_DS = OFF_V + NS * KV_BYTES;
  static constexpr int OFF_BAR = OFF_DS + DS_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int COL_DQ = COL_ACC;
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmO, const BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sO = sb + C::OFF_DO, sK = sb + C::OFF_K, sV = sb + C::OFF_V,
                 sS = sb + C::OFF_DS;
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t qo_full = bar;          // Q, dO loaded              (tx)
  const uint32_t kv_full0 = bar + 8;     // [3] K/V stage loaded      (tx)
  const uint32_t kv_empty0 = bar + 32;   // [3] stage read by dQ      (commit)
  const uint32_t sp_full0 = bar + 56;    // [2] S/dP ready            (commit)
  const uint32_t ds_full = bar + 72;     // dS written                (256 arrivals)
  const uint32_t ds_empty = bar + 80;    // dQ read it                (commit)
  const uint32_t acc_done = bar + 88;    // all products done         (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 128);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 132);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqt = (p.S + TR - 1) / TR;
  const int qt = nqt - 1 - (int)blockIdx.y;  // longest causal rows first
  const int h = blockIdx.x % p.nq, b = blockIdx.x / p.nq;
  const int g = h / (p.nq / p.nkv);
  const int q0 = qt * TR;
  const int kv_end = p.causal ? min(p.S, q0 + TR) : p.S;
  const int nkt = (kv_end + TC - 1) / TC;
  const int grow0 = b * p.S;

  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
    for (int i = 0; i < 9; ++i) mbar_init(bar + 8 * i, 1);
    mbar_init(ds_full, NCOMPUTE);
    mbar_init(ds_empty, 1);
    mbar_init(acc_done, 1);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(qo_full, 2 * C::QO_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_2d(sQ + kb * (TR * 128), &tmQ, h * D + kb * 64, grow0 + q0, qo_full);
        tma_load_2d(sO + kb * (TR * 128), &tmO, h * D + kb * 64, grow0 + q0, qo_full);
      }
      for (int j = 0; j < nkt && !*abort; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(kv_empty0 + 8 * s, ((j - NS) / NS) & 1, p.err)) {
          *abort = 1;
          break;
        }
        const uint32_t fb = kv_full0 + 8 * s;
        mbar_arrive_expect_tx(fb, 2 * C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_2d(sK + s * C::KV_BYTES + kb * 8192, &tmK, g * D + kb * 64, grow0 + j * TC, fb);
          tma_load_2d(sV + s * C::KV_BYTES + kb * 8192, &tmV, g * D + kb * 64, grow0 + j * TC, fb);
        }
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_sp = idesc_bf16_f32(TR, TC, 0, 0);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(TR, D, 0, 1);
      auto issue_sp = [&](int j) -> bool {
        const int s = j % NS;
        if (!mbar_wait(kv_full0 + 8 * s, (j / NS) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t tb = tmem + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (TR * 128) + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * 8192 + (kk & 3) * 32;
          tc_mma_f16(tb, smem_desc_sw128(sQ + off, 16, 1024),
                     smem_desc_sw128(sK + s * C::KV_BYTES + offk, 16, 1024), idesc_sp, kk > 0);
          tc_mma_f16(tb + 64, smem_desc_sw128(sO + off, 16, 1024),
                     smem_desc_sw128(sV + s * C::KV_BYTES + offk, 16, 1024), idesc_sp, kk > 0);
        }
        tc_commit(sp_full0 + 8 * (j & 1));
        return true;
      };
      bool good = mbar_wait(qo_full, 0, p.err) && issue_sp(0) && (nkt < 2 || issue_sp(1));
      for (int j = 0; j < nkt && good && !*abort; ++j) {
        if (!mbar_wait(ds_full, j & 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        const int s = j % NS;
#pragma unroll
        for (int kk = 0; kk < TC / 16; ++kk)
          tc_mma_f16(tmem + C::COL_DQ, smem_desc_sw128(sS + kk * 32, 16, 1024),
                     smem_desc_sw128(sK + s * C::KV_BYTES + kk * 2048, 8192, 1024), idesc_acc,
                     (j > 0 || kk > 0));
        tc_commit(kv_empty0 + 8 * s);
        tc_commit(ds_empty);
        if (j + 2 < nkt && !issue_sp(j + 2)) good = false;
      }
      if (good && !*abort) tc_commit(acc_done);
      else *abort = 1;
    }
  } else {
    // ---------------- compute warps 0-7
    const int rrow = (warp & 3) * 32 + lane, half = warp >> 2;
    const int row = q0 + rrow;
    const int64_t lrow = ((int64_t)b * p.nq + h) * p.S;
    const float L2 = row < p.S ? p.lse[lrow + row] * LOG2E : INFINITY;
    const float Dr = row < p.S ? p.delta[lrow + row] : 0.0f;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t col0 = half * 32;
    bool good = true;
    for (int j = 0; j < nkt; ++j) {
      if (warp_aborted(abort) || !warp_wait(sp_full0 + 8 * (j & 1), (j >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      float sc[32], dp[32];
      const uint32_t tb = tmem + (j & 1) * 128;
      ld_cols32(tb + lane_base + col0, sc);
      ld_cols32(tb + lane_base + 64 + col0, dp);
      const int kv0 = j * TC + col0;  // first key of this thread's columns
      // mask-free when every query row of the CTA sees every key of the half-tile
      const bool full = kv0 + 32 <= p.S && (!p.causal || kv0 + 31 <= q0);
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) dp[c] = exp2f(fmaf(sc[c], p.sl2, -L2)) * (dp[c] - Dr);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int kv = kv0 + c;
          const bool vis = kv < p.S && !(p.causal && kv > row);
          const float pr = vis ? exp2f(fmaf(sc[c], p.sl2, -L2)) : 0.0f;
          dp[c] = pr * (dp[c] - Dr);
        }
      }
      if (j >= 1 && !warp_wait(ds_empty, (j - 1) & 1, p.err)) {
        good = false;
        break;
      }
      store_half_row_sw128(smem + C::OFF_DS + rrow * 128, rrow, half, dp);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (!good) *abort = 1;
    if (good && warp_wait(acc_done, 0, p.err) && !warp_aborted(abort)) {
      tc_fence_after();
      const bool row_ok = row < p.S;
      const int c0 = half * (D / 2);
      store_tmem_row<D / 2>(tmem + lane_base + C::COL_DQ + c0, p.scale,
                            row_ok ? p.d0 + (int64_t)(grow0 + row) * p.ld_out + h * D + c0
                                   : nullptr);
    } else {
      *abort = 1;
    }
  }
  __syncthreads();
  if (*abort && tid == 0) spin_10ms();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
mgb_status bwd_tc_d(const AttnArgs& a, cudaStream_t st) {
  const uint64_t T = (uint64_t)a.B * a.S;
  BwdParams p{};
  p.B = a.B; p.S = a.S; p.nq = a.nq; p.nkv = a.nkv; p.causal = a.causal;
  p.lse = a.lse; p.delta = a.delta;
  p.err = device_error_word();
  p.sl2 = LOG2E / sqrtf((float)D);
  p.scale = 1.0f / sqrtf((float)D);
  // kernel A: K/V rows of 128, Q/dO tiles of 64
  {
    using C = DkvCfg<D>;
    CUtensorMap tq, tk, tv, to;
    if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TC) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&to, a.dout, (uint64_t)a.nq * D, T, a.ld_do, 64, TC) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TR) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TR) != CUDA_SUCCESS)
      return MGB_ERR_CUDA;
    p.d0 = reinterpret_cast<bf16*>(a.dk);
    p.d1 = reinterpret_cast<bf16*>(a.dv);
    p.ld_out = a.ld_dkv;
    auto k = attn_bwd_dkdv_tc_kernel<D>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return MGB_ERR_CUDA;
    dim3 grid(a.nkv * a.B, (a.S + TR - 1) / TR);
    k<<<grid, NTHREADS, C::SMEM, st>>>(tq, tk, tv, to, p);
  }
  // kernel B: Q/dO rows of 128, K/V tiles of 64
  {
    using C = DqCfg<D>;
    CUtensorMap tq, tk, tv, to;
    if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TR) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&to, a.dout, (uint64_t)a.nq * D, T, a.ld_do, 64, TR) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TC) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TC) != CUDA_SUCCESS)
      return MGB_ERR_CUDA;
    p.d0 = reinterpret_cast<bf16*>(a.dq);
    p.d1 = nullptr;
    p.ld_out = a.ld_dq;
    auto k = attn_bwd_dq_tc_kernel<D>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return MGB_ERR_CUDA;
    dim3 grid(a.nq * a.B, (a.S + TR - 1) / TR);
    k<<<grid, NTHREADS, C::SMEM, st>>>(tq, tk, tv, to, p);
  }
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

mgb_status attention_tc_bwd_main(const AttnArgs& a, cudaStream_t st) {
  if (a.d == 64) return bwd_tc_d<64>(a, st);
  if (a.d == 128) return bwd_tc_d<128>(a, st);
  return MGB_ERR_UNSUPPORTED;
}

}  // namespace mgb

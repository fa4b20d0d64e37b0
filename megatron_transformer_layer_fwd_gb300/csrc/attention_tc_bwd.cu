// bf16 attention backward on the 5th-generation tensor cores (tcgen05).
//
// From the saved LSE ("02 - How a whole Transformer block is split",
// section 2 defines the forward; page 1, section 2 asks for the end-to-end
// backward): with s = q.k / sqrt(d), P = exp(s - LSE) recomputed, dP = dO V^T,
// delta = rowsum(dO * O) (precomputed), dS = P * (dP - delta):
//   dV_g = sum_h P^T dO_h,   dK_g = sum_h dS^T Q_h / sqrt(d),   dQ_h = dS K_g / sqrt(d),
// summing over the query heads h of the GQA group g.
//
// The per-query inputs come from a workspace the pre-pass fills: two planes
// [B * nq][s_pad] of float32, LSE * log2(e) (+inf past the sequence end) and
// delta (0 there), rows padded to a multiple of 128 so that any query tile is
// one aligned, in-bounds 16-byte-multiple block.
//
// Kernel A (dK, dV): one CTA = 128 keys of one KV head (key row = TMEM lane).
// It loops over every query head of the group and every 64-query tile that
// can see its keys (Q, dO and that tile's LSE/delta in a 4-stage TMA ring):
//   S^T  = K Q^T     M=128 N=64 K=d     TMEM columns [0, 64)
//   dP^T = V dO^T    M=128 N=64 K=d     TMEM columns [64, 128)
//   registers: P^T = exp2(S^T*log2e/sqrt(d) - LSE*log2e), dS^T = P^T (dP^T - delta)
//   as bf16 pairs into TMEM buffer i & 1 (columns [128, 256)), the A operands of
//   dV  += P^T dO    M=128 N=d K=64     TMEM [256, 256+d)
//   dK  += dS^T Q    M=128 N=d K=64     TMEM [256+d, 256+2d)
// The Q and dO tiles are read as K-major operands by the first two products and
// as MN-major operands (d contiguous) by the last two: the same smem bytes.
// dK and dV stay in TMEM across the whole loop, so the GQA sum costs nothing.
//
// Kernel B (dQ): one CTA = 128 queries of one head; per 64-key tile (K/V in a
// 5-stage ring): S = Q K^T, dP = dO V^T (TMEM [0, 128); Q and dO are copied once
// into TMEM [384, 512) and read from there, so the products read only K and V
// from shared memory), dS in registers -> TMEM buffer j & 1 (bf16 pairs,
// [128, 192)), dQ += dS K (TMEM [256, 256+d), A from TMEM, the K tile read as
// MN-major).
//
// Warp-specialised, 18 warps:
//   warps 0-15 compute, in two groups of 8 that take alternate tiles (group
//              g the tiles i with i & 1 == g): one group's exponentials and
//              stores overlap the other's. In a group, warps w and w+4 share
//              TMEM lane quarter w%4 (32 rows) and take one 32-column half of
//              each 64-column tile
//   warp 16    producer (one lane): TMA ring refills
//   warp 17    MMA issuer: the whole warp runs the loop (warp-uniform values)
//              and one elected lane issues each tcgen05 instruction from
//              shared-memory descriptors built once (base + offset / 16)
// The score products have one TMEM buffer: a group releases it as soon as it
// has loaded its tile's scores into registers, and the next tile's products
// are issued right then, so they run while the group computes. Products whose
// A operand is a tile of the compute warps read it from TMEM, which keeps
// those tiles out of shared memory (whose bandwidth the other operands and the
// TMA copies need) and leaves room for deep copy rings. No CTA barrier inside
// the loop: the roles hand tiles to each other through mbarriers only. Every
// wait is bounded; a wait that runs out sets a shared abort flag and every role
// leaves its loop (warp-uniformly) before the single closing barrier.
//
// Dropout on the probabilities (the DROP variants): the forward wrote one keep
// bit per (query, key). With keep mask M and scale s: dV uses P o M s, the
// gradient reaching P is dP o M s, and dS = P (dP o M s - delta) (delta =
// rowsum(dO o O) of the dropped output). Kernel A stages each tile's 64 x 128
// bits with its Q/dO stage (a TMA box of 4 words x 64 query rows); kernel B
// loads one word per 32 keys.
#include "common.cuh"
#include "internal.h"

namespace mgb {

CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer);
// 2-D uint32 tensor map without swizzle (gemm_tc.cu)
CUresult tmap_encode_u32_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                            int64_t ld, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int TR = 128;        // rows (keys in A, queries in B) per CTA
constexpr int TC = 64;         // columns per inner tile (queries in A, keys in B)
constexpr int NSA = 4;         // Q/dO ring stages (kernel A)
constexpr int NSB = 5;         // K/V ring stages (kernel B)
constexpr int COL_ACC = 256;   // first TMEM column of the accumulators
constexpr int NGROUP = 256;    // compute threads of one group (8 warps)
constexpr int NTHREADS = 576;  // 2 compute groups + producer warp + MMA warp
constexpr int W_PROD = 16, W_MMA = 17;

struct BwdParams {
  int B, S, nq, nkv, causal, s_pad;
  const uint32_t* dmask;  // keep bits [B*nq*S][mw] (DROP variants)
  int mw;
  float dscale;
  const float* lse2;   // [B * nq][s_pad]: LSE * log2(e)
  const float* delta;  // [B * nq][s_pad]
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
  static constexpr int LD_BYTES = 2 * TC * 4;   // a tile's LSE*log2e and delta
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;          // NSA stages
  static constexpr int OFF_DO = OFF_Q + NSA * QT_BYTES;   // NSA stages
  static constexpr int OFF_LD = OFF_DO + NSA * QT_BYTES;  // NSA stages
  static constexpr int M_BYTES = TC * 16;                 // a tile's keep bits: [64 queries][4 words]
  static constexpr int OFF_M = OFF_LD + NSA * LD_BYTES;   // NSA stages (DROP)
  static constexpr int OFF_BAR = OFF_M + NSA * M_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  // TMEM: scores [0, 128), P^T/dS^T buffers [128, 256) (64 columns each: P^T
  // then dS^T, 32 columns = 64 bf16 queries apiece), dV, dK
  static constexpr int COL_PDS = 128, COL_DV = COL_ACC, COL_DK = COL_ACC + D;
};

template <int D, bool DROP>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO,
                            const __grid_constant__ CUtensorMap tmM, const BwdParams p) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V, sQ = sb + C::OFF_Q, sO = sb + C::OFF_DO,
                 sLDa = sb + C::OFF_LD;
  const float* sLD = reinterpret_cast<const float*>(smem + C::OFF_LD);
  const uint32_t* sM = reinterpret_cast<const uint32_t*>(smem + C::OFF_M);
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t kv_full = bar;          // K, V loaded                       (tx)
  const uint32_t qd_full0 = bar + 8;     // [4] Q/dO/LSE/delta stage loaded   (tx)
  const uint32_t qd_empty0 = bar + 40;   // [4] stage read by dV/dK           (commit)
  const uint32_t sp_full0 = bar + 72;    // [2] S^T/dP^T of tile i ready      (commit)
  const uint32_t sp_free0 = bar + 88;    // [2] group read them out of TMEM   (256 arrivals)
  const uint32_t pds_full0 = bar + 104;  // [2] P^T/dS^T buffer written       (256 arrivals)
  const uint32_t pds_empty0 = bar + 120; // [2] dV/dK read the buffer         (commit)
  const uint32_t acc_done = bar + 136;   // all products done                 (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 160);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 164);

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

  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
    mbar_init(kv_full, 1);
    for (int i = 0; i < NSA; ++i) {
      mbar_init(qd_full0 + 8 * i, 1);
      mbar_init(qd_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sp_full0 + 8 * i, 1);
      mbar_init(sp_free0 + 8 * i, NGROUP);
      mbar_init(pds_full0 + 8 * i, NGROUP);
      mbar_init(pds_empty0 + 8 * i, 1);
    }
    mbar_init(acc_done, 1);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_PROD) {
    // ---------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_2d(sK + kb * (TR * 128), &tmK, g * D + kb * 64, grow0 + kv0, kv_full);
        tma_load_2d(sV + kb * (TR * 128), &tmV, g * D + kb * 64, grow0 + kv0, kv_full);
      }
      int h = g * rep, qt = qt_start;  // head and query tile of iteration it
      for (int it = 0; it < n_it && !*abort; ++it) {
        // Q/dO of tile it into stage it % NSA once dV/dK of the tile before read it
        const int s = it % NSA;
        if (it >= NSA && !mbar_wait(qd_empty0 + 8 * s, ((it - NSA) / NSA) & 1, p.err)) {
          *abort = 1;
          break;
        }
        const uint32_t fb = qd_full0 + 8 * s;
        const int q0 = qt * TC;
        mbar_arrive_expect_tx(fb, 2 * C::QT_BYTES + C::LD_BYTES + (DROP ? C::M_BYTES : 0));
        if constexpr (DROP)  // keep bits of queries q0.. (rows of head h) x keys kv0..kv0+127
          tma_load_2d(sb + C::OFF_M + s * C::M_BYTES, &tmM, kv0 >> 5,
                      (int)(((int64_t)b * p.nq + h) * p.S + q0), fb);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_2d(sQ + s * C::QT_BYTES + kb * 8192, &tmQ, h * D + kb * 64, grow0 + q0, fb);
          tma_load_2d(sO + s * C::QT_BYTES + kb * 8192, &tmO, h * D + kb * 64, grow0 + q0, fb);
        }
        const int64_t lrow = ((int64_t)b * p.nq + h) * p.s_pad + q0;
        bulk_load(sLDa + s * C::LD_BYTES, p.lse2 + lrow, TC * 4, fb);
        bulk_load(sLDa + s * C::LD_BYTES + TC * 4, p.delta + lrow, TC * 4, fb);
        if (++qt == nqt) {
          qt = qt_start;
          ++h;
        }
      }
    }
  } else if (warp == W_MMA) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc_sp = idesc_bf16_f32(TR, TC, 0, 0);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(TR, D, 0, 1);
    const uint64_t dk = smem_desc_sw128(sK, 16, 1024), dv = smem_desc_sw128(sV, 16, 1024);
    const uint64_t dqk = smem_desc_sw128(sQ, 16, 1024), dok = smem_desc_sw128(sO, 16, 1024);
    const uint64_t dqm = smem_desc_sw128(sQ, 8192, 1024), dom = smem_desc_sw128(sO, 8192, 1024);
    // S^T / dP^T of tile it into the score columns
    auto issue_sp = [&](int it) -> bool {
      const int s = it % NSA;
      if (!warp_wait(qd_full0 + 8 * s, (it / NSA) & 1, p.err)) return false;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * (TR * 128) + (kk & 3) * 32) >> 4;
          const uint32_t offq = (s * C::QT_BYTES + (kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          tc_mma_f16(tmem, dk + off, dqk + offq, idesc_sp, kk > 0);
          tc_mma_f16(tmem + 64, dv + off, dok + offq, idesc_sp, kk > 0);
        }
        tc_commit(sp_full0 + 8 * (it & 1));
      }
      __syncwarp();
      return true;
    };
    bool good = warp_wait(kv_full, 0, p.err) && issue_sp(0);
    for (int it = 0; it < n_it && good; ++it) {
      // the group of tile it has its scores in registers: the next tile's go in
      // (no abort-flag poll here: a role that gave up stops arriving, so this
      // warp's next bounded wait runs out as well)
      if (!warp_wait(sp_free0 + 8 * (it & 1), (it >> 1) & 1, p.err) ||
          (it + 1 < n_it && !issue_sp(it + 1)) ||
          !warp_wait(pds_full0 + 8 * (it & 1), (it >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      const int s = it % NSA;
      const uint32_t ta = tmem + C::COL_PDS + (it & 1) * 64;  // P^T, then dS^T at + 32
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < TC / 16; ++kk) {
          const uint32_t b_off = (s * C::QT_BYTES + kk * 2048) >> 4;
          tc_mma_f16_ts(tmem + C::COL_DV, ta + kk * 8, dom + b_off, idesc_acc, (it > 0 || kk > 0));
          tc_mma_f16_ts(tmem + C::COL_DK, ta + 32 + kk * 8, dqm + b_off, idesc_acc,
                        (it > 0 || kk > 0));
        }
        tc_commit(qd_empty0 + 8 * s);
        tc_commit(pds_empty0 + 8 * (it & 1));
        if (it == n_it - 1) tc_commit(acc_done);
      }
      __syncwarp();
    }
    if (!good) *abort = 1;
  } else {
    // ---------------- compute warps 0-15 (group grp takes the tiles it & 1 == grp)
    const int grp = warp >> 3, half = (warp >> 2) & 1;
    const int rrow = (warp & 3) * 32 + lane;
    const int kr = kv0 + rrow;  // this thread's key position
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t col0 = half * 32;  // this warp's columns of the 64-wide tiles
    bool good = true;
    int qt = qt_start + grp;  // query tile of iteration it (it mod per_head past qt_start)
    while (qt >= nqt) qt -= per_head;
    for (int it = grp; it < n_it; it += 2) {
      if (warp_aborted(abort) || !warp_wait(sp_full0 + 8 * grp, (it >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      float st[32], dp[32];
      {
        uint32_t rs[32], rd[32];
        tmem_ld32(tmem + lane_base + col0, rs);
        tmem_ld32(tmem + lane_base + 64 + col0, rd);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          st[c] = __uint_as_float(rs[c]);
          dp[c] = __uint_as_float(rd[c]);
        }
      }
      // the scores are in registers: the MMA warp may overwrite them
      tc_fence_before();
      mbar_arrive(sp_free0 + 8 * grp);
      const float* ldp = sLD + (it % NSA) * (2 * TC) + col0;
      // this key's keep bits against the tile's queries: word (warp & 3) of each
      // query row of the staged [64][4] tile (the same word for the whole warp)
      const uint32_t* mq = sM + (it % NSA) * (TC * 4) + col0 * 4 + (warp & 3);
      // P^T and dS^T of this key row against its 32 queries of the tile (past
      // the sequence end the workspace holds LSE = +inf, so P = 0 there);
      // LSE/delta are read from smem four at a time
      const int q0 = qt * TC + col0;
      const bool full = kr < p.S && (!p.causal || q0 >= kv0 + TR - 1);
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 L = *reinterpret_cast<const float4*>(ldp + c);
        const float4 Dl = *reinterpret_cast<const float4*>(ldp + TC + c);
        const float l4[4] = {L.x, L.y, L.z, L.w}, d4[4] = {Dl.x, Dl.y, Dl.z, Dl.w};
        if (full) {
          fma2(st[c], st[c + 1], st[c], st[c + 1], p.sl2, p.sl2, -l4[0], -l4[1]);
          fma2(st[c + 2], st[c + 3], st[c + 2], st[c + 3], p.sl2, p.sl2, -l4[2], -l4[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) st[c + e] = ex2_ftz(st[c + e]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const bool vis = kr < p.S && !(p.causal && q0 + c + e < kr);
            st[c + e] = vis ? ex2_ftz(fmaf(st[c + e], p.sl2, -l4[e])) : 0.0f;
          }
        }
        if constexpr (DROP) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const bool kp = (mq[(c + e) * 4] >> lane) & 1u;
            dp[c + e] = st[c + e] * ((kp ? dp[c + e] * p.dscale : 0.0f) - d4[e]);
            st[c + e] = kp ? st[c + e] * p.dscale : 0.0f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) dp[c + e] = st[c + e] * (dp[c + e] - d4[e]);
        }
      }
      uint32_t pp[16], pd[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        pp[c] = pack_bf16x2(st[2 * c], st[2 * c + 1]);
        pd[c] = pack_bf16x2(dp[2 * c], dp[2 * c + 1]);
      }
      // P^T / dS^T buffer grp was last read by dV/dK of tile it - 2
      if (it >= 2 && !warp_wait(pds_empty0 + 8 * grp, ((it - 2) >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      const uint32_t tpd = tmem + lane_base + C::COL_PDS + grp * 64 + half * 16;
      tmem_st16(tpd, pp);
      tmem_st16(tpd + 32, pd);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(pds_full0 + 8 * grp);
      qt += 2;
      while (qt >= nqt) qt -= per_head;
    }
    if (!good) *abort = 1;
    // ---- all products done: group 0 stores dK (scaled), group 1 dV, out of TMEM
    if (good && warp_wait(acc_done, 0, p.err) && !warp_aborted(abort)) {
      tc_fence_after();
      const bool row_ok = kr < p.S;
      const int64_t orow = (int64_t)(grow0 + kr) * p.ld_out + g * D;
      const int c0 = half * (D / 2);  // the two warps of a quarter split the d columns
      if (grp == 0)
        store_tmem_row<D / 2>(tmem + lane_base + C::COL_DK + c0, p.scale,
                              row_ok ? p.d0 + orow + c0 : nullptr);
      else
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
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + QO_BYTES;
  static constexpr int OFF_K = OFF_DO + QO_BYTES;        // NSB stages
  static constexpr int OFF_V = OFF_K + NSB * KV_BYTES;   // NSB stages
  static constexpr int OFF_BAR = OFF_V + NSB * KV_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  // TMEM: scores [0, 128), dS buffers [128, 192) (32 columns = 64 bf16 keys each), dQ,
  // and the CTA's Q and dO rows (bf16 pairs) as the A operands of the score products
  static constexpr int COL_DS = 128, COL_DQ = COL_ACC;
  static constexpr int COL_QT = 384, COL_OT = 384 + D / 2;
  static_assert(COL_DQ + D <= COL_QT && COL_OT + D / 2 <= 512, "TMEM columns");
};

template <int D, bool DROP>
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
  const uint32_t sQ = sb + C::OFF_Q, sO = sb + C::OFF_DO, sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t qo_full = bar;          // Q, dO loaded                  (tx)
  const uint32_t kv_full0 = bar + 8;     // [5] K/V stage loaded          (tx)
  const uint32_t kv_empty0 = bar + 48;   // [5] stage read by dQ          (commit)
  const uint32_t sp_full0 = bar + 88;    // [2] S/dP of tile j ready      (commit)
  const uint32_t sp_free0 = bar + 104;   // [2] group read them out       (256 arrivals)
  const uint32_t ds_full0 = bar + 120;   // [2] dS buffer written         (256 arrivals)
  const uint32_t ds_empty0 = bar + 136;  // [2] dQ read the buffer        (commit)
  const uint32_t acc_done = bar + 152;   // all products done             (commit)
  const uint32_t qo_tmem = bar + 160;    // Q, dO copied into TMEM        (128 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 176);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 180);

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
    mbar_init(qo_full, 1);
    for (int i = 0; i < NSB; ++i) {
      mbar_init(kv_full0 + 8 * i, 1);
      mbar_init(kv_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sp_full0 + 8 * i, 1);
      mbar_init(sp_free0 + 8 * i, NGROUP);
      mbar_init(ds_full0 + 8 * i, NGROUP);
      mbar_init(ds_empty0 + 8 * i, 1);
    }
    mbar_init(acc_done, 1);
    mbar_init(qo_tmem, 128);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_PROD) {
    // ---------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(qo_full, 2 * C::QO_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_2d(sQ + kb * (TR * 128), &tmQ, h * D + kb * 64, grow0 + q0, qo_full);
        tma_load_2d(sO + kb * (TR * 128), &tmO, h * D + kb * 64, grow0 + q0, qo_full);
      }
      for (int j = 0; j < nkt && !*abort; ++j) {
        const int s = j % NSB;
        if (j >= NSB && !mbar_wait(kv_empty0 + 8 * s, ((j - NSB) / NSB) & 1, p.err)) {
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
  } else if (warp == W_MMA) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc_sp = idesc_bf16_f32(TR, TC, 0, 0);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(TR, D, 0, 1);
    const uint64_t dkk = smem_desc_sw128(sK, 16, 1024), dvk = smem_desc_sw128(sV, 16, 1024);
    const uint64_t dkm = smem_desc_sw128(sK, 8192, 1024);
    auto issue_sp = [&](int j) -> bool {
      const int s = j % NSB;
      if (!warp_wait(kv_full0 + 8 * s, (j / NSB) & 1, p.err)) return false;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offk = (s * C::KV_BYTES + (kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          tc_mma_f16_ts(tmem, tmem + C::COL_QT + kk * 8, dkk + offk, idesc_sp, kk > 0);
          tc_mma_f16_ts(tmem + 64, tmem + C::COL_OT + kk * 8, dvk + offk, idesc_sp, kk > 0);
        }
        tc_commit(sp_full0 + 8 * (j & 1));
      }
      __syncwarp();
      return true;
    };
    bool good = warp_wait(qo_tmem, 0, p.err) && issue_sp(0);
    for (int j = 0; j < nkt && good; ++j) {
      // the group of tile j has its scores in registers: the next tile's go in
      if (!warp_wait(sp_free0 + 8 * (j & 1), (j >> 1) & 1, p.err) ||
          (j + 1 < nkt && !issue_sp(j + 1)) ||
          !warp_wait(ds_full0 + 8 * (j & 1), (j >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      const int s = j % NSB;
      const uint32_t ta = tmem + C::COL_DS + (j & 1) * 32;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < TC / 16; ++kk)
          tc_mma_f16_ts(tmem + C::COL_DQ, ta + kk * 8, dkm + ((s * C::KV_BYTES + kk * 2048) >> 4),
                        idesc_acc, (j > 0 || kk > 0));
        tc_commit(kv_empty0 + 8 * s);
        tc_commit(ds_empty0 + 8 * (j & 1));
        if (j == nkt - 1) tc_commit(acc_done);
      }
      __syncwarp();
    }
    if (!good) *abort = 1;
  } else {
    // ---------------- compute warps 0-15 (group grp takes the tiles j & 1 == grp)
    const int grp = warp >> 3, half = (warp >> 2) & 1;
    const int rrow = (warp & 3) * 32 + lane;
    const int row = q0 + rrow;
    const int64_t lrow = ((int64_t)b * p.nq + h) * p.s_pad + row;
    const float L2 = p.lse2[lrow];  // +inf past the sequence end
    const float Dr = p.delta[lrow];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t col0 = half * 32;
    bool good = true;
    if (warp < 4) {
      // Q and dO rows of this lane quarter from the (128-byte swizzled) smem
      // tiles into TMEM, bf16 pairs in column order: the score products then
      // read them from TMEM instead of shared memory for every key tile
      if (!warp_wait(qo_full, 0, p.err)) {
        good = false;
      } else {
        const uint32_t r = (uint32_t)rrow, sw = r & 7;
#pragma unroll
        for (int mtx = 0; mtx < 2; ++mtx) {
          const uint8_t* base = smem + (mtx == 0 ? C::OFF_Q : C::OFF_DO) + r * 128;
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb) {
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 w = *reinterpret_cast<const uint4*>(base + kb * (TR * 128) + ((c ^ sw) << 4));
              v[4 * c] = w.x; v[4 * c + 1] = w.y; v[4 * c + 2] = w.z; v[4 * c + 3] = w.w;
            }
            tmem_st32(tmem + lane_base + (mtx == 0 ? C::COL_QT : C::COL_OT) + kb * 32, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(qo_tmem);
      }
    }
    for (int j = grp; j < nkt && good; j += 2) {
      // keep bits of this query row against the thread's 32 keys (issued before
      // the wait so the load overlaps it)
      uint32_t kbits = 0;
      if constexpr (DROP) {
        if (row < p.S)
          kbits = p.dmask[(((int64_t)b * p.nq + h) * p.S + row) * p.mw + ((j * TC + col0) >> 5)];
      }
      if (warp_aborted(abort) || !warp_wait(sp_full0 + 8 * grp, (j >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      float sc[32], dp[32];
      {
        uint32_t rs[32], rd[32];
        tmem_ld32(tmem + lane_base + col0, rs);
        tmem_ld32(tmem + lane_base + 64 + col0, rd);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sc[c] = __uint_as_float(rs[c]);
          dp[c] = __uint_as_float(rd[c]);
        }
      }
      // the scores are in registers: the MMA warp may overwrite them
      tc_fence_before();
      mbar_arrive(sp_free0 + 8 * grp);
      const int kv0 = j * TC + col0;  // first key of this thread's columns
      // mask-free when every query row of the CTA sees every key of the half-tile
      const bool full = kv0 + 32 <= p.S && (!p.causal || kv0 + 31 <= q0);
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          fma2(sc[c], sc[c + 1], sc[c], sc[c + 1], p.sl2, p.sl2, -L2, -L2);
          sc[c] = ex2_ftz(sc[c]);
          sc[c + 1] = ex2_ftz(sc[c + 1]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int kv = kv0 + c;
          const bool vis = kv < p.S && !(p.causal && kv > row);
          sc[c] = vis ? ex2_ftz(fmaf(sc[c], p.sl2, -L2)) : 0.0f;
        }
      }
      if constexpr (DROP) {
#pragma unroll
        for (int c = 0; c < 32; ++c) dp[c] = (kbits >> c) & 1u ? dp[c] * p.dscale : 0.0f;
      }
      uint32_t pd[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        pd[c] = pack_bf16x2(sc[2 * c] * (dp[2 * c] - Dr), sc[2 * c + 1] * (dp[2 * c + 1] - Dr));
      // dS buffer grp was last read by dQ of tile j - 2
      if (j >= 2 && !warp_wait(ds_empty0 + 8 * grp, ((j - 2) >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tmem_st16(tmem + lane_base + C::COL_DS + grp * 32 + half * 16, pd);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_full0 + 8 * grp);
    }
    if (!good) *abort = 1;
    // ---- all products done: dQ (scaled) out of TMEM, the warps of each lane
    // quarter taking 32-column slices (all four for d = 128, two for d = 64)
    if (good && warp_wait(acc_done, 0, p.err) && !warp_aborted(abort)) {
      tc_fence_after();
      const bool row_ok = row < p.S;
      constexpr int NW = D / 32;  // warps per quarter with a slice
      const int slice = grp * 2 + half;
      if (slice < NW) {
        const int c0 = slice * 32;
        store_tmem_row<32>(tmem + lane_base + C::COL_DQ + c0, p.scale,
                           row_ok ? p.d0 + (int64_t)(grow0 + row) * p.ld_out + h * D + c0
                                  : nullptr);
      }
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

template <int D, bool DROP>
mgb_status bwd_tc_d(const AttnArgs& a, cudaStream_t st, cudaStream_t st_dq) {
  const uint64_t T = (uint64_t)a.B * a.S;
  BwdParams p{};
  p.B = a.B; p.S = a.S; p.nq = a.nq; p.nkv = a.nkv; p.causal = a.causal;
  p.s_pad = attn_bwd_row_pad(a.S);
  p.lse2 = a.delta;
  p.delta = a.delta + (size_t)a.B * a.nq * p.s_pad;
  p.err = device_error_word();
  p.sl2 = 1.4426950408889634f / sqrtf((float)D);
  p.scale = 1.0f / sqrtf((float)D);
  p.dmask = a.drop_mask;
  p.mw = attn_mask_words(a.S);
  p.dscale = a.drop_scale;
  // kernel A: K/V rows of 128, Q/dO tiles of 64
  {
    using C = DkvCfg<D>;
    CUtensorMap tq, tk, tv, to, tm;
    // keep bits: [B*nq*S rows][mw words], boxes of 4 words x 64 query rows
    // (without dropout a harmless map over the same rows of the output)
    if ((DROP ? tmap_encode_u32_2d(&tm, a.drop_mask, p.mw, (uint64_t)a.B * a.nq * a.S, p.mw, 4, TC)
              : tmap_encode_u32_2d(&tm, a.dk, 4, T, 4, 4, TC)) != CUDA_SUCCESS)
      return MGB_ERR_CUDA;
    if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TC) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&to, a.dout, (uint64_t)a.nq * D, T, a.ld_do, 64, TC) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TR) != CUDA_SUCCESS ||
        tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TR) != CUDA_SUCCESS)
      return MGB_ERR_CUDA;
    p.d0 = reinterpret_cast<bf16*>(a.dk);
    p.d1 = reinterpret_cast<bf16*>(a.dv);
    p.ld_out = a.ld_dkv;
    auto k = attn_bwd_dkdv_tc_kernel<D, DROP>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return MGB_ERR_CUDA;
    dim3 grid(a.nkv * a.B, (a.S + TR - 1) / TR);
    k<<<grid, NTHREADS, C::SMEM, st>>>(tq, tk, tv, to, tm, p);
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
    auto k = attn_bwd_dq_tc_kernel<D, DROP>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return MGB_ERR_CUDA;
    dim3 grid(a.nq * a.B, (a.S + TR - 1) / TR);
    k<<<grid, NTHREADS, C::SMEM, st_dq>>>(tq, tk, tv, to, p);
  }
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

// dK/dV on st, dQ on st_dq (which the caller has made wait for the inputs).
mgb_status attention_tc_bwd_main(const AttnArgs& a, cudaStream_t st, cudaStream_t st_dq) {
  const bool drop = a.drop_thr < 256;
  if (drop && a.drop_mask == nullptr) return MGB_ERR_INVALID_ARG;
  if (a.d == 64)
    return drop ? bwd_tc_d<64, true>(a, st, st_dq) : bwd_tc_d<64, false>(a, st, st_dq);
  if (a.d == 128)
    return drop ? bwd_tc_d<128, true>(a, st, st_dq) : bwd_tc_d<128, false>(a, st, st_dq);
  return MGB_ERR_UNSUPPORTED;
}

}  // namespace mgb

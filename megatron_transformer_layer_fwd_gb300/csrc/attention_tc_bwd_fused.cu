// bf16 attention backward in one pass over key blocks (tcgen05): dK, dV and
// dQ from the same score tiles, head dimension 128, no dropout.
//
// The products are those of the two-kernel backward ("02 - How a whole
// Transformer block is split", section 2 defines the forward; page 1,
// section 2 asks for the end-to-end backward): P = exp(s - LSE), dP = dO V^T,
// dS = P (dP - delta), dV_g = sum_h P^T dO_h, dK_g = sum_h dS^T Q_h / sqrt(d),
// dQ_h = dS K_g / sqrt(d). Here the CTA that owns 128 keys of one KV head also
// forms each query tile's share of dQ,
//   dQ^T(tile) = K^T dS^T      M = d (TMEM lanes), N = 64 queries, K = 128 keys
// and adds it into a float32 accumulator [B * S][nq * d] in global memory with
// TMA reduce-add copies (the additions happen in L2). The score products are
// not computed twice, as the separate dQ kernel does; the price is that the
// float32 sums of dQ arrive in no fixed order (results differ run to run at
// float32 rounding level), which is why the two-kernel path stays available
// for deterministic runs (and serves dropout and head dimension 64).
//
// One CTA = 128 keys (TMEM lane = key) of one KV head, looping over every
// query head of the group and every 64-query tile that can see its keys.
// TMEM (512 columns):
//   [0, 64)    S^T  = K Q^T      [64, 128)  dP^T = V dO^T      (one buffer)
//   [128, 192) P^T as bf16 pairs, two buffers of 32 columns (tile i & 1)
//   [192, 256) dQ^T of one tile (lanes = head-dim index)
//   [256, 384) dV     [384, 512) dK   (accumulated over the whole loop)
// Shared memory: K and V (the CTA's rows), a 3-stage ring of Q / dO / LSE /
// delta tiles, dS^T of tiles i & 1 as [128 keys][64 queries] bf16 tiles with
// the 128-byte swizzle (the A operand of dK += dS^T Q read K-major, the B
// operand of dQ^T read MN-major), and eight float32 boxes [32 queries][32 d]
// for the reduce-add copies, box w % 8 taken by compute warp w (the warps w
// and w + 8 of the two groups in turn, handed over by a barrier per box).
//
// Warps (18): 0-15 compute, in two groups of 8 taking alternate tiles; 16
// producer (TMA); 17 MMA issuer. A group, after handing tile i's P^T (TMEM)
// and dS^T (shared memory) to the MMA warp, reads dQ^T of tile i - 1 out of
// TMEM (warp w: lane quarter w % 4, i.e. d = 32 (w % 4) + lane, and the 32
// queries of its half), stages it transposed in its box and adds the box to
// the accumulator; the MMA warp issues dQ^T of tile i once that read is done,
// after dV and dK of tile i. The group that would take tile n reads the last
// tile's dQ^T after its loop. Every wait is bounded; a wait that runs out
// sets the shared abort flag and every role leaves its loop before the
// closing barrier.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace mgb {

CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer);
CUresult tmap_encode_f32_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                            int64_t ld, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int D = 128;          // head dimension of this kernel
constexpr int TR = 128;         // keys per CTA
constexpr int TC = 64;          // queries per tile
constexpr int NS = 3;           // Q/dO ring stages
constexpr int NGROUP = 256;     // compute threads per group
constexpr int NTHREADS = 576;   // 16 compute warps, producer, MMA
constexpr int W_PROD = 16, W_MMA = 17;

struct FusedParams {
  int B, S, nq, nkv, causal, s_pad;
  const float* lse2;   // [B * nq][s_pad]: LSE * log2(e)
  const float* delta;  // [B * nq][s_pad]
  bf16 *dk, *dv;
  int64_t ld_dkv;
  int* err;
  float sl2, scale;
};

struct FCfg {
  static constexpr int KV_BYTES = TR * D * 2;   // K or V rows of this CTA
  static constexpr int QT_BYTES = TC * D * 2;   // one Q or dO tile
  static constexpr int DS_BYTES = TR * TC * 2;  // one dS^T tile
  static constexpr int DQ_BOX = 32 * 32 * 4;    // one [32][32] float32 box
  static constexpr int LD_BYTES = 2 * TC * 4;   // a tile's LSE*log2e and delta
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;
  static constexpr int OFF_DO = OFF_Q + NS * QT_BYTES;
  static constexpr int OFF_DS = OFF_DO + NS * QT_BYTES;
  static constexpr int OFF_DQ = OFF_DS + 2 * DS_BYTES;
  static constexpr int OFF_LD = OFF_DQ + 8 * DQ_BOX;
  static constexpr int OFF_BAR = OFF_LD + NS * LD_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int COL_P = 128, COL_DQ = 192, COL_DV = 256, COL_DK = 384;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(OFF_DS % 1024 == 0 && OFF_DQ % 1024 == 0, "swizzled tiles 1024-byte aligned");
};

// dQ^T of tile j out of TMEM and into the accumulator, for one compute warp:
// 32 lanes of TMEM from column tcol (d = lane of this warp's quarter) x 32
// queries, written transposed into the warp's box ([query][d], 128-byte rows,
// 16-byte chunk c of row q at q * 128 + ((c ^ (q % 8)) * 16): the 32 lanes of
// a row hit 32 different banks), then one reduce-add copy at (x, y) of the
// accumulator. Arrives on dq_free once the TMEM read is done. The box was
// last filled for tile j - 1 by the other group's warp: box_free has passed
// phase j - 1 once that copy has read it; this warp's copy, once it has read
// the box, completes phase j. Returns false if a wait ran out.
__device__ __forceinline__ bool dq_out(int j, uint32_t tcol, uint32_t box, uint32_t box_free,
                                       uint32_t dq_free, const CUtensorMap* tm, int x, int y,
                                       int* err) {
  const int lane = threadIdx.x & 31;
  uint32_t r[32];
  tmem_ld32(tcol, r);
  tmem_ld_wait();
  tc_fence_before();
  mbar_arrive(dq_free);  // the MMA warp may write the next tile's dQ^T
  if (j > 0 && !warp_wait(box_free, (j - 1) & 1, err)) return false;
  const uint32_t wo = (uint32_t)(lane & 3) * 4;
  const uint32_t ch = (uint32_t)(lane >> 2);
#pragma unroll
  for (int q = 0; q < 32; ++q)
    st_shared_f32(box + q * 128 + ((ch ^ (q & 7)) << 4) + wo, __uint_as_float(r[q]));
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    if (dcheck((x & 31) == 0 && x >= 0 && y >= 0, err)) {
      tma_reduce_add_2d(tm, box, x, y);
      bulk_commit();
      bulk_wait_read<0>();  // the copy has read the box: the other group may refill it
    }
    mbar_arrive(box_free);
  }
  return true;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmO,
                          const __grid_constant__ CUtensorMap tmDQ, const FusedParams p) {
  using C = FCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V, sQ = sb + C::OFF_Q, sO = sb + C::OFF_DO,
                 sDS = sb + C::OFF_DS, sDQ = sb + C::OFF_DQ, sLDa = sb + C::OFF_LD;
  const float* sLD = reinterpret_cast<const float*>(smem + C::OFF_LD);
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t kv_full = bar;           // K, V loaded                          (tx)
  const uint32_t qd_full0 = bar + 8;      // [3] Q/dO/LSE/delta stage loaded      (tx)
  const uint32_t qd_empty0 = bar + 32;    // [3] stage read by dV/dK              (commit)
  const uint32_t sp_full0 = bar + 56;     // [2] S^T/dP^T of tile i ready         (commit)
  const uint32_t sp_free0 = bar + 72;     // [2] group read them out of TMEM      (256)
  const uint32_t pds_full0 = bar + 88;    // [2] P^T (TMEM), dS^T (smem) written   (256)
  const uint32_t pds_empty0 = bar + 104;  // [2] dV/dK/dQ^T read them             (commit)
  const uint32_t dq_full = bar + 120;     // dQ^T of a tile complete              (commit)
  const uint32_t dq_free = bar + 128;     // a group read dQ^T out of TMEM        (256)
  const uint32_t acc_done = bar + 136;    // all products done                    (commit)
  const uint32_t box_free0 = bar + 176;   // [8] the last copy out of box b read it (1)
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
    tma_prefetch_desc(&tmDQ);
    mbar_init(kv_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(qd_full0 + 8 * i, 1);
      mbar_init(qd_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 8; ++i) mbar_init(box_free0 + 8 * i, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(sp_full0 + 8 * i, 1);
      mbar_init(sp_free0 + 8 * i, NGROUP);
      mbar_init(pds_full0 + 8 * i, NGROUP);
      mbar_init(pds_empty0 + 8 * i, 1);
    }
    mbar_init(dq_full, 1);
    mbar_init(dq_free, NGROUP);
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
      for (int kb = 0; kb < D / 64; ++kb) {
        tma_load_2d(sK + kb * (TR * 128), &tmK, g * D + kb * 64, grow0 + kv0, kv_full);
        tma_load_2d(sV + kb * (TR * 128), &tmV, g * D + kb * 64, grow0 + kv0, kv_full);
      }
      int h = g * rep, qt = qt_start;  // head and query tile of iteration it
      for (int it = 0; it < n_it && !*abort; ++it) {
        const int s = it % NS;
        if (it >= NS && !mbar_wait(qd_empty0 + 8 * s, ((it - NS) / NS) & 1, p.err)) {
          *abort = 1;
          break;
        }
        const uint32_t fb = qd_full0 + 8 * s;
        const int q0 = qt * TC;
        if (!dcheck(h < p.nq && q0 < p.S, p.err)) {
          *abort = 1;
          break;
        }
        mbar_arrive_expect_tx(fb, 2 * C::QT_BYTES + C::LD_BYTES);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) {
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
    constexpr uint32_t idesc_sp = idesc_bf16_f32(TR, TC, 0, 0);   // S^T, dP^T
    constexpr uint32_t idesc_acc = idesc_bf16_f32(TR, D, 0, 1);   // dV, dK
    constexpr uint32_t idesc_dq = idesc_bf16_f32(D, TC, 1, 1);    // dQ^T = K^T dS^T
    const uint64_t dk = smem_desc_sw128(sK, 16, 1024), dv = smem_desc_sw128(sV, 16, 1024);
    const uint64_t dkm = smem_desc_sw128(sK, TR * 128, 1024);     // K as MN-major A (d inner)
    const uint64_t dqk = smem_desc_sw128(sQ, 16, 1024), dok = smem_desc_sw128(sO, 16, 1024);
    const uint64_t dqm = smem_desc_sw128(sQ, 8192, 1024), dom = smem_desc_sw128(sO, 8192, 1024);
    const uint64_t dsk = smem_desc_sw128(sDS, 16, 1024);          // dS^T as K-major A
    const uint64_t dsm = smem_desc_sw128(sDS, 8192, 1024);        // dS^T as MN-major B
    auto issue_sp = [&](int it) -> bool {
      const int s = it % NS;
      if (!warp_wait(qd_full0 + 8 * s, (it / NS) & 1, p.err)) return false;
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
      if (!warp_wait(sp_free0 + 8 * (it & 1), (it >> 1) & 1, p.err) ||
          (it + 1 < n_it && !issue_sp(it + 1)) ||
          !warp_wait(pds_full0 + 8 * (it & 1), (it >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      const int s = it % NS;
      const uint32_t ta = tmem + C::COL_P + (it & 1) * 32;     // P^T of tile it
      const uint32_t ds_off = ((it & 1) * C::DS_BYTES) >> 4;   // its dS^T tile
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < TC / 16; ++kk) {
          const uint32_t b_off = (s * C::QT_BYTES + kk * 2048) >> 4;
          tc_mma_f16_ts(tmem + C::COL_DV, ta + kk * 8, dom + b_off, idesc_acc, (it > 0 || kk > 0));
          tc_mma_f16(tmem + C::COL_DK, dsk + ds_off + ((kk * 32) >> 4), dqm + b_off, idesc_acc,
                     (it > 0 || kk > 0));
        }
        tc_commit(qd_empty0 + 8 * s);
      }
      __syncwarp();
      // dQ^T of tile it - 1 read out of TMEM by the group of tile it
      if (it > 0 && !warp_wait(dq_free, (it - 1) & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < TR / 16; ++kk)
          tc_mma_f16(tmem + C::COL_DQ, dkm + ((kk * 2048) >> 4), dsm + ds_off + ((kk * 2048) >> 4),
                     idesc_dq, kk > 0);
        tc_commit(pds_empty0 + 8 * (it & 1));
        tc_commit(dq_full);
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
    const uint32_t box = sDQ + (warp & 7) * C::DQ_BOX, box_free = box_free0 + 8 * (warp & 7);
    // dQ^T of tile j to the accumulator. Inside the loop the reader of tile j
    // holds tile j + 1's scores, so dq_full has completed phase j - 1 and
    // cannot complete phase j + 1 before this read (its parity names phase j
    // alone). The last tile's reader, after its loop, may come two phases
    // early: it waits for all products instead.
    auto dq_tile = [&](int j) -> bool {
      if (!(j == n_it - 1 ? warp_wait(acc_done, 0, p.err) : warp_wait(dq_full, j & 1, p.err)))
        return false;
      tc_fence_after();
      const int hj = g * rep + j / per_head, qj = qt_start + j % per_head;
      return dq_out(j, tmem + lane_base + C::COL_DQ + col0, box, box_free, dq_free, &tmDQ,
                    hj * D + 32 * (warp & 3), grow0 + qj * TC + (int)col0, p.err);
    };
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
      // P^T / dS^T buffers grp were last read by dV/dK/dQ^T of tile it - 2
      if (it >= 2 && !warp_wait(pds_empty0 + 8 * grp, ((it - 2) >> 1) & 1, p.err)) {
        good = false;
        break;
      }
      const float* ldp = sLD + (it % NS) * (2 * TC) + col0;
      const int q0 = qt * TC + col0;
      const bool full = kr < p.S && (!p.causal || q0 >= kv0 + TR - 1);
      // dS^T row rrow, this warp's 32 queries: 16-byte chunks half*4 .. of the
      // 128-byte-swizzled [128 keys][64 queries] tile, written 8 queries at a time
      uint8_t* dsrow = smem + C::OFF_DS + grp * C::DS_BYTES + rrow * 128;
      uint32_t pp[16];
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
#pragma unroll
        for (int e = 0; e < 4; ++e) dp[c + e] = st[c + e] * (dp[c + e] - d4[e]);
        pp[c / 2] = pack_bf16x2(st[c], st[c + 1]);
        pp[c / 2 + 1] = pack_bf16x2(st[c + 2], st[c + 3]);
        if (c & 4) {
          const int j = c - 4;
          uint4 v;
          v.x = pack_bf16x2(dp[j], dp[j + 1]);
          v.y = pack_bf16x2(dp[j + 2], dp[j + 3]);
          v.z = pack_bf16x2(dp[j + 4], dp[j + 5]);
          v.w = pack_bf16x2(dp[j + 6], dp[j + 7]);
          *reinterpret_cast<uint4*>(dsrow + (((half * 4 + (c >> 3)) ^ (rrow & 7)) << 4)) = v;
        }
      }
      tmem_st16(tmem + lane_base + C::COL_P + grp * 32 + half * 16, pp);
      fence_proxy_async();  // dS^T (generic writes) visible to the tensor core
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(pds_full0 + 8 * grp);
      // the other group's tile before this one: its dQ^T out of TMEM
      if (it > 0 && !dq_tile(it - 1)) {
        good = false;
        break;
      }
      qt += 2;
      while (qt >= nqt) qt -= per_head;
    }
    // the group that would take tile n_it reads the last tile's dQ^T
    if (good && (n_it & 1) == grp && !warp_aborted(abort) && !dq_tile(n_it - 1)) good = false;
    if (!good) *abort = 1;
    // ---- all products done: group 0 stores dK (scaled), group 1 dV, out of TMEM
    if (good && warp_wait(acc_done, 0, p.err) && !warp_aborted(abort)) {
      tc_fence_after();
      const bool row_ok = kr < p.S;
      const int64_t orow = (int64_t)(grow0 + kr) * p.ld_dkv + g * D;
      const int c0 = half * (D / 2);  // the two warps of a quarter split the d columns
      if (grp == 0)
        store_tmem_row<D / 2>(tmem + lane_base + C::COL_DK + c0, p.scale,
                              row_ok ? p.dk + orow + c0 : nullptr);
      else
        store_tmem_row<D / 2>(tmem + lane_base + C::COL_DV + c0, 1.0f,
                              row_ok ? p.dv + orow + c0 : nullptr);
    } else {
      *abort = 1;
    }
    if (lane == 0) bulk_wait<0>();  // this warp's reduce-add copies complete before exit
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

// dq[t][h*d + j] = bf16(acc[t][h*d + j] * scale): 8 columns per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(int64_t rows, int cols, const float* acc,
                                                         float scale, bf16* dq, int64_t ld) {
  const int nv = cols / 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * nv;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nv;
    const int c = (int)(i % nv) * 8;
    const float4 a = *reinterpret_cast<const float4*>(acc + r * cols + c);
    const float4 b2 = *reinterpret_cast<const float4*>(acc + r * cols + c + 4);
    uint4 w;
    w.x = pack_bf16x2(a.x * scale, a.y * scale);
    w.y = pack_bf16x2(a.z * scale, a.w * scale);
    w.z = pack_bf16x2(b2.x * scale, b2.y * scale);
    w.w = pack_bf16x2(b2.z * scale, b2.w * scale);
    *reinterpret_cast<uint4*>(dq + r * ld + c) = w;
  }
}

mgb_status fused_go(const AttnArgs& a, float* dq_acc, cudaStream_t st) {
  using C = FCfg;
  const uint64_t T = (uint64_t)a.B * a.S;
  FusedParams p{};
  p.B = a.B; p.S = a.S; p.nq = a.nq; p.nkv = a.nkv; p.causal = a.causal;
  p.s_pad = attn_bwd_row_pad(a.S);
  p.lse2 = a.delta;
  p.delta = a.delta + (size_t)a.B * a.nq * p.s_pad;
  p.err = device_error_word();
  p.sl2 = 1.4426950408889634f / sqrtf((float)D);
  p.scale = 1.0f / sqrtf((float)D);
  p.dk = reinterpret_cast<bf16*>(a.dk);
  p.dv = reinterpret_cast<bf16*>(a.dv);
  p.ld_dkv = a.ld_dkv;
  CUtensorMap tq, tk, tv, to, tdq;
  if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TC) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&to, a.dout, (uint64_t)a.nq * D, T, a.ld_do, 64, TC) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TR) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TR) != CUDA_SUCCESS ||
      tmap_encode_f32_2d(&tdq, dq_acc, (uint64_t)a.nq * D, T, (int64_t)a.nq * D, 32, 32) !=
          CUDA_SUCCESS)
    return MGB_ERR_CUDA;
  auto k = attn_bwd_fused_kernel;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 grid(a.nkv * a.B, (a.S + TR - 1) / TR);
  k<<<grid, NTHREADS, C::SMEM, st>>>(tq, tk, tv, to, tdq, p);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

bool attention_bwd_fused_ok(const AttnArgs& a) {
  if (a.d != D || a.dtype != MGB_BF16 || a.drop_thr < 256) return false;
  const char* det = getenv("MGB_DETERMINISTIC");
  if (det != nullptr && det[0] == '1') return false;
  const char* e = getenv("MGB_ATTN_BWD");
  return e == nullptr || strcmp(e, "split") != 0;
}

// dK/dV and the float32 dQ accumulator (in the workspace after the LSE/delta
// planes, zeroed by the pre-pass) in one pass, then dQ = bf16(accumulator /
// sqrt(d)).
mgb_status attention_tc_bwd_fused(const AttnArgs& a, cudaStream_t st) {
  float* acc = a.delta + 2 * (size_t)a.B * a.nq * attn_bwd_row_pad(a.S);
  const int64_t rows = (int64_t)a.B * a.S;
  const int cols = a.nq * D;
  const mgb_status r = fused_go(a, acc, st);
  if (r != MGB_OK) return r;
  const int64_t n = rows * (cols / 8);
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 8 * 152);
  dq_convert_kernel<<<blocks, 256, 0, st>>>(rows, cols, acc, 1.0f / sqrtf((float)D),
                                            reinterpret_cast<bf16*>(a.dq), a.ld_dq);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace mgb

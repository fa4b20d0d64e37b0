// bf16 attention forward on the tensor cores (tcgen05), two query tiles per
// work item taking turns.
//
// Definition ("LLM Lab 06: build a Megatron-style Transformer Block from
// scratch", section 2; "02 - How a whole Transformer block is split",
// section 2): O_h = softmax(Q_h K_g^T / sqrt(d)) V_g per batch and query head h,
// g = h / (nq / nkv), optional causal mask; LSE = log sum_j exp(s_j) is saved
// for the backward. Online softmax over key tiles (FlashAttention, which
// page 1, section 5 points to): the [S, S] score matrix never leaves the chip.
//
// A work item is 256 query rows of one (batch, head): tile A (rows q0 ..
// q0 + 127) and tile B (q0 + 128 .. q0 + 255), both against the same key /
// value tiles of 128 keys. TMEM (512 columns) holds S_A, S_B, O_A and O_B; a
// tile's probabilities P (bf16 pairs, 64 columns) are written over the first
// half of its own score columns and read from there by the PV product, so the
// score buffer of a tile is free again once its PV product has run. The MMA
// warp issues, per key tile j:
//     PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// (tcgen05.mma operations of one thread run in issue order, so S_X(j+1) writes
// the columns PV_X(j) has read). While the softmax warps of tile A work on
// S_A(j+1), the tensor core runs PV_B(j) and S_B(j+1), and the other way
// round: each tile's softmax overlaps the other tile's products.
//
// Ten warps:
//   warp 0     MMA issuer (whole warp runs the loop; one elected lane issues)
//   warp 1     producer: each item's two Q tiles, then K_0, V_0, K_1, V_1, ...
//              by TMA (128-byte swizzle) into a 2-stage K ring and a 2-stage V
//              ring; a stage is refilled once its last reader is done
//   warps 2-5  softmax of tile A, warps 6-9 softmax of tile B: one thread per
//              query row (warp w reads TMEM lane quarter w % 4) over all 128
//              keys, in chunks of 64 (32 with dropout): on a row's first key
//              tile a pass for the row maximum, then one pass for the
//              exponentials, the row sum and P; then, at the item's end, O / l
//              and LSE to global memory
// Online softmax in the log2 domain with a lazy reference: a row's reference
// maximum moves only when a tile's maximum exceeds it by more than TAU, and
// only then are its row sum and TMEM O row rescaled (P stays below 2^TAU).
// When S_X(j) is complete, PV_X(j - 1) is too (it was issued earlier), so the
// rescale of O_X before PV_X(j) needs no further wait.
// Every wait is bounded; one that runs out sets a shared abort flag, every role
// leaves its loop, and the CTA waits for work in flight before freeing TMEM.
// Dropout on the probabilities (DROP): the row sums take the undropped P; each
// softmax thread draws its 128 keys' keep bytes (element ((b*nq + h)*S + row) *
// Sp + key of the site's stream), drops and scales P as it is packed, and
// writes the 128 keep bits for the backward.
#include "common.cuh"
#include "internal.h"

namespace mgb {

CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int TQ = 128;         // query rows per tile (TMEM lanes)
constexpr int TK = 128;         // keys per KV tile
constexpr int NSK = 2;          // K ring stages
constexpr int NSV = 2;          // V ring stages
constexpr int NSOFT = 128;      // softmax threads per tile
constexpr int NTHREADS = 320;   // MMA warp, producer warp, 2 x 4 softmax warps
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float TAU = 8.0f;

template <int D>
struct Cfg2 {
  static constexpr int KB = D / 64;                     // 64-wide d boxes
  static constexpr int BOX = 128 * 128;                 // bytes of one [128][64] box
  static constexpr int Q_BYTES = TQ * D * 2;
  static constexpr int KV_BYTES = TK * D * 2;
  static constexpr int OFF_QA = 0;
  static constexpr int OFF_QB = Q_BYTES;
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NSV * KV_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;     // barriers, alignment slack
  static constexpr int COL_S = 0;                       // S_A at 0, S_B at TK
  static constexpr int COL_O = 2 * TK;                  // O_A, then O_B at + D
  static constexpr int TMEM_COLS = 512;
  static_assert(COL_O + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Params {
  int B, S, nq, nkv, causal, n_items;
  bf16* o;
  int64_t ld_o;
  float* lse;
  int* err;
  float sl2;  // log2(e) / sqrt(d)
  uint64_t dseed, doff;
  uint32_t dthr;
  float dscale;
  uint32_t* dmask;
  int mw, sp;
};

struct Item {
  int q0, h, b, n[2];  // first query row; head; batch; key tiles of tile A and B
};

// Item i: 256-row query blocks from the last (longest causal rows) to the
// first; within a block, the heads of a GQA group next to each other.
__device__ __forceinline__ Item item_of(int i, const Params& p) {
  const int nqp = (p.S + 2 * TQ - 1) / (2 * TQ), per = p.nq * p.B;
  Item it;
  it.q0 = (nqp - 1 - i / per) * 2 * TQ;
  const int hb = i % per;
  it.h = hb % p.nq;
  it.b = hb / p.nq;
  const int all = (p.S + TK - 1) / TK;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int r0 = it.q0 + x * TQ;
    if (r0 >= p.S) {
      it.n[x] = 0;
    } else {
      const int end = p.causal ? min(p.S, r0 + TQ) : p.S;
      it.n[x] = p.causal ? (end + TK - 1) / TK : all;
    }
  }
  return it;
}

// The item a CTA takes in its k-th round. Round k covers items k G .. k G +
// G - 1 (G CTAs); CTA c takes item k G + c in even rounds and k G + G - 1 - c
// in odd ones. With the items ordered from the longest causal rows down, a
// CTA that took a longer item in one round takes a shorter one in the next,
// so the CTAs' totals come out nearly equal (plain strides hand the first
// CTAs the longest item of every round: on 16 query blocks of a 4096-long
// causal sequence the busiest CTA then has 14 % more key tiles than the
// mean, against 1 % this way). Once k G + c passes the item count, every
// later round does too.
__device__ __forceinline__ int item_index(int k) {
  const int g = (int)gridDim.x, c = (int)blockIdx.x;
  return k * g + ((k & 1) ? g - 1 - c : c);
}

template <int D, bool DROP>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg2<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ[2] = {sb + C::OFF_QA, sb + C::OFF_QB};
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t q_full = bar;         // both Q tiles loaded                   (tx)
  const uint32_t q_empty = bar + 8;    // the item's last S product done        (commit)
  const uint32_t k_full0 = bar + 16;   // [2] K stage loaded                    (tx)
  const uint32_t k_empty0 = bar + 32;  // [2] S products with it done           (commit)
  const uint32_t v_full0 = bar + 48;   // [2] V stage loaded                    (tx)
  const uint32_t v_empty0 = bar + 64;  // [2] PV products with it done          (commit)
  const uint32_t s_full0 = bar + 80;   // [tile] S_X(j) complete                (commit)
  const uint32_t p_full0 = bar + 96;   // [tile] P_X(j) written, O_X rescaled   (4: one per warp)
  const uint32_t o_full0 = bar + 112;  // [tile] the item's last PV_X done      (commit)
  const uint32_t o_empty0 = bar + 128; // [tile] O_X read out                   (4: one per warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 240);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 244);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full0 + 8 * i, 1);
      mbar_init(k_empty0 + 8 * i, 1);
      mbar_init(v_full0 + 8 * i, 1);
      mbar_init(v_empty0 + 8 * i, 1);
      mbar_init(s_full0 + 8 * i, 1);
      mbar_init(p_full0 + 8 * i, NSOFT / 32);
      mbar_init(o_full0 + 8 * i, 1);
      mbar_init(o_empty0 + 8 * i, NSOFT / 32);
    }
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 1) {
    // ---------------- producer: per item Q_A, Q_B, then K_0, V_0, K_1, V_1, ...
    if (lane == 0) {
      int nk = 0, nv = 0;  // K / V tiles loaded so far (ring positions)
      for (int k = 0, i = item_index(0); i < p.n_items && !*abort; ++k, i = item_index(k)) {
        const Item w = item_of(i, p);
        const int grow0 = w.b * p.S;
        const int xcol = (w.h / (p.nq / p.nkv)) * D;
        // the item lies in the problem and the TMA x coordinates are 16-byte
        // multiples (head columns: multiples of 64)
        if (!dcheck(w.q0 >= 0 && w.q0 < p.S && w.b < p.B && w.h < p.nq && (xcol & 7) == 0 &&
                        ((w.h * D) & 7) == 0,
                    p.err)) {
          *abort = 1;
          break;
        }
        if (k >= 1 && !mbar_wait(q_empty, (k - 1) & 1, p.err)) {
          *abort = 1;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sQ[x] + kb * C::BOX, &tmQ, w.h * D + kb * 64, grow0 + w.q0 + x * TQ,
                        q_full);
        const int nt = max(w.n[0], w.n[1]);
        bool good = true;
        for (int j = 0; j < nt && good; ++j) {
          // K_j
          {
            const int s = nk % NSK;
            if (nk >= NSK && !mbar_wait(k_empty0 + 8 * s, ((nk - NSK) / NSK) & 1, p.err)) {
              good = false;
              break;
            }
            mbar_arrive_expect_tx(k_full0 + 8 * s, C::KV_BYTES);
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(sK + s * C::KV_BYTES + kb * C::BOX, &tmK, xcol + kb * 64, grow0 + j * TK,
                          k_full0 + 8 * s);
            ++nk;
          }
          // V_j
          {
            const int s = nv % NSV;
            if (nv >= NSV && !mbar_wait(v_empty0 + 8 * s, ((nv - NSV) / NSV) & 1, p.err)) {
              good = false;
              break;
            }
            mbar_arrive_expect_tx(v_full0 + 8 * s, C::KV_BYTES);
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(sV + s * C::KV_BYTES + kb * C::BOX, &tmV, xcol + kb * 64, grow0 + j * TK,
                          v_full0 + 8 * s);
            ++nv;
          }
        }
        if (!good) {
          *abort = 1;
          break;
        }
      }
    }
  } else if (warp == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(TQ, TK, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(TQ, D, 0, 1);
    const uint64_t dq0[2] = {smem_desc_sw128(sQ[0], 16, 1024), smem_desc_sw128(sQ[1], 16, 1024)};
    const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sV, C::BOX, 1024);
    int nk = 0, nv = 0;     // K / V tiles consumed so far
    int np[2] = {0, 0};     // PV products of each tile so far (p_full phases)
    int no[2] = {0, 0};     // items with a non-empty tile X so far (o_full / o_empty phases)
    bool good = true;
    // S_X = Q_X K^T into tile X's score columns (K stage sk)
    auto issue_s = [&](int x, int sk) {
      const uint64_t db = dk0 + (uint64_t)((sk * C::KV_BYTES) >> 4);
      const uint32_t td = tmem + C::COL_S + x * TK;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BOX + (kk & 3) * 32;
          tc_mma_f16(td, dq0[x] + (uint64_t)(off >> 4), db + (uint64_t)(off >> 4), idesc_s, kk > 0);
        }
        tc_commit(s_full0 + 8 * x);
      }
      __syncwarp();
    };
    // O_X += P_X V (P from tile X's score columns, V stage sv)
    auto issue_pv = [&](int x, int sv, bool acc) {
      const uint64_t db = dv0 + (uint64_t)((sv * C::KV_BYTES) >> 4);
      const uint32_t ta = tmem + C::COL_S + x * TK;
      const uint32_t to = tmem + C::COL_O + x * D;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < TK / 16; ++kk)
          tc_mma_f16_ts(to, ta + kk * 8, db + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                        (acc || kk > 0) ? 1u : 0u);
      }
      __syncwarp();
      ++np[x];
    };
    for (int k = 0, i = item_index(0); i < p.n_items && good; ++k, i = item_index(k)) {
      const Item w = item_of(i, p);
      const int nt = max(w.n[0], w.n[1]);
      if (warp_aborted(abort) || !warp_wait(q_full, k & 1, p.err)) {
        good = false;
        break;
      }
      // K_0 for both tiles' first scores
      {
        const int s = nk % NSK;
        if (!warp_wait(k_full0 + 8 * s, (nk / NSK) & 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (w.n[x] > 0) issue_s(x, s);
        if (elect_one()) {
          tc_commit(k_empty0 + 8 * s);
          if (nt == 1) tc_commit(q_empty);
        }
        __syncwarp();
        ++nk;
      }
      for (int j = 0; j < nt && good; ++j) {
        const int sv = nv % NSV;
        if (warp_aborted(abort) || !warp_wait(v_full0 + 8 * sv, (nv / NSV) & 1, p.err)) {
          good = false;
          break;
        }
        const bool next = j + 1 < nt;
        const int sk = nk % NSK;
        if (next && !warp_wait(k_full0 + 8 * sk, (nk / NSK) & 1, p.err)) {
          good = false;
          break;
        }
        for (int x = 0; x < 2 && good; ++x) {
          if (j >= w.n[x]) continue;
          // O_X of the previous item read out before this item's first PV_X
          if (j == 0 && no[x] >= 1 && !warp_wait(o_empty0 + 8 * x, (no[x] - 1) & 1, p.err)) {
            good = false;
            break;
          }
          if (!warp_wait(p_full0 + 8 * x, np[x] & 1, p.err)) {
            good = false;
            break;
          }
          tc_fence_after();
          issue_pv(x, sv, j > 0);
          if (j == w.n[x] - 1) {
            if (elect_one()) tc_commit(o_full0 + 8 * x);
            __syncwarp();
            ++no[x];
          } else {
            issue_s(x, sk);
          }
        }
        if (!good) break;
        if (elect_one()) {
          tc_commit(v_empty0 + 8 * sv);
          if (next) tc_commit(k_empty0 + 8 * sk);
        }
        __syncwarp();
        ++nv;
        if (next) ++nk;
        // the item's last score product has been issued once j + 1 == nt - 1
        if (next && j + 2 == nt) {
          if (elect_one()) tc_commit(q_empty);
          __syncwarp();
        }
      }
    }
    if (!good) *abort = 1;
  } else {
    // ---------------- softmax: warps 2-5 tile A, 6-9 tile B
    const int x = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                // row of the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t ts = tmem + C::COL_S + x * TK + lane_base;
    const uint32_t t_o = tmem + C::COL_O + x * D + lane_base;
    const uint32_t sfull = s_full0 + 8 * x, pfull = p_full0 + 8 * x;
    const uint32_t ofull = o_full0 + 8 * x, oempty = o_empty0 + 8 * x;
    bool good = true;
    int n = 0;   // S_X products consumed so far
    int ko = 0;  // items with a non-empty tile X so far
    for (int k = 0, i = item_index(0); i < p.n_items && good; ++k, i = item_index(k)) {
      const Item w = item_of(i, p);
      if (w.n[x] == 0) continue;  // tile past the sequence end: nothing to do
      const int row = w.q0 + x * TQ + r;
      const int row0 = w.q0 + x * TQ;  // first row of the tile
      float m_ref = -INFINITY, l = 0.0f;
      for (int j = 0; j < w.n[x]; ++j, ++n) {
        const int kv0 = j * TK;
        uint32_t kb[4] = {0u, 0u, 0u, 0u};
        if constexpr (DROP) {
          // keep bits of this row's 128 keys (8 blocks of the site's stream)
          const int64_t bh = (int64_t)w.b * p.nq + w.h;
          const uint64_t q = (p.doff + ((uint64_t)(bh * p.S + row)) * p.sp + kv0) >> 4;
#pragma unroll
          for (int gq = 0; gq < 8; ++gq) {
            const uint4 wd = philox_block(p.dseed, q + gq);
            const uint32_t ws[4] = {wd.x, wd.y, wd.z, wd.w};
            uint32_t bits = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) bits |= (uint32_t)keep_byte(ws[e >> 2], e & 3, p.dthr) << e;
            kb[gq >> 1] |= bits << (16 * (gq & 1));
          }
          const int wi = kv0 >> 5;
          if (row < p.S && wi < p.mw)
            *reinterpret_cast<uint4*>(p.dmask + (bh * p.S + row) * p.mw + wi) =
                make_uint4(kb[0], kb[1], kb[2], kb[3]);
        }
        if (warp_aborted(abort) || !warp_wait(sfull, n & 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        const bool interior = kv0 + TK <= p.S && (!p.causal || kv0 + TK - 1 <= row0);
        // The scores are read in chunks of CW keys (64 without dropout: two
        // TMEM round trips per pass; 32 with dropout, whose keep bits need
        // the registers). From the second key tile on (m_ref is then finite:
        // the first tile holds a visible key of every row) one pass: each
        // chunk's maximum is checked against the reference as it is read, and
        // only a chunk that exceeds it by more than TAU moves it, by a whole
        // number k of log2 units, so that the P already written for this tile
        // and the O row scale by 2^-k exactly. The first tile takes the row
        // maximum in a pass of its own.
        constexpr int CW = DROP ? 32 : 64;
        auto load_chunk = [&](int c, float (&sc)[CW]) {
          uint32_t qa[32];
          tmem_ld32(ts + c * CW, qa);
          if constexpr (CW == 64) {
            uint32_t qb[32];
            tmem_ld32(ts + c * CW + 32, qb);
            tmem_ld_wait();
            tmem_regs_ready(qb);
#pragma unroll
            for (int e = 0; e < 32; ++e) sc[32 + e] = __uint_as_float(qb[e]);
          } else {
            tmem_ld_wait();
          }
          tmem_regs_ready(qa);
#pragma unroll
          for (int e = 0; e < 32; ++e) sc[e] = __uint_as_float(qa[e]);
          if (!interior) {
#pragma unroll
            for (int e = 0; e < CW; ++e) {
              const int key = kv0 + c * CW + e;
              if (key >= p.S || (p.causal && key > row)) sc[e] = -INFINITY;
            }
          }
        };
        auto chunk_max = [&](const float (&sc)[CW], float m0) {
          float m4[4] = {m0, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < CW; e += 8) {
            m4[0] = fmax3(m4[0], sc[e], sc[e + 1]);
            m4[1] = fmax3(m4[1], sc[e + 2], sc[e + 3]);
            m4[2] = fmax3(m4[2], sc[e + 4], sc[e + 5]);
            m4[3] = fmax3(m4[3], sc[e + 6], sc[e + 7]);
          }
          return fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        };
        const bool one_pass = j > 0 && __all_sync(0xffffffffu, m_ref > -INFINITY);
        bool need = false;
        float alpha = 1.0f;
        if (!one_pass) {
          // pass 1: the row maximum over the 128 scores
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < TK / CW; ++c) {
            float sc[CW];
            load_chunk(c, sc);
            mx = chunk_max(sc, mx);
          }
          mx *= p.sl2;
          need = mx > m_ref + TAU;
          if (need) {
            alpha = exp2f(m_ref - mx);
            m_ref = mx;
            l *= alpha;
          }
        }
        float nref = m_ref == -INFINITY ? 0.0f : -m_ref;
        // pass 2: P = 2^(s log2e / sqrt(d) - m_ref) as bf16 pairs over the
        // tile's first 64 score columns (chunk c's keys -> columns c CW / 2 ..),
        // which only ever cover scores already read in this pass
        float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f, r3 = 0.0f;
#pragma unroll
        for (int c = 0; c < TK / CW; ++c) {
          float sc[CW];
          load_chunk(c, sc);
          if (one_pass) {
            const float cm = chunk_max(sc, -INFINITY) * p.sl2;
            const bool up = cm > m_ref + TAU;
            if (__any_sync(0xffffffffu, up)) {
              // this row's reference moves up by k: l, the P chunks already
              // written for this tile and (after the pass) O scale by 2^-k
              float a = 1.0f;
              if (up) {
                const float k = ceilf(cm - m_ref);
                a = k < 126.0f ? __int_as_float((127 - (int)k) << 23) : 0.0f;
                m_ref += k;
                l *= a;
                r0 *= a; r1 *= a; r2 *= a; r3 *= a;
                alpha *= a;
                need = true;
              }
              tmem_st_wait();  // the chunks' P stores have landed
              for (int g = 0; g < c * CW / 32; ++g) {
                uint32_t pw[16];
                tmem_ld16(ts + g * 16, pw);
                tmem_ld_wait();
                tmem_regs_ready(pw);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const float2 f = unpack_bf16x2(pw[e]);
                  pw[e] = pack_bf16x2(f.x * a, f.y * a);
                }
                tmem_st16(ts + g * 16, pw);
              }
              nref = -m_ref;
            }
          }
#pragma unroll
          for (int e = 0; e < CW; e += 4) {
            fma2(sc[e], sc[e + 1], sc[e], sc[e + 1], p.sl2, p.sl2, nref, nref);
            fma2(sc[e + 2], sc[e + 3], sc[e + 2], sc[e + 3], p.sl2, p.sl2, nref, nref);
            sc[e] = ex2_ftz(sc[e]);
            sc[e + 1] = ex2_ftz(sc[e + 1]);
            sc[e + 2] = ex2_ftz(sc[e + 2]);
            sc[e + 3] = ex2_ftz(sc[e + 3]);
            add2(r0, r1, r0, r1, sc[e], sc[e + 1]);
            add2(r2, r3, r2, r3, sc[e + 2], sc[e + 3]);
          }
          uint32_t pk[CW / 2];
          if constexpr (DROP) {
            const uint32_t kw = kb[c];
#pragma unroll
            for (int e = 0; e < CW / 2; ++e)
              pk[e] = pack_bf16x2((kw >> (2 * e)) & 1u ? sc[2 * e] * p.dscale : 0.0f,
                                  (kw >> (2 * e + 1)) & 1u ? sc[2 * e + 1] * p.dscale : 0.0f);
            tmem_st16(ts + c * 16, pk);
          } else {
#pragma unroll
            for (int e = 0; e < CW / 2; ++e) pk[e] = pack_bf16x2(sc[2 * e], sc[2 * e + 1]);
            tmem_st32(ts + c * 32, pk);
          }
        }
        l += (r0 + r1) + (r2 + r3);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // rescale this O_X row (PV_X(j - 1) completed before S_X(j) did)
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ro[32];
            tmem_ld32(t_o + c * 32, ro);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
            tmem_st32(t_o + c * 32, ro);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // the warp's P stores are done: one arrival for the warp
        if (lane == 0) mbar_arrive(pfull);
      }
      if (!good) break;
      // ---- tile done: O / l and LSE
      if (!warp_wait(ofull, ko & 1, p.err)) {
        good = false;
        break;
      }
      ++ko;
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const bool row_ok = row < p.S;
      bf16* out = p.o + (int64_t)(w.b * p.S + row) * p.ld_o + w.h * D;
      store_tmem_row<D>(t_o, inv, row_ok ? out : nullptr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(oempty);
      if (row_ok) p.lse[((int64_t)w.b * p.nq + w.h) * p.S + row] = (m_ref + log2f(l)) * LN2;
    }
    if (!good) *abort = 1;
  }
  __syncthreads();
  if (*abort && tid == 0) spin_10ms();  // let work and copies still in flight finish
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool DROP>
mgb_status fwd2_d(const AttnArgs& a, cudaStream_t st) {
  using C = Cfg2<D>;
  const uint64_t T = (uint64_t)a.B * a.S;
  const int n_items = a.B * a.nq * ((a.S + 2 * TQ - 1) / (2 * TQ));
  if (n_items == 0) return MGB_OK;
  CUtensorMap tq, tk, tv;
  if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TQ) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TK) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TK) != CUDA_SUCCESS)
    return MGB_ERR_CUDA;
  Params p{};
  p.B = a.B; p.S = a.S; p.nq = a.nq; p.nkv = a.nkv; p.causal = a.causal;
  p.n_items = n_items;
  p.o = reinterpret_cast<bf16*>(a.o); p.ld_o = a.ld_o; p.lse = a.lse;
  p.err = device_error_word();
  p.sl2 = LOG2E / sqrtf((float)D);
  p.dseed = a.drop_seed; p.doff = a.drop_offset; p.dthr = a.drop_thr; p.dscale = a.drop_scale;
  p.dmask = a.drop_mask; p.mw = attn_mask_words(a.S); p.sp = (a.S + 15) / 16 * 16;
  auto k = attn_fwd2_kernel<D, DROP>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return MGB_ERR_CUDA;
  const int grid = n_items < device_sm_count() ? n_items : device_sm_count();
  k<<<grid, NTHREADS, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

mgb_status attention_tc2_fwd(const AttnArgs& a, cudaStream_t st) {
  const bool drop = a.drop_thr < 256;
  if (drop && (a.drop_mask == nullptr || a.drop_offset % 16 || a.drop_thr == 0))
    return MGB_ERR_INVALID_ARG;
  if (a.d == 64) return drop ? fwd2_d<64, true>(a, st) : fwd2_d<64, false>(a, st);
  if (a.d == 128) return drop ? fwd2_d<128, true>(a, st) : fwd2_d<128, false>(a, st);
  return MGB_ERR_UNSUPPORTED;
}

}  // namespace mgb

// bf16 attention forward on the 5th-generation tensor cores (tcgen05).
//
// Definition ("LLM Lab 06: build a Megatron-style Transformer Block from
// scratch", section 2; "02 - How a whole Transformer block is split",
// section 2): O_h = softmax(Q_h K_g^T / sqrt(d)) V_g per batch and query head h,
// g = h / (nq / nkv), optional causal mask; LSE = log sum_j exp(s_j) is saved
// for the backward. FlashAttention-style (page 1, section 5): the [S, S] score
// matrix never leaves the chip.
//
// Persistent and warp-specialised. A work item is 128 query rows of one
// (batch, head); items are ordered longest causal rows first and dealt
// round-robin to one CTA per SM. Keys come in tiles of 128, so every product
// is a full-width tcgen05.mma (N = 128: N = 64 products run at two thirds of
// the rate) and each hand-off between the warps moves 128 keys of work.
// Ten warps:
//   warp 0     MMA issuer; the whole warp runs the loop (its values stay
//              warp-uniform) and one elected lane issues each instruction:
//                S = Q K^T   M=128 N=128 K=d  -> TMEM score buffer n & 1
//                O += P V    M=128 N=d K=128  -> TMEM O, with P read from TMEM
//              S(n+2) is issued as soon as the softmax warps have loaded S(n)
//              out of TMEM, so it runs while they exponentiate tile n
//   warp 1     producer: each item's Q and its K and V tiles by TMA with
//              128-byte swizzle, in separate rings (K: 3 stages, V: 2), K up to
//              three tiles ahead of V (the score products run ahead of the PV
//              products); a slot is refilled as soon as its own reader is done
//   warps 2-9  softmax: warps w and w+4 own TMEM lane quarter w % 4 (32 query
//              rows, thread = row). Both read the whole 128-column score row,
//              so they take the same running-max decision without exchanging
//              it; each exponentiates its own 64 columns into P (bf16 pairs
//              stored to a double-buffered TMEM tile, the A operand of PV) and
//              keeps its own partial row sum.
// Online softmax in the log2 domain with a lazy reference: the reference max of
// a row moves only when a tile's max exceeds it by more than TAU, so P stays
// below 2^TAU (harmless for bf16 P and the float32 accumulator). Only then are
// the row sums and the TMEM O row rescaled. O / l and LSE = ln2 (m_ref +
// log2 l) do not depend on which reference was used. When an item's last PV
// lands, the softmax warps normalise O out of TMEM, store it (bf16) and LSE,
// and release O; the MMA warp has meanwhile started the next item's score
// products. Q and K are K-major operands; the V tile bytes are read as an
// MN-major operand (d contiguous). Every wait is bounded: one that runs out
// sets a shared abort flag and every role leaves its loop before the closing
// barrier.
// Dropout on the probabilities ("02 - How a whole Transformer block is split",
// section 5: inside the tensor-parallel region), the DROP variant: after the
// row sums take the undropped P, each softmax thread draws its 64 keys' keep
// bytes (element ((b*nq + h)*S + row)*Sp + key of the site's Philox stream:
// four 16-byte blocks), zeroes the dropped probabilities and scales the kept
// ones before P goes to TMEM, and writes the 64 keep bits for the backward.
#include "common.cuh"
#include "internal.h"

namespace mgb {

CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int TQ = 128;        // query rows per item (TMEM lanes)
constexpr int TK = 128;        // keys per KV tile
constexpr int NSK = 3;         // K ring stages
constexpr int NSV = 2;         // V ring stages
constexpr int NCOMPUTE = 256;  // softmax threads (warps 2-9)
constexpr int NTHREADS = 320;  // + MMA warp 0 + producer warp 1
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float TAU = 8.0f;    // lazy-rescale threshold (log2 units)

template <int D>
struct FwdCfg {
  static constexpr int KB = D / 64;                     // 64-wide d blocks
  static constexpr int Q_BYTES = TQ * D * 2;            // KB boxes of [128 rows][64]
  static constexpr int KV_BYTES = TK * D * 2;           // KB boxes of [128 keys][64]
  static constexpr int BOX = 128 * 128;                 // bytes of one [128][64] box
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;         // NSK stages
  static constexpr int OFF_V = OFF_K + NSK * KV_BYTES;  // NSV stages
  static constexpr int OFF_L = OFF_V + NSV * KV_BYTES;  // [2 items][2 halves][128] f32
  static constexpr int OFF_BAR = OFF_L + 4 * TQ * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;     // barriers + alignment slack
  // TMEM columns: two score buffers, O, two P buffers (128 bf16 keys = 64 columns)
  static constexpr int COL_O = 2 * TK;
  static constexpr int COL_P = 384;
  static constexpr int TMEM_COLS = 512;
  static_assert(COL_O + D <= COL_P, "O overlaps P in TMEM");
};

struct FwdParams {
  int B, S, nq, nkv, causal, n_items;
  bf16* o;
  int64_t ld_o;
  float* lse;
  int* err;
  float sl2;  // log2(e) / sqrt(d)
  // dropout (DROP variant)
  uint64_t dseed, doff;
  uint32_t dthr;
  float dscale;
  uint32_t* dmask;
  int mw, sp;  // mask words per row; Sp
};

struct Item {
  int q0, h, b, nkt;
};

// Item i: query tile from the last (longest causal rows) to the first; within
// a tile, heads of a GQA group next to each other so they share K/V in L2.
__device__ __forceinline__ Item item_of(int i, const FwdParams& p) {
  const int nqt = (p.S + TQ - 1) / TQ, per = p.nq * p.B;
  Item it;
  it.q0 = (nqt - 1 - i / per) * TQ;
  const int hb = i % per;
  it.h = hb % p.nq;
  it.b = hb / p.nq;
  const int kv_end = p.causal ? min(p.S, it.q0 + TQ) : p.S;
  it.nkt = (kv_end + TK - 1) / TK;
  return it;
}

template <int D, bool DROP>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  float* sL = reinterpret_cast<float*>(smem + C::OFF_L);
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t q_full = bar;          // Q loaded                        (tx)
  const uint32_t q_empty = bar + 8;     // last S of its item done         (commit)
  const uint32_t k_full0 = bar + 16;    // [3] K stage loaded              (tx)
  const uint32_t k_empty0 = bar + 40;   // [3] score product of it done    (commit)
  const uint32_t v_full0 = bar + 64;    // [2] V stage loaded              (tx)
  const uint32_t v_empty0 = bar + 80;   // [2] PV product of it done       (commit)
  const uint32_t s_full0 = bar + 96;    // [2] score buffer ready          (commit)
  const uint32_t s_free0 = bar + 112;   // [2] score buffer read out       (256 arrivals)
  const uint32_t p_full0 = bar + 128;   // [2] P buffer written            (256 arrivals)
  const uint32_t pv_done0 = bar + 144;  // [2] PV that read P buffer done  (commit)
  const uint32_t o_full = bar + 160;    // item's last PV done             (commit)
  const uint32_t o_empty = bar + 168;   // O read out                      (256 arrivals)
  const uint32_t l_ready0 = bar + 176;  // [4 quarters][2] row sums exchanged (64 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 240);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 244);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int stride = gridDim.x;

  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NSK; ++i) {
      mbar_init(k_full0 + 8 * i, 1);
      mbar_init(k_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(v_full0 + 8 * i, 1);
      mbar_init(v_empty0 + 8 * i, 1);
      mbar_init(s_full0 + 8 * i, 1);
      mbar_init(s_free0 + 8 * i, NCOMPUTE);
      mbar_init(p_full0 + 8 * i, NCOMPUTE);
      mbar_init(pv_done0 + 8 * i, 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, NCOMPUTE);
    for (int i = 0; i < 8; ++i) mbar_init(l_ready0 + 8 * i, 64);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 1) {
    // ---------------- producer
    if (lane == 0) {
      // two cursors over this CTA's (item, tile) sequence: K runs up to NSK
      // tiles ahead of V; an item's Q is loaded right before its first K tile (the
      // item decode, integer divisions, is done once per item)
      struct Cursor {
        int i, k, j, n;
        Item w;
        int grow0, xcol;  // first token row of the batch; first K/V column of the group
      };
      auto set_item = [&](Cursor& c) {
        if (c.i >= p.n_items) return;
        c.w = item_of(c.i, p);
        c.grow0 = c.w.b * p.S;
        c.xcol = (c.w.h / (p.nq / p.nkv)) * D;
      };
      Cursor ck{(int)blockIdx.x, 0, 0, 0, {}, 0, 0};
      set_item(ck);
      Cursor cv = ck;
      auto advance = [&](Cursor& c) {
        ++c.n;
        if (++c.j == c.w.nkt) {
          c.j = 0;
          ++c.k;
          c.i += stride;
          set_item(c);
        }
      };
      while ((ck.i < p.n_items || cv.i < p.n_items) && !*abort) {
        const bool do_k = ck.i < p.n_items && ck.n < cv.n + NSK;
        Cursor& c = do_k ? ck : cv;
        if (do_k) {
          if (c.j == 0) {
            // Q of item k once the last score product of item k - 1 is done
            if (c.k >= 1 && !mbar_wait(q_empty, (c.k - 1) & 1, p.err)) {
              *abort = 1;
              break;
            }
            mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(sQ + kb * C::BOX, &tmQ, c.w.h * D + kb * 64, c.grow0 + c.w.q0, q_full);
          }
          const int s = c.n % NSK;
          if (c.n >= NSK && !mbar_wait(k_empty0 + 8 * s, ((c.n - NSK) / NSK) & 1, p.err)) {
            *abort = 1;
            break;
          }
          const uint32_t fb = k_full0 + 8 * s;
          mbar_arrive_expect_tx(fb, C::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sK + s * C::KV_BYTES + kb * C::BOX, &tmK, c.xcol + kb * 64,
                        c.grow0 + c.j * TK, fb);
        } else {
          const int s = c.n % NSV;
          if (c.n >= NSV && !mbar_wait(v_empty0 + 8 * s, ((c.n - NSV) / NSV) & 1, p.err)) {
            *abort = 1;
            break;
          }
          const uint32_t fb = v_full0 + 8 * s;
          mbar_arrive_expect_tx(fb, C::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sV + s * C::KV_BYTES + kb * C::BOX, &tmV, c.xcol + kb * 64,
                        c.grow0 + c.j * TK, fb);
        }
        advance(c);
      }
    }
  } else if (warp == 0) {
    // ---------------- MMA issuer
    // Shared-memory descriptors are built once: a tile's descriptor is the
    // base descriptor plus its byte offset / 16 (a constant per MMA).
    constexpr uint32_t idesc_s = idesc_bf16_f32(TQ, TK, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(TQ, D, 0, 1);
    const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024), dk0 = smem_desc_sw128(sK, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sV, C::BOX, 1024);
    const uint32_t t_o = tmem + C::COL_O;
    // score-product cursor: item index si (k-th of this CTA), tile sj, global tile sn
    int si = blockIdx.x, sk = 0, sj = 0, sn = 0;
    int s_nkt = si < p.n_items ? item_of(si, p).nkt : 0;
    auto issue_s = [&]() -> bool {
      if (si >= p.n_items) return true;
      if (sj == 0 && !warp_wait(q_full, sk & 1, p.err)) return false;
      const int s = sn % NSK;
      if (!warp_wait(k_full0 + 8 * s, (sn / NSK) & 1, p.err)) return false;
      tc_fence_after();
      const uint64_t da = dq0;
      const uint64_t db = dk0 + (uint64_t)((s * C::KV_BYTES) >> 4);
      const uint32_t td = tmem + (sn & 1) * TK;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BOX + (kk & 3) * 32;  // d block, K step inside it
          tc_mma_f16(td, da + (uint64_t)(off >> 4), db + (uint64_t)(off >> 4), idesc_s, kk > 0);
        }
        tc_commit(s_full0 + 8 * (sn & 1));
        tc_commit(k_empty0 + 8 * s);
        if (sj == s_nkt - 1) tc_commit(q_empty);
      }
      __syncwarp();
      ++sn;
      if (++sj == s_nkt) {
        sj = 0;
        ++sk;
        si += stride;
        s_nkt = si < p.n_items ? item_of(si, p).nkt : 0;
      }
      return true;
    };
    bool good = issue_s() && issue_s();
    int n = 0;  // global tile of the PV product
    for (int k = 0, i = blockIdx.x; i < p.n_items && good; ++k, i += stride) {
      const int nkt = item_of(i, p).nkt;
      for (int j = 0; j < nkt; ++j, ++n) {
        // score buffer n & 1 read out by the softmax warps: S(n + 2) goes into it
        if (warp_aborted(abort) || !warp_wait(s_free0 + 8 * (n & 1), (n >> 1) & 1, p.err) ||
            !issue_s()) {
          good = false;
          break;
        }
        // O of the previous item read out (before this item's first PV)
        if (j == 0 && k >= 1 && !warp_wait(o_empty, (k - 1) & 1, p.err)) {
          good = false;
          break;
        }
        if (!warp_wait(p_full0 + 8 * (n & 1), (n >> 1) & 1, p.err) ||
            !warp_wait(v_full0 + 8 * (n % NSV), (n / NSV) & 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        const uint64_t db = dv0 + (uint64_t)(((n % NSV) * C::KV_BYTES) >> 4);
        const uint32_t ta = tmem + C::COL_P + (n & 1) * (TK / 2);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk)
            tc_mma_f16_ts(t_o, ta + kk * 8, db + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                          (j > 0 || kk > 0));
          tc_commit(pv_done0 + 8 * (n & 1));
          tc_commit(v_empty0 + 8 * (n % NSV));
          if (j == nkt - 1) tc_commit(o_full);
        }
        __syncwarp();
      }
    }
    if (!good) *abort = 1;
  } else {
    // ---------------- softmax warps 2-9
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // this thread's row of the item
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int c_own = half * 64, c_oth = (1 - half) * 64;  // column halves of a tile
    bool good = true;
    int n = 0;
    for (int k = 0, i = blockIdx.x; i < p.n_items && good; ++k, i += stride) {
      const Item w = item_of(i, p);
      const int row = w.q0 + r;
      const uint32_t t_o = tmem + C::COL_O + half * (D / 2) + lane_base;
      float m_ref = -INFINITY, l_part = 0.0f;
      for (int j = 0; j < w.nkt; ++j, ++n) {
        const int kv0 = j * TK;
        // dropout: keep bits of this thread's 64 keys (4 blocks of the site's
        // stream), drawn while the scores are computed and stored for the
        // backward (bit c of kb0 / kb1: key kv0 + c_own + c / 32 + c)
        uint32_t kb0 = 0, kb1 = 0;
        if constexpr (DROP) {
          const int64_t bh = (int64_t)w.b * p.nq + w.h;
          const uint64_t q = (p.doff + ((uint64_t)(bh * p.S + row)) * p.sp + kv0 + c_own) >> 4;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const uint4 wd = philox_block(p.dseed, q + gq);
            const uint32_t ws[4] = {wd.x, wd.y, wd.z, wd.w};
            uint32_t bits = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) bits |= (uint32_t)keep_byte(ws[i >> 2], i & 3, p.dthr) << i;
            if (gq < 2) kb0 |= bits << (16 * gq);
            else kb1 |= bits << (16 * (gq - 2));
          }
          const int wi = (kv0 + c_own) >> 5;
          if (row < p.S && wi < p.mw)
            *reinterpret_cast<uint2*>(p.dmask + (bh * p.S + row) * p.mw + wi) = make_uint2(kb0, kb1);
        }
        if (warp_aborted(abort) || !warp_wait(s_full0 + 8 * (n & 1), (n >> 1) & 1, p.err)) {
          good = false;
          break;
        }
        tc_fence_after();
        // the partner's 64 columns first, reduced to their max (so only 64
        // scores are live at a time), then this thread's own 64
        const uint32_t ts = tmem + (n & 1) * TK + lane_base;
        const bool interior = kv0 + TK <= p.S && (!p.causal || kv0 + TK - 1 <= w.q0);
        float mo;
        {
          float sx[64];
          ld_cols32(ts + c_oth, *reinterpret_cast<float(*)[32]>(&sx[0]));
          ld_cols32(ts + c_oth + 32, *reinterpret_cast<float(*)[32]>(&sx[32]));
          if (!interior) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int kx = kv0 + c_oth + c;
              if (kx >= p.S || (p.causal && kx > row)) sx[c] = -INFINITY;
            }
          }
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            m4[0] = fmax3(m4[0], sx[c], sx[c + 1]);
            m4[1] = fmax3(m4[1], sx[c + 2], sx[c + 3]);
            m4[2] = fmax3(m4[2], sx[c + 4], sx[c + 5]);
            m4[3] = fmax3(m4[3], sx[c + 6], sx[c + 7]);
          }
          mo = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        }
        float so[64];
        ld_cols32(ts + c_own, *reinterpret_cast<float(*)[32]>(&so[0]));
        ld_cols32(ts + c_own + 32, *reinterpret_cast<float(*)[32]>(&so[32]));
        if (!interior) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int ko = kv0 + c_own + c;
            if (ko >= p.S || (p.causal && ko > row)) so[c] = -INFINITY;
          }
        }
        // score buffer n & 1 is read out: the MMA warp may compute S(n + 2) into it
        tc_fence_before();
        mbar_arrive(s_free0 + 8 * (n & 1));
        // row max over all 128 columns: four independent three-input chains
        float m4[4] = {mo, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          m4[0] = fmax3(m4[0], so[c], so[c + 1]);
          m4[1] = fmax3(m4[1], so[c + 2], so[c + 3]);
          m4[2] = fmax3(m4[2], so[c + 4], so[c + 5]);
          m4[3] = fmax3(m4[3], so[c + 6], so[c + 7]);
        }
        const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]) * p.sl2;
        const bool need = mx > m_ref + TAU;
        float alpha = 1.0f;
        if (need) {
          alpha = exp2f(m_ref - mx);
          m_ref = mx;
          l_part *= alpha;
        }
        const float nref = m_ref == -INFINITY ? 0.0f : -m_ref;
        // P = 2^(s * log2e / sqrt(d) - m_ref), two columns per float32x2 op
        float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f, r3 = 0.0f;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          fma2(so[c], so[c + 1], so[c], so[c + 1], p.sl2, p.sl2, nref, nref);
          fma2(so[c + 2], so[c + 3], so[c + 2], so[c + 3], p.sl2, p.sl2, nref, nref);
          so[c] = ex2_ftz(so[c]);
          so[c + 1] = ex2_ftz(so[c + 1]);
          so[c + 2] = ex2_ftz(so[c + 2]);
          so[c + 3] = ex2_ftz(so[c + 3]);
          add2(r0, r1, r0, r1, so[c], so[c + 1]);
          add2(r2, r3, r2, r3, so[c + 2], so[c + 3]);
        }
        l_part += (r0 + r1) + (r2 + r3);
        // this half's 64 keys of P as bf16 pairs: 32 TMEM columns of P buffer n & 1
        uint32_t pk[32];
        if constexpr (DROP) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t kw = c < 16 ? kb0 : kb1, sh = (2 * c) & 31;
            pk[c] = pack_bf16x2((kw >> sh) & 1u ? so[2 * c] * p.dscale : 0.0f,
                                (kw >> (sh + 1)) & 1u ? so[2 * c + 1] * p.dscale : 0.0f);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(so[2 * c], so[2 * c + 1]);
        }
        // P buffer n & 1 was last read by the PV product of tile n - 2
        if (n >= 2 && !warp_wait(pv_done0 + 8 * (n & 1), ((n - 2) >> 1) & 1, p.err)) {
          good = false;
          break;
        }
        tmem_st32(tmem + C::COL_P + (n & 1) * (TK / 2) + half * 32 + lane_base, pk);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // rescale this half of the O rows once PV of tile n - 1 has landed
          if (!warp_wait(pv_done0 + 8 * ((n - 1) & 1), ((n - 1) >> 1) & 1, p.err)) {
            good = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t ro[32];
            tmem_ld32(t_o + c * 32, ro);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) ro[q] = __float_as_uint(__uint_as_float(ro[q]) * alpha);
            tmem_st32(t_o + c * 32, ro);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full0 + 8 * (n & 1));
      }
      if (!good) break;
      // ---- item done: exchange the half row sums, normalise and store O, LSE
      const uint32_t lr = l_ready0 + 8 * (quarter * 2 + (k & 1));
      float* lsl = sL + (k & 1) * 2 * TQ;
      lsl[half * TQ + r] = l_part;
      mbar_arrive(lr);
      if (!warp_wait(lr, (k >> 1) & 1, p.err) || !warp_wait(o_full, k & 1, p.err)) {
        good = false;
        break;
      }
      tc_fence_after();
      const float l = lsl[r] + lsl[TQ + r];
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const bool row_ok = row < p.S;
      bf16* out = p.o + (int64_t)(w.b * p.S + row) * p.ld_o + w.h * D + half * (D / 2);
      store_tmem_row<D / 2>(t_o, inv, row_ok ? out : nullptr);
      tc_fence_before();
      mbar_arrive(o_empty);
      if (half == 0 && row_ok)
        p.lse[((int64_t)w.b * p.nq + w.h) * p.S + row] = (m_ref + log2f(l)) * LN2;
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
mgb_status fwd_tc_d(const AttnArgs& a, cudaStream_t st) {
  using C = FwdCfg<D>;
  const uint64_t T = (uint64_t)a.B * a.S;
  const int n_items = a.B * a.nq * ((a.S + TQ - 1) / TQ);
  if (n_items == 0) return MGB_OK;
  CUtensorMap tq, tk, tv;
  if (tmap_encode_bf16_2d(&tq, a.q, (uint64_t)a.nq * D, T, a.ld_q, 64, TQ) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tk, a.k, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TK) != CUDA_SUCCESS ||
      tmap_encode_bf16_2d(&tv, a.v, (uint64_t)a.nkv * D, T, a.ld_kv, 64, TK) != CUDA_SUCCESS)
    return MGB_ERR_CUDA;
  FwdParams p{};
  p.B = a.B; p.S = a.S; p.nq = a.nq; p.nkv = a.nkv; p.causal = a.causal;
  p.n_items = n_items;
  p.o = reinterpret_cast<bf16*>(a.o); p.ld_o = a.ld_o; p.lse = a.lse;
  p.err = device_error_word();
  p.sl2 = LOG2E / sqrtf((float)D);
  p.dseed = a.drop_seed; p.doff = a.drop_offset; p.dthr = a.drop_thr; p.dscale = a.drop_scale;
  p.dmask = a.drop_mask; p.mw = attn_mask_words(a.S); p.sp = (a.S + 15) / 16 * 16;
  auto k = attn_fwd_tc_kernel<D, DROP>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return MGB_ERR_CUDA;
  const int grid = n_items < device_sm_count() ? n_items : device_sm_count();
  k<<<grid, NTHREADS, C::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

mgb_status attention_tc2_fwd(const AttnArgs& a, cudaStream_t st);

// Two query tiles per work item (attention_tc2.cu) unless MGB_ATTN_FWD=1 picks
// the one-tile kernel above.
mgb_status attention_tc_fwd(const AttnArgs& a, cudaStream_t st) {
  const char* v = getenv("MGB_ATTN_FWD");
  if (!(v != nullptr && v[0] == '1')) return attention_tc2_fwd(a, st);
  const bool drop = a.drop_thr < 256;
  if (drop && (a.drop_mask == nullptr || a.drop_offset % 16 || a.drop_thr == 0))
    return MGB_ERR_INVALID_ARG;
  if (a.d == 64) return drop ? fwd_tc_d<64, true>(a, st) : fwd_tc_d<64, false>(a, st);
  if (a.d == 128) return drop ? fwd_tc_d<128, true>(a, st) : fwd_tc_d<128, false>(a, st);
  return MGB_ERR_UNSUPPORTED;
}

}  // namespace mgb

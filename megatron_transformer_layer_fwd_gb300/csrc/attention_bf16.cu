// bf16 attention core: fused online-softmax forward and recompute backward.
//
// Definition ("LLM Lab 06: build a Megatron-style Transformer Block from
// scratch", section 2; "02 - How a whole Transformer block is split",
// section 2): per batch b and query head h, O_h = softmax(Q_h K_g^T / sqrt(d)) V_g
// with g = h / (nq / nkv) (GQA), optional causal mask (key j visible to query i
// iff j <= i). Page 1 section 5 points at FlashAttention for this step: the
// [S, S] score matrix never leaves the chip. KV tiles of 64 keys stream
// through shared memory; each query row keeps a running max m and sum l, and
// the output accumulator is rescaled by exp(m_old - m_new) when the max grows.
// The forward saves LSE = m + log l per row.
//
// Backward from the saved LSE (P = exp(S - LSE) recomputed; D = rowsum(dO*O)):
//   dV_g = sum_h P^T dO_h,  dS = P * (dO V^T - D),
//   dK_g = sum_h dS^T Q_h / sqrt(d),  dQ_h = dS K_g / sqrt(d).
// Kernel A (one CTA per 64-key tile of one KV head) loops over every query
// head of its group and every query tile, so the GQA sum happens on chip and
// needs no atomics. Kernel B (one CTA per 64-query tile of one head) forms dQ.
//
// Matrix products use the warp-level bf16 tensor-core instruction
// (mma.sync m16n8k16, float32 accumulate); each warp owns 16 rows of the tile.
// Shared-memory tiles are [64 rows][d] bf16 with 16-byte chunks XOR-swizzled
// by (row & 7), so 8-row ldmatrix accesses hit distinct banks.
#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

constexpr int BT = 64;  // rows of a Q tile and of a KV tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// byte offset of 16-byte chunk `ch` of row `r` in a swizzled [*, D] bf16 tile
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  return (uint32_t)(r * D * 2 + ((ch ^ (r & 7)) << 4));
}

// Async copy of rows [row0, row0+BT) of a [*, D] slice (row stride ld elements)
// into a swizzled tile; rows >= nrows are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t tile, const bf16* base, int64_t ld, int row0,
                                          int nrows) {
  constexpr int CH = D / 8;
  for (int i = threadIdx.x; i < BT * CH; i += blockDim.x) {
    const int r = i / CH, ch = i % CH;
    const int gr = row0 + r;
    const bool ok = gr < nrows;
    const bf16* src = base + (int64_t)(ok ? gr : 0) * ld + ch * 8;
    cp_async16(tile + swz<D>(r, ch), src, ok);
  }
}

// A fragments (16 rows x 16 k) of a warp's 16-row strip of a swizzled tile.
template <int D>
__device__ __forceinline__ void ld_a(uint32_t tile, int row_base, int kstep, uint32_t (&a)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = row_base + (lane & 15);
  const int ch = kstep * 2 + (lane >> 4);
  ldsm_x4(tile + swz<D>(r, ch), a[0], a[1], a[2], a[3]);
}
// B fragments for two n8 tiles (rows n0..n0+15 of the tile are the n index,
// columns = k), i.e. B = tile^T: returns {b0,b1} of n-tile 0 and of n-tile 1.
template <int D>
__device__ __forceinline__ void ld_b_nt(uint32_t tile, int n0, int kstep, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = n0 + ((lane >> 4) << 3) + (lane & 7);
  const int ch = kstep * 2 + ((lane >> 3) & 1);
  ldsm_x4(tile + swz<D>(r, ch), b[0], b[1], b[2], b[3]);
}
// B fragments where the tile rows are the k index and columns (d) the n index:
// k rows k0..k0+15, n columns n0..n0+15 (two n8 tiles).
template <int D>
__device__ __forceinline__ void ld_b_kn(uint32_t tile, int k0, int n0, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const int r = k0 + (((lane >> 3) & 1) << 3) + (lane & 7);
  const int ch = (n0 >> 3) + (lane >> 4);
  ldsm_x4_t(tile + swz<D>(r, ch), b[0], b[1], b[2], b[3]);
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Copy a warp's 16 x D float accumulator strip (mma C layout) to global bf16
// through the warp's rows of a swizzled smem tile.
template <int D>
__device__ __forceinline__ void store_strip(uint32_t tile, int row_base, const float (*acc)[4],
                                            float scale_a, float scale_b, bf16* out, int64_t ld,
                                            int grow0, int nrows) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint8_t* base = reinterpret_cast<uint8_t*>(__cvta_shared_to_generic(tile));
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + 2 * t;
    const int ra = row_base + g, rb = ra + 8;
    *reinterpret_cast<uint32_t*>(base + swz<D>(ra, col >> 3) + (col & 7) * 2) =
        pack_bf16x2(acc[nt][0] * scale_a, acc[nt][1] * scale_a);
    *reinterpret_cast<uint32_t*>(base + swz<D>(rb, col >> 3) + (col & 7) * 2) =
        pack_bf16x2(acc[nt][2] * scale_b, acc[nt][3] * scale_b);
  }
  __syncwarp();
  constexpr int CH = D / 8;
  for (int i = lane; i < 16 * CH; i += 32) {
    const int r = i / CH, ch = i % CH;
    const int gr = grow0 + row_base + r;
    if (gr < nrows)
      *reinterpret_cast<uint4*>(out + (int64_t)gr * ld + ch * 8) =
          *reinterpret_cast<const uint4*>(base + swz<D>(row_base + r, ch));
  }
}

// ------------------------------------------------------------------ forward
template <int D>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sQ = smem_u32(sm);
  const uint32_t sK0 = sQ + BT * D * 2;
  const uint32_t sV0 = sK0 + 2 * BT * D * 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nqt = (a.S + BT - 1) / BT;
  const int qt = nqt - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (a.nq / a.nkv);
  const int q0 = qt * BT;
  const bf16* Q = reinterpret_cast<const bf16*>(a.q) + (int64_t)b * a.S * a.ld_q + h * D;
  const bf16* K = reinterpret_cast<const bf16*>(a.k) + (int64_t)b * a.S * a.ld_kv + kvh * D;
  const bf16* V = reinterpret_cast<const bf16*>(a.v) + (int64_t)b * a.S * a.ld_kv + kvh * D;
  const int kv_end = a.causal ? min(a.S, q0 + BT) : a.S;
  const int nkt = (kv_end + BT - 1) / BT;
  const float sl2 = rsqrtf((float)D) * LOG2E;

  load_tile<D>(sQ, Q, a.ld_q, q0, a.S);
  load_tile<D>(sK0, K, a.ld_kv, 0, a.S);
  load_tile<D>(sV0, V, a.ld_kv, 0, a.S);
  cp_commit();

  uint32_t qf[D / 16][4];
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;

  for (int j = 0; j < nkt; ++j) {
    const int buf = j & 1;
    if (j + 1 < nkt) {
      load_tile<D>(sK0 + (buf ^ 1) * BT * D * 2, K, a.ld_kv, (j + 1) * BT, a.S);
      load_tile<D>(sV0 + (buf ^ 1) * BT * D * 2, V, a.ld_kv, (j + 1) * BT, a.S);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) ld_a<D>(sQ, warp * 16, ks, qf[ks]);
    }
    const uint32_t sK = sK0 + buf * BT * D * 2, sV = sV0 + buf * BT * D * 2;
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        ld_b_nt<D>(sK, np * 16, ks, bb);
        mma16816(s[2 * np], qf[ks], bb[0], bb[1]);
        mma16816(s[2 * np + 1], qf[ks], bb[2], bb[3]);
      }
    }
    // scale, mask, row max
    const int kv0 = j * BT;
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kv = kv0 + nt * 8 + 2 * t + e;
        const bool bad = kv >= a.S;
        s[nt][e] = (bad || (a.causal && kv > row_a)) ? -INFINITY : s[nt][e] * sl2;
        s[nt][2 + e] = (bad || (a.causal && kv > row_b)) ? -INFINITY : s[nt][2 + e] * sl2;
        mx_a = fmaxf(mx_a, s[nt][e]);
        mx_b = fmaxf(mx_b, s[nt][2 + e]);
      }
    }
    mx_a = quad_max(mx_a);
    mx_b = quad_max(mx_b);
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float ref_a = mn_a == -INFINITY ? 0.0f : mn_a;
    const float ref_b = mn_b == -INFINITY ? 0.0f : mn_b;
    const float al_a = exp2f(m_a - ref_a), al_b = exp2f(m_b - ref_b);
    m_a = mn_a;
    m_b = mn_b;
    float rs_a = 0.0f, rs_b = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - ref_a);
      s[nt][1] = exp2f(s[nt][1] - ref_a);
      s[nt][2] = exp2f(s[nt][2] - ref_b);
      s[nt][3] = exp2f(s[nt][3] - ref_b);
      rs_a += s[nt][0] + s[nt][1];
      rs_b += s[nt][2] + s[nt][3];
    }
    l_a = l_a * al_a + quad_sum(rs_a);
    l_b = l_b * al_b + quad_sum(rs_b);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= al_a; o[i][1] *= al_a;
      o[i][2] *= al_b; o[i][3] *= al_b;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t bb[4];
        ld_b_kn<D>(sV, kk * 16, dp * 16, bb);
        mma16816(o[2 * dp], pa, bb[0], bb[1]);
        mma16816(o[2 * dp + 1], pa, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  const float inv_a = l_a > 0.0f ? 1.0f / l_a : 0.0f;
  const float inv_b = l_b > 0.0f ? 1.0f / l_b : 0.0f;
  bf16* O = reinterpret_cast<bf16*>(a.o) + (int64_t)b * a.S * a.ld_o + h * D;
  store_strip<D>(sQ, warp * 16, o, inv_a, inv_b, O, a.ld_o, q0, a.S);
  if (t == 0) {
    float* L = a.lse + ((int64_t)b * a.nq + h) * a.S;
    if (row_a < a.S) L[row_a] = (m_a + log2f(l_a)) * LN2;
    if (row_b < a.S) L[row_b] = (m_b + log2f(l_b)) * LN2;
  }
}

// ------------------------------------------------------- delta = rowsum(dO*O)
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

// ------------------------------------------------------- dK, dV (per KV tile)
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  constexpr int TB = BT * D * 2;
  const uint32_t sK = smem_u32(sm);
  const uint32_t sV = sK + TB;
  const uint32_t sQ0 = sV + TB;            // 2 buffers
  const uint32_t sO0 = sQ0 + 2 * TB;       // dO, 2 buffers
  float* sL = reinterpret_cast<float*>(sm + 6 * TB);  // [2][BT] lse*log2e
  float* sD = sL + 2 * BT;                            // [2][BT] delta
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int rep = a.nq / a.nkv;
  const int kv0 = kt * BT;
  const int nqt = (a.S + BT - 1) / BT;
  const int qt_start = a.causal ? kt : 0;
  const int per_head = nqt - qt_start;
  const int n_it = per_head * rep;
  const float scale = rsqrtf((float)D);
  const float sl2 = scale * LOG2E;
  const bf16* Kg = reinterpret_cast<const bf16*>(a.k) + (int64_t)b * a.S * a.ld_kv + kvh * D;
  const bf16* Vg = reinterpret_cast<const bf16*>(a.v) + (int64_t)b * a.S * a.ld_kv + kvh * D;

  auto issue = [&](int it, int buf) {
    const int h = kvh * rep + it / per_head;
    const int qt = qt_start + it % per_head;
    const bf16* Q = reinterpret_cast<const bf16*>(a.q) + (int64_t)b * a.S * a.ld_q + h * D;
    const bf16* dO = reinterpret_cast<const bf16*>(a.dout) + (int64_t)b * a.S * a.ld_do + h * D;
    load_tile<D>(sQ0 + buf * TB, Q, a.ld_q, qt * BT, a.S);
    load_tile<D>(sO0 + buf * TB, dO, a.ld_do, qt * BT, a.S);
  };
  load_tile<D>(sK, Kg, a.ld_kv, kv0, a.S);
  load_tile<D>(sV, Vg, a.ld_kv, kv0, a.S);
  if (n_it > 0) issue(0, 0);
  cp_commit();

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.0f;
  const int kr_a = kv0 + warp * 16 + g, kr_b = kr_a + 8;

  for (int it = 0; it < n_it; ++it) {
    const int buf = it & 1;
    const int h = kvh * rep + it / per_head;
    const int qt = qt_start + it % per_head;
    const int q0 = qt * BT;
    // per-row lse / delta of this query tile into smem
    for (int i = threadIdx.x; i < BT; i += blockDim.x) {
      const int qi = q0 + i;
      const int64_t off = ((int64_t)b * a.nq + h) * a.S + qi;
      sL[buf * BT + i] = qi < a.S ? a.lse[off] * LOG2E : INFINITY;
      sD[buf * BT + i] = qi < a.S ? a.delta[off] : 0.0f;
    }
    if (it + 1 < n_it) {
      issue(it + 1, buf ^ 1);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const uint32_t sQ = sQ0 + buf * TB, sO = sO0 + buf * TB;
    // S^T = K Q^T  (rows: this warp's 16 keys, cols: 64 queries)
    float st[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) st[i][0] = st[i][1] = st[i][2] = st[i][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t af[4];
      ld_a<D>(sK, warp * 16, ks, af);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        ld_b_nt<D>(sQ, np * 16, ks, bb);
        mma16816(st[2 * np], af, bb[0], bb[1]);
        mma16816(st[2 * np + 1], af, bb[2], bb[3]);
      }
    }
    // P^T = exp2(S^T * scale*log2e - lse*log2e), masked
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int ql = nt * 8 + 2 * t + e;
        const int qi = q0 + ql;
        const float L = sL[buf * BT + ql];
        const bool bad_q = qi >= a.S;
        st[nt][e] = (bad_q || (a.causal && qi < kr_a) || kr_a >= a.S) ? 0.0f
                                                                         : exp2f(st[nt][e] * sl2 - L);
        st[nt][2 + e] = (bad_q || (a.causal && qi < kr_b) || kr_b >= a.S)
                            ? 0.0f
                            : exp2f(st[nt][2 + e] * sl2 - L);
      }
    }
    // dV += P^T dO
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(st[2 * kk][0], st[2 * kk][1]);
      pa[1] = pack_bf16x2(st[2 * kk][2], st[2 * kk][3]);
      pa[2] = pack_bf16x2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t bb[4];
        ld_b_kn<D>(sO, kk * 16, dp * 16, bb);
        mma16816(dv[2 * dp], pa, bb[0], bb[1]);
        mma16816(dv[2 * dp + 1], pa, bb[2], bb[3]);
      }
    }
    // dP^T = V dO^T
    float dpt[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t af[4];
      ld_a<D>(sV, warp * 16, ks, af);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        ld_b_nt<D>(sO, np * 16, ks, bb);
        mma16816(dpt[2 * np], af, bb[0], bb[1]);
        mma16816(dpt[2 * np + 1], af, bb[2], bb[3]);
      }
    }
    // dS^T = P^T (dP^T - delta)  ->  dK += dS^T Q
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      float v[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int nt = 2 * kk + u;
        const float d0 = sD[buf * BT + nt * 8 + 2 * t], d1 = sD[buf * BT + nt * 8 + 2 * t + 1];
        v[u][0] = st[nt][0] * (dpt[nt][0] - d0);
        v[u][1] = st[nt][1] * (dpt[nt][1] - d1);
        v[u][2] = st[nt][2] * (dpt[nt][2] - d0);
        v[u][3] = st[nt][3] * (dpt[nt][3] - d1);
      }
      pa[0] = pack_bf16x2(v[0][0], v[0][1]);
      pa[1] = pack_bf16x2(v[0][2], v[0][3]);
      pa[2] = pack_bf16x2(v[1][0], v[1][1]);
      pa[3] = pack_bf16x2(v[1][2], v[1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t bb[4];
        ld_b_kn<D>(sQ, kk * 16, dp * 16, bb);
        mma16816(dk[2 * dp], pa, bb[0], bb[1]);
        mma16816(dk[2 * dp + 1], pa, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  // write dK (scaled) and dV through the (now idle) Q buffers
  bf16* dK = reinterpret_cast<bf16*>(a.dk) + (int64_t)b * a.S * a.ld_dkv + kvh * D;
  bf16* dV = reinterpret_cast<bf16*>(a.dv) + (int64_t)b * a.S * a.ld_dkv + kvh * D;
  store_strip<D>(sQ0, warp * 16, dk, scale, scale, dK, a.ld_dkv, kv0, a.S);
  store_strip<D>(sQ0 + TB, warp * 16, dv, 1.0f, 1.0f, dV, a.ld_dkv, kv0, a.S);
}

// ---------------------------------------------------------- dQ (per Q tile)
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  constexpr int TB = BT * D * 2;
  const uint32_t sQ = smem_u32(sm);
  const uint32_t sO = sQ + TB;
  const uint32_t sK0 = sO + TB;        // 2 buffers
  const uint32_t sV0 = sK0 + 2 * TB;   // 2 buffers
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nqt = (a.S + BT - 1) / BT;
  const int qt = nqt - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / (a.nq / a.nkv);
  const int q0 = qt * BT;
  const float scale = rsqrtf((float)D);
  const float sl2 = scale * LOG2E;
  const bf16* Q = reinterpret_cast<const bf16*>(a.q) + (int64_t)b * a.S * a.ld_q + h * D;
  const bf16* dO = reinterpret_cast<const bf16*>(a.dout) + (int64_t)b * a.S * a.ld_do + h * D;
  const bf16* K = reinterpret_cast<const bf16*>(a.k) + (int64_t)b * a.S * a.ld_kv + kvh * D;
  const bf16* V = reinterpret_cast<const bf16*>(a.v) + (int64_t)b * a.S * a.ld_kv + kvh * D;
  const int kv_end = a.causal ? min(a.S, q0 + BT) : a.S;
  const int nkt = (kv_end + BT - 1) / BT;

  load_tile<D>(sQ, Q, a.ld_q, q0, a.S);
  load_tile<D>(sO, dO, a.ld_do, q0, a.S);
  load_tile<D>(sK0, K, a.ld_kv, 0, a.S);
  load_tile<D>(sV0, V, a.ld_kv, 0, a.S);
  cp_commit();

  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;
  const int64_t lrow = ((int64_t)b * a.nq + h) * a.S;
  const float L_a = row_a < a.S ? a.lse[lrow + row_a] * LOG2E : INFINITY;
  const float L_b = row_b < a.S ? a.lse[lrow + row_b] * LOG2E : INFINITY;
  const float D_a = row_a < a.S ? a.delta[lrow + row_a] : 0.0f;
  const float D_b = row_b < a.S ? a.delta[lrow + row_b] : 0.0f;

  uint32_t qf[D / 16][4], of[D / 16][4];
  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.0f;

  for (int j = 0; j < nkt; ++j) {
    const int buf = j & 1;
    if (j + 1 < nkt) {
      load_tile<D>(sK0 + (buf ^ 1) * TB, K, a.ld_kv, (j + 1) * BT, a.S);
      load_tile<D>(sV0 + (buf ^ 1) * TB, V, a.ld_kv, (j + 1) * BT, a.S);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        ld_a<D>(sQ, warp * 16, ks, qf[ks]);
        ld_a<D>(sO, warp * 16, ks, of[ks]);
      }
    }
    const uint32_t sK = sK0 + buf * TB, sV = sV0 + buf * TB;
    float s[8][4], dp[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[i][e] = dp[i][e] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        ld_b_nt<D>(sK, np * 16, ks, bb);
        mma16816(s[2 * np], qf[ks], bb[0], bb[1]);
        mma16816(s[2 * np + 1], qf[ks], bb[2], bb[3]);
        ld_b_nt<D>(sV, np * 16, ks, bb);
        mma16816(dp[2 * np], of[ks], bb[0], bb[1]);
        mma16816(dp[2 * np + 1], of[ks], bb[2], bb[3]);
      }
    }
    const int kv0 = j * BT;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      float v[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int nt = 2 * kk + u;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kv = kv0 + nt * 8 + 2 * t + e;
          const bool bad = kv >= a.S;
          const float pa_ = (bad || (a.causal && kv > row_a)) ? 0.0f : exp2f(s[nt][e] * sl2 - L_a);
          const float pb_ =
              (bad || (a.causal && kv > row_b)) ? 0.0f : exp2f(s[nt][2 + e] * sl2 - L_b);
          v[u][e] = pa_ * (dp[nt][e] - D_a);
          v[u][2 + e] = pb_ * (dp[nt][2 + e] - D_b);
        }
      }
      pa[0] = pack_bf16x2(v[0][0], v[0][1]);
      pa[1] = pack_bf16x2(v[0][2], v[0][3]);
      pa[2] = pack_bf16x2(v[1][0], v[1][1]);
      pa[3] = pack_bf16x2(v[1][2], v[1][3]);
#pragma unroll
      for (int dpi = 0; dpi < D / 16; ++dpi) {
        uint32_t bb[4];
        ld_b_kn<D>(sK, kk * 16, dpi * 16, bb);
        mma16816(dq[2 * dpi], pa, bb[0], bb[1]);
        mma16816(dq[2 * dpi + 1], pa, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  bf16* dQ = reinterpret_cast<bf16*>(a.dq) + (int64_t)b * a.S * a.ld_dq + h * D;
  store_strip<D>(sQ, warp * 16, dq, scale, scale, dQ, a.ld_dq, q0, a.S);
}

template <int D>
mgb_status fwd_d(const AttnArgs& a, cudaStream_t st) {
  const int smem = 5 * BT * D * 2;
  auto k = attn_fwd_kernel<D>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 grid((a.S + BT - 1) / BT, a.nq, a.B);
  k<<<grid, 128, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

template <int D>
mgb_status bwd_d(const AttnArgs& a, cudaStream_t st) {
  const int T = a.B * a.S;
  const int warps = T * a.nq;
  attn_delta_kernel<D><<<(warps + 7) / 8, 256, 0, st>>>(a);
  const int smem_kv = 6 * BT * D * 2 + 4 * BT * 4;
  auto k1 = attn_bwd_dkdv_kernel<D>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 g1((a.S + BT - 1) / BT, a.nkv, a.B);
  k1<<<g1, 128, smem_kv, st>>>(a);
  const int smem_q = 6 * BT * D * 2;
  auto k2 = attn_bwd_dq_kernel<D>;
  if (cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q) != cudaSuccess)
    return MGB_ERR_CUDA;
  dim3 g2((a.S + BT - 1) / BT, a.nq, a.B);
  k2<<<g2, 128, smem_q, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

}  // namespace

mgb_status attention_bf16_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.d == 64) return fwd_d<64>(a, st);
  if (a.d == 128) return fwd_d<128>(a, st);
  return MGB_ERR_UNSUPPORTED;
}
mgb_status attention_bf16_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.d == 64) return bwd_d<64>(a, st);
  if (a.d == 128) return bwd_d<128>(a, st);
  return MGB_ERR_UNSUPPORTED;
}

}  // namespace mgb
